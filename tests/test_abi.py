"""C ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import _binding, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sinkattn.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return _binding.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SINKATTN_API\s+[\w\s\*]*?\b(sinkattn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("sinkattn_prefill", "sinkattn_decode_split", "sinkattn_merge", "sinkattn_decode",
              "sinkattn_decode_workspace_bytes", "sinkattn_status_string", "sinkattn_last_error",
              "sinkattn_debug_status"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
    # and nothing else from the library namespace leaks out
    out = os.popen("nm -D --defined-only %s" % _binding.LIB_PATH).read()
    exported = set(re.findall(r"\b(sinkattn_\w+)\b", out))
    assert exported == set(declared_symbols())


def test_status_strings(L):
    assert sa.sinkattn_status_string(0) == "SINKATTN_OK"
    assert sa.sinkattn_status_string(1) == "SINKATTN_INVALID_ARG"
    assert sa.sinkattn_status_string(2) == "SINKATTN_UNSUPPORTED"
    assert sa.sinkattn_status_string(4) == "SINKATTN_TIMEOUT"
    assert sa.sinkattn_status_string(99) == "SINKATTN_UNKNOWN_STATUS"


# Fake, 16-byte aligned, never dereferenced: every case below is rejected
# before any CUDA call.
A, B, C, O = 0x1000, 0x2000, 0x3000, 0x4000


def prefill(L, **kw):
    args = dict(q=A, k=B, v=C, sinks=None, cuq=0x5000, cuk=0x6000, batch=1, total_q=16,
                maxq=16, maxk=128, hq=4, hkv=1, d=64, scale=0.125, causal=1, window=0, out=O,
                lse=None)
    args.update(kw)
    return L.sinkattn_prefill(args["q"], args["k"], args["v"], args["sinks"], args["cuq"],
                              args["cuk"], args["batch"], args["total_q"], args["maxq"],
                              args["maxk"], args["hq"], args["hkv"], args["d"], args["scale"],
                              args["causal"], args["window"], args["out"], args["lse"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1),
    (dict(out=None), 1),
    (dict(cuq=None), 1),
    (dict(q=A + 8), 1),              # misaligned (16-byte rule)
    (dict(out=O + 2), 1),
    (dict(hq=6, hkv=4), 2),          # Hq % Hkv != 0
    (dict(d=96), 2),                 # head_dim not 64/128
    (dict(causal=0, window=8), 2),   # window without causal
    (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(batch=-1), 1),
    (dict(maxq=200, maxk=128), 1),   # q longer than k
    (dict(causal=2), 1),
    (dict(batch=70000), 2),
])
def test_prefill_rejects_bad_arguments(L, kw, status):
    assert prefill(L, **kw) == status
    assert sa.sinkattn_last_error() != ""


def test_prefill_empty_problem_is_a_no_op(L):
    assert prefill(L, batch=0) == 0
    assert prefill(L, total_q=0) == 0


def split(L, **kw):
    args = dict(q=A, k=B, v=C, ind=0x5000, batch=2, qlen=1, maxk=100, hq=8, hkv=1, d=128,
                scale=0.1, causal=1, window=0, S=4, acc=0x7000, md=0x8000)
    args.update(kw)
    return L.sinkattn_decode_split(args["q"], args["k"], args["v"], args["ind"], args["batch"],
                                   args["qlen"], args["maxk"], args["hq"], args["hkv"], args["d"],
                                   args["scale"], args["causal"], args["window"], args["S"],
                                   args["acc"], args["md"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(ind=None), 1),
    (dict(acc=None), 1),
    (dict(md=0x8004), 1),
    (dict(S=0), 1),
    (dict(qlen=0), 1),
    (dict(qlen=200, maxk=100), 1),   # q_len > kv_len
    (dict(hq=130, hkv=2), 2),        # GQA group beyond 64
    (dict(d=32), 2),
    (dict(hq=9, hkv=2), 2),
])
def test_decode_split_rejects_bad_arguments(L, kw, status):
    assert split(L, **kw) == status


def test_merge_rejects_bad_arguments(L):
    assert L.sinkattn_merge(None, 0x1000, None, 4, 8, 64, 2, O, None, None) == 1
    assert L.sinkattn_merge(0x1000, 0x2000, None, 4, 8, 80, 2, O, None, None) == 2
    assert L.sinkattn_merge(0x1000, 0x2000, None, 4, 8, 64, 0, O, None, None) == 1


def test_workspace_bytes(L):
    n = sa.sinkattn_decode_workspace_bytes(256, 3, 64, 128, 16)
    slots = 256 * 3 * 64 * 16
    assert n >= slots * 128 * 4 + slots * 2 * 4
    assert n - slots * 2 * 4 == ((slots * 128 * 4 + 255) // 256) * 256
    with pytest.raises(sa.SinkAttnError):
        sa.sinkattn_decode_workspace_bytes(1, 1, 8, 96, 1)


def test_decode_checks_workspace_before_launch(L):
    need = sa.sinkattn_decode_workspace_bytes(2, 1, 8, 128, 4)
    rc = L.sinkattn_decode(A, B, C, 0x5000, 2, 1, 100, 8, 1, 128, 0.1, 1, 0, 4, None, 0x10000,
                           need - 1, O, None, None)
    assert rc == 1 and "workspace" in sa.sinkattn_last_error()
    rc = L.sinkattn_decode(A, B, C, 0x5000, 2, 1, 100, 8, 1, 128, 0.1, 1, 0, 4, None, 0x10010,
                           need, O, None, None)
    assert rc == 1   # workspace not 256-byte aligned


def test_default_splits_bounds(L):
    s = sa.sinkattn_decode_default_splits(64, 1, 64, 8, 64, 8192)
    assert 1 <= s <= 64
    assert sa.sinkattn_decode_default_splits(1, 1, 8, 1, 64, 100) == 1   # short: no split


def prefill_paged(L, **kw):
    args = dict(q=A, k=B, v=C, sinks=None, cuq=0x5000, cuk=0x6000, pind=0x9000, pidx=0xA000,
                npages=8, psize=64, batch=1, total_q=16, maxq=16, maxk=128, hq=4, hkv=1, d=64,
                scale=0.125, causal=1, window=0, out=O, lse=None)
    args.update(kw)
    return L.sinkattn_prefill_paged(
        args["q"], args["k"], args["v"], args["sinks"], args["cuq"], args["cuk"], args["pind"],
        args["pidx"], args["npages"], args["psize"], args["batch"], args["total_q"], args["maxq"],
        args["maxk"], args["hq"], args["hkv"], args["d"], args["scale"], args["causal"],
        args["window"], args["out"], args["lse"], None)


def split_paged(L, **kw):
    args = dict(q=A, k=B, v=C, ind=0x5000, pind=0x9000, pidx=0xA000, npages=8, psize=64, batch=2,
                qlen=1, maxk=100, hq=8, hkv=1, d=128, scale=0.1, causal=1, window=0, S=4,
                acc=0x7000, md=0x8000)
    args.update(kw)
    return L.sinkattn_decode_split_paged(
        args["q"], args["k"], args["v"], args["ind"], args["pind"], args["pidx"], args["npages"],
        args["psize"], args["batch"], args["qlen"], args["maxk"], args["hq"], args["hkv"],
        args["d"], args["scale"], args["causal"], args["window"], args["S"], args["acc"],
        args["md"], None)


PAGED_BAD = [
    (dict(pind=None), 1),
    (dict(pidx=None), 1),
    (dict(psize=8), 2),              # below 16
    (dict(psize=48), 2),             # not a power of two
    (dict(psize=512), 2),            # above 256
    (dict(npages=0), 1),
    (dict(npages=1 << 24, psize=256), 2),   # pool rows reach 2^31
    (dict(k=B + 8), 1),              # misaligned pool
]


@pytest.mark.parametrize("kw,status", PAGED_BAD)
def test_prefill_paged_rejects_bad_arguments(L, kw, status):
    assert prefill_paged(L, **kw) == status
    assert sa.sinkattn_last_error() != ""


@pytest.mark.parametrize("kw,status", PAGED_BAD + [(dict(S=0), 1), (dict(d=32), 2)])
def test_decode_split_paged_rejects_bad_arguments(L, kw, status):
    assert split_paged(L, **kw) == status


def test_decode_paged_checks_workspace_before_launch(L):
    need = sa.sinkattn_decode_workspace_bytes(2, 1, 8, 128, 4)
    rc = L.sinkattn_decode_paged(A, B, C, 0x5000, 0x9000, 0xA000, 8, 64, 2, 1, 100, 8, 1, 128, 0.1,
                                 1, 0, 4, None, 0x10000, need - 1, O, None, None)
    assert rc == 1 and "workspace" in sa.sinkattn_last_error()
    rc = L.sinkattn_decode_paged(A, B, C, 0x5000, 0x9000, 0xA000, 8, 16, 2, 1, 100, 8, 1, 128, 0.1,
                                 1, 0, 4, None, 0x10000, need, O, None, None)
    assert rc != 1 or "workspace" not in sa.sinkattn_last_error()


def test_prefill_kernel_switch(L):
    assert L.sinkattn_set_prefill_kernel(3) == 1
    assert L.sinkattn_set_prefill_kernel(-1) == 1
    for k in (1, 2, 0):
        assert L.sinkattn_set_prefill_kernel(k) == 0


def test_decode_split_fp8_rejects_missing_scales(L):
    rc = L.sinkattn_decode_split_fp8(A, B, C, None, 0x9000, 0x5000, 2, 1, 100, 8, 1, 128, 0.1, 1,
                                     0, 4, 0x7000, 0x8000, None)
    assert rc == 1 and "scale" in sa.sinkattn_last_error()
    rc = L.sinkattn_decode_split_fp8(A, B, C, 0x9002, 0x9000, 0x5000, 2, 1, 100, 8, 1, 128, 0.1,
                                     1, 0, 4, 0x7000, 0x8000, None)
    assert rc == 1

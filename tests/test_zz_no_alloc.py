"""sinkattn_decode_noalloc: decode for callers that cannot allocate device
memory (the partials live in the library's fixed scratch array instead of a
caller workspace). Its results must match sinkattn_decode's, call after call,
since every call reuses the same scratch; one case is also checked against
the float64 oracle directly.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes
import math

import pytest
import torch

import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import workloads
from gqa_attention_softmax_gb300._binding import INVALID_ARG, UNSUPPORTED
from _helpers import compare, to_dev

SCRATCH_BYTES = 32 * 2**20


def _inputs(B, q_len, Hq, Hkv, d, kv_range, seed):
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=B, q_len=q_len,
                           kv_range=kv_range, sink_dist="uniform2", seed=seed)
    return workloads.make_inputs(w)


def _raw_call(batch, q_len, Hq, Hkv, d, S):
    """The C entry point with null pointers: every outcome is decided on the
    host (a null q is rejected before anything could launch)."""
    L = sa.lib()
    return L.sinkattn_decode_noalloc(None, None, None, None, batch, q_len, 4096, Hq, Hkv, d, 0.1,
                                     1, 0, S, None, None, None, None)


def test_noalloc_scratch_boundary_is_host_side():
    """Largest accepted and smallest rejected partial sizes around the 32 MiB
    scratch. Accepted sizes go on to the other checks (here: no device on a
    CPU host, or the null q on a GPU host), rejected ones stop with
    SINKATTN_UNSUPPORTED naming the scratch. Nothing launches either way."""
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    Hq, S, d = 4, 25, 64
    lo, hi = 1, 1 << 20   # the largest batch whose partials fit, by bisection
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if sa.sinkattn_decode_workspace_bytes(mid, 1, Hq, d, S) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    fit = lo
    assert sa.sinkattn_decode_workspace_bytes(fit, 1, Hq, d, S) <= SCRATCH_BYTES
    assert sa.sinkattn_decode_workspace_bytes(fit + 1, 1, Hq, d, S) > SCRATCH_BYTES
    rc = _raw_call(fit, 1, Hq, 1, d, S)
    assert rc != UNSUPPORTED, sa.lib().sinkattn_last_error().decode()
    assert rc in (INVALID_ARG, 3)   # null q on a GPU host; no device (CUDA error) here
    rc = _raw_call(fit + 1, 1, Hq, 1, d, S)
    assert rc == UNSUPPORTED
    assert "scratch" in sa.lib().sinkattn_last_error().decode()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [
    (16, 1, 64, 8, 64, (100, 3000), 3),     # gpt-oss-like decode
    (8, 3, 64, 4, 128, (50, 2000), 16),     # MTP-like, 16 chunks
    (12, 1, 64, 8, 64, (64, 2500), 0),      # the library's default split count
])
def test_noalloc_matches_decode_two_calls_in_a_row(shape):
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    B, q_len, Hq, Hkv, d, kvr, S = shape
    scale = 1.0 / math.sqrt(d)
    for call in range(2):
        g = to_dev(_inputs(B, q_len, Hq, Hkv, d, kvr, seed=100 + call))
        max_kv = max(g["kv_lens"])
        ref_out, ref_lse = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len,
                                              max_kv, Hkv, num_splits=S, sm_scale=scale)
        out = torch.full_like(g["q"], float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), device="cuda")
        sa.sinkattn_decode_noalloc(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                   Hkv, num_splits=S, sm_scale=scale, out=out, lse=lse)
        torch.cuda.synchronize()
        compare(out, lse, ref_out.float().cpu().numpy(), ref_lse.cpu().numpy(),
                "noalloc call %d" % call)


@pytest.mark.gpu
def test_noalloc_matches_oracle():
    import oracle
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    oracle.build()
    B, q_len, Hq, Hkv, d = 6, 3, 64, 4, 128
    inp = _inputs(B, q_len, Hq, Hkv, d, (40, 1500), seed=5)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, 1.0 / math.sqrt(d), True, 0)
    g = to_dev(inp)
    out, lse = sa.sinkattn_decode_noalloc(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len,
                                          max(inp["kv_lens"]), Hkv, num_splits=16)
    torch.cuda.synchronize()
    compare(out, lse, want_out, want_lse, "noalloc vs oracle")


@pytest.mark.gpu
def test_noalloc_rejects_partials_beyond_its_scratch():
    g = to_dev(_inputs(2, 1, 8, 1, 64, (10, 20), seed=7))
    need = sa.sinkattn_decode_workspace_bytes(4096, 16, 64, 128, 64)
    assert need > SCRATCH_BYTES
    # host-side sizes too large for the scratch: rejected before any launch
    with pytest.raises(sa.SinkAttnError) as e:
        L = sa.lib()
        rc = L.sinkattn_decode_noalloc(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(),
                                       g["cu_k"].data_ptr(), 4096, 16, 4096, 64, 4, 128, 0.1, 1, 0,
                                       64, None, g["q"].data_ptr(), None, None)
        from gqa_attention_softmax_gb300._binding import _check
        _check(rc)
    assert e.value.status == UNSUPPORTED and "scratch" in str(e.value)


@pytest.mark.gpu
def test_noalloc_rejects_a_stream_of_another_device():
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    g = to_dev(_inputs(2, 1, 8, 1, 64, (10, 20), seed=7), "cuda:0")
    s1 = torch.cuda.Stream(device="cuda:1")
    with torch.cuda.device(0):
        L = sa.lib()
        rc = L.sinkattn_decode_noalloc(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(),
                                       g["cu_k"].data_ptr(), 2, 1, 20, 8, 1, 64, 0.125, 1, 0, 3,
                                       None, g["q"].data_ptr(), None,
                                       ctypes.c_void_p(s1.cuda_stream))
    assert rc == INVALID_ARG
    assert "stream" in L.sinkattn_last_error().decode()

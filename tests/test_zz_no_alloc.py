"""sinkattn_decode_noalloc: decode for callers that cannot allocate device
memory (the partials live in the library's fixed scratch array instead of a
caller workspace). Its results must match sinkattn_decode's, call after call,
since every call reuses the same scratch.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import math

import pytest
import torch

import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import workloads
from _helpers import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    assert torch.cuda.is_available()


def _inputs(B, q_len, Hq, Hkv, d, kv_range, seed):
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=B, q_len=q_len,
                           kv_range=kv_range, sink_dist="uniform2", seed=seed)
    return to_dev(workloads.make_inputs(w))


@pytest.mark.parametrize("shape", [
    (16, 1, 64, 8, 64, (100, 3000), 3),     # gpt-oss-like decode
    (8, 3, 64, 4, 128, (50, 2000), 16),     # MTP-like, 16 chunks
])
def test_noalloc_matches_decode_two_calls_in_a_row(shape):
    B, q_len, Hq, Hkv, d, kvr, S = shape
    scale = 1.0 / math.sqrt(d)
    for call in range(2):
        g = _inputs(B, q_len, Hq, Hkv, d, kvr, seed=100 + call)
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


def test_noalloc_rejects_partials_beyond_its_scratch():
    g = _inputs(2, 1, 8, 1, 64, (10, 20), seed=7)
    need = sa.sinkattn_decode_workspace_bytes(4096, 16, 64, 128, 64)
    assert need > 32 * 2**20
    # host-side sizes too large for the scratch: rejected before any launch
    with pytest.raises(sa.SinkAttnError) as e:
        L = sa.lib()
        rc = L.sinkattn_decode_noalloc(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(),
                                       g["cu_k"].data_ptr(), 4096, 16, 4096, 64, 4, 128, 0.1, 1, 0,
                                       64, None, g["q"].data_ptr(), None, None)
        from gqa_attention_softmax_gb300._binding import _check
        _check(rc)
    assert e.value.status == 2 and "scratch" in str(e.value)

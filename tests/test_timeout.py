"""Failure detection without a GPU fault: a bounded wait that runs out.

A test hook (sinkattn_debug_set_hooks) shortens every bounded wait to about
10 ms and makes the TMA producer of the grid's first thread block leave out
the copies of one KV tile, so the waits for that tile run out. The kernel
must record SINKATTN_TIMEOUT in its status word, drain its copies and MMAs,
free its tensor memory and exit; the host reads the status, clears it, and
the next normal call on the same context must match the oracle. One case
per kernel family: the prefill kernel in both launches, the warp-level
split-KV kernel and the tcgen05 split-KV kernel.
"""
import math

import pytest
import torch

import oracle
import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import workloads
from gqa_attention_softmax_gb300._binding import TIMEOUT
from _helpers import compare, to_dev

pytestmark = pytest.mark.gpu

LIMIT_CYCLES = 20_000_000   # ~10 ms at 2 GHz: far above any legitimate wait here


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    oracle.build()
    assert torch.cuda.is_available()
    yield
    sa.sinkattn_debug_set_hooks(0, -1)
    sa.sinkattn_set_prefill_kernel("auto")
    sa.sinkattn_set_decode_kernel("auto")


def _prefill_case():
    inp = workloads.explicit_inputs([300], [300], 8, 1, 64, seed=11)
    g = to_dev(inp)

    def run():
        return sa.sinkattn_prefill(g["q"], g["k"], g["v"], g["sinks"], g["cu_q"], g["cu_k"], 300,
                                   300, 1, 0.125, True, 0)
    want = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"], inp["cu_k"], 8,
                         1, 64, 0.125, True, 0)
    return run, want


def _decode_case(Hq, Hkv, d, q_len, S):
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=4, q_len=q_len,
                           kv_range=(500, 900), sink_dist="uniform2", seed=12)
    inp = workloads.make_inputs(w)
    g = to_dev(inp)
    max_kv = max(inp["kv_lens"])

    def run():
        return sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                  Hkv, num_splits=S, sm_scale=1.0 / math.sqrt(d))
    want = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"], inp["cu_k"], Hq,
                         Hkv, d, 1.0 / math.sqrt(d), True, 0)
    return run, want


CASES = {
    "prefill_one_block": ("prefill", "one_block", lambda: _prefill_case()),
    "prefill_persistent": ("prefill", "persistent", lambda: _prefill_case()),
    "decode_warp": ("decode", "warp", lambda: _decode_case(8, 1, 64, 1, 2)),
    "decode_tcgen05": ("decode", "tcgen05", lambda: _decode_case(64, 4, 128, 3, 2)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_clean(name):
    kind, launch, make = CASES[name]
    if kind == "prefill":
        sa.sinkattn_set_prefill_kernel(launch)
    else:
        sa.sinkattn_set_decode_kernel(launch)
    try:
        run, (want_out, want_lse) = make()
        torch.cuda.synchronize()
        assert sa.sinkattn_debug_status() == 0   # nothing recorded before
        sa.sinkattn_debug_set_hooks(LIMIT_CYCLES, 1)
        try:
            run()
            torch.cuda.synchronize()
            status = sa.sinkattn_debug_status()
        finally:
            sa.sinkattn_debug_set_hooks(0, -1)
        assert status == TIMEOUT, sa.sinkattn_status_string(status)
        assert sa.sinkattn_debug_status() == 0   # read and cleared
        out, lse = run()
        torch.cuda.synchronize()
        compare(out, lse, want_out, want_lse, "%s after a timeout" % name)
        assert sa.sinkattn_debug_status() == 0
    finally:
        sa.sinkattn_set_prefill_kernel("auto")
        sa.sinkattn_set_decode_kernel("auto")


def test_hooks_reject_a_bad_tile():
    with pytest.raises(sa.SinkAttnError):
        sa.sinkattn_debug_set_hooks(0, -2)

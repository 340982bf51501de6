"""Host-side arithmetic of the benchmark (no GPU): the visible-pair count
behind every TFLOP/s figure against brute force, the algorithmic byte
count against a hand count, and the kernel and traffic-record selection."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gqa_attention_softmax_gb300 import workloads  # noqa: E402


def _pairs_brute(q_lens, kv_lens, causal, window):
    n = 0
    for lq, lk in zip(q_lens, kv_lens):
        for i in range(lq):
            pos = lk - lq + i
            for j in range(lk):
                if causal and j > pos:
                    continue
                if window > 0 and j <= pos - window:
                    continue
                n += 1
    return n


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 1), (True, 5), (True, 64)])
def test_visible_pairs_matches_brute_force(causal, window):
    rng = np.random.default_rng(3)
    kv = rng.integers(0, 90, 7).tolist()
    q = [int(rng.integers(0, k + 1)) for k in kv]
    assert bench.visible_pairs(q, kv, causal, window) == _pairs_brute(q, kv, causal, window)


def test_decode_bytes_by_hand():
    """Q, K and V read once, out and lse written, plus sinks and kv_indptr;
    FP8 halves K/V and adds the two scale vectors; pages add their lists."""
    w = workloads.Workload("t", "decode", 8, 2, 64, True, batch=3, q_len=2,
                           kv_range=(5, 40), seed=1)
    inp = workloads.make_inputs(w)
    B, Hq, Hkv, d, tq = 3, 8, 2, 64, 6
    kv_tok = sum(inp["kv_lens"])
    small = Hq * 4 + (B + 1) * 4
    want = tq * Hq * d * 2 + 2 * Hkv * kv_tok * d * 2 + tq * Hq * d * 2 + tq * Hq * 4 + small
    total, flops, split = bench.work(w, inp)
    assert total == want
    assert split == tq * Hq * d * 2 + 2 * Hkv * kv_tok * d * 2
    assert flops == 4.0 * d * Hq * _pairs_brute(inp["q_lens"], inp["kv_lens"], True, 0)

    w8 = workloads.Workload("t", "decode", 8, 2, 64, True, batch=3, q_len=2,
                            kv_range=(5, 40), seed=1, kv_fp8=True)
    t8, _, s8 = bench.work(w8, workloads.make_inputs(w8))
    assert s8 == tq * Hq * d * 2 + 2 * Hkv * kv_tok * d
    assert t8 == want - 2 * Hkv * kv_tok * d + 2 * Hkv * 4

    wp = workloads.Workload("t", "decode", 8, 2, 64, True, batch=3, q_len=2,
                            kv_range=(5, 40), seed=1, page_size=16)
    tp, _, _ = bench.work(wp, workloads.make_inputs(wp))
    pages = sum(-(-lk // 16) for lk in inp["kv_lens"])
    assert tp == want + 4 * (B + 1 + pages)


def test_decode_kernel_selection_names():
    W = workloads.WORKLOADS
    assert "attn_mma" in bench.decode_kernel_name(W["gptoss_decode"])
    assert "decode_tc" in bench.decode_kernel_name(W["qwen_mtp_decode"])
    assert "decode_tc" in bench.decode_kernel_name(W["qwen_mtp_decode_fp8"])   # 48 rows per tile
    assert "attn_mma" in bench.decode_kernel_name(W["gptoss_decode_fp8"])      # head_dim 64


def test_traffic_records_name_their_capture():
    """Every DRAM-traffic record points at a committed ncu summary that names
    its command, and carries the hash of the sources it was taken on."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    with open(path) as f:
        t = json.load(f)
    assert t
    for key, e in t.items():
        assert e["dram_bytes_per_launch"] > 0, key
        assert len(e["source_sha"]) == 16, key
        cap = os.path.join(ROOT, e["capture"])
        assert os.path.exists(cap), key
        with open(cap) as f:
            assert "ncu " in f.read(), key

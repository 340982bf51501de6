"""Pins for the float64 oracle (no GPU).

Each test checks the oracle against something that is not the oracle:
hand-derived worked examples, the library SDPA routine (to which the method
reduces exactly), closed forms, identities, a second implementation with
exactly rounded sums, and brute-force enumeration of KV splits. The method is
the one in "GPT-OSS on Day 0" (Perplexity), section "Kernels for GPT-OSS /
Sink attention".
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from gqa_attention_softmax_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sink_worked_examples.json")


def _num(x):
    if isinstance(x, str):
        if x == "-inf":
            return -math.inf
        if x.startswith("ln"):
            return math.log(float(x[2:]))
    return float(x)


def _to_bf16(a):
    t = torch.tensor(np.asarray(a, dtype=np.float64), dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), "golden inputs must be exact in bf16"
    return b


# --------------------------------------------------------------------------
# hand-derived worked examples
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_worked_examples(oracle_lib, case):
    q = _to_bf16(case["q"])
    k = _to_bf16(case["k"])
    v = _to_bf16(case["v"])
    sinks = np.array([_num(s) for s in case["sinks"]])
    scale = _num(case["sm_scale"])
    out, lse = oracle.attend(q, k, v, sinks, case["cu_q"], case["cu_k"], case["Hq"], case["Hkv"],
                             case["d"], scale, case["causal"], case["window"])
    want_out = np.array(case["out"], dtype=np.float64).reshape(out.shape)
    want_lse = np.array([[_num(x) for x in r] for r in case["lse"]]).reshape(lse.shape)
    np.testing.assert_allclose(out, want_out, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-14)

    # the pure-Python implementation agrees on the same worked examples
    bo, bl = brute.attend_fsum(q.double().tolist(), k.double().flatten().tolist(),
                               v.double().flatten().tolist(), sinks.tolist(), case["cu_q"],
                               case["cu_k"], case["Hq"], case["Hkv"], case["d"], scale,
                               case["causal"], case["window"])
    np.testing.assert_allclose(np.array(bo).reshape(out.shape), want_out, rtol=0, atol=1e-14)
    np.testing.assert_allclose(np.array(bl).reshape(lse.shape), want_lse, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# reduction to the library routine (SDPA, float64)
# --------------------------------------------------------------------------
SHAPES = [
    # (q_lens, kv_lens, Hq, Hkv, d)
    ([16], [128], 4, 1, 64),           # the tiny workload's shape
    ([3, 1, 5], [7, 1, 9], 6, 3, 8),   # varlen, GQA 2:1, three KV heads
    ([4, 4], [4, 12], 8, 2, 16),       # GQA 4:1
    ([2, 0, 3], [5, 2, 3], 4, 4, 4),   # MHA, one sequence with no queries
]


def _sdpa_rows(inp, Hq, Hkv, d, scale, causal, window, sinks):
    """Library SDPA per sequence; the sink, when given, as an extra key whose
    key and value rows are zero and whose additive mask entry is s_h."""
    G = Hq // Hkv
    outs = []
    cu_q, cu_k = inp["cu_q"].tolist(), inp["cu_k"].tolist()
    for b in range(len(cu_q) - 1):
        Lq, Lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        if Lq == 0:
            continue
        q = inp["q"][cu_q[b]:cu_q[b + 1]].double().permute(1, 0, 2).unsqueeze(0)   # [1,Hq,Lq,d]
        kb = inp["k"][Hkv * cu_k[b]:Hkv * cu_k[b + 1]].double().view(Hkv, Lk, d)
        vb = inp["v"][Hkv * cu_k[b]:Hkv * cu_k[b + 1]].double().view(Hkv, Lk, d)
        kb = kb.repeat_interleave(G, dim=0).unsqueeze(0)
        vb = vb.repeat_interleave(G, dim=0).unsqueeze(0)
        keep = torch.ones(Lq, Lk, dtype=torch.bool)
        if causal:
            keep = keep.tril(diagonal=Lk - Lq)
        if window > 0:
            keep = keep.triu(diagonal=Lk - Lq - window + 1)
        add = torch.zeros(Lq, Lk, dtype=torch.float64).masked_fill(~keep, -math.inf)
        add = add.expand(Hq, Lq, Lk)
        if sinks is not None:
            kb = torch.cat([kb, torch.zeros(1, Hq, 1, d, dtype=torch.float64)], dim=2)
            vb = torch.cat([vb, torch.zeros(1, Hq, 1, d, dtype=torch.float64)], dim=2)
            col = torch.as_tensor(sinks, dtype=torch.float64).view(Hq, 1, 1).expand(Hq, Lq, 1)
            add = torch.cat([add, col], dim=2)
        o = torch.nn.functional.scaled_dot_product_attention(q, kb, vb, attn_mask=add.unsqueeze(0),
                                                             scale=scale)
        outs.append(o[0].permute(1, 0, 2))   # [Lq, Hq, d]
    return torch.cat(outs, 0).numpy()


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mask", [(False, 0), (True, 0), (True, 1), (True, 3)])
def test_no_sink_reduces_to_softmax_attention(oracle_lib, shape, mask):
    q_lens, kv_lens, Hq, Hkv, d = shape
    causal, window = mask
    inp = workloads.explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=1)
    scale = 1.0 / math.sqrt(d)
    want = _sdpa_rows(inp, Hq, Hkv, d, scale, causal, window, None)
    for sinks in (None, np.full(Hq, -np.inf)):
        out, _ = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"], inp["cu_k"],
                               Hq, Hkv, d, scale, causal, window)
        np.testing.assert_allclose(out.reshape(want.shape), want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mask", [(False, 0), (True, 0), (True, 2)])
def test_sink_reduces_to_sdpa_with_extra_zero_column(oracle_lib, shape, mask):
    q_lens, kv_lens, Hq, Hkv, d = shape
    causal, window = mask
    inp = workloads.explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=2)
    scale = 1.0 / math.sqrt(d)
    sinks = np.linspace(-3.0, 3.0, Hq)
    want = _sdpa_rows(inp, Hq, Hkv, d, scale, causal, window, sinks)
    out, _ = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"], inp["cu_k"],
                           Hq, Hkv, d, scale, causal, window)
    np.testing.assert_allclose(out.reshape(want.shape), want, rtol=0, atol=1e-12)


def test_gqa_head_mapping_is_contiguous_groups(oracle_lib):
    """KV head of query head h is floor(h / G): make KV heads differ only in V
    and check each query head reads its group's V (q = 0 -> mean of V)."""
    Hq, Hkv, d, Lk = 6, 3, 4, 5
    q = torch.zeros(1, Hq, d, dtype=torch.bfloat16)
    k = torch.zeros(Hkv * Lk, d, dtype=torch.bfloat16)
    v = torch.zeros(Hkv, Lk, d)
    for g in range(Hkv):
        v[g] = float(g + 1)
    out, _ = oracle.attend(q, k, v.view(Hkv * Lk, d).to(torch.bfloat16), None, [0, 1], [0, Lk],
                           Hq, Hkv, d, 0.5, True)
    got = out.reshape(Hq, d)[:, 0]
    np.testing.assert_array_equal(got, [1, 1, 2, 2, 3, 3])


# --------------------------------------------------------------------------
# closed forms and identities
# --------------------------------------------------------------------------
def test_weight_sum_identity(oracle_lib):
    """Weights over real tokens sum to 1/(1 + e^{s-M}/sum_j e^{l_j-M}) = 1 - e^{s - lse}:
    with V = 1 the output is exactly that sum."""
    inp = workloads.explicit_inputs([5, 9], [11, 9], 8, 2, 16, seed=3, q_scale=3.0)
    v1 = torch.ones_like(inp["v"])
    sinks = np.array([-5.0, -1.0, -0.25, 0.0, 0.5, 1.5, 3.0, 8.0])
    out, lse = oracle.attend(inp["q"], inp["k"], v1, sinks, inp["cu_q"], inp["cu_k"], 8, 2, 16,
                             0.25, True, 0)
    hs = np.arange(out.shape[0]) % 8
    want = 1.0 - np.exp(sinks[hs] - lse)
    np.testing.assert_allclose(out[:, 0], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, np.repeat(want[:, None], 16, 1), rtol=0, atol=1e-12)


def test_zero_query_closed_form(oracle_lib):
    """q = 0: every visible logit is 0, so out = sum(v_vis)/(n + e^s), lse = ln(n + e^s)."""
    Hq, Hkv, d = 4, 2, 8
    inp = workloads.explicit_inputs([3], [10], Hq, Hkv, d, seed=4)
    q0 = torch.zeros_like(inp["q"])
    sinks = np.array([0.3, -1.2, 2.0, -np.inf])
    W = 4
    out, lse = oracle.attend(q0, inp["k"], inp["v"], sinks, inp["cu_q"], inp["cu_k"], Hq, Hkv, d,
                             0.7, True, W)
    out = out.reshape(3, Hq, d)
    lse = lse.reshape(3, Hq)
    v = inp["v"].double().view(Hkv, 10, d).numpy()
    # hand-listed visible keys: positions 7, 8, 9 with window 4
    vis = {0: [4, 5, 6, 7], 1: [5, 6, 7, 8], 2: [6, 7, 8, 9]}
    for i in range(3):
        for h in range(Hq):
            n = len(vis[i])
            es = math.exp(sinks[h]) if np.isfinite(sinks[h]) else 0.0
            want = v[h // 2, vis[i]].sum(0) / (n + es)
            np.testing.assert_allclose(out[i, h], want, rtol=0, atol=1e-13)
            assert abs(lse[i, h] - math.log(n + es)) < 1e-13


def test_visible_sets_by_one_hot_values(oracle_lib):
    """With q = 0 and V rows one-hot in the key index, out[i][j] > 0 exactly
    for the visible keys; compare with hand-listed sets (bottom-right causal,
    window W counts the query's own position)."""
    Lq, Lk, d = 4, 6, 8
    q = torch.zeros(Lq, 1, d, dtype=torch.bfloat16)
    k = torch.zeros(Lk, d, dtype=torch.bfloat16)
    v = torch.eye(Lk, d, dtype=torch.bfloat16)
    hand = {
        (False, 0): [[0, 1, 2, 3, 4, 5]] * 4,
        (True, 0): [[0, 1, 2], [0, 1, 2, 3], [0, 1, 2, 3, 4], [0, 1, 2, 3, 4, 5]],
        (True, 3): [[0, 1, 2], [1, 2, 3], [2, 3, 4], [3, 4, 5]],
        (True, 1): [[2], [3], [4], [5]],
        (True, 100): [[0, 1, 2], [0, 1, 2, 3], [0, 1, 2, 3, 4], [0, 1, 2, 3, 4, 5]],
    }
    for (causal, W), sets in hand.items():
        out, _ = oracle.attend(q, k, v, [0.0], [0, Lq], [0, Lk], 1, 1, d, 1.0, causal, W)
        for i in range(Lq):
            got = [j for j in range(Lk) if out[i, j] > 0]
            assert got == sets[i], (causal, W, i, got)
            np.testing.assert_allclose(out[i, sets[i]], 1.0 / (len(sets[i]) + 1.0), atol=1e-15)


def test_tiny_workload_pair_count(oracle_lib):
    """The tiny workload (q_len 16 against 128 keys, causal) has
    16*113 + (0+1+...+15) = 1928 visible pairs per head. Recover each row's
    visible count n from the oracle with q = 0, V = 1, sink 0:
    out = n/(n+1)."""
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(w)
    out, _ = oracle.attend(torch.zeros_like(inp["q"]), inp["k"], torch.ones_like(inp["v"]),
                           np.zeros(4), inp["cu_q"], inp["cu_k"], 4, 1, 64, w.scale, True, 0)
    n = out[:, 0] / (1.0 - out[:, 0])
    assert np.allclose(n, np.round(n), atol=1e-9)
    assert int(np.round(n).sum()) == 1928 * 4


def test_single_key_closed_form(oracle_lib):
    """One visible key: out = v/(1 + e^{s-l}), lse = l + ln(1 + e^{s-l})."""
    inp = workloads.explicit_inputs([1], [1], 3, 1, 8, seed=5)
    sinks = np.array([-2.0, 0.0, 1.0])
    out, lse = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"], inp["cu_k"], 3, 1,
                             8, 0.35, True)
    qd = inp["q"].double().numpy()[0]
    kd = inp["k"].double().numpy()[0]
    vd = inp["v"].double().numpy()[0]
    for h in range(3):
        l = 0.35 * float(qd[h] @ kd)
        np.testing.assert_allclose(out[h], vd / (1.0 + math.exp(sinks[h] - l)), atol=1e-14)
        assert abs(lse[h] - (l + math.log1p(math.exp(sinks[h] - l)))) < 1e-13


def test_huge_sink_absorbs_everything(oracle_lib):
    inp = workloads.explicit_inputs([4], [64], 2, 1, 16, seed=6)
    out, lse = oracle.attend(inp["q"], inp["k"], inp["v"], [60.0, 60.0], inp["cu_q"], inp["cu_k"],
                             2, 1, 16, 0.25, True)
    assert np.abs(out).max() < 1e-15
    np.testing.assert_allclose(lse, 60.0, atol=1e-12)


def test_no_keys(oracle_lib):
    """A sequence with queries but no keys is rejected (Lq > Lk); a sequence
    with neither is skipped; with keys absent and no sink the row is empty."""
    q = torch.ones(1, 1, 4, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.attend(q, torch.zeros(0, 4, dtype=torch.bfloat16), torch.zeros(0, 4, dtype=torch.bfloat16),
                      [0.5], [0, 1], [0, 0], 1, 1, 4, 1.0, True)
    # fully masked row: window excludes nothing here, so emulate "no keys" via merge of empty chunks
    acc = np.zeros((1, 1, 3, 4))
    m = np.full((1, 1, 3), -np.inf)
    dd = np.zeros((1, 1, 3))
    out, lse = oracle.merge(acc, m, dd, [0.5], 1, 4)
    np.testing.assert_array_equal(out, 0.0)
    assert lse[0, 0] == 0.5
    out, lse = oracle.merge(acc, m, dd, None, 1, 4)
    np.testing.assert_array_equal(out, 0.0)
    assert lse[0, 0] == -np.inf


# --------------------------------------------------------------------------
# split invariance: every contiguous partition, folded with the sink once
# --------------------------------------------------------------------------
def _compositions(n, parts):
    """All ways to cut range(n) into `parts` contiguous (possibly empty) chunks."""
    for cuts in itertools.combinations_with_replacement(range(n + 1), parts - 1):
        yield (0,) + cuts + (n,)


@pytest.mark.parametrize("Lk", [1, 2, 5, 8])
def test_split_invariance_every_partition(oracle_lib, Lk):
    Hq, Hkv, d = 2, 1, 8
    inp = workloads.explicit_inputs([1], [Lk], Hq, Hkv, d, seed=7 + Lk, q_scale=2.0)
    sinks = np.array([0.75, -np.inf])
    args = (inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"], Hq, Hkv, d, 0.4, True, 0)
    full_out, full_lse = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"], inp["cu_k"],
                                       Hq, Hkv, d, 0.4, True, 0)
    n_checked = 0
    for h in range(Hq):
        for parts in range(1, 5):
            for bounds in _compositions(Lk, parts):
                acc = np.zeros((1, 1, parts, d))
                m = np.zeros((1, 1, parts))
                dd = np.zeros((1, 1, parts))
                for s in range(parts):
                    acc[0, 0, s], m[0, 0, s], dd[0, 0, s] = oracle.chunk_partial(
                        *args, h, bounds[s], bounds[s + 1])
                out, lse = oracle.merge(acc, m, dd, sinks[h:h + 1], 1, d)
                np.testing.assert_allclose(out[0, 0], full_out[h], rtol=0, atol=1e-12)
                assert abs(lse[0, 0] - full_lse[h]) < 1e-12
                n_checked += 1
    assert n_checked > 0


@pytest.mark.parametrize("S", [1, 2, 3, 7, 16, 40])
def test_split_rule_then_merge_equals_unsplit(oracle_lib, S):
    """Chunks of c = 64 * ceil(Lk / (64 S)) keys (ceil(Lk / S) rounded up to a
    whole number of 64-key tiles): each chunk's partial is the partial of its
    key range, chunks past the end are empty, and the merge of all chunks is
    the unsplit result."""
    Hq, Hkv, d = 8, 2, 16
    kv_lens = [3, 170, 333]
    inp = workloads.explicit_inputs([3, 1, 2], kv_lens, Hq, Hkv, d, seed=11)
    sinks = np.linspace(-2, 2, Hq)
    acc, m, dd = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"], Hq,
                                       Hkv, d, 0.25, True, 0, S)
    out, lse = oracle.merge(acc, m, dd, sinks, Hq, d)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, 0.25, True, 0)
    np.testing.assert_allclose(out.reshape(want_out.shape), want_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(want_lse.shape), want_lse, rtol=0, atol=1e-12)
    args = (inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"], Hq, Hkv, d, 0.25, True, 0)
    for b, Lk in enumerate(kv_lens):
        c = 64 * (-(-Lk // (64 * S)))
        assert c % 64 == 0 and c * S >= Lk and (c - 64) * S < Lk
        tok = [2, 3, 5][b]   # last query of each sequence sees every key
        for s in range(S):
            lo, hi = min(s * c, Lk), min((s + 1) * c, Lk)
            for h in (0, Hq - 1):
                a1, m1, d1 = oracle.chunk_partial(*args, tok * Hq + h, lo, hi)
                assert (m[tok, h, s] == m1) and (dd[tok, h, s] == d1)
                np.testing.assert_array_equal(acc[tok, h, s], a1)
            assert np.isfinite(m[tok, 0, s]) == (lo < hi)


def test_merge_is_invariant_to_rescaled_partials(oracle_lib):
    """A chunk's partial (m, d, acc) is a softmax state up to a common scale:
    (m + c, d e^-c, acc e^-c) describes the same chunk, so the merge must give
    the same out and lse for any c per (row, head, chunk)."""
    Hq, Hkv, d = 6, 2, 8
    inp = workloads.explicit_inputs([2, 3], [40, 25], Hq, Hkv, d, seed=14)
    sinks = np.linspace(-1, 3, Hq)
    acc, m, dd = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"], Hq,
                                       Hkv, d, 0.3, True, 0, 5)
    out, lse = oracle.merge(acc, m, dd, sinks, Hq, d)
    c = np.random.default_rng(3).uniform(-6, 6, size=m.shape)
    fin = np.isfinite(m)
    m2 = np.where(fin, m + c, m)
    d2 = np.where(fin, dd * np.exp(-c), dd)
    acc2 = np.where(fin[..., None], acc * np.exp(-c)[..., None], acc)
    out2, lse2 = oracle.merge(acc2, m2, d2, sinks, Hq, d)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# second implementation (exactly rounded sums)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", [
    ([2, 3], [5, 3], 4, 2, 8, True, 0, 1.0),
    ([4], [9], 6, 3, 4, True, 3, 1.0),
    ([3, 2], [3, 6], 4, 1, 8, False, 0, 4.0),   # peaky logits
])
def test_cpp_oracle_matches_fsum_oracle(oracle_lib, case):
    q_lens, kv_lens, Hq, Hkv, d, causal, W, qs = case
    inp = workloads.explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=12, q_scale=qs)
    sinks = np.linspace(-1.5, 2.5, Hq)
    out, lse = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"], inp["cu_k"], Hq,
                             Hkv, d, 0.3, causal, W)
    bo, bl = brute.attend_fsum(inp["q"].double().tolist(), inp["k"].double().flatten().tolist(),
                               inp["v"].double().flatten().tolist(), sinks.tolist(),
                               inp["cu_q"].tolist(), inp["cu_k"].tolist(), Hq, Hkv, d, 0.3, causal, W)
    np.testing.assert_allclose(out, np.array(bo).reshape(out.shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl).reshape(lse.shape), rtol=0, atol=1e-12)


def test_row_subset_matches_full(oracle_lib):
    inp = workloads.explicit_inputs([5, 7], [9, 7], 4, 2, 8, seed=13)
    s = np.array([0.1, 0.2, -0.3, 1.0])
    full, lf = oracle.attend(inp["q"], inp["k"], inp["v"], s, inp["cu_q"], inp["cu_k"], 4, 2, 8, 0.3, True)
    rows = [0, 5, 17, 47, 30]
    sub, ls = oracle.attend(inp["q"], inp["k"], inp["v"], s, inp["cu_q"], inp["cu_k"], 4, 2, 8, 0.3,
                            True, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(ls, lf[rows])


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV: the decode of the codes, and the scales' use
# ---------------------------------------------------------------------------
def test_e4m3_decode_matches_torch_float8(oracle_lib):
    """Every e4m3 code decodes to torch's float8_e4m3fn value (NaN codes to NaN)."""
    got = oracle.e4m3_table()
    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert (np.isnan(got) == np.isnan(want)).all()
    fin = ~np.isnan(want)
    np.testing.assert_array_equal(got[fin], want[fin])
    # a few values fixed by the format: largest normal, smallest normal and subnormal
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9


def _fp8_case(seed, Hkv):
    """Random e4m3 codes (no NaN) for K and V and power-of-two scales per KV
    head, plus the bf16 tensors of exactly the dequantised values."""
    inp = workloads.explicit_inputs([3, 1, 5], [40, 7, 90], 4 * Hkv, Hkv, 64, seed=seed)
    g = torch.Generator().manual_seed(seed)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
    valid = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    kc = valid[torch.randint(len(valid), inp["k"].shape, generator=g)]
    vc = valid[torch.randint(len(valid), inp["v"].shape, generator=g)]
    ks = torch.tensor([2.0 ** (-3 + (i % 4)) for i in range(Hkv)], dtype=torch.float64)
    vs = torch.tensor([2.0 ** (1 - (i % 3)) for i in range(Hkv)], dtype=torch.float64)
    cu = inp["cu_k"].tolist()
    heads = torch.cat([torch.arange(Hkv).repeat_interleave(cu[b + 1] - cu[b])
                       for b in range(len(cu) - 1)])
    kb = (table[kc.long()] * ks[heads][:, None]).to(torch.bfloat16)
    vb = (table[vc.long()] * vs[heads][:, None]).to(torch.bfloat16)
    # the dequantised values are exact in bf16 (4 significant bits, small exponents)
    assert torch.equal(kb.double(), table[kc.long()] * ks[heads][:, None])
    return inp, kc, vc, ks, vs, kb, vb


def test_fp8_oracle_equals_bf16_oracle_on_exactly_representable_values(oracle_lib):
    """With power-of-two scales the dequantised K/V are exact bf16 values: the
    FP8 path (codes x per-head scales) must give the bf16 path's result on
    them, for full rows and for split partials; distinct key / value scales
    per KV head check which scale goes where."""
    Hkv = 3
    inp, kc, vc, ks, vs, kb, vb = _fp8_case(5, Hkv)
    Hq, d = 4 * Hkv, 64
    args = (inp["cu_q"], inp["cu_k"], Hq, Hkv, d, 0.2, True, 0)
    o8, l8 = oracle.attend(inp["q"], kc, vc, inp["sinks"], *args, k_scale=ks, v_scale=vs)
    ob, lb = oracle.attend(inp["q"], kb, vb, inp["sinks"], *args)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, lb, rtol=0, atol=1e-12)
    a8, m8, d8 = oracle.split_partials(inp["q"], kc, vc, inp["cu_q"], inp["cu_k"], Hq, Hkv, d,
                                       0.2, True, 0, 3, k_scale=ks, v_scale=vs)
    ab, mb, db = oracle.split_partials(inp["q"], kb, vb, inp["cu_q"], inp["cu_k"], Hq, Hkv, d,
                                       0.2, True, 0, 3)
    np.testing.assert_allclose(a8, ab, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(m8, mb)
    np.testing.assert_allclose(d8, db, rtol=0, atol=1e-12)

"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle,
element by element, on the same seeded bf16 inputs.

Small shapes span several KV tiles and ragged tails; edge cases cover empty
sequences, chunked prefill (Lq < Lk), windows of 1, empty KV chunks, sinks of
-inf / +-30, and peaky logits. Split decode is checked step by step: the
per-chunk partials against the oracle's partials, the merge on the oracle's
own partials, and the whole call against the unsplit oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import workloads
from _helpers import TOL_LSE, TOL_MAX, TOL_MEAN, compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    oracle.build()
    assert torch.cuda.is_available()
    yield
    assert sa.sinkattn_debug_status() == 0


def _sinks(kind, Hq, base):
    if kind == "given":
        return base
    if kind == "none":
        return None
    if kind == "mixed":
        vals = [-math.inf, -30.0, -2.0, 0.0, 1.5, 30.0]
        return torch.tensor([vals[h % len(vals)] for h in range(Hq)], dtype=torch.float32)
    return torch.full((Hq,), float(kind), dtype=torch.float32)


def _run_prefill(inp, Hq, Hkv, d, scale, causal, window, sinks):
    g = to_dev(inp)
    s_dev = None if sinks is None else sinks.cuda()
    out, lse = sa.sinkattn_prefill(g["q"], g["k"], g["v"], s_dev, g["cu_q"], g["cu_k"],
                                   max(inp["q_lens"]), max(inp["kv_lens"]), Hkv, scale, causal,
                                   window)
    torch.cuda.synchronize()
    return out, lse


PREFILL_CASES = [
    # q_lens, kv_lens, Hq, Hkv, d, causal, window, sinks, q_scale
    ([130, 1, 67], [130, 1, 67], 8, 1, 64, True, 0, "given", 1.0),
    ([200, 33], [200, 300], 16, 2, 128, True, 0, "given", 1.0),       # chunked prefill
    ([129, 64], [129, 64], 64, 4, 128, True, 0, "given", 1.0),         # GQA 16, d 128
    ([100, 257], [100, 257], 64, 8, 64, True, 128, "given", 1.0),      # window 128
    ([70], [70], 4, 4, 64, True, 1, "given", 1.0),                     # MHA, window 1
    ([90, 45], [90, 120], 6, 2, 64, False, 0, "given", 1.0),           # non-causal, G = 3
    ([0, 50, 0, 3], [10, 50, 0, 3], 8, 2, 64, True, 0, "given", 1.0),  # empty sequences
    ([96], [96], 8, 1, 128, True, 0, "none", 1.0),
    ([96], [96], 8, 1, 64, True, 0, "mixed", 1.0),
    ([150], [150], 16, 1, 64, True, 0, "given", 4.0),                  # peaky logits
    ([81], [81], 32, 2, 128, True, 17, "mixed", 3.0),
    ([1, 2, 3], [1, 2, 3], 4, 1, 128, True, 0, "given", 1.0),          # tiny sequences
    ([40, 7], [40, 7], 128, 1, 64, True, 0, "given", 1.0),            # G = 128: one token per tile
    ([33], [60], 32, 1, 128, True, 0, "given", 1.0),                   # G = 32, chunked
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "q%s_k%s_h%d-%d_d%d_c%d_w%d_%s_x%g" % (
    "-".join(map(str, c[0])), "-".join(map(str, c[1])), c[2], c[3], c[4], c[5], c[6], c[7], c[8]))
@pytest.mark.parametrize("launch", ["one_block", "persistent"])
def test_prefill_matches_oracle(case, launch):
    q_lens, kv_lens, Hq, Hkv, d, causal, window, sk, qs = case
    inp = workloads.explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=21, q_scale=qs)
    sinks = _sinks(sk, Hq, inp["sinks"])
    scale = 1.0 / math.sqrt(d)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], sinks, inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, causal, window)
    sa.sinkattn_set_prefill_kernel(launch)
    try:
        out, lse = _run_prefill(inp, Hq, Hkv, d, scale, causal, window, sinks)
    finally:
        sa.sinkattn_set_prefill_kernel("auto")
    compare(out, lse, want_out, want_lse, "prefill " + launch)


@pytest.mark.parametrize("d,Hq,Hkv,window,page", [(64, 16, 8, 0, 0), (128, 16, 4, 0, 0),
                                                  (64, 8, 2, 40, 0), (64, 16, 8, 0, 32),
                                                  (128, 8, 8, 0, 16)])
@pytest.mark.parametrize("launch", ["one_block", "persistent"])
def test_prefill_many_items_per_cta(d, Hq, Hkv, window, page, launch):
    """More (query block, KV head, sequence) items than SMs, so every CTA of
    the persistent prefill runs several items back to back (the K/V ring, S
    buffers and barrier phases carry over); varied lengths, some sequences
    with fewer queries than keys and some with none."""
    sa.sinkattn_set_prefill_kernel(launch)
    try:
        _many_items(d, Hq, Hkv, window, page)
    finally:
        sa.sinkattn_set_prefill_kernel("auto")


def _many_items(d, Hq, Hkv, window, page):
    rng = np.random.default_rng(17 + d + window + page)
    B = 64
    kv_lens = rng.integers(1, 320, size=B).tolist()
    q_lens = [int(min(k, max(0, rng.integers(-20, k + 1)))) for k in kv_lens]
    inp = workloads.explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=29)
    scale = 1.0 / math.sqrt(d)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, window)
    g = to_dev(inp)
    if page:
        pg = to_dev(workloads.to_paged(inp, Hkv, page, seed=3))
        out, lse = sa.sinkattn_prefill_paged(g["q"], pg["k_pages"], pg["v_pages"], g["sinks"],
                                             g["cu_q"], g["cu_k"], pg["page_indptr"],
                                             pg["page_indices"], max(q_lens), max(kv_lens),
                                             scale, True, window)
    else:
        out, lse = sa.sinkattn_prefill(g["q"], g["k"], g["v"], g["sinks"], g["cu_q"], g["cu_k"],
                                       max(q_lens), max(kv_lens), Hkv, scale, True, window)
    torch.cuda.synchronize()
    compare(out, lse, want_out, want_lse, "prefill, many items per CTA")


def test_tiny_workload_prefill_and_decode():
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(w)
    Hq, Hkv, d = w.num_qo_heads, w.num_kv_heads, w.head_dim
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, w.scale, True, 0)
    out, lse = _run_prefill(inp, Hq, Hkv, d, w.scale, True, 0, inp["sinks"])
    compare(out, lse, want_out, want_lse, "tiny prefill")
    g = to_dev(inp)
    for S in (1, 3, 8, 200):
        out, lse = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], 16, 128, Hkv,
                                      num_splits=S, sm_scale=w.scale)
        torch.cuda.synchronize()
        compare(out, lse, want_out, want_lse, "tiny decode S=%d" % S)


def check_partials(acc, md, acc_o, m_o, d_o):
    """Split partials against the oracle's. A partial (m, d, acc) is defined
    up to a common rescale, so compare what is unique: which chunks are
    empty, the chunk's log-sum-exp m + ln d, and its normalised output acc / d."""
    acc_g, md_g = acc.cpu().numpy(), md.cpu().numpy()
    m_g, d_g = md_g[..., 0], md_g[..., 1]
    empty = np.isneginf(m_o)
    assert (np.isneginf(m_g) == empty).all()
    assert (d_g[empty] == 0).all() and (acc_g[empty] == 0).all()
    ne = ~empty
    lse_g = m_g[ne] + np.log(d_g[ne])
    lse_o = m_o[ne] + np.log(d_o[ne])
    assert np.abs(lse_g - lse_o).max() <= TOL_LSE
    og = acc_g[ne] / d_g[ne][:, None]
    oo = acc_o[ne] / d_o[ne][:, None]
    assert np.abs(og - oo).max() <= TOL_MAX and np.abs(og - oo).mean() <= TOL_MEAN


def _decode_inputs(B, q_len, Hq, Hkv, d, kv_range, seed, q_scale=1.0):
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=B, q_len=q_len,
                           kv_range=kv_range, sink_dist="uniform2", seed=seed)
    return workloads.make_inputs(w, q_scale=q_scale)


DECODE_CASES = [
    # B, q_len, Hq, Hkv, d, kv_range, S, window
    (3, 1, 64, 8, 64, (1, 300), 4, 0),
    (4, 3, 64, 4, 128, (3, 500), 16, 0),
    (2, 16, 4, 1, 64, (16, 200), 2, 0),
    (3, 4, 32, 2, 128, (4, 129), 40, 0),     # more chunks than keys: empty chunks
    (2, 2, 8, 8, 64, (2, 100), 3, 16),       # window 16
    (1, 1, 64, 1, 64, (50, 70), 1, 0),       # GQA 64: four warp tiles
    (2, 5, 16, 1, 128, (5, 90), 2, 0),       # 80 rows: two query blocks
    (5, 2, 12, 3, 64, (2, 333), 5, 0),       # GQA 4 with odd head count
    (2, 1, 32, 2, 128, (1, 700), 3, 0),      # 16 rows per block (tcgen05 N = 16)
    (2, 2, 64, 4, 128, (2, 1500), 2, 64),    # 32 rows, window 64
    (1, 3, 64, 4, 128, (1900, 2100), 1, 0),  # one chunk of 16 tiles: 4 TMEM groups
    (2, 8, 64, 4, 128, (600, 1500), 1, 0),   # 128 rows over many tiles: two-stage ring
    (64, 3, 64, 4, 128, (100, 1200), 8, 0),  # many items per CTA, chunks of 0-3 tiles
    # MTP / speculative drafts at the gpt-oss layout (64/8, d 64) ...
    (3, 2, 64, 8, 64, (2, 900), 4, 0),
    (3, 3, 64, 8, 64, (3, 900), 4, 0),
    (3, 4, 64, 8, 64, (4, 1200), 3, 0),
    # ... and at the Qwen layout (64/4, d 128), up to 16 drafts (256 rows: two query blocks)
    (3, 2, 64, 4, 128, (2, 1400), 16, 0),
    (3, 4, 64, 4, 128, (4, 1400), 16, 0),
    (2, 16, 64, 4, 128, (16, 900), 4, 0),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "b%d_q%d_h%d-%d_d%d_k%d-%d_s%d_w%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5][0], c[5][1], c[6], c[7]))
@pytest.mark.parametrize("kernel", ["auto", "warp"])
def test_decode_split_merge_matches_oracle(case, kernel):
    sa.sinkattn_set_decode_kernel(kernel)
    try:
        _decode_split_merge(case)
    finally:
        sa.sinkattn_set_decode_kernel("auto")


def _decode_split_merge(case):
    B, q_len, Hq, Hkv, d, kvr, S, window = case
    inp = _decode_inputs(B, q_len, Hq, Hkv, d, kvr, seed=31 + S)
    scale = 1.0 / math.sqrt(d)
    g = to_dev(inp)
    max_kv = max(inp["kv_lens"])

    # step 1: partials against the oracle's own partials
    acc, md = sa.sinkattn_decode_split(g["q"], g["k"], g["v"], g["cu_k"], q_len, max_kv, Hkv, S,
                                       scale, True, window)
    torch.cuda.synchronize()
    acc_o, m_o, d_o = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"],
                                            Hq, Hkv, d, scale, True, window, S)
    check_partials(acc, md, acc_o, m_o, d_o)

    # step 2: the merge alone, fed the oracle's partials
    mo, lo = oracle.merge(acc_o, m_o, d_o, inp["sinks"], Hq, d)
    part_acc = torch.from_numpy(acc_o.astype(np.float32)).cuda()
    part_md = torch.from_numpy(np.stack([m_o, d_o], -1).astype(np.float32)).cuda()
    out, lse = sa.sinkattn_merge(part_acc, part_md, g["sinks"])
    torch.cuda.synchronize()
    compare(out, lse, mo.reshape(-1, d), lo.reshape(-1), "merge")

    # the whole call against the unsplit oracle
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, window)
    out, lse = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                  Hkv, num_splits=S, sm_scale=scale, window=window)
    torch.cuda.synchronize()
    compare(out, lse, want_out, want_lse, "decode")


def test_merge_accepts_rescaled_partials():
    """sinkattn_merge reads a partial only through the invariant m + ln d and
    acc / d: the oracle's partials rescaled by a random c per chunk give the
    oracle's unsplit result."""
    B, q_len, Hq, Hkv, d, S = 3, 3, 32, 2, 128, 6
    inp = _decode_inputs(B, q_len, Hq, Hkv, d, (3, 700), seed=91)
    scale = 1.0 / math.sqrt(d)
    acc_o, m_o, d_o = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"],
                                            Hq, Hkv, d, scale, True, 0, S)
    c = np.random.default_rng(5).uniform(-10, 10, size=m_o.shape)
    fin = np.isfinite(m_o)
    m2 = np.where(fin, m_o + c, m_o)
    d2 = np.where(fin, d_o * np.exp(-c), d_o)
    acc2 = np.where(fin[..., None], acc_o * np.exp(-c)[..., None], acc_o)
    part_acc = torch.from_numpy(acc2.astype(np.float32)).cuda()
    part_md = torch.from_numpy(np.stack([m2, d2], -1).astype(np.float32)).cuda()
    out, lse = sa.sinkattn_merge(part_acc, part_md, inp["sinks"].cuda())
    torch.cuda.synchronize()
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, 0)
    compare(out, lse, want_out, want_lse, "merge of rescaled partials")


TC_DECODE_CASES = [
    # B, q_len, Hq, Hkv, kv_range, S, window, q_scale   (rows per item = G x tokens)
    (3, 1, 64, 4, (1, 900), 2, 0, 3.0),        # 16 rows
    (2, 4, 64, 8, (4, 1300), 1, 0, 3.0),       # GQA 8 x 4 tokens: 32 rows, one long chunk
    (4, 3, 64, 4, (3, 2600), 2, 0, 4.0),       # 48 rows, peaky logits (lazy rescales)
    (2, 4, 32, 2, (4, 700), 3, 100, 1.0),      # 64 rows, window 100
    (3, 7, 32, 2, (7, 400), 2, 0, 1.0),        # 112 rows: one query block of 7 tokens
    (2, 12, 32, 2, (12, 300), 3, 0, 1.0),      # 128-row tiles: query blocks of 8 and 4 tokens
    (2, 3, 24, 2, (3, 500), 4, 0, 1.0),        # GQA 12: 36 real rows in a 48-row Q tile
    (1, 2, 8, 8, (2, 200), 5, 9, 1.0),         # MHA (G 1), window 9, mostly empty chunks
    (300, 3, 64, 4, (3, 64), 16, 0, 1.0),      # many short items per CTA, most chunks empty
    (7, 3, 64, 4, (3000, 9000), 16, 0, 8.0),   # very peaky logits: rescales every few tiles
]


@pytest.mark.parametrize("case", TC_DECODE_CASES, ids=lambda c: "b%d_q%d_h%d-%d_k%d-%d_s%d_w%d_x%g" % (
    c[0], c[1], c[2], c[3], c[4][0], c[4][1], c[5], c[6], c[7]))
def test_tcgen05_decode_partials(case):
    """The tcgen05 split kernel forced on, partials against the oracle's;
    peaky logits and chunks longer than one TMEM group of tiles."""
    B, q_len, Hq, Hkv, kvr, S, window, qs = case
    d = 128
    inp = _decode_inputs(B, q_len, Hq, Hkv, d, kvr, seed=71 + S, q_scale=qs)
    scale = 1.0 / math.sqrt(d)
    g = to_dev(inp)
    max_kv = max(inp["kv_lens"])
    sa.sinkattn_set_decode_kernel("tcgen05")
    try:
        acc, md = sa.sinkattn_decode_split(g["q"], g["k"], g["v"], g["cu_k"], q_len, max_kv, Hkv,
                                           S, scale, True, window)
        out, lse = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                      Hkv, num_splits=S, sm_scale=scale, window=window)
        torch.cuda.synchronize()
    finally:
        sa.sinkattn_set_decode_kernel("auto")
    acc_o, m_o, d_o = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"],
                                            Hq, Hkv, d, scale, True, window, S)
    check_partials(acc, md, acc_o, m_o, d_o)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, window)
    compare(out, lse, want_out, want_lse, "tcgen05 decode")


def test_tcgen05_decode_without_staged_kv_indptr():
    """More sequences than the kernel stages in shared memory (2048): every
    role reads kv_indptr from global memory instead."""
    B, q_len, Hq, Hkv, d, S = 2100, 1, 16, 1, 128, 2
    inp = _decode_inputs(B, q_len, Hq, Hkv, d, (1, 40), seed=99)
    scale = 1.0 / math.sqrt(d)
    g = to_dev(inp)
    max_kv = max(inp["kv_lens"])
    sa.sinkattn_set_decode_kernel("tcgen05")
    try:
        out, lse = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                      Hkv, num_splits=S, sm_scale=scale)
        torch.cuda.synchronize()
    finally:
        sa.sinkattn_set_decode_kernel("auto")
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, 0)
    compare(out, lse, want_out, want_lse, "tcgen05 decode, 2100 sequences")


def test_tcgen05_decode_rejects_unsupported_shape():
    inp = _decode_inputs(2, 1, 64, 8, 64, (10, 100), seed=3)
    g = to_dev(inp)
    sa.sinkattn_set_decode_kernel("tcgen05")
    try:
        with pytest.raises(sa.SinkAttnError) as e:
            sa.sinkattn_decode_split(g["q"], g["k"], g["v"], g["cu_k"], 1, 100, 8, 2, 0.125,
                                     True, 0)
        assert e.value.status == 2
    finally:
        sa.sinkattn_set_decode_kernel("auto")


def test_decode_default_splits_and_no_sink():
    inp = _decode_inputs(6, 1, 64, 8, 64, (100, 2000), seed=41)
    g = to_dev(inp)
    scale = 0.125
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], None, inp["cu_q"], inp["cu_k"],
                                       64, 8, 64, scale, True, 0)
    out, lse = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], None, 1,
                                  max(inp["kv_lens"]), 8, num_splits=0, sm_scale=scale)
    torch.cuda.synchronize()
    compare(out, lse, want_out, want_lse, "decode default splits")


def test_outputs_are_deterministic():
    inp = _decode_inputs(4, 3, 64, 4, 128, (200, 900), seed=51)
    g = to_dev(inp)
    r1 = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], 3, 900, 4, num_splits=7)
    r2 = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], 3, 900, 4, num_splits=7)
    torch.cuda.synchronize()
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "b%d_q%d_h%d-%d_d%d_k%d-%d_s%d_w%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5][0], c[5][1], c[6], c[7]))
def test_fused_decode_matches_oracle(case):
    """The cluster-fused decode (merge on chip through distributed shared
    memory) against the unsplit oracle; more than 16 chunks is rejected."""
    B, q_len, Hq, Hkv, d, kvr, S, window = case
    inp = _decode_inputs(B, q_len, Hq, Hkv, d, kvr, seed=61 + S)
    scale = 1.0 / math.sqrt(d)
    g = to_dev(inp)
    max_kv = max(inp["kv_lens"])
    if S > 16:
        with pytest.raises(sa.SinkAttnError) as e:
            sa.sinkattn_decode_fused(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                     Hkv, num_splits=S, sm_scale=scale, window=window)
        assert e.value.status == 2
        S = 16
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, window)
    out, lse = sa.sinkattn_decode_fused(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                        Hkv, num_splits=S, sm_scale=scale, window=window)
    torch.cuda.synchronize()
    compare(out, lse, want_out, want_lse, "fused decode S=%d" % S)
    # and it equals split + merge up to rounding
    out2, lse2 = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv,
                                    Hkv, num_splits=S, sm_scale=scale, window=window)
    torch.cuda.synchronize()
    assert (out.float() - out2.float()).abs().max().item() <= 1e-2
    assert (lse - lse2).abs().max().item() <= 1e-4


def test_fused_decode_no_sink_and_default_splits():
    inp = _decode_inputs(5, 2, 32, 4, 64, (2, 3000), seed=71)
    g = to_dev(inp)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], None, inp["cu_q"], inp["cu_k"],
                                       32, 4, 64, 0.125, True, 0)
    out, lse = sa.sinkattn_decode_fused(g["q"], g["k"], g["v"], g["cu_k"], None, 2,
                                        max(inp["kv_lens"]), 4, num_splits=0, sm_scale=0.125)
    torch.cuda.synchronize()
    compare(out, lse, want_out, want_lse, "fused decode, no sink")

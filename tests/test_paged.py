"""GPU parity of the paged-KV entry points against the float64 oracle.

The oracle reads the contiguous ragged HND K/V; the CUDA path reads the same
values scattered into page pools (seeded random page order, spare pages, and
unused page slots filled with large finite values so a mask leak shows).
Page sizes cover every supported power of two (16..256), both below and
above the kernels' 64/128-key tiles.
"""
import math

import pytest
import torch

import oracle
import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import workloads
from gqa_attention_softmax_gb300._binding import BAD_LENGTHS
from _helpers import compare, to_dev
from test_parity import check_partials

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    oracle.build()
    assert torch.cuda.is_available()
    yield
    assert sa.sinkattn_debug_status() == 0


def _decode_inputs(B, q_len, Hq, Hkv, d, kv_range, seed, q_scale=1.0):
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=B, q_len=q_len,
                           kv_range=kv_range, sink_dist="uniform2", seed=seed)
    return workloads.make_inputs(w, q_scale=q_scale)


PAGED_DECODE_CASES = [
    # B, q_len, Hq, Hkv, d, kv_range, S, window, page_size, q_scale
    (3, 1, 64, 8, 64, (1, 300), 4, 0, 16, 1.0),
    (4, 3, 64, 4, 128, (3, 500), 3, 0, 32, 1.0),
    (2, 4, 32, 2, 128, (4, 700), 2, 100, 64, 1.0),     # window across page boundaries
    (3, 2, 64, 8, 64, (2, 900), 2, 0, 128, 1.0),
    (2, 3, 64, 4, 128, (3, 1300), 5, 0, 256, 3.0),     # pages longer than a tile, peaky
    (5, 1, 16, 1, 128, (1, 40), 8, 0, 16, 1.0),        # short sequences, empty chunks
    (2, 16, 4, 1, 64, (16, 200), 2, 0, 64, 1.0),
    (2, 7, 32, 2, 128, (7, 600), 2, 33, 16, 1.0),      # 112 rows, window 33
    (3, 4, 64, 4, 128, (2000, 3000), 1, 0, 16, 1.0),   # long chunk over many 16-key pages
    (2, 6, 32, 2, 128, (400, 900), 1, 0, 32, 1.0),     # 96 rows over many tiles: two-stage ring
]


@pytest.mark.parametrize("case", PAGED_DECODE_CASES,
                         ids=lambda c: "b%d_q%d_h%d-%d_d%d_k%d-%d_s%d_w%d_p%d_x%g" % (
                             c[0], c[1], c[2], c[3], c[4], c[5][0], c[5][1], c[6], c[7], c[8],
                             c[9]))
@pytest.mark.parametrize("kernel", ["auto", "warp"])
def test_paged_decode_matches_oracle(case, kernel):
    B, q_len, Hq, Hkv, d, kvr, S, window, P, qs = case
    inp = _decode_inputs(B, q_len, Hq, Hkv, d, kvr, seed=131 + S + P, q_scale=qs)
    pg = to_dev(workloads.to_paged(inp, Hkv, P, seed=P))
    g = to_dev(inp)
    scale = 1.0 / math.sqrt(d)
    max_kv = max(inp["kv_lens"])
    sa.sinkattn_set_decode_kernel(kernel)
    try:
        acc, md = sa.sinkattn_decode_split_paged(g["q"], pg["k_pages"], pg["v_pages"], g["cu_k"],
                                                 pg["page_indptr"], pg["page_indices"], q_len,
                                                 max_kv, S, scale, True, window)
        out, lse = sa.sinkattn_decode_paged(g["q"], pg["k_pages"], pg["v_pages"], g["cu_k"],
                                            pg["page_indptr"], pg["page_indices"], g["sinks"],
                                            q_len, max_kv, num_splits=S, sm_scale=scale,
                                            window=window)
        torch.cuda.synchronize()
    finally:
        sa.sinkattn_set_decode_kernel("auto")
    acc_o, m_o, d_o = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"],
                                            Hq, Hkv, d, scale, True, window, S)
    check_partials(acc, md, acc_o, m_o, d_o)
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, True, window)
    compare(out, lse, want_out, want_lse, "paged decode")


PAGED_PREFILL_CASES = [
    # q_lens, kv_lens, Hq, Hkv, d, causal, window, page_size
    ([130, 1, 67], [130, 1, 67], 8, 1, 64, True, 0, 16),
    ([200, 33], [200, 300], 16, 2, 128, True, 0, 32),      # chunked prefill
    ([129, 64], [129, 64], 64, 4, 128, True, 0, 64),
    ([100, 257], [100, 257], 64, 8, 64, True, 128, 128),   # window 128
    ([90, 45], [90, 120], 6, 2, 64, False, 0, 256),        # non-causal
    ([0, 50, 0, 3], [10, 50, 0, 3], 8, 2, 64, True, 0, 16),  # empty sequences
    ([300], [300], 16, 1, 128, True, 37, 16),              # window 37 over 16-key pages
]


@pytest.mark.parametrize("case", PAGED_PREFILL_CASES,
                         ids=lambda c: "q%s_k%s_h%d-%d_d%d_c%d_w%d_p%d" % (
                             "-".join(map(str, c[0])), "-".join(map(str, c[1])), c[2], c[3], c[4],
                             c[5], c[6], c[7]))
def test_paged_prefill_matches_oracle(case):
    q_lens, kv_lens, Hq, Hkv, d, causal, window, P = case
    inp = workloads.explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=23)
    pg = to_dev(workloads.to_paged(inp, Hkv, P, seed=7))
    g = to_dev(inp)
    scale = 1.0 / math.sqrt(d)
    out, lse = sa.sinkattn_prefill_paged(g["q"], pg["k_pages"], pg["v_pages"], g["sinks"],
                                         g["cu_q"], g["cu_k"], pg["page_indptr"],
                                         pg["page_indices"], max(q_lens), max(kv_lens), scale,
                                         causal, window)
    torch.cuda.synchronize()
    want_out, want_lse = oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"],
                                       inp["cu_k"], Hq, Hkv, d, scale, causal, window)
    compare(out, lse, want_out, want_lse, "paged prefill")


@pytest.mark.parametrize("page_size", [32, 128])
@pytest.mark.parametrize("kernel", ["auto", "warp"])
def test_paged_decode_with_too_few_pages_records_bad_lengths(kernel, page_size):
    """A sequence given fewer pages than its key count needs: the kernel
    reads only pool pages and records SINKATTN_BAD_LENGTHS (pages smaller
    than a tile and pages holding whole tiles)."""
    inp = _decode_inputs(3, 1, 16, 1, 128, (100, 200) if page_size < 64 else (300, 600), seed=5)
    pg = workloads.to_paged(inp, 1, page_size, seed=1)
    # drop the last page of sequence 1
    ind = pg["page_indptr"].tolist()
    idx = pg["page_indices"].tolist()
    idx = idx[:ind[2] - 1] + idx[ind[2]:]
    ind = ind[:2] + [x - 1 for x in ind[2:]]
    pg["page_indptr"] = torch.tensor(ind, dtype=torch.int32)
    pg["page_indices"] = torch.tensor(idx, dtype=torch.int32)
    pg, g = to_dev(pg), to_dev(inp)
    assert sa.sinkattn_debug_status() == 0
    sa.sinkattn_set_decode_kernel(kernel)
    try:
        sa.sinkattn_decode_split_paged(g["q"], pg["k_pages"], pg["v_pages"], g["cu_k"],
                                       pg["page_indptr"], pg["page_indices"], 1,
                                       max(inp["kv_lens"]), 2)
        torch.cuda.synchronize()
    finally:
        sa.sinkattn_set_decode_kernel("auto")
    assert sa.sinkattn_debug_status() == BAD_LENGTHS


def test_paged_prefill_with_too_few_pages_records_bad_lengths():
    inp = workloads.explicit_inputs([40, 70], [40, 70], 8, 1, 64, seed=9)
    pg = workloads.to_paged(inp, 1, 16, seed=2)
    ind = pg["page_indptr"].tolist()
    pg["page_indptr"] = torch.tensor([0, ind[1], ind[2] - 1], dtype=torch.int32)
    pg["page_indices"] = pg["page_indices"][:ind[2] - 1].clone()
    pg, g = to_dev(pg), to_dev(inp)
    assert sa.sinkattn_debug_status() == 0
    sa.sinkattn_prefill_paged(g["q"], pg["k_pages"], pg["v_pages"], g["sinks"], g["cu_q"],
                              g["cu_k"], pg["page_indptr"], pg["page_indices"], 70, 70)
    torch.cuda.synchronize()
    assert sa.sinkattn_debug_status() == BAD_LENGTHS


def test_paged_decode_agrees_with_contiguous():
    """The same cache read through pages and contiguously gives the same
    result within the tolerance (tile boundaries differ, so not bit for bit)."""
    B, q_len, Hq, Hkv, d, P = 4, 2, 64, 4, 128, 64
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=B, q_len=q_len,
                           kv_range=(P, 8 * P), seed=3)
    inp = workloads.make_inputs(w)
    pg = to_dev(workloads.to_paged(inp, Hkv, P, seed=0, spare_pages=0))
    g = to_dev(inp)
    max_kv = max(inp["kv_lens"])
    o1, l1 = sa.sinkattn_decode_paged(g["q"], pg["k_pages"], pg["v_pages"], g["cu_k"],
                                      pg["page_indptr"], pg["page_indices"], g["sinks"], q_len,
                                      max_kv, num_splits=3)
    o2, l2 = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], q_len, max_kv, Hkv,
                                num_splits=3)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3

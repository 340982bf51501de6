"""GPU parity of the FP8 (e4m3) KV decode against the float64 oracle.

K and V are drawn in bf16, quantised per KV head (amax / 448 scales, round to
nearest even), and both sides read the same codes and the same fp32 scales:
the oracle decodes each code from the E4M3 definition and multiplies by the
scale in float64. The partials are checked chunk by chunk, and the whole
decode against the unsplit oracle.
"""
import math

import pytest
import torch

import oracle
import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import workloads
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


FP8_CASES = [
    # B, q_len, Hq, Hkv, d, kv_range, S, window, q_scale
    (3, 1, 64, 8, 64, (1, 300), 4, 0, 1.0),        # gpt-oss shape: 8 rows per KV head
    (4, 3, 64, 4, 128, (3, 500), 3, 0, 1.0),       # MTP shape: 48 rows
    (2, 2, 32, 2, 128, (2, 700), 2, 100, 1.0),     # 32 rows, window 100
    (2, 4, 64, 8, 64, (4, 1300), 5, 0, 3.0),       # 32 rows, peaky logits
    (5, 1, 16, 1, 128, (1, 40), 8, 0, 1.0),        # short sequences, empty chunks
    (2, 16, 4, 1, 64, (16, 200), 2, 0, 1.0),       # 64 rows
    (1, 1, 8, 8, 64, (2000, 2000), 1, 0, 1.0),     # MHA, one long chunk
    (2, 3, 64, 8, 64, (3, 900), 4, 50, 1.0),       # 24 rows, window 50: masks in the permuted key order
    (2, 8, 64, 8, 64, (8, 700), 3, 0, 1.0),        # 64 rows: four row tiles, two token groups
    # head_dim 128 shapes for the tcgen05 kernel (tiles of 16..64 rows, ragged q blocks)
    (3, 4, 64, 4, 128, (4, 900), 3, 0, 1.0),       # 64 rows: the MTP shape
    (2, 5, 32, 4, 128, (5, 1100), 2, 0, 3.0),      # 40 rows, peaky logits
    (3, 7, 32, 2, 128, (7, 600), 2, 33, 1.0),      # 16 heads x 4 tokens + a ragged block
    (4, 1, 16, 16, 128, (1, 3000), 4, 0, 1.0),     # MHA: one row per item
    (2, 2, 128, 2, 128, (2, 400), 2, 0, 1.0),      # 64 heads per group, one token per tile
    (2, 16, 64, 8, 128, (16, 2500), 6, 200, 1.0),  # 8 heads x 8 tokens, window 200
    # many items per CTA, chunks of 0 to 3 tiles (items that end within the S look-ahead)
    (64, 3, 64, 4, 128, (100, 1200), 8, 0, 1.0),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "b%d_q%d_h%d-%d_d%d_k%d-%d_s%d_w%d_x%g" % (
    c[0], c[1], c[2], c[3], c[4], c[5][0], c[5][1], c[6], c[7], c[8]))
@pytest.mark.parametrize("kernel", ["auto", "warp"])
def test_fp8_decode_matches_oracle(case, kernel):
    B, q_len, Hq, Hkv, d, kvr, S, window, qs = case
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=B, q_len=q_len,
                           kv_range=kvr, sink_dist="uniform2", seed=61 + S)
    inp = workloads.make_inputs(w, q_scale=qs)
    f8 = workloads.to_fp8(inp, Hkv)
    g, gf = to_dev(inp), to_dev(f8)
    scale = 1.0 / math.sqrt(d)
    max_kv = max(inp["kv_lens"])
    sa.sinkattn_set_decode_kernel(kernel)
    try:
        acc, md = sa.sinkattn_decode_split_fp8(g["q"], gf["k_fp8"], gf["v_fp8"], gf["k_scale"],
                                               gf["v_scale"], g["cu_k"], q_len, max_kv, S, scale,
                                               True, window)
        out, lse = sa.sinkattn_decode_fp8(g["q"], gf["k_fp8"], gf["v_fp8"], gf["k_scale"],
                                          gf["v_scale"], g["cu_k"], g["sinks"], q_len, max_kv,
                                          num_splits=S, sm_scale=scale, window=window)
        torch.cuda.synchronize()
    finally:
        sa.sinkattn_set_decode_kernel("auto")
    acc_o, m_o, d_o = oracle.split_partials(inp["q"], f8["k_fp8"], f8["v_fp8"], inp["cu_q"],
                                            inp["cu_k"], Hq, Hkv, d, scale, True, window, S,
                                            k_scale=f8["k_scale"], v_scale=f8["v_scale"])
    check_partials(acc, md, acc_o, m_o, d_o)
    want_out, want_lse = oracle.attend(inp["q"], f8["k_fp8"], f8["v_fp8"], inp["sinks"],
                                       inp["cu_q"], inp["cu_k"], Hq, Hkv, d, scale, True, window,
                                       k_scale=f8["k_scale"], v_scale=f8["v_scale"])
    compare(out, lse, want_out, want_lse, "fp8 decode")


def test_fp8_decode_close_to_bf16_decode():
    """The quantisation error itself: FP8 K/V against the bf16 values they
    were rounded from stays small (a few percent of the outputs' scale)."""
    w = workloads.Workload("t", "decode", 64, 8, 64, True, batch=4, q_len=1,
                           kv_range=(500, 1500), sink_dist="uniform2", seed=4)
    inp = workloads.make_inputs(w)
    f8 = workloads.to_fp8(inp, 8)
    g, gf = to_dev(inp), to_dev(f8)
    o1, _ = sa.sinkattn_decode(g["q"], g["k"], g["v"], g["cu_k"], g["sinks"], 1, 1500, 8,
                               num_splits=2)
    o2, _ = sa.sinkattn_decode_fp8(g["q"], gf["k_fp8"], gf["v_fp8"], gf["k_scale"],
                                   gf["v_scale"], g["cu_k"], g["sinks"], 1, 1500, num_splits=2)
    torch.cuda.synchronize()
    err = (o1.float() - o2.float()).abs()
    assert err.max().item() < 0.05 and err.mean().item() < 0.005


@pytest.mark.parametrize("shape", [(16, 2, 64), (256, 2, 128)], ids=["d64", "g128"])
def test_fp8_tcgen05_rejects_unsupported_shapes(shape):
    """Forcing the tcgen05 kernel on an FP8 shape it does not cover (head_dim
    64, or more than 64 heads per group) is SINKATTN_UNSUPPORTED."""
    Hq, Hkv, d = shape
    w = workloads.Workload("t", "decode", Hq, Hkv, d, True, batch=2, q_len=1,
                           kv_range=(10, 50), seed=2)
    inp = workloads.make_inputs(w)
    f8 = workloads.to_fp8(inp, Hkv)
    g, gf = to_dev(inp), to_dev(f8)
    sa.sinkattn_set_decode_kernel("tcgen05")
    try:
        with pytest.raises(sa.SinkAttnError) as e:
            sa.sinkattn_decode_split_fp8(g["q"], gf["k_fp8"], gf["v_fp8"], gf["k_scale"],
                                         gf["v_scale"], g["cu_k"], 1, 50, 2)
        assert e.value.status == 2
    finally:
        sa.sinkattn_set_decode_kernel("auto")


def test_fp8_tcgen05_and_warp_kernels_agree():
    """The two FP8 kernels on the MTP shape: both within the tolerance of each
    other (different tilings, same codes and scales)."""
    w = workloads.Workload("t", "decode", 64, 4, 128, True, batch=6, q_len=4,
                           kv_range=(2000, 6000), sink_dist="uniform2", seed=8)
    inp = workloads.make_inputs(w)
    f8 = workloads.to_fp8(inp, 4)
    g, gf = to_dev(inp), to_dev(f8)
    outs = []
    for kernel in ("tcgen05", "warp"):
        sa.sinkattn_set_decode_kernel(kernel)
        try:
            outs.append(sa.sinkattn_decode_fp8(g["q"], gf["k_fp8"], gf["v_fp8"], gf["k_scale"],
                                               gf["v_scale"], g["cu_k"], g["sinks"], 4, 6000,
                                               num_splits=4))
            torch.cuda.synchronize()
        finally:
            sa.sinkattn_set_decode_kernel("auto")
    (o1, l1), (o2, l2) = outs
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3

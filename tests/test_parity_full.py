"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: sampled rows (first and last query of each checked
sequence for every head, plus random rows) against the float64 oracle, and
properties that hold at any size on every row."""
import numpy as np
import pytest
import torch

import oracle
import gqa_attention_softmax_gb300 as sa
from gqa_attention_softmax_gb300 import runner, workloads
from _helpers import compare, sampled_rows, sub_problem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["gptoss_decode", "qwen_mtp_decode", "gptoss_prefill",
                                  "gptoss_prefill_w128", "qwen_prefill", "gptoss_decode_paged",
                                  "qwen_mtp_decode_paged", "gptoss_decode_fp8",
                                  "qwen_mtp_decode_fp8", "gptoss_mtp2_decode",
                                  "gptoss_mtp4_decode", "qwen_mtp2_decode", "qwen_mtp4_decode",
                                  "qwen_mtp16_decode"])
def test_full_size_sampled_rows(name):
    from gqa_attention_softmax_gb300 import _build
    _build.build()
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda")
    run = runner.Runner(w, inp)
    out, lse = run()
    torch.cuda.synchronize()
    assert sa.sinkattn_debug_status() == 0

    # every row: finite, and |out| bounded by the largest |v| (a convex
    # combination of value rows, shrunk by the sink's share)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert out.float().abs().max().item() <= inp["v"].float().abs().max().item() * 1.01

    Hq, Hkv, d = w.num_qo_heads, w.num_kv_heads, w.head_dim
    B = inp["batch"]
    rng = np.random.default_rng(7)
    seqs = list(range(B)) if B <= 4 else sorted({0, B - 1, *rng.choice(B, 4, replace=False).tolist()})
    scales = {}
    if w.kv_fp8:   # the oracle reads the same e4m3 codes and per-KV-head scales
        sub = sub_problem(dict(inp, k=inp["k_fp8"], v=inp["v_fp8"]), Hkv, d, seqs)
        scales = dict(k_scale=inp["k_scale"].cpu(), v_scale=inp["v_scale"].cpu())
    else:
        sub = sub_problem(inp, Hkv, d, seqs)
    _, rows = sampled_rows(sub, Hq, 384, seed=3)
    want_out, want_lse = oracle.attend(sub["q"], sub["k"], sub["v"], sub["sinks"], sub["cu_q"],
                                       sub["cu_k"], Hq, Hkv, d, w.scale, w.causal, w.window,
                                       rows=rows, **scales)
    orig = sub["tok_map"][rows // Hq] * Hq + rows % Hq
    got_out = out.view(-1, d)[torch.from_numpy(orig).cuda()]
    got_lse = lse.view(-1)[torch.from_numpy(orig).cuda()]
    compare(got_out, got_lse, want_out, want_lse, name)

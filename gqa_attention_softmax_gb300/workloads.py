"""Workload registry and seeded synthetic input generator.

This module holds no attention arithmetic: it only draws random tensors in
the layouts the library consumes, so both the CUDA path's tests/bench and the
float64 oracle can be fed the very same bf16 values.

Layouts (heads-leading KV cache, "Hosting Qwen on Blackwell", section
"Deployment on GB200 NVL72"):

* ``q``, ``out``: bf16 ``[total_q, Hq, d]`` (token-major). For decode,
  ``total_q = B * q_len`` and token ``b * q_len + t`` is draft ``t`` of
  sequence ``b``.
* ``k``, ``v``: bf16 ragged HND ``[Hkv * total_k, d]``: sequence ``b`` is the
  contiguous block ``[Hkv, Lk_b, d]`` starting at row ``Hkv * cu_k[b]``.
* ``sinks``: fp32 ``[Hq]``; ``cu_q``, ``cu_k``: int32 ``[B + 1]``.
* paged KV (``to_paged``): pools ``k_pages``, ``v_pages`` bf16
  ``[num_pages, Hkv, page_size, d]``; sequence ``b``'s keys
  ``[e * page_size, (e + 1) * page_size)`` sit in page
  ``page_indices[page_indptr[b] + e]``.

Draw order (fixed, so a seed names one input set): key lengths, then Q, K, V,
sinks. Q/K/V are drawn as fp32 normals then rounded to bf16 (round to nearest
even). Key lengths are always drawn on the CPU, so a seed gives the same
lengths whatever device the tensors are drawn on.

The workload shapes are those of gpt-oss-style (64 query / 8 KV heads, d 64)
and Qwen3-235B-style (64 query / 4 KV heads, d 128) attention; the pages these
follow run no public benchmark or dataset for attention, so these synthetic
draws are the whole workload.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str                       # "prefill" or "decode"
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    causal: bool
    window: int = 0                 # <= 0: no sliding window
    # prefill: explicit per-sequence lengths (q_len == kv_len unless q_lens given)
    kv_lens: Optional[Sequence[int]] = None
    q_lens: Optional[Sequence[int]] = None
    # decode: batch, q_len, kv_len range (inclusive)
    batch: int = 0
    q_len: int = 1
    kv_range: Optional[tuple] = None
    num_splits: int = 0             # 0: library heuristic
    sink_dist: str = "normal"       # "normal" -> N(0,1); "uniform2" -> U(-2, 2)
    sm_scale: Optional[float] = None  # None -> 1/sqrt(head_dim)
    seed: int = 0
    page_size: int = 0              # > 0: K/V also scattered into page pools (paged decode)
    kv_fp8: bool = False            # K/V also quantised to e4m3 codes (FP8 decode)

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def gqa(self) -> int:
        return self.num_qo_heads // self.num_kv_heads


WORKLOADS = {
    # 1 sequence, GQA 4:1, q_len 16 against 128 keys, causal.
    "tiny": Workload("tiny", "prefill", 4, 1, 64, True, kv_lens=[128], q_lens=[16],
                     sink_dist="normal", sm_scale=1.0 / 8.0),
    # gpt-oss-120b-shaped decode.
    "gptoss_decode": Workload("gptoss_decode", "decode", 64, 8, 64, True, batch=64, q_len=1,
                              kv_range=(1024, 8192), sink_dist="uniform2", sm_scale=1.0 / 8.0),
    # gpt-oss-120b-shaped varlen prefill, full causal and 128-key window.
    "gptoss_prefill": Workload("gptoss_prefill", "prefill", 64, 8, 64, True,
                               kv_lens=[4096, 3000, 2048, 1024], sink_dist="uniform2"),
    "gptoss_prefill_w128": Workload("gptoss_prefill_w128", "prefill", 64, 8, 64, True, window=128,
                                    kv_lens=[4096, 3000, 2048, 1024], sink_dist="uniform2"),
    # Qwen3-235B-shaped prefill, GQA 16:1, d 128.
    "qwen_prefill": Workload("qwen_prefill", "prefill", 64, 4, 128, True, kv_lens=[6000, 6000],
                             sink_dist="normal"),
    # Qwen3-235B-shaped MTP speculative decode: 3 drafts, 16 KV chunks.
    "qwen_mtp_decode": Workload("qwen_mtp_decode", "decode", 64, 4, 128, True, batch=256, q_len=3,
                                kv_range=(4000, 8000), num_splits=16, sink_dist="uniform2"),
    # Wider MTP / speculative drafts ("Hosting Qwen on Blackwell", section
    # "Decoders"): 2 and 4 drafts at both layouts, 16 drafts at the Qwen one.
    "gptoss_mtp2_decode": Workload("gptoss_mtp2_decode", "decode", 64, 8, 64, True, batch=64,
                                   q_len=2, kv_range=(1024, 8192), sink_dist="uniform2",
                                   sm_scale=1.0 / 8.0),
    "gptoss_mtp4_decode": Workload("gptoss_mtp4_decode", "decode", 64, 8, 64, True, batch=64,
                                   q_len=4, kv_range=(1024, 8192), sink_dist="uniform2",
                                   sm_scale=1.0 / 8.0),
    "qwen_mtp2_decode": Workload("qwen_mtp2_decode", "decode", 64, 4, 128, True, batch=256,
                                 q_len=2, kv_range=(4000, 8000), num_splits=16,
                                 sink_dist="uniform2"),
    "qwen_mtp4_decode": Workload("qwen_mtp4_decode", "decode", 64, 4, 128, True, batch=256,
                                 q_len=4, kv_range=(4000, 8000), num_splits=16,
                                 sink_dist="uniform2"),
    "qwen_mtp16_decode": Workload("qwen_mtp16_decode", "decode", 64, 4, 128, True, batch=256,
                                  q_len=16, kv_range=(4000, 8000), num_splits=16,
                                  sink_dist="uniform2"),
    # The two decodes over an FP8 (e4m3) KV cache with per-KV-head scales.
    "gptoss_decode_fp8": Workload("gptoss_decode_fp8", "decode", 64, 8, 64, True, batch=64,
                                  q_len=1, kv_range=(1024, 8192), sink_dist="uniform2",
                                  sm_scale=1.0 / 8.0, kv_fp8=True),
    "qwen_mtp_decode_fp8": Workload("qwen_mtp_decode_fp8", "decode", 64, 4, 128, True,
                                    batch=256, q_len=3, kv_range=(4000, 8000), num_splits=16,
                                    sink_dist="uniform2", kv_fp8=True),
    # The two decodes over a paged KV cache (pages in seeded random order).
    "gptoss_decode_paged": Workload("gptoss_decode_paged", "decode", 64, 8, 64, True, batch=64,
                                    q_len=1, kv_range=(1024, 8192), sink_dist="uniform2",
                                    sm_scale=1.0 / 8.0, page_size=16),
    "qwen_mtp_decode_paged": Workload("qwen_mtp_decode_paged", "decode", 64, 4, 128, True,
                                      batch=256, q_len=3, kv_range=(4000, 8000), num_splits=16,
                                      sink_dist="uniform2", page_size=64),
}


def _randn_bf16(n_rows: int, d: int, gen: torch.Generator, device) -> torch.Tensor:
    """Draw N(0,1) fp32 in row chunks and round to bf16 (bounded fp32 scratch)."""
    out = torch.empty((n_rows, d), dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 26) // max(d, 1))
    for r0 in range(0, n_rows, chunk):
        r1 = min(n_rows, r0 + chunk)
        out[r0:r1] = torch.randn((r1 - r0, d), generator=gen, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None,
                batch: Optional[int] = None, q_scale: float = 1.0) -> dict:
    """Draw one input set for workload ``w``.

    ``batch`` overrides the decode batch (used for bounded samples of a
    workload); ``q_scale`` multiplies Q before rounding (peaky logits).
    Returns a dict of tensors on ``device`` plus host-side sizes.
    """
    seed = w.seed if seed is None else seed
    device = torch.device(device)
    cpu_gen = torch.Generator(device="cpu").manual_seed(seed)
    gen = cpu_gen if device.type == "cpu" else torch.Generator(device=device).manual_seed(seed)

    if w.kind == "decode":
        B = w.batch if batch is None else batch
        lo, hi = w.kv_range
        kv_lens = torch.randint(lo, hi + 1, (B,), generator=cpu_gen).tolist()
        q_lens = [w.q_len] * B
    else:
        kv_lens = list(w.kv_lens)
        q_lens = list(w.q_lens) if w.q_lens is not None else list(kv_lens)
        B = len(kv_lens)
    cu_q = [0]
    cu_k = [0]
    for lq, lk in zip(q_lens, kv_lens):
        cu_q.append(cu_q[-1] + lq)
        cu_k.append(cu_k[-1] + lk)
    total_q, total_k = cu_q[-1], cu_k[-1]
    Hq, Hkv, d = w.num_qo_heads, w.num_kv_heads, w.head_dim

    if q_scale == 1.0:
        q = _randn_bf16(total_q * Hq, d, gen, device)
    else:
        q = (torch.randn((total_q * Hq, d), generator=gen, device=device) * q_scale).to(torch.bfloat16)
    q = q.view(total_q, Hq, d)
    k = _randn_bf16(Hkv * total_k, d, gen, device)
    v = _randn_bf16(Hkv * total_k, d, gen, device)
    if w.sink_dist == "uniform2":
        sinks = torch.rand((Hq,), generator=gen, device=device, dtype=torch.float32) * 4.0 - 2.0
    else:
        sinks = torch.randn((Hq,), generator=gen, device=device, dtype=torch.float32)

    inp = dict(
        q=q, k=k, v=v, sinks=sinks,
        cu_q=torch.tensor(cu_q, dtype=torch.int32, device=device),
        cu_k=torch.tensor(cu_k, dtype=torch.int32, device=device),
        q_lens=q_lens, kv_lens=kv_lens, batch=B, total_q=total_q, total_k=total_k,
        max_q=max(q_lens) if q_lens else 0, max_k=max(kv_lens) if kv_lens else 0,
    )
    if w.page_size > 0:
        inp.update(to_paged(inp, Hkv, w.page_size, seed=seed, spare_pages=0, fill_scale=0.0))
    if w.kv_fp8:
        inp.update(to_fp8(inp, Hkv))
    return inp


def explicit_inputs(q_lens, kv_lens, Hq, Hkv, d, seed=0, device="cpu",
                    sink_dist="normal", q_scale=1.0) -> dict:
    """Inputs for an ad-hoc shape (tests): explicit per-sequence lengths."""
    w = Workload("adhoc", "prefill", Hq, Hkv, d, True, kv_lens=list(kv_lens),
                 q_lens=list(q_lens), sink_dist=sink_dist, seed=seed)
    return make_inputs(w, device=device, q_scale=q_scale)



def to_paged(inp: dict, Hkv: int, page_size: int, seed: int = 0, spare_pages: int = 3,
             fill_scale: float = 100.0, shuffle: bool = True) -> dict:
    """Scatter the ragged HND ``k``/``v`` of ``inp`` into page pools.

    Pages are handed out in a seeded random order (in pool order if not
    ``shuffle``), plus ``spare_pages`` that no sequence uses; every slot that
    holds no key of a sequence -- the tail of each sequence's last page and
    the spare pages -- is filled with large finite values (N(0, fill_scale^2),
    bf16; zeros if fill_scale is 0), so a kernel that lets such a slot through
    its mask shows it. Returns k_pages, v_pages, page_indptr, page_indices on
    the device of ``inp["k"]``. Pure data movement.
    """
    k, v = inp["k"], inp["v"]
    dev = k.device
    d = k.shape[1]
    kv_lens = torch.tensor(list(inp["kv_lens"]), dtype=torch.int64)
    n_b = (kv_lens + page_size - 1) // page_size
    used = int(n_b.sum())
    total = used + spare_pages
    gen = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(total, generator=gen) if shuffle else torch.arange(total)
    shape = (total, Hkv, page_size, d)
    if fill_scale == 0:
        kp = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        vp = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    else:
        fgen = gen if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(seed)
        kp = (torch.randn(shape, generator=fgen, device=dev) * fill_scale).to(torch.bfloat16)
        vp = (torch.randn(shape, generator=fgen, device=dev) * fill_scale).to(torch.bfloat16)
    indptr = torch.zeros(len(n_b) + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(n_b, 0)
    # destination row of every source row (sequence b, head h, key t) of the
    # ragged HND layout: slot t % P of head h in page perm[indptr[b] + t // P]
    rows_b = Hkv * kv_lens
    b_of = torch.repeat_interleave(torch.arange(len(kv_lens)), rows_b).to(dev)
    start = (torch.cumsum(rows_b, 0) - rows_b).to(dev)
    o = torch.arange(int(rows_b.sum()), device=dev) - start[b_of]
    L = kv_lens.to(dev)[b_of]
    h, t = o // L, o % L
    page = perm.to(dev)[indptr.to(dev)[b_of] + t // page_size]
    dest = (page * Hkv + h) * page_size + t % page_size
    kp.view(-1, d)[dest] = k
    vp.view(-1, d)[dest] = v
    return dict(k_pages=kp, v_pages=vp, page_indptr=indptr.to(torch.int32).to(dev),
                page_indices=perm[:used].to(torch.int32).to(dev))


def to_fp8(inp: dict, Hkv: int) -> dict:
    """An FP8 (e4m3) copy of the ragged HND ``k``/``v`` of ``inp``: per KV head
    g, scale[g] = max |x| over that head's keys (or values) / 448 (the largest
    e4m3 magnitude), codes = x / scale[g] rounded to nearest even e4m3 (torch's
    float8_e4m3fn conversion), stored as uint8. Returns k_fp8, v_fp8 (uint8,
    same layout) and k_scale, v_scale (fp32 [Hkv]) on the device of
    ``inp["k"]``. Pure data preparation."""
    out = {}
    cu = inp["cu_k"].cpu().tolist()
    for name in ("k", "v"):
        x = inp[name].float()
        heads = torch.zeros_like(x[:, 0], dtype=torch.int64)
        for b in range(len(cu) - 1):
            L = cu[b + 1] - cu[b]
            r0 = Hkv * cu[b]
            heads[r0:r0 + Hkv * L] = torch.arange(Hkv, device=x.device).repeat_interleave(L)
        amax = torch.zeros(Hkv, dtype=torch.float32, device=x.device)
        amax = amax.scatter_reduce(0, heads, x.abs().amax(dim=1), reduce="amax")
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        codes = (x / scale[heads][:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        out[name + "_fp8"] = codes
        out[name + "_scale"] = scale
    return out

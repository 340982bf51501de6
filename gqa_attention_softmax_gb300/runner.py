"""One pass of the hot path for a named workload, through the C ABI.

The benchmark and the full-size parity tests both call ``run`` so they time
and check the same launch configuration. Argument marshalling only.
"""
from __future__ import annotations

import torch

from . import _binding as B
from .workloads import Workload


def splits_for(w: Workload, inp: dict) -> int:
    """Split count of a decode workload: the one it states, else the library's default."""
    if w.kind != "decode":
        return 1
    if w.num_splits > 0:
        return w.num_splits
    return B.sinkattn_decode_default_splits(inp["batch"], w.q_len, w.num_qo_heads, w.num_kv_heads,
                                            w.head_dim, inp["max_k"])


class Runner:
    """Holds the output / workspace buffers of one workload so repeated calls
    allocate nothing."""

    def __init__(self, w: Workload, inp: dict, fused: bool = False):
        self.w, self.inp = w, inp
        dev = inp["q"].device
        self.out = torch.empty_like(inp["q"])
        self.lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=dev)
        self.num_splits = splits_for(w, inp)
        # decode: split + merge through a workspace. The cluster-fused form
        # (sinkattn_decode_fused) is available but measured slower on the
        # gpt-oss- and Qwen-shaped decodes, so it is opt-in.
        self.fused = (w.kind == "decode" and fused and self.num_splits <= 16
                      and w.page_size == 0 and not w.kv_fp8)
        self.workspace = None
        if w.kind == "decode" and not self.fused:
            n = B.sinkattn_decode_workspace_bytes(inp["batch"], w.q_len, w.num_qo_heads, w.head_dim,
                                                  self.num_splits)
            self.workspace = torch.empty((max(n, 256),), dtype=torch.uint8, device=dev)

    @property
    def launches_per_call(self) -> int:
        return 2 if (self.w.kind == "decode" and not self.fused) else 1

    def __call__(self, stream=None):
        w, i = self.w, self.inp
        if w.kind == "decode" and self.fused:
            return B.sinkattn_decode_fused(i["q"], i["k"], i["v"], i["cu_k"], i["sinks"], w.q_len,
                                           i["max_k"], w.num_kv_heads, num_splits=self.num_splits,
                                           sm_scale=w.scale, causal=w.causal, window=w.window,
                                           out=self.out, lse=self.lse, stream=stream)
        if w.kind == "decode" and w.kv_fp8:
            return B.sinkattn_decode_fp8(i["q"], i["k_fp8"], i["v_fp8"], i["k_scale"],
                                         i["v_scale"], i["cu_k"], i["sinks"], w.q_len, i["max_k"],
                                         num_splits=self.num_splits, sm_scale=w.scale,
                                         causal=w.causal, window=w.window,
                                         workspace=self.workspace, out=self.out, lse=self.lse,
                                         stream=stream)
        if w.kind == "decode" and w.page_size > 0:
            return B.sinkattn_decode_paged(i["q"], i["k_pages"], i["v_pages"], i["cu_k"],
                                           i["page_indptr"], i["page_indices"], i["sinks"],
                                           w.q_len, i["max_k"], num_splits=self.num_splits,
                                           sm_scale=w.scale, causal=w.causal, window=w.window,
                                           workspace=self.workspace, out=self.out, lse=self.lse,
                                           stream=stream)
        if w.kind == "decode":
            return B.sinkattn_decode(i["q"], i["k"], i["v"], i["cu_k"], i["sinks"], w.q_len,
                                     i["max_k"], w.num_kv_heads, num_splits=self.num_splits,
                                     sm_scale=w.scale, causal=w.causal, window=w.window,
                                     workspace=self.workspace, out=self.out, lse=self.lse,
                                     stream=stream)
        return B.sinkattn_prefill(i["q"], i["k"], i["v"], i["sinks"], i["cu_q"], i["cu_k"],
                                  i["max_q"], i["max_k"], w.num_kv_heads, w.scale, w.causal,
                                  w.window, out=self.out, lse=self.lse, stream=stream)


# ----------------------------------------------------------------------------
# multi-rank host logic (one process per GPU; the path needs no exchange)
# ----------------------------------------------------------------------------
def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank serves its own independent requests: rank r draws its batch
    with seed base + r (weak scaling, no data-path collective)."""
    return int(base_seed) + int(rank)


def max_over_ranks(x: float) -> float:
    """Largest value of `x` over all ranks (identity without a process group).
    Uses a CUDA tensor under NCCL and a CPU tensor under gloo."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_sequences(batch: int, rank: int, world: int) -> range:
    """Contiguous block of sequence indices owned by `rank` when one batch is
    split over `world` ranks (sizes differ by at most one)."""
    base, extra = divmod(batch, world)
    lo = rank * base + min(rank, extra)
    return range(lo, lo + base + (1 if rank < extra else 0))


def slice_sequences(inp: dict, num_kv_heads: int, seqs) -> dict:
    """Input set restricted to the sequences `seqs` (contiguous), re-based
    cu_seqlens; tensors stay on their device."""
    seqs = list(seqs)
    cu_q = inp["cu_q"].cpu().tolist()
    cu_k = inp["cu_k"].cpu().tolist()
    if not seqs:
        raise ValueError("empty shard")
    b0, b1 = seqs[0], seqs[-1] + 1
    q = inp["q"][cu_q[b0]:cu_q[b1]]
    k = inp["k"][num_kv_heads * cu_k[b0]:num_kv_heads * cu_k[b1]]
    v = inp["v"][num_kv_heads * cu_k[b0]:num_kv_heads * cu_k[b1]]
    dev = inp["q"].device
    ncq = torch.tensor([c - cu_q[b0] for c in cu_q[b0:b1 + 1]], dtype=torch.int32, device=dev)
    nck = torch.tensor([c - cu_k[b0] for c in cu_k[b0:b1 + 1]], dtype=torch.int32, device=dev)
    q_lens = inp["q_lens"][b0:b1]
    kv_lens = inp["kv_lens"][b0:b1]
    return dict(q=q, k=k, v=v, sinks=inp["sinks"], cu_q=ncq, cu_k=nck, q_lens=q_lens,
                kv_lens=kv_lens, batch=b1 - b0, total_q=sum(q_lens), total_k=sum(kv_lens),
                max_q=max(q_lens), max_k=max(kv_lens))

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

    def __init__(self, w: Workload, inp: dict):
        self.w, self.inp = w, inp
        dev = inp["q"].device
        self.out = torch.empty_like(inp["q"])
        self.lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=dev)
        self.num_splits = splits_for(w, inp)
        self.workspace = None
        if w.kind == "decode":
            n = B.sinkattn_decode_workspace_bytes(inp["batch"], w.q_len, w.num_qo_heads, w.head_dim,
                                                  self.num_splits)
            self.workspace = torch.empty((max(n, 256),), dtype=torch.uint8, device=dev)

    def __call__(self, stream=None):
        w, i = self.w, self.inp
        if w.kind == "decode":
            return B.sinkattn_decode(i["q"], i["k"], i["v"], i["cu_k"], i["sinks"], w.q_len,
                                     i["max_k"], w.num_kv_heads, num_splits=self.num_splits,
                                     sm_scale=w.scale, causal=w.causal, window=w.window,
                                     workspace=self.workspace, out=self.out, lse=self.lse,
                                     stream=stream)
        return B.sinkattn_prefill(i["q"], i["k"], i["v"], i["sinks"], i["cu_q"], i["cu_k"],
                                  i["max_q"], i["max_k"], w.num_kv_heads, w.scale, w.causal,
                                  w.window, out=self.out, lse=self.lse, stream=stream)

"""Second, independent oracle: pure-Python loops with exactly rounded sums.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``). For tiny shapes.

It states the definition from "GPT-OSS on Day 0" (Perplexity), section
"Kernels for GPT-OSS / Sink attention" -- softmax over the scaled logits plus
one sink logit per query head, whose value row is zero -- with every sum taken
by ``math.fsum`` (exactly rounded), so it shares neither code nor summation
order with the C++ oracle.
"""
from __future__ import annotations

import math


def attend_fsum(q, k, v, sinks, cu_q, cu_k, Hq, Hkv, d, sm_scale, causal, window=0):
    """q: nested lists/array [total_q][Hq][d] of floats; k, v: flat sequences in
    ragged HND order; sinks: list of Hq floats or None.

    Returns (out [total_q][Hq][d], lse [total_q][Hq]) as Python floats.
    """
    G = Hq // Hkv
    B = len(cu_q) - 1
    T = cu_q[-1]
    out = [[[0.0] * d for _ in range(Hq)] for _ in range(T)]
    lse = [[0.0] * Hq for _ in range(T)]
    for b in range(B):
        Lq = cu_q[b + 1] - cu_q[b]
        Lk = cu_k[b + 1] - cu_k[b]
        base = Hkv * cu_k[b] * d
        for i in range(Lq):
            tok = cu_q[b] + i
            pos = Lk - Lq + i
            for h in range(Hq):
                kvh = h // G
                # the whole row: visible keys, then the sink column
                logits, vrows = [], []
                for j in range(Lk):
                    if causal and j > pos:
                        continue
                    if window > 0 and pos - j >= window:
                        continue
                    off = base + (kvh * Lk + j) * d
                    dot = math.fsum(float(q[tok][h][c]) * float(k[off + c]) for c in range(d))
                    logits.append(sm_scale * dot)
                    vrows.append([float(v[off + c]) for c in range(d)])
                s = -math.inf if sinks is None else float(sinks[h])
                row = logits + [s]
                M = max(row)
                if M == -math.inf:
                    lse[tok][h] = -math.inf
                    continue
                w = [math.exp(x - M) for x in logits]
                Z = math.fsum(w + [math.exp(s - M)])
                for c in range(d):
                    out[tok][h][c] = math.fsum(wj * vr[c] for wj, vr in zip(w, vrows)) / Z
                lse[tok][h] = M + math.log(Z)
    return out, lse

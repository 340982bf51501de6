"""Shared test helpers: tolerances, comparison, sub-problem slicing for
sampled-row oracle checks. Holds no attention arithmetic."""
import numpy as np
import torch

# Tolerances on unit-scale outputs: max-abs 1e-2 and mean-abs 1e-3 on out,
# 1e-3 on the per-row log-sum-exp.
TOL_MAX = 1e-2
TOL_MEAN = 1e-3
TOL_LSE = 1e-3


# Every comparison's errors, also relative to the RMS of the expected output
# (informational: at thousands of keys with N(0,1) values |out| is ~1e-2, the
# size of the absolute bound, so the relative figure is the one that shows a
# scale regression). Printed at the end of the session by conftest.py.
REPORT = []


def compare(out_gpu, lse_gpu, want_out, want_lse, what=""):
    o = out_gpu.detach().float().cpu().numpy().reshape(want_out.shape)
    err = np.abs(o - want_out)
    assert np.isfinite(o).all(), "%s: non-finite output" % what
    rms = float(np.sqrt(np.mean(np.square(want_out)))) if want_out.size else 0.0
    rel = float(err.max() / rms) if rms > 0 else 0.0
    rel_mean = float(err.mean() / rms) if rms > 0 else 0.0
    REPORT.append((what, float(err.max()) if err.size else 0.0,
                   float(err.mean()) if err.size else 0.0, rms, rel, rel_mean))
    assert err.max() <= TOL_MAX, "%s: max-abs %.3g (%.3g of the output RMS)" % (what, err.max(), rel)
    assert err.mean() <= TOL_MEAN, "%s: mean-abs %.3g (%.3g of the output RMS)" % (
        what, err.mean(), rel_mean)
    if lse_gpu is not None and want_lse is not None:
        l = lse_gpu.detach().cpu().numpy().reshape(want_lse.shape)
        both_inf = np.isneginf(l) & np.isneginf(want_lse)
        lerr = np.where(both_inf, 0.0, np.abs(l - want_lse))
        assert lerr.max() <= TOL_LSE, "%s: lse max-abs %.3g" % (what, lerr.max())
    return float(err.max()), float(err.mean())


def to_dev(inp, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}


def sub_problem(inp, Hkv, d, seqs):
    """Slice sequences `seqs` out of an input set (any device) into a CPU
    input set with its own cu_q/cu_k, plus the map from the sub-problem's
    token index to the original one."""
    cu_q = inp["cu_q"].cpu().tolist()
    cu_k = inp["cu_k"].cpu().tolist()
    qs, ks, vs, tok_map = [], [], [], []
    ncq, nck = [0], [0]
    for b in seqs:
        qs.append(inp["q"][cu_q[b]:cu_q[b + 1]].cpu())
        ks.append(inp["k"][Hkv * cu_k[b]:Hkv * cu_k[b + 1]].cpu())
        vs.append(inp["v"][Hkv * cu_k[b]:Hkv * cu_k[b + 1]].cpu())
        tok_map.extend(range(cu_q[b], cu_q[b + 1]))
        ncq.append(ncq[-1] + cu_q[b + 1] - cu_q[b])
        nck.append(nck[-1] + cu_k[b + 1] - cu_k[b])
    return dict(q=torch.cat(qs), k=torch.cat(ks), v=torch.cat(vs), sinks=inp["sinks"].cpu(),
                cu_q=torch.tensor(ncq, dtype=torch.int32), cu_k=torch.tensor(nck, dtype=torch.int32),
                tok_map=np.array(tok_map, dtype=np.int64))


def sampled_rows(inp, Hq, n_random, seed=0, seqs=None):
    """(sequence list, flat row ids) covering the first and last token of each
    chosen sequence for every head, plus random rows."""
    rng = np.random.default_rng(seed)
    cu_q = inp["cu_q"].cpu().tolist()
    B = len(cu_q) - 1
    if seqs is None:
        seqs = list(range(B))
    rows = []
    for b in seqs:
        if cu_q[b + 1] == cu_q[b]:
            continue
        for t in {cu_q[b], cu_q[b + 1] - 1}:
            rows.extend(t * Hq + h for h in range(Hq))
        toks = rng.integers(cu_q[b], cu_q[b + 1], size=max(1, n_random // len(seqs)))
        heads = rng.integers(0, Hq, size=len(toks))
        rows.extend((toks * Hq + heads).tolist())
    return seqs, np.unique(np.array(rows, dtype=np.int64))

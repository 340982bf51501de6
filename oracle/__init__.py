"""Float64 CPU oracle for GQA attention with a per-head softmax sink.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The CUDA
path never imports it, and it imports nothing from the CUDA path; the two
share only the seeded input generator, which holds none of the method's
arithmetic.

Two independent implementations live here:

* ``attend`` / ``split_partials`` also take K/V as e4m3 codes (uint8) with
  per-KV-head scales (the FP8 KV cache), decoded from the E4M3 format's
  definition (``e4m3_table`` exposes the decode);
* ``attend`` / ``split_partials`` / ``chunk_partial`` / ``merge``: a C++
  float64 library (``sinkattn_oracle.cpp``, OpenMP over rows) that
  materialises every visible logit row plus the sink column, following
  "GPT-OSS on Day 0" (Perplexity), section "Kernels for GPT-OSS / Sink
  attention": attn = softmax(q @ k^T * sm_scale + sink) * V, with the sink
  read as one extra logit column whose value row is zero;
* ``brute.attend_fsum``: pure-Python loops with ``math.fsum``, for tiny shapes.

Inputs are the exact bf16 values the GPU sees (passed as raw bf16 bits);
widening bf16 to float64 is exact. Sinks and sm_scale are passed as float64
(widened from the float32 values the GPU receives).

Parity status: every function here is pinned by ``tests/test_oracle.py``
against results that do not come from this code (library SDPA, closed forms,
a hand-derived golden fixture, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sinkattn_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library in place with g++ (-O2, OpenMP, strict IEEE)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB_OVERRIDE: a library built with a planted mistake, used
            # only by the test that checks the pins catch such mistakes.
            path = os.environ.get("ORACLE_LIB_OVERRIDE")
            if not path:
                build()
                path = _LIB
            lib = ctypes.CDLL(path)
            P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_attend_rows.argtypes = [P, P, P, P, P, P, I, I, I, I, D, I, I, I64, P, P, P]
            lib.oracle_split_partials.argtypes = [P, P, P, P, P, I, I, I, I, D, I, I, I, P, P, P]
            lib.oracle_chunk_partial.argtypes = [P, P, P, P, P, I, I, I, I, D, I, I, I64, I64, I64, P, P, P]
            lib.oracle_merge.argtypes = [P, P, P, P, I64, I, I, I, P, P]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_attend_rows_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, D, I, I, I64,
                                                   P, P, P]
            lib.oracle_split_partials_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, D, I, I, I,
                                                      P, P, P]
            lib.oracle_e4m3_table.argtypes = [P]
            for f in (lib.oracle_attend_rows, lib.oracle_split_partials,
                      lib.oracle_chunk_partial, lib.oracle_merge, lib.oracle_num_threads,
                      lib.oracle_attend_rows_fp8, lib.oracle_split_partials_fp8,
                      lib.oracle_e4m3_table):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array of raw bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _codes(x) -> np.ndarray:
    """uint8 tensor / array of e4m3 codes -> contiguous uint8 numpy array."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint8
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.uint8, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().numpy())


def _is_codes(x) -> bool:
    if isinstance(x, np.ndarray):
        return x.dtype == np.uint8
    import torch
    return x.dtype == torch.uint8


def _f64(x) -> np.ndarray | None:
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 e4m3 codes (NaN codes: NaN), float64."""
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def attend(q, k, v, sinks, cu_q, cu_k, num_qo_heads, num_kv_heads, head_dim,
           sm_scale, causal, window=0, rows=None, k_scale=None, v_scale=None):
    """Full-row float64 attention with sink.

    q: bf16 [total_q, Hq, d]; k, v: bf16 ragged HND (sequence b is a contiguous
    [Hkv, Lk_b, d] block starting at element Hkv*cu_k[b]*d), or uint8 e4m3
    codes in that layout with per-KV-head scales k_scale, v_scale [Hkv];
    sinks: [Hq] or None; cu_q, cu_k: int [B+1]. rows: optional array of flat
    row ids (token * Hq + head). Returns (out [n, d] float64, lse [n]
    float64), with n = len(rows) or total_q * Hq.
    """
    lib = _load()
    fp8 = _is_codes(k)
    qb = _bits(q)
    kb, vb = (_codes(k), _codes(v)) if fp8 else (_bits(k), _bits(v))
    s = _f64(sinks)
    cq, ck = _i32(cu_q), _i32(cu_k)
    B = len(cq) - 1
    if rows is None:
        n = int(cq[-1]) * num_qo_heads
        r = None
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(r)
    out = np.zeros((n, head_dim), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    if fp8:
        ks, vs = _f64(k_scale), _f64(v_scale)
        rc = lib.oracle_attend_rows_fp8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(ks), _ptr(vs), _ptr(s),
                                        _ptr(cq), _ptr(ck), B, num_qo_heads, num_kv_heads,
                                        head_dim, float(sm_scale), int(bool(causal)),
                                        int(window), n, _ptr(r), _ptr(out), _ptr(lse))
    else:
        rc = lib.oracle_attend_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(s), _ptr(cq), _ptr(ck),
                                    B, num_qo_heads, num_kv_heads, head_dim, float(sm_scale),
                                    int(bool(causal)), int(window), n, _ptr(r), _ptr(out),
                                    _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attend_rows rejected the problem")
    return out, lse


def split_partials(q, k, v, cu_q, cu_k, num_qo_heads, num_kv_heads, head_dim,
                   sm_scale, causal, window, num_splits, k_scale=None, v_scale=None):
    """Per-chunk (acc, m, d) of the split-KV method, no sink.

    Returns acc [total_q, Hq, S, d], m [total_q, Hq, S], d [total_q, Hq, S],
    all float64, chunks of 64 * ceil(Lk_b / (64 S)) keys (the last may be
    shorter, later ones empty).
    """
    lib = _load()
    fp8 = _is_codes(k)
    qb = _bits(q)
    kb, vb = (_codes(k), _codes(v)) if fp8 else (_bits(k), _bits(v))
    cq, ck = _i32(cu_q), _i32(cu_k)
    B = len(cq) - 1
    T = int(cq[-1])
    S = int(num_splits)
    acc = np.zeros((T, num_qo_heads, S, head_dim), dtype=np.float64)
    m = np.zeros((T, num_qo_heads, S), dtype=np.float64)
    dd = np.zeros((T, num_qo_heads, S), dtype=np.float64)
    if fp8:
        ks, vs = _f64(k_scale), _f64(v_scale)
        rc = lib.oracle_split_partials_fp8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(ks), _ptr(vs),
                                           _ptr(cq), _ptr(ck), B, num_qo_heads, num_kv_heads,
                                           head_dim, float(sm_scale), int(bool(causal)),
                                           int(window), S, _ptr(acc), _ptr(m), _ptr(dd))
    else:
        rc = lib.oracle_split_partials(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cq), _ptr(ck), B,
                                       num_qo_heads, num_kv_heads, head_dim, float(sm_scale),
                                       int(bool(causal)), int(window), S, _ptr(acc), _ptr(m),
                                       _ptr(dd))
    if rc != 0:
        raise ValueError("oracle_split_partials rejected the problem")
    return acc, m, dd


def chunk_partial(q, k, v, cu_q, cu_k, num_qo_heads, num_kv_heads, head_dim,
                  sm_scale, causal, window, row, lo, hi):
    """(acc [d], m, d) of keys [lo, hi) for one flat row id, no sink."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cq, ck = _i32(cu_q), _i32(cu_k)
    acc = np.zeros((head_dim,), dtype=np.float64)
    m = np.zeros((1,), dtype=np.float64)
    dd = np.zeros((1,), dtype=np.float64)
    rc = lib.oracle_chunk_partial(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cq), _ptr(ck), len(cq) - 1,
                                  num_qo_heads, num_kv_heads, head_dim, float(sm_scale),
                                  int(bool(causal)), int(window), int(row), int(lo), int(hi),
                                  _ptr(acc), _ptr(m), _ptr(dd))
    if rc != 0:
        raise ValueError("oracle_chunk_partial rejected the problem")
    return acc, float(m[0]), float(dd[0])


def merge(part_acc, part_m, part_d, sinks, num_qo_heads, head_dim):
    """Fold partials [rows, Hq, S, ...] with the sink counted once.

    Returns out [rows, Hq, d], lse [rows, Hq] (float64).
    """
    lib = _load()
    a, m, dd = _f64(part_acc), _f64(part_m), _f64(part_d)
    s = _f64(sinks)
    rows, Hq, S = m.shape
    assert Hq == num_qo_heads and a.shape == (rows, Hq, S, head_dim) and dd.shape == m.shape
    out = np.zeros((rows, Hq, head_dim), dtype=np.float64)
    lse = np.zeros((rows, Hq), dtype=np.float64)
    rc = lib.oracle_merge(_ptr(a), _ptr(m), _ptr(dd), _ptr(s), rows, Hq, head_dim, S,
                          _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_merge rejected the input")
    return out, lse

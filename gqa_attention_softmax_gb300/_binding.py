"""Thin ctypes binding of libsinkattn (argument marshalling only).

Every function here has the name of the C entry point it calls and does
nothing but turn torch tensors into pointers and sizes, allocate outputs the
caller did not pass (torch device memory), and raise on a non-zero status.
All arithmetic runs in the CUDA kernels behind the C ABI; there is no
fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsinkattn.so")
_lock = threading.Lock()
_lib = None

OK, INVALID_ARG, UNSUPPORTED, CUDA_ERROR, TIMEOUT, BAD_LENGTHS = range(6)


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (status_name(status), message))
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libsinkattn.so (built in-tree by ``_build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libsinkattn.so is not built (%s); build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            P, I32, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            L.sinkattn_prefill.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, I32, F,
                                           I32, I32, P, P, P]
            L.sinkattn_decode_split.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, I32, F, I32, I32,
                                                I32, P, P, P]
            L.sinkattn_merge.argtypes = [P, P, P, I32, I32, I32, I32, P, P, P]
            L.sinkattn_decode.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, I32, F, I32, I32, I32,
                                          P, P, SZ, P, P, P]
            L.sinkattn_decode_fused.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, I32, F, I32,
                                                I32, I32, P, P, P, P]
            L.sinkattn_decode_noalloc.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, I32, F, I32,
                                                  I32, I32, P, P, P, P]
            L.sinkattn_decode_workspace_bytes.argtypes = [I32, I32, I32, I32, I32,
                                                          ctypes.POINTER(SZ)]
            L.sinkattn_decode_default_splits.argtypes = [I32, I32, I32, I32, I32, I32,
                                                         ctypes.POINTER(I32)]
            L.sinkattn_prefill_paged.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I32, I32, I32,
                                                 I32, I32, I32, I32, F, I32, I32, P, P, P]
            L.sinkattn_decode_split_paged.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32,
                                                      I32, I32, I32, F, I32, I32, I32, P, P, P]
            L.sinkattn_decode_paged.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32,
                                                I32, I32, F, I32, I32, I32, P, P, SZ, P, P, P]
            L.sinkattn_status_string.argtypes = [ctypes.c_int]
            L.sinkattn_status_string.restype = ctypes.c_char_p
            L.sinkattn_last_error.argtypes = []
            L.sinkattn_last_error.restype = ctypes.c_char_p
            L.sinkattn_debug_status.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
            L.sinkattn_debug_set_hooks.argtypes = [ctypes.c_longlong, ctypes.c_int]
            L.sinkattn_set_decode_kernel.argtypes = [ctypes.c_int]
            L.sinkattn_set_prefill_kernel.argtypes = [ctypes.c_int]
            L.sinkattn_decode_split_fp8.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32,
                                                    F, I32, I32, I32, P, P, P]
            L.sinkattn_decode_fp8.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, F,
                                              I32, I32, I32, P, P, SZ, P, P, P]
            for name in ("sinkattn_prefill", "sinkattn_decode_split", "sinkattn_merge",
                         "sinkattn_decode", "sinkattn_decode_fused", "sinkattn_decode_noalloc",
                         "sinkattn_decode_workspace_bytes", "sinkattn_decode_default_splits",
                         "sinkattn_debug_status", "sinkattn_debug_set_hooks",
                         "sinkattn_set_decode_kernel",
                         "sinkattn_set_prefill_kernel", "sinkattn_decode_split_fp8",
                         "sinkattn_decode_fp8",
                         "sinkattn_prefill_paged", "sinkattn_decode_split_paged",
                         "sinkattn_decode_paged"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def status_name(status: int) -> str:
    return lib().sinkattn_status_string(int(status)).decode()


def _check(rc: int):
    if rc != OK:
        raise SinkAttnError(rc, lib().sinkattn_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t, stream):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _scale(sm_scale, d):
    return float(1.0 / math.sqrt(d) if sm_scale is None else sm_scale)


def sinkattn_prefill(q, k, v, sinks, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                     num_kv_heads, sm_scale=None, causal=True, window=0, out=None, lse=None,
                     return_lse=True, stream=None):
    """Varlen prefill with sink. q [total_q, Hq, d] bf16; k, v ragged HND
    [Hkv * total_k, d] bf16; sinks [Hq] fp32 or None; cu_seqlens int32 [B+1]
    on the device. Returns (out, lse) with lse None unless requested."""
    total_q, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens_q),
                                _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, total_q,
                                int(max_seqlen_q), int(max_seqlen_k), Hq, int(num_kv_heads), d,
                                _scale(sm_scale, d), int(bool(causal)), int(window), _ptr(out),
                                _ptr(lse), _stream(q, stream))
    _check(rc)
    return out, lse


def sinkattn_decode_split(q, k, v, kv_indptr, q_len, max_kv_len, num_kv_heads, num_splits,
                          sm_scale=None, causal=True, window=0, part_acc=None, part_md=None,
                          stream=None):
    """Split-KV step 1. q [B*q_len, Hq, d]. Returns (part_acc [B*q_len, Hq, S, d],
    part_md [B*q_len, Hq, S, 2]) fp32, without the sink."""
    rows, Hq, d = q.shape
    batch = kv_indptr.numel() - 1
    if part_acc is None:
        part_acc = torch.empty((rows, Hq, num_splits, d), dtype=torch.float32, device=q.device)
    if part_md is None:
        part_md = torch.empty((rows, Hq, num_splits, 2), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode_split(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), batch, int(q_len),
                                     int(max_kv_len), Hq, int(num_kv_heads), d,
                                     _scale(sm_scale, d), int(bool(causal)), int(window),
                                     int(num_splits), _ptr(part_acc), _ptr(part_md),
                                     _stream(q, stream))
    _check(rc)
    return part_acc, part_md


def sinkattn_merge(part_acc, part_md, sinks, out=None, lse=None, return_lse=True, stream=None):
    """Split-KV step 2: fold partials with the sink counted once. Returns (out, lse)."""
    rows, Hq, S, d = part_acc.shape
    if out is None:
        out = torch.empty((rows, Hq, d), dtype=torch.bfloat16, device=part_acc.device)
    if lse is None and return_lse:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=part_acc.device)
    rc = lib().sinkattn_merge(_ptr(part_acc), _ptr(part_md), _ptr(sinks), rows, Hq, d, S,
                              _ptr(out), _ptr(lse), _stream(part_acc, stream))
    _check(rc)
    return out, lse


def sinkattn_decode_workspace_bytes(batch, q_len, num_qo_heads, head_dim, num_splits) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().sinkattn_decode_workspace_bytes(int(batch), int(q_len), int(num_qo_heads),
                                                 int(head_dim), int(num_splits), ctypes.byref(n)))
    return int(n.value)


def sinkattn_decode_default_splits(batch, q_len, num_qo_heads, num_kv_heads, head_dim,
                                   max_kv_len) -> int:
    s = ctypes.c_int32(0)
    _check(lib().sinkattn_decode_default_splits(int(batch), int(q_len), int(num_qo_heads),
                                                int(num_kv_heads), int(head_dim), int(max_kv_len),
                                                ctypes.byref(s)))
    return int(s.value)


def sinkattn_decode(q, k, v, kv_indptr, sinks, q_len, max_kv_len, num_kv_heads, num_splits=0,
                    sm_scale=None, causal=True, window=0, workspace=None, out=None, lse=None,
                    return_lse=True, stream=None):
    """Split-KV decode / MTP in one call (split then merge on one stream).
    ``workspace``: a uint8 device tensor of at least
    sinkattn_decode_workspace_bytes() bytes (allocated here if None)."""
    rows, Hq, d = q.shape
    batch = kv_indptr.numel() - 1
    if num_splits <= 0:
        num_splits = sinkattn_decode_default_splits(batch, q_len, Hq, num_kv_heads, d, max_kv_len)
    need = sinkattn_decode_workspace_bytes(batch, q_len, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), batch, int(q_len),
                               int(max_kv_len), Hq, int(num_kv_heads), d, _scale(sm_scale, d),
                               int(bool(causal)), int(window), int(num_splits), _ptr(sinks),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(out), _ptr(lse), _stream(q, stream))
    _check(rc)
    return out, lse


def sinkattn_decode_fused(q, k, v, kv_indptr, sinks, q_len, max_kv_len, num_kv_heads,
                          num_splits=0, sm_scale=None, causal=True, window=0, out=None, lse=None,
                          return_lse=True, stream=None):
    """Split-KV decode / MTP with the merge done on chip by a thread-block
    cluster (num_splits <= 16; no workspace). Returns (out, lse)."""
    rows, Hq, d = q.shape
    batch = kv_indptr.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), batch,
                                     int(q_len), int(max_kv_len), Hq, int(num_kv_heads), d,
                                     _scale(sm_scale, d), int(bool(causal)), int(window),
                                     int(num_splits), _ptr(sinks), _ptr(out), _ptr(lse),
                                     _stream(q, stream))
    _check(rc)
    return out, lse


def sinkattn_decode_noalloc(q, k, v, kv_indptr, sinks, q_len, max_kv_len, num_kv_heads,
                            num_splits=0, sm_scale=None, causal=True, window=0, out=None, lse=None,
                            return_lse=True, stream=None):
    """sinkattn_decode without a workspace, for callers that cannot allocate
    device memory: the partials go to the library's fixed 32 MiB scratch
    array. Pass ``out`` (and ``lse``) to allocate nothing here either."""
    rows, Hq, d = q.shape
    batch = kv_indptr.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    # the library looks the scratch address up in the current device's
    # context and rejects a stream of another device: make q's device current
    with torch.cuda.device(q.device):
        rc = lib().sinkattn_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), batch,
                                           int(q_len), int(max_kv_len), Hq, int(num_kv_heads), d,
                                           _scale(sm_scale, d), int(bool(causal)), int(window),
                                           int(num_splits), _ptr(sinks), _ptr(out), _ptr(lse),
                                           _stream(q, stream))
    _check(rc)
    return out, lse


DECODE_KERNELS = {"auto": 0, "warp": 1, "tcgen05": 2}


def _pages(k_pages):
    """(num_pages, Hkv, page_size, d) of a page pool."""
    num_pages, Hkv, page_size, d = k_pages.shape
    return num_pages, Hkv, page_size, d


def sinkattn_prefill_paged(q, k_pages, v_pages, sinks, cu_seqlens_q, cu_seqlens_k, page_indptr,
                           page_indices, max_seqlen_q, max_seqlen_k, sm_scale=None, causal=True,
                           window=0, out=None, lse=None, return_lse=True, stream=None):
    """sinkattn_prefill over a paged KV cache: k_pages, v_pages bf16
    [num_pages, Hkv, page_size, d]; sequence b's pages are
    page_indices[page_indptr[b]:page_indptr[b+1]] (int32, device); key
    counts come from cu_seqlens_k. Returns (out, lse)."""
    total_q, Hq, d = q.shape
    num_pages, Hkv, page_size, _ = _pages(k_pages)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_prefill_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(sinks), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        _ptr(page_indptr), _ptr(page_indices), num_pages, page_size, cu_seqlens_q.numel() - 1,
        total_q, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, d, _scale(sm_scale, d),
        int(bool(causal)), int(window), _ptr(out), _ptr(lse), _stream(q, stream))
    _check(rc)
    return out, lse


def sinkattn_decode_split_paged(q, k_pages, v_pages, kv_indptr, page_indptr, page_indices, q_len,
                                max_kv_len, num_splits, sm_scale=None, causal=True, window=0,
                                part_acc=None, part_md=None, stream=None):
    """sinkattn_decode_split over a paged KV cache (layout as in
    sinkattn_prefill_paged). Returns (part_acc, part_md) without the sink."""
    rows, Hq, d = q.shape
    num_pages, Hkv, page_size, _ = _pages(k_pages)
    batch = kv_indptr.numel() - 1
    if part_acc is None:
        part_acc = torch.empty((rows, Hq, num_splits, d), dtype=torch.float32, device=q.device)
    if part_md is None:
        part_md = torch.empty((rows, Hq, num_splits, 2), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode_split_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indptr), _ptr(page_indptr),
        _ptr(page_indices), num_pages, page_size, batch, int(q_len), int(max_kv_len), Hq, Hkv, d,
        _scale(sm_scale, d), int(bool(causal)), int(window), int(num_splits), _ptr(part_acc),
        _ptr(part_md), _stream(q, stream))
    _check(rc)
    return part_acc, part_md


def sinkattn_decode_paged(q, k_pages, v_pages, kv_indptr, page_indptr, page_indices, sinks, q_len,
                          max_kv_len, num_splits=0, sm_scale=None, causal=True, window=0,
                          workspace=None, out=None, lse=None, return_lse=True, stream=None):
    """sinkattn_decode over a paged KV cache (layout as in
    sinkattn_prefill_paged). Returns (out, lse)."""
    rows, Hq, d = q.shape
    num_pages, Hkv, page_size, _ = _pages(k_pages)
    batch = kv_indptr.numel() - 1
    if num_splits <= 0:
        num_splits = sinkattn_decode_default_splits(batch, q_len, Hq, Hkv, d, max_kv_len)
    need = sinkattn_decode_workspace_bytes(batch, q_len, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indptr), _ptr(page_indptr),
        _ptr(page_indices), num_pages, page_size, batch, int(q_len), int(max_kv_len), Hq, Hkv, d,
        _scale(sm_scale, d), int(bool(causal)), int(window), int(num_splits), _ptr(sinks),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        _stream(q, stream))
    _check(rc)
    return out, lse


def sinkattn_set_decode_kernel(kind) -> None:
    """Selects the split-KV partial kernel process-wide: "auto", "warp" or
    "tcgen05" (or the integer codes of include/sinkattn.h)."""
    code = DECODE_KERNELS[kind] if isinstance(kind, str) else int(kind)
    _check(lib().sinkattn_set_decode_kernel(code))


def sinkattn_decode_split_fp8(q, k, v, k_scale, v_scale, kv_indptr, q_len, max_kv_len,
                              num_splits, sm_scale=None, causal=True, window=0, part_acc=None,
                              part_md=None, stream=None):
    """sinkattn_decode_split over an FP8 KV cache: k, v uint8 e4m3 codes in
    the ragged HND layout [Hkv * total_k, d]; k_scale, v_scale fp32 [Hkv]
    per-KV-head scales (device). Returns (part_acc, part_md) without the sink."""
    rows, Hq, d = q.shape
    Hkv = k_scale.numel()
    batch = kv_indptr.numel() - 1
    if part_acc is None:
        part_acc = torch.empty((rows, Hq, num_splits, d), dtype=torch.float32, device=q.device)
    if part_md is None:
        part_md = torch.empty((rows, Hq, num_splits, 2), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode_split_fp8(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_scale), _ptr(v_scale), _ptr(kv_indptr), batch,
        int(q_len), int(max_kv_len), Hq, Hkv, d, _scale(sm_scale, d), int(bool(causal)),
        int(window), int(num_splits), _ptr(part_acc), _ptr(part_md), _stream(q, stream))
    _check(rc)
    return part_acc, part_md


def sinkattn_decode_fp8(q, k, v, k_scale, v_scale, kv_indptr, sinks, q_len, max_kv_len,
                        num_splits=0, sm_scale=None, causal=True, window=0, workspace=None,
                        out=None, lse=None, return_lse=True, stream=None):
    """sinkattn_decode over an FP8 KV cache (layout as in
    sinkattn_decode_split_fp8). Returns (out, lse)."""
    rows, Hq, d = q.shape
    Hkv = k_scale.numel()
    batch = kv_indptr.numel() - 1
    if num_splits <= 0:
        num_splits = sinkattn_decode_default_splits(batch, q_len, Hq, Hkv, d, max_kv_len)
    need = sinkattn_decode_workspace_bytes(batch, q_len, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    rc = lib().sinkattn_decode_fp8(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_scale), _ptr(v_scale), _ptr(kv_indptr), batch,
        int(q_len), int(max_kv_len), Hq, Hkv, d, _scale(sm_scale, d), int(bool(causal)),
        int(window), int(num_splits), _ptr(sinks), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(q, stream))
    _check(rc)
    return out, lse


PREFILL_KERNELS = {"auto": 0, "one_block": 1, "persistent": 2}


def sinkattn_set_prefill_kernel(kind) -> None:
    """Selects the prefill launch process-wide: "auto", "one_block" or
    "persistent" (or the integer codes of include/sinkattn.h)."""
    code = PREFILL_KERNELS[kind] if isinstance(kind, str) else int(kind)
    _check(lib().sinkattn_set_prefill_kernel(code))


def sinkattn_status_string(status: int) -> str:
    return status_name(status)


def sinkattn_last_error() -> str:
    return lib().sinkattn_last_error().decode()


def sinkattn_debug_status(stream=None) -> int:
    st = ctypes.c_int(0)
    s = ctypes.c_void_p(0) if stream is None and not torch.cuda.is_available() else (
        _stream(torch.empty(0, device="cuda"), stream))
    _check(lib().sinkattn_debug_status(s, ctypes.byref(st)))
    return int(st.value)


def sinkattn_debug_set_hooks(wait_limit_cycles: int = 0, skip_tile: int = -1) -> None:
    """Test only: bounded-wait limit in SM clock cycles (0: the default) and
    the KV tile the first thread block's producer leaves out (-1: none)."""
    _check(lib().sinkattn_debug_set_hooks(int(wait_limit_cycles), int(skip_tile)))

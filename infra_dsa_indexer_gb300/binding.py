"""Thin ctypes binding over the C ABI in include/dsa_indexer.h.

Same entry-point names as the C library; this module only marshals torch
tensors into pointers and shape structs and raises on a non-zero status. All
arithmetic runs in the CUDA library. If the library has not been built
(infra_dsa_indexer_gb300/_build/libdsa_indexer.so), every call raises; there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

IDX_FMT_BF16, IDX_FMT_E4M3, IDX_FMT_MXFP8, IDX_FMT_MXFP4 = 0, 1, 2, 3
IDX_W_F32, IDX_W_BF16 = 0, 1
IDX_FLAG_GROUP_ROWS = 1
IDX_FLAG_OUT_BF16 = 2
IDX_OK = 0
IDX_ERR_TIMEOUT = 8

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build",
                         "libdsa_indexer.so")
_lock = threading.Lock()
_lib = None


class IndexerError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({indexer_status_string(status)})")


class idx_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("N", ctypes.c_int32),
                ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("w_fmt", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("q_row_bytes", ctypes.c_int64), ("k_row_bytes", ctypes.c_int64),
                ("k_batch_bytes", ctypes.c_int64), ("out_row_stride", ctypes.c_int64)]


class idx_paged(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("table_stride", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Open the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {_LIB_PATH} is missing "
                "(run `python -m infra_dsa_indexer_gb300.build`)")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.indexer_logits.restype = i32
        lib.indexer_logits.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, i32,
                                       vp, ctypes.POINTER(idx_shape), vp]
        lib.indexer_logits_noalloc.restype = i32
        lib.indexer_logits_noalloc.argtypes = lib.indexer_logits.argtypes
        lib.indexer_status_string.restype = ctypes.c_char_p
        lib.indexer_status_string.argtypes = [i32]
        lib.indexer_get_last_error.restype = i32
        lib.indexer_get_last_error.argtypes = [vp]
        lib.indexer_set_wait_limit_ns.restype = i64
        lib.indexer_set_wait_limit_ns.argtypes = [i64]
        lib.indexer_paged_logits.restype = i32
        lib.indexer_paged_logits.argtypes = lib.indexer_logits.argtypes[:12] + [
            ctypes.POINTER(idx_paged), vp]
        lib.indexer_topk.restype = i32
        lib.indexer_topk.argtypes = [vp, i32, i64, i32, i64, i32, vp, i64, vp]
        lib.indexer_logits_topk_workspace_bytes.restype = i64
        lib.indexer_logits_topk_workspace_bytes.argtypes = [ctypes.POINTER(idx_shape)]
        lib.indexer_logits_topk.restype = i32
        lib.indexer_logits_topk.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                            ctypes.POINTER(idx_shape), i32, vp, i64, vp, i64, vp]
        lib.indexer_thd_windows.restype = i32
        lib.indexer_thd_windows.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
        lib.indexer_selftest_wait_timeout.restype = i32
        lib.indexer_selftest_wait_timeout.argtypes = [i64, vp]
        lib.indexer_noalloc_get_last_error.restype = i32
        lib.indexer_noalloc_get_last_error.argtypes = [vp]
        lib.indexer_noalloc_selftest_wait_timeout.restype = i32
        lib.indexer_noalloc_selftest_wait_timeout.argtypes = [i64, vp]
        lib.indexer_stream_release.restype = i32
        lib.indexer_stream_release.argtypes = [vp]
        lib.indexer_launches_per_call.restype = i32
        lib.indexer_launches_per_call.argtypes = [ctypes.POINTER(idx_shape)]
        lib.indexer_shutdown.restype = i32
        lib.indexer_shutdown.argtypes = []
        lib.indexer_version.restype = i32
        lib.indexer_version.argtypes = []
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("indexer_logits takes CUDA tensors (device pointers)")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_shape(B, S, N, H, D, fmt, w_fmt, *, q_row_bytes=0, k_row_bytes=0,
               k_batch_bytes=0, out_row_stride=0, flags=0) -> idx_shape:
    return idx_shape(B, S, N, H, D, fmt, w_fmt, flags, q_row_bytes, k_row_bytes,
                     k_batch_bytes, out_row_stride)


def indexer_logits(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, clean, out,
                   shape: idx_shape, stream=None) -> None:
    """Enqueue one logits call. Tensors are CUDA tensors holding the raw
    layouts of include/dsa_indexer.h (q [B,S,H,row], k [B,N,row], w [B,S,H],
    ks/ke [B,S] int32, out [B,S,>=N] float32, or bfloat16 with IDX_FLAG_OUT_BF16);
    q_sf/k_sf/k_scales may be None."""
    lib = load()
    st = lib.indexer_logits(_ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf), _ptr(k_scales), _ptr(w),
                            _ptr(ks), _ptr(ke), ctypes.c_float(sm_scale), int(bool(clean)),
                            _ptr(out), ctypes.byref(shape), _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_logits")


def indexer_logits_noalloc(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, clean, out,
                           shape: idx_shape, stream=None) -> None:
    """indexer_logits for callers that may not allocate device memory: the
    library keeps its scratch in one fixed device array instead (see the
    declaration in include/dsa_indexer.h for the sharing rules)."""
    lib = load()
    st = lib.indexer_logits_noalloc(_ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf), _ptr(k_scales),
                                    _ptr(w), _ptr(ks), _ptr(ke), ctypes.c_float(sm_scale),
                                    int(bool(clean)), _ptr(out), ctypes.byref(shape),
                                    _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_logits_noalloc")


def indexer_status_string(status: int) -> str:
    return load().indexer_status_string(int(status)).decode()


def indexer_get_last_error(stream=None) -> int:
    return load().indexer_get_last_error(_stream(stream))


def indexer_set_wait_limit_ns(ns: int) -> int:
    return load().indexer_set_wait_limit_ns(int(ns))


def indexer_paged_logits(q, q_sf, k_cache, k_sf_cache, k_scales_cache, w, ks, ke, sm_scale,
                         clean, out, shape: idx_shape, block_table, page_size: int,
                         num_pages: int, table_stride: int, stream=None) -> None:
    """indexer_logits with the keys in a page cache (see idx_paged in
    include/dsa_indexer.h): k_cache [num_pages, page_size, row bytes],
    block_table [B, table_stride] int32, all CUDA tensors."""
    lib = load()
    pg = idx_paged(ctypes.c_void_p(_ptr(block_table).value if block_table is not None else None),
                   int(table_stride), int(page_size), int(num_pages), 0)
    st = lib.indexer_paged_logits(_ptr(q), _ptr(q_sf), _ptr(k_cache), _ptr(k_sf_cache),
                                  _ptr(k_scales_cache), _ptr(w), _ptr(ks), _ptr(ke),
                                  ctypes.c_float(sm_scale), int(bool(clean)), _ptr(out),
                                  ctypes.byref(shape), ctypes.byref(pg), _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_paged_logits")


def indexer_topk(logits, k: int, idx=None, n=None, stream=None):
    """Top-k column indices of every row of a CUDA logits tensor (float32 or
    bfloat16, last dimension the columns, rows contiguous at a fixed stride):
    returns (or fills) an int32 tensor [..., k]; -1 pads rows with fewer than
    k finite values. `n` limits the columns (default: the last dimension)."""
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("logits must be float32 or bfloat16")
    flat = logits.reshape(-1, logits.shape[-1]) if logits.is_contiguous() else None
    if flat is None:
        if logits.dim() < 2 or logits.stride(-1) != 1:
            raise ValueError("logits rows must be contiguous")
        flat = logits.view(-1, logits.shape[-1]) if logits.dim() == 2 else None
        if flat is None:
            raise ValueError("logits must be 2-D or contiguous")
    rows, cols = flat.shape
    stride = flat.stride(0)
    n = cols if n is None else int(n)
    if idx is None:
        idx = torch.empty(logits.shape[:-1] + (k,), dtype=torch.int32, device=logits.device)
    idx_flat = idx.view(-1, idx.shape[-1])
    st = load().indexer_topk(_ptr(flat), int(logits.dtype == torch.bfloat16), int(rows), int(n),
                             int(stride), int(k), _ptr(idx_flat), int(idx_flat.stride(0)),
                             _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_topk")
    return idx


def indexer_logits_topk_workspace_bytes(shape: idx_shape) -> int:
    return load().indexer_logits_topk_workspace_bytes(ctypes.byref(shape))


def indexer_logits_topk(q, q_sf, k, k_sf, k_scales, w, ks, ke, sm_scale, shape: idx_shape,
                        topk: int, idx, workspace, stream=None) -> None:
    """Top-k key columns of every row straight from the inputs, without the
    logits (see include/dsa_indexer.h): idx is an int32 CUDA tensor
    [B*S, >= topk] (rows contiguous at a fixed stride), workspace a uint8
    CUDA tensor of indexer_logits_topk_workspace_bytes(shape) bytes."""
    flat = idx.view(-1, idx.shape[-1])
    st = load().indexer_logits_topk(_ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf), _ptr(k_scales),
                                    _ptr(w), _ptr(ks), _ptr(ke), ctypes.c_float(sm_scale),
                                    ctypes.byref(shape), int(topk), _ptr(flat),
                                    int(flat.stride(0)), _ptr(workspace),
                                    int(workspace.numel() * workspace.element_size()),
                                    _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_logits_topk")


def topk_case(case, t, topk: int, idx=None, workspace=None, stream=None):
    """indexer_logits_topk on tensors made by case_to_device (contiguous keys,
    FP32 logits shape); allocates idx and the workspace when not given."""
    shape = make_shape(case.B, case.S, case.N, case.H, case.D, case.fmt, case.w_fmt,
                       flags=IDX_FLAG_GROUP_ROWS if case.group_rows else 0)
    dev = t["q"].device
    if idx is None:
        idx = torch.empty(case.B * case.S, topk, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(indexer_logits_topk_workspace_bytes(shape), dtype=torch.uint8,
                                device=dev)
    indexer_logits_topk(t["q"], t["q_sf"], t["k"], t["k_sf"], t["k_scales"], t["w"], t["ks"],
                        t["ke"], case.sm_scale, shape, topk, idx, workspace, stream)
    return idx


def indexer_thd_windows(cu_seqlens_q, cu_seqlens_k, total_q: int, causal=True, ks=None,
                        ke=None, stream=None):
    """Absolute per-row windows of packed sequences from cumulative lengths
    (int32 CUDA tensors [num_seqs + 1]); returns (ks, ke) int32 [1, total_q]."""
    dev = cu_seqlens_q.device
    if ks is None:
        ks = torch.empty(1, total_q, dtype=torch.int32, device=dev)
    if ke is None:
        ke = torch.empty(1, total_q, dtype=torch.int32, device=dev)
    st = load().indexer_thd_windows(_ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                    int(cu_seqlens_q.numel() - 1), int(total_q),
                                    int(bool(causal)), _ptr(ks), _ptr(ke), _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_thd_windows")
    return ks, ke


def indexer_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    st = load().indexer_selftest_wait_timeout(int(limit_ns), _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_selftest_wait_timeout")


def indexer_noalloc_get_last_error(stream=None) -> int:
    return load().indexer_noalloc_get_last_error(_stream(stream))


def indexer_noalloc_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    st = load().indexer_noalloc_selftest_wait_timeout(int(limit_ns), _stream(stream))
    if st != IDX_OK:
        raise IndexerError(st, "indexer_noalloc_selftest_wait_timeout")


def indexer_stream_release(stream=None) -> int:
    return load().indexer_stream_release(_stream(stream))


def indexer_launches_per_call(shape: idx_shape) -> int:
    return load().indexer_launches_per_call(ctypes.byref(shape))


def indexer_shutdown() -> int:
    return load().indexer_shutdown()


def indexer_version() -> int:
    return load().indexer_version()


# ---------------------------------------------------------------------------
# convenience: a synth.Case on the device
# ---------------------------------------------------------------------------

def case_to_device(case, device="cuda", out_row_stride=None, out_bf16=False):
    """Copy a synth.Case's input bytes to `device`; allocate the FP32 (or,
    with out_bf16, BF16) output."""
    def dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:          # bf16 codes travel as int16 bit patterns
            a = a.view(np.int16)
        return torch.from_numpy(np.require(a, requirements=["C", "W"])).to(device)
    t = dict(q=dev(case.q), k=dev(case.k), w=dev(case.w), ks=dev(case.ks), ke=dev(case.ke),
             q_sf=dev(case.q_sf), k_sf=dev(case.k_sf), k_scales=dev(case.k_tok))
    if getattr(case, "page_size", 0):
        from . import synth
        pl = synth.paged_layout(case, case.page_size, seed=7)
        t.update(k=dev(pl["k_cache"]), k_sf=dev(pl["k_sf_cache"]),
                 k_scales=dev(pl["k_scales_cache"]), block_table=dev(pl["block_table"]),
                 page_size=case.page_size, num_pages=pl["num_pages"],
                 table_stride=pl["table_stride"])
    stride = out_row_stride or case.N
    t["out"] = torch.empty((case.B, case.S, stride),
                           dtype=torch.bfloat16 if out_bf16 else torch.float32, device=device)
    flags = (IDX_FLAG_GROUP_ROWS if case.group_rows else 0) | (IDX_FLAG_OUT_BF16 if out_bf16 else 0)
    t["shape"] = make_shape(case.B, case.S, case.N, case.H, case.D, case.fmt, case.w_fmt,
                            out_row_stride=stride, flags=flags)
    return t


def run_case(case, t, stream=None, clean=None):
    """indexer_logits (indexer_paged_logits for a paged case) on tensors made
    by case_to_device."""
    clean = case.clean if clean is None else clean
    if "block_table" in t:
        indexer_paged_logits(t["q"], t["q_sf"], t["k"], t["k_sf"], t["k_scales"], t["w"],
                             t["ks"], t["ke"], case.sm_scale, clean, t["out"], t["shape"],
                             t["block_table"], t["page_size"], t["num_pages"],
                             t["table_stride"], stream)
    else:
        indexer_logits(t["q"], t["q_sf"], t["k"], t["k_sf"], t["k_scales"], t["w"], t["ks"],
                       t["ke"], case.sm_scale, clean, t["out"], t["shape"], stream)
    return t["out"]

"""Float64 CPU oracle for the lightning-indexer MQA logits (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only code allowed to import this package. The product
path (the CUDA library and its Python binding) never loads it, and the two
share no code: this package decodes the raw input bytes itself, in float64,
in `dsa_oracle.c`.

What it computes, and the pages it follows, is documented at the top of
`dsa_oracle.c`: logits[b,i,j] = sum_h w[b,i,h]*max(0, sm_scale*q[b,i,h,:].k[b,j,:])
inside the half-open window [ks, ke) (DeepGEMM pull request 435, "Standalone
performance reproducer"; cuDNN-frontend pull request 416, "Precision /
determinism"), -inf outside.

Every function here has pins in tests/test_oracle_pins.py (decoders against
library dtype casts, closed forms, invariants, a library-matmul route); none
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_BF16, FMT_E4M3, FMT_MXFP8, FMT_MXFP4 = 0, 1, 2, 3
W_F32, W_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into oracle/_build/liboracle.so with gcc + OpenMP."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so every product and sum is a
    # separately rounded float64 operation in source order.
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dbl, i32, i64 = ctypes.c_double, ctypes.c_int, ctypes.c_int64
        vp = ctypes.c_void_p
        lib.orc_decode_bf16.restype = dbl
        lib.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        for name in ("orc_decode_e4m3", "orc_decode_e2m1", "orc_decode_e8m0"):
            getattr(lib, name).restype = dbl
            getattr(lib, name).argtypes = [ctypes.c_uint8]
        lib.orc_logits.restype = i32
        lib.orc_logits.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                   i32, i32, i32, i32, i32, dbl, vp, i64,
                                   vp, vp, vp, i32]
        lib.orc_num_threads.restype = i32
        lib.orc_dequant_row.restype = i32
        lib.orc_dequant_row.argtypes = [i32, vp, vp, i32, dbl, vp]
        _lib = lib
        return lib


def decode_bf16(code: int) -> float:
    return _load().orc_decode_bf16(code)


def decode_e4m3(code: int) -> float:
    return _load().orc_decode_e4m3(code)


def decode_e2m1(code: int) -> float:
    return _load().orc_decode_e2m1(code)


def decode_e8m0(code: int) -> float:
    return _load().orc_decode_e8m0(code)


def dequant_row(fmt, data, sf, D, extra=1.0):
    """Dequantise one row of D elements (raw bytes, E8M0 scales) to float64."""
    data = np.ascontiguousarray(data)
    sf = None if sf is None else np.ascontiguousarray(sf, dtype=np.uint8)
    dst = np.empty(D, dtype=np.float64)
    if _load().orc_dequant_row(fmt, _ptr(data), _ptr(sf), D, float(extra), _ptr(dst)) != 0:
        raise ValueError("oracle rejected its arguments")
    return dst


def num_threads() -> int:
    return _load().orc_num_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def logits(fmt, q, k, w, ks, ke, sm_scale, *, q_sf=None, k_sf=None,
           k_tok=None, w_fmt=W_F32, H=None, D=None, rows=None,
           want_den=True, want_den_abs=False, nthreads=0):
    """Evaluate the oracle on raw input bytes.

    q: uint8/uint16 array [B,S,H,row] (row = D bf16 codes, D e4m3 bytes, or
       D/2 packed e2m1 bytes); k: [B,N,row]; q_sf [B,S,H,D/32], k_sf [B,N,D/32]
       uint8 E8M0 (MX formats); k_tok float32 [B,N] (FP8 per-token) or None;
    w: float32 [B,S,H] (w_fmt=W_F32) or uint16 bf16 codes (w_fmt=W_BF16);
    ks, ke int32 [B,S]; rows: optional int64 flattened row ids b*S+i.
    Returns (out [R,N], den [R,N] or None, den_abs [R,N] or None), float64.
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    B, S = q.shape[0], q.shape[1]
    H = q.shape[2] if H is None else H
    N = k.shape[1]
    if D is None:
        row = q.shape[3]
        D = {FMT_BF16: row, FMT_E4M3: row, FMT_MXFP8: row, FMT_MXFP4: 2 * row}[fmt]
    w = np.ascontiguousarray(w)
    ks = np.ascontiguousarray(ks, dtype=np.int32)
    ke = np.ascontiguousarray(ke, dtype=np.int32)
    q_sf = None if q_sf is None else np.ascontiguousarray(q_sf, dtype=np.uint8)
    k_sf = None if k_sf is None else np.ascontiguousarray(k_sf, dtype=np.uint8)
    k_tok = None if k_tok is None else np.ascontiguousarray(k_tok, dtype=np.float32)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows.shape[0]
    else:
        R = B * S
    out = np.empty((R, N), dtype=np.float64)
    den = np.empty((R, N), dtype=np.float64) if want_den else None
    den_abs = np.empty((R, N), dtype=np.float64) if want_den_abs else None
    rc = lib.orc_logits(fmt, w_fmt, _ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf),
                        _ptr(k_tok), _ptr(w), _ptr(ks), _ptr(ke), B, S, N, H, D,
                        float(sm_scale), _ptr(rows), R, _ptr(out), _ptr(den),
                        _ptr(den_abs), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (status {rc})")
    return out, den, den_abs

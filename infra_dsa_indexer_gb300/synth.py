"""Seeded synthetic inputs for the lightning-indexer MQA logits.

This module makes input bytes and nothing else: Gaussian draws, their
quantisation into the input formats (BF16, E4M3, MXFP8 = E4M3 + E8M0 per
32-element block, MXFP4 = E2M1 + E8M0) and the per-row key windows. It holds
none of the logits arithmetic; the CUDA path and the float64 oracle both
consume exactly the bytes made here.

Quantisation recipe (it shapes the inputs only, never parity):
  * BF16: round-to-nearest-even of the float32 draw.
  * FP8 per-token: per key row, scale = amax/448 (amax 0 -> 1), element =
    e4m3(x/scale). Q gets one scale per query row (all heads), folded into W.
  * MX (OCP Microscaling v1.0): per 32-element block, shared exponent
    X = floor(log2(amax)) - emax_elem (emax 8 for E4M3, 2 for E2M1), stored as
    the E8M0 byte X+127; element = x / 2^X rounded to nearest-even and
    saturated to the element format's largest finite value.
  * E2M1 packs two elements per byte, the even element in the low nibble.

Random draws use numpy's PCG64 so the same seed gives the same bytes on every
machine.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

FMT_BF16, FMT_E4M3, FMT_MXFP8, FMT_MXFP4 = 0, 1, 2, 3
W_F32, W_BF16 = 0, 1
FMT_NAMES = {FMT_BF16: "bf16", FMT_E4M3: "e4m3", FMT_MXFP8: "mxfp8", FMT_MXFP4: "mxfp4"}

E4M3_MAX = 448.0


@dataclasses.dataclass
class Case:
    """One problem instance: raw input bytes plus its shape and scalars."""
    name: str
    fmt: int
    B: int
    S: int
    N: int
    H: int
    D: int
    sm_scale: float               # exactly representable in float32
    q: np.ndarray                 # [B,S,H,row]  uint16 (bf16) / uint8
    k: np.ndarray                 # [B,N,row]
    w: np.ndarray                 # [B,S,H] float32, or uint16 bf16 codes
    w_fmt: int
    ks: np.ndarray                # [B,S] int32
    ke: np.ndarray                # [B,S] int32
    q_sf: np.ndarray | None = None  # [B,S,H,D/32] uint8 E8M0
    k_sf: np.ndarray | None = None  # [B,N,D/32] uint8 E8M0
    k_tok: np.ndarray | None = None  # [B,N] float32 per-token K scale
    clean: bool = True
    group_rows: bool = False      # windows are irregular: ask the call to group rows
    page_size: int = 0            # > 0: the keys go to the GPU through a paged cache

    def in_window_pairs(self) -> int:
        lo = np.clip(self.ks.astype(np.int64), 0, self.N)
        hi = np.clip(self.ke.astype(np.int64), 0, self.N)
        return int(np.maximum(hi - lo, 0).sum())

    def in_window_flops(self) -> float:
        return 2.0 * self.H * self.D * self.in_window_pairs()


# ----------------------------------------------------------------------------
# element encoders
# ----------------------------------------------------------------------------

def to_bf16_codes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even into OCP E4M3, saturating at +-448."""
    x = np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# E2M1 magnitudes by code: 0, 0.5, 1, 1.5, 2, 3, 4, 6. Midpoints between
# neighbours, and whether a value exactly on a midpoint rounds up (to the
# even code above) or stays on the even code below.
_E2M1_MIDPOINTS = ((0.25, False), (0.75, True), (1.25, False), (1.75, True),
                   (2.5, False), (3.5, True), (5.0, False))


def to_e2m1_codes(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even into E2M1 (one code per uint8), saturating at 6."""
    x = np.asarray(x, dtype=np.float32)
    ax = np.abs(x)
    code = np.zeros(x.shape, dtype=np.uint8)
    for mid, tie_up in _E2M1_MIDPOINTS:
        code += (ax >= mid) if tie_up else (ax > mid)
    code |= (np.signbit(x) & (code != 0)).astype(np.uint8) << 3
    return code


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[..., D] codes -> [..., D/2] bytes, element 2k in the low nibble."""
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).astype(np.uint8)


def mx_quantize(x: np.ndarray, elem: str):
    """OCP MX quantisation along the last axis (blocks of 32).

    Returns (element codes [..., D] for e4m3 / packed [..., D/2] for e2m1,
    E8M0 scale bytes [..., D/32])."""
    emax = {"e4m3": 8, "e2m1": 2}[elem]
    D = x.shape[-1]
    assert D % 32 == 0
    xb = x.reshape(*x.shape[:-1], D // 32, 32)
    amax = np.abs(xb).max(axis=-1)
    _, e = np.frexp(amax)                     # amax = m * 2^e, m in [0.5, 1)
    X = (e.astype(np.int32) - 1) - emax      # floor(log2(amax)) - emax
    X = np.where(amax > 0, X, 0)
    X = np.clip(X, -127, 127)
    sf = (X + 127).astype(np.uint8)
    scaled = xb / np.exp2(X.astype(np.float32))[..., None]
    scaled = scaled.reshape(x.shape)
    if elem == "e4m3":
        return to_e4m3_codes(scaled), sf
    return pack_e2m1(to_e2m1_codes(scaled)), sf


# ----------------------------------------------------------------------------
# windows
# ----------------------------------------------------------------------------

def causal_windows(B, S, N, offset):
    """Row i sees [0, offset + i)."""
    ke = (np.arange(S, dtype=np.int64) + offset)
    ke = np.broadcast_to(ke, (B, S)).astype(np.int32)
    return np.zeros((B, S), dtype=np.int32), np.ascontiguousarray(ke)


FORCED_EMPTY_ROWS = (0, 1, 127, 128, 4095, 4096, 8190, 8191)


def irregular_windows(rng, B, S, N, forced_empty=FORCED_EMPTY_ROWS):
    """ks ~ U[0, N/2), length ~ U[0, N/2] inclusive, ke = ks + length; rows in
    `forced_empty` (those below S) get length 0."""
    ks = rng.integers(0, N // 2, size=(B, S), dtype=np.int64)
    ln = rng.integers(0, N // 2 + 1, size=(B, S), dtype=np.int64)
    for r in forced_empty:
        if r < S:
            ln[:, r] = 0
    return ks.astype(np.int32), (ks + ln).astype(np.int32)


def decode_windows(rng, B, S, N, min_context):
    """Decode: batch b has a context of ctx_b ~ U[min_context, N] keys and S
    new query tokens at its end; token t sees [0, ctx_b - S + t + 1)."""
    ctx = rng.integers(min_context, N + 1, size=B, dtype=np.int64)
    t = np.arange(S, dtype=np.int64)
    ke = np.clip(ctx[:, None] - S + t[None, :] + 1, 0, N)
    return np.zeros((B, S), dtype=np.int32), ke.astype(np.int32)


def paged_layout(case, page_size, seed=0, spare_pages=3):
    """Scatter the case's keys (and key scales) into a page cache: batch b's
    pages get distinct page numbers in a random order, with `spare_pages`
    pages no key maps to; rows past N in the last page of a batch and the
    spare pages hold random bytes (no window reads them). Returns a dict with
    k_cache and k_sf_cache as bytes [num_pages, page_size, bytes per key]
    (k_sf_cache None for plain formats), k_scales_cache FP32 [num_pages,
    page_size] or None, block_table [B, stride] int32, num_pages and
    table_stride."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, N = case.B, case.N
    per = -(-N // page_size)
    num_pages = B * per + spare_pages
    order = rng.permutation(num_pages)[: B * per].reshape(B, per).astype(np.int32)
    stride = per + 1
    table = np.full((B, stride), -5, dtype=np.int32)       # one entry past the keys, never read
    table[:, :per] = order

    def scatter(src):
        """[B, N, ...] array -> random-filled byte cache [num_pages, page_size, bytes]."""
        if src is None:
            return None
        sb = np.ascontiguousarray(src).view(np.uint8).reshape(B, N, -1)
        cache = rng.integers(0, 256, size=(num_pages, page_size, sb.shape[-1]), dtype=np.uint8)
        for b in range(B):
            for i in range(per):
                n = min(page_size, N - i * page_size)
                cache[order[b, i], :n] = sb[b, i * page_size: i * page_size + n]
        return cache

    k_cache = scatter(case.k)
    k_sf_cache = scatter(case.k_sf)
    k_scales_cache = None
    if case.k_tok is not None:
        # random bytes could be NaN scales: spare rows get 1.0 instead
        k_scales_cache = np.ones((num_pages, page_size), dtype=np.float32)
        for b in range(B):
            for i in range(per):
                n = min(page_size, N - i * page_size)
                k_scales_cache[order[b, i], :n] = case.k_tok[b, i * page_size: i * page_size + n]
    return dict(k_cache=k_cache, k_sf_cache=k_sf_cache, k_scales_cache=k_scales_cache,
                block_table=table, num_pages=num_pages, table_stride=stride)


def thd_windows(seqlens_q, seqlens_k, causal=True):
    """Windows of sequences packed along the row and key axes of one batch
    (the THD layout: cu_seqlens are the prefix sums of the lengths). Query
    row i of sequence s sees that sequence's keys only: [cu_k[s], cu_k[s] +
    n_k - n_q + i + 1) when causal (the last query row sees every key of its
    sequence), else [cu_k[s], cu_k[s] + n_k). Returns ks, ke as int32 [1, T_q]."""
    ks, ke = [], []
    k0 = 0
    for nq, nk in zip(seqlens_q, seqlens_k):
        i = np.arange(nq, dtype=np.int64)
        ks.append(np.full(nq, k0, dtype=np.int64))
        ln = np.clip(nk - nq + i + 1, 0, nk) if causal else np.full(nq, nk, dtype=np.int64)
        ke.append(k0 + ln)
        k0 += nk
    return (np.concatenate(ks).astype(np.int32)[None, :],
            np.concatenate(ke).astype(np.int32)[None, :])


# ----------------------------------------------------------------------------
# case builder
# ----------------------------------------------------------------------------

def make_case(fmt, B, S, N, H=64, D=128, *, seed=0, windows="full",
              w_fmt=W_F32, w_std=1.0 / 8.0, sm_scale=None, ks=None, ke=None,
              zero=False, name=None, mx_unit_scales=False, group_rows=False,
              thd=None, page_size=0, min_context=1) -> Case:
    """Draw Q, K ~ N(0,1), W ~ N(0, w_std^2), quantise to `fmt`.

    windows: "full" ([0,N)), "causal" ([0, N-S+i+1)), "causal_excl"
    ([0, N-S+i)), "irregular" (random, see irregular_windows), "thd" (packed
    sequences, thd = (seqlens_q, seqlens_k) summing to S and N; see
    thd_windows), "decode" (S new tokens at the end of a context of
    U[min_context, N] keys per batch; see decode_windows), or give ks/ke.
    page_size > 0 marks the case for the paged-key entry point (see
    paged_layout); the logical keys stay in `k`.
    zero=True makes all-zero Q/K/W (MX scales = 1), as in the pages' timing
    workload."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    sm_scale = float(np.float32(sm_scale))

    def draw(shape):
        if zero:
            return np.zeros(shape, dtype=np.float32)
        return rng.standard_normal(shape, dtype=np.float32)

    qf = draw((B, S, H, D))
    kf = draw((B, N, D))
    wf = draw((B, S, H)) * np.float32(w_std)

    q_sf = k_sf = k_tok = None
    if fmt == FMT_BF16:
        q, k = to_bf16_codes(qf), to_bf16_codes(kf)
    elif fmt == FMT_E4M3:
        # per-key scale amax/448; per-query-row scale folded into W
        kam = np.abs(kf).max(axis=-1)
        k_tok = np.where(kam > 0, kam / np.float32(E4M3_MAX), 1.0).astype(np.float32)
        k = to_e4m3_codes(kf / k_tok[..., None])
        qam = np.abs(qf).max(axis=(-1, -2))
        q_row = np.where(qam > 0, qam / np.float32(E4M3_MAX), 1.0).astype(np.float32)
        q = to_e4m3_codes(qf / q_row[..., None, None])
        wf = (wf * q_row[..., None]).astype(np.float32)
    elif fmt in (FMT_MXFP8, FMT_MXFP4):
        elem = "e4m3" if fmt == FMT_MXFP8 else "e2m1"
        q, q_sf = mx_quantize(qf, elem)
        k, k_sf = mx_quantize(kf, elem)
        if zero or mx_unit_scales:
            q_sf = np.full_like(q_sf, 0x7F)
            k_sf = np.full_like(k_sf, 0x7F)
    else:
        raise ValueError(f"unknown format {fmt}")

    w = to_bf16_codes(wf) if w_fmt == W_BF16 else wf.astype(np.float32)

    if ks is None or ke is None:
        if windows == "full":
            ks = np.zeros((B, S), dtype=np.int32)
            ke = np.full((B, S), N, dtype=np.int32)
        elif windows == "causal":
            ks, ke = causal_windows(B, S, N, N - S + 1)
        elif windows == "causal_excl":
            ks, ke = causal_windows(B, S, N, N - S)
        elif windows == "irregular":
            ks, ke = irregular_windows(rng, B, S, N)
        elif windows == "decode":
            ks, ke = decode_windows(rng, B, S, N, min_context)
        elif windows == "thd":
            lq, lk = thd
            if B != 1 or sum(lq) != S or sum(lk) != N:
                raise ValueError("thd: one batch, lengths summing to S and N")
            ks, ke = thd_windows(lq, lk)
        else:
            raise ValueError(windows)
    ks = np.ascontiguousarray(np.broadcast_to(np.asarray(ks, dtype=np.int32), (B, S)))
    ke = np.ascontiguousarray(np.broadcast_to(np.asarray(ke, dtype=np.int32), (B, S)))
    return Case(name=name or f"{FMT_NAMES[fmt]}_B{B}_S{S}_N{N}", fmt=fmt, B=B,
                S=S, N=N, H=H, D=D, sm_scale=sm_scale, q=q, k=k, w=w,
                w_fmt=w_fmt, ks=ks, ke=ke, q_sf=q_sf, k_sf=k_sf, k_tok=k_tok,
                group_rows=group_rows, page_size=page_size)


# The five workloads, by what they are. Seed = position in this list.
WORKLOADS = {
    "tiny_causal_bf16": dict(fmt=FMT_BF16, B=1, S=128, N=1024, windows="causal",
                             w_fmt=W_F32, seed=0),
    "bf16_batched_causal_4096": dict(fmt=FMT_BF16, B=2, S=4096, N=4096,
                                     windows="causal", w_fmt=W_BF16, seed=1),
    "fp8_per_token_2048x32768": dict(fmt=FMT_E4M3, B=1, S=2048, N=32768,
                                     windows="causal_excl", w_fmt=W_F32, seed=2),
    "mxfp8_8192x65536": dict(fmt=FMT_MXFP8, B=1, S=8192, N=65536,
                             windows="causal_excl", w_fmt=W_F32, seed=3),
    "mxfp4_irregular_8192x65536": dict(fmt=FMT_MXFP4, B=1, S=8192, N=65536,
                                       windows="irregular", w_fmt=W_F32, seed=4,
                                       group_rows=True),
    # The DeepGEMM MX reproducer's shapes (window [0, N - S + i)), for a
    # like-for-like reading of its published times.
    "mxfp8_2048x32768": dict(fmt=FMT_MXFP8, B=1, S=2048, N=32768,
                             windows="causal_excl", w_fmt=W_F32, seed=5),
    "mxfp4_2048x32768": dict(fmt=FMT_MXFP4, B=1, S=2048, N=32768,
                             windows="causal_excl", w_fmt=W_F32, seed=6),
    "mxfp4_8192x65536": dict(fmt=FMT_MXFP4, B=1, S=8192, N=65536,
                             windows="causal_excl", w_fmt=W_F32, seed=7),
    # Three causal sequences packed along rows and keys (THD), 4 keys per
    # query, 8192 query rows in all; the output has global key columns.
    "thd_bf16_3seq_8192x32768": dict(fmt=FMT_BF16, B=1, S=8192, N=32768, windows="thd",
                                     thd=((4096, 2560, 1536), (16384, 10240, 6144)),
                                     w_fmt=W_F32, seed=8),
    # Decode: 64 sequences, 2 new tokens each, contexts U[16384, 32768], keys
    # E4M3 with per-key scales in a cache of 64-key pages in random order.
    "paged_fp8_decode_64x2_32768": dict(fmt=FMT_E4M3, B=64, S=2, N=32768, windows="decode",
                                        min_context=16384, page_size=64, w_fmt=W_F32, seed=9),
}


def make_workload(name: str, **overrides) -> Case:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return make_case(name=name, **kw)

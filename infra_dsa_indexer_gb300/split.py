"""Query-row split of one logits problem across GPUs (host logic only).

Every query row of the indexer is independent: its logits need that row's
Q, head weights and window, and the keys of its batch. So one problem splits
across W processes (one GPU each) by query rows: rank r takes a contiguous
range of the flattened B*S rows, keeps the keys (and key scales) of the
batches it touches whole, and writes its own slice of the output rows.
Nothing is exchanged between ranks: no collective on the data path.

The ranges are balanced by work, not by row count: a causal or irregular
window makes some rows far longer than others, so the split points are
placed where the running sum of in-window keys (plus one per row, for the
rows' fixed cost) reaches r/W of the total.

A range that crosses a batch boundary becomes one slice per batch, because
one indexer_logits call covers rows of a single batch layout: slice
(b, s0, s1) is a B=1 call on rows [s0, s1) of batch b with the keys of b.
"""
from __future__ import annotations

import numpy as np


def row_split(ks, ke, N: int, world: int):
    """Split the rows of a [B, S] window layout into `world` contiguous work
    ranges. Returns, per rank, a list of (b, s0, s1) slices (possibly empty
    when there are fewer rows than ranks)."""
    ks = np.asarray(ks, dtype=np.int64)
    ke = np.asarray(ke, dtype=np.int64)
    if ks.shape != ke.shape or ks.ndim != 2:
        raise ValueError("ks and ke must be [B, S]")
    if world < 1:
        raise ValueError("world must be >= 1")
    B, S = ks.shape
    lo = np.clip(ks, 0, N)
    hi = np.clip(ke, 0, N)
    cost = (np.maximum(hi - lo, 0) + 1).reshape(-1).astype(np.float64)
    cum = np.concatenate([[0.0], np.cumsum(cost)])
    total = cum[-1]
    # first flattened row of each rank; monotone, so ranges never overlap
    cuts = [0]
    for r in range(1, world):
        cuts.append(int(np.searchsorted(cum, total * r / world, side="left")))
    cuts.append(B * S)
    cuts = np.maximum.accumulate(np.clip(cuts, 0, B * S))
    out = []
    for r in range(world):
        a, b_end = int(cuts[r]), int(cuts[r + 1])
        slices = []
        while a < b_end:
            b = a // S
            s0 = a - b * S
            s1 = min(S, s0 + (b_end - a))
            slices.append((b, s0, s1))
            a += s1 - s0
        out.append(slices)
    return out


def slice_tensors(t: dict, b: int, s0: int, s1: int) -> dict:
    """Views of a device problem (the dict binding.case_to_device makes) for
    rows [s0, s1) of batch b: a B=1 problem whose pointers start at that
    slice. Q, W, its Q scales, windows and output rows are offset; the keys
    of batch b are taken whole."""
    v = dict(t)
    for key in ("q", "q_sf", "w", "ks", "ke", "out"):
        if t.get(key) is not None:
            v[key] = t[key][b:b + 1, s0:s1]
    for key in ("k", "k_sf", "k_scales"):
        if t.get(key) is not None:
            v[key] = t[key][b:b + 1]
    return v

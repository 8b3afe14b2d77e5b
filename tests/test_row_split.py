"""The query-row split of one problem across ranks, on CPU with two gloo ranks.

Each rank takes a contiguous, work-balanced range of the query rows, the keys
of its batches whole, and writes its own output rows; nothing is exchanged on
the data path. Checked here: the ranges of all ranks cover every row exactly
once, the work is balanced, and the float64 oracle run slice by slice (each a
B=1 problem on the sliced arrays, as the ranks' calls see them) gives the
oracle's logits of the whole problem, bit for bit.
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

from infra_dsa_indexer_gb300 import split, synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    rng = np.random.default_rng(5)
    B, S, N = 3, 9, 300
    ks = rng.integers(-10, N // 2, size=(B, S))
    ke = ks + rng.integers(-5, N, size=(B, S))
    ke[1, 4] = ks[1, 4]                           # an empty row
    return synth.make_case(synth.FMT_MXFP8, B, S, N, H=4, seed=77, ks=ks, ke=ke)


def _oracle_slice(case, b, s0, s1):
    """The oracle on rows [s0, s1) of batch b as a B=1 problem."""
    import oracle
    sl = lambda a: None if a is None else a[b:b + 1, s0:s1]
    kb = lambda a: None if a is None else a[b:b + 1]
    out, _, _ = oracle.logits(case.fmt, sl(case.q), kb(case.k), sl(case.w), sl(case.ks),
                              sl(case.ke), case.sm_scale, q_sf=sl(case.q_sf), k_sf=kb(case.k_sf),
                              k_tok=kb(case.k_tok), w_fmt=case.w_fmt, H=case.H, D=case.D,
                              want_den=False, nthreads=1)
    return out


def _rank_main(rank, world, port, out):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = _case()
        mine = split.row_split(case.ks, case.ke, case.N, world)[rank]
        pieces = [(b, s0, s1, _oracle_slice(case, b, s0, s1)) for b, s0, s1 in mine]
        gathered = [None] * world
        dist.all_gather_object(gathered, pieces)
        out.put((rank, gathered if rank == 0 else None))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_cover_rows_once_and_match_the_whole_problem():
    import oracle
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    case = _case()
    whole, _, _ = oracle.logits(case.fmt, case.q, case.k, case.w, case.ks, case.ke,
                                case.sm_scale, q_sf=case.q_sf, k_sf=case.k_sf, k_tok=case.k_tok,
                                w_fmt=case.w_fmt, H=case.H, D=case.D, want_den=False, nthreads=1)
    whole = whole.reshape(case.B, case.S, case.N)
    seen = np.zeros((case.B, case.S), dtype=np.int64)
    for rank_pieces in got[0]:
        for b, s0, s1, logits in rank_pieces:
            seen[b, s0:s1] += 1
            # same rows, same float64 loops: the same bits, -inf included
            assert np.array_equal(logits.view(np.int64), whole[b, s0:s1].view(np.int64))
    assert np.all(seen == 1)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 40])
def test_row_split_is_a_balanced_partition(world):
    rng = np.random.default_rng(world)
    B, S, N = 2, 20, 4096
    ks = np.zeros((B, S), dtype=np.int64)
    ke = np.tile(np.arange(1, S + 1) * (N // S), (B, 1))          # causal staircase
    ke[1] = rng.integers(0, N, size=S)
    parts = split.row_split(ks, ke, N, world)
    assert len(parts) == world
    seen = np.zeros((B, S), dtype=np.int64)
    cost = []
    for slices in parts:
        c = 0
        for b, s0, s1 in slices:
            assert 0 <= b < B and 0 <= s0 < s1 <= S
            seen[b, s0:s1] += 1
            c += int((np.clip(ke[b, s0:s1], 0, N) + 1).sum())
        cost.append(c)
    assert np.all(seen == 1)
    if world <= B * S:
        # each range ends at most one row past its share
        share = sum(cost) / world
        assert max(cost) <= share + N + 1


def test_slice_tensors_offsets_rows_and_keeps_keys():
    torch = pytest.importorskip("torch")
    B, S, N, H = 2, 8, 50, 64
    t = {"q": torch.arange(B * S * H * 4).reshape(B, S, H, 4),
         "k": torch.arange(B * N * 4).reshape(B, N, 4),
         "w": torch.zeros(B, S, H), "ks": torch.zeros(B, S, dtype=torch.int32),
         "ke": torch.ones(B, S, dtype=torch.int32), "out": torch.zeros(B, S, N),
         "q_sf": None, "k_sf": None, "k_scales": None}
    v = split.slice_tensors(t, 1, 3, 7)
    assert v["q"].shape == (1, 4, H, 4) and v["q"].data_ptr() == t["q"][1, 3].data_ptr()
    assert v["out"].data_ptr() == t["out"][1, 3].data_ptr() and v["out"].shape == (1, 4, N)
    assert v["k"].shape == (1, N, 4) and v["k"].data_ptr() == t["k"][1].data_ptr()
    assert v["ks"].is_contiguous() and v["ks"].shape == (1, 4)

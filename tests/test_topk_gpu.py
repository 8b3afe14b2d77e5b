"""Top-k selection over logits (indexer_topk).

Several answers are correct when values tie at the threshold, so the check is
on what is unique: with T the k-th largest finite value of a row (numpy on
the very same values), the selection holds k distinct valid columns (or every
finite column and -1 padding when there are fewer than k), every value above
T, and only values >= T. End to end, the columns selected from the GPU
logits of a call must be a top-k of the float64 oracle's logits up to the
logits tolerance.
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import REL_TOL, check_topk, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,k", [(1, 1), (100, 7), (100, 150), (5000, 2048), (65536, 2048),
                                 (3000, 2999), (65536, 4096), (8192, 5000)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_topk_random_rows(N, k, dtype):
    g = torch.Generator(device="cuda").manual_seed(N + k)
    rows = 37
    x = torch.randn(rows, N, device="cuda", generator=g)
    # -inf outside random windows, a few empty rows, and heavy ties
    lo = torch.randint(0, N, (rows, 1), device="cuda", generator=g)
    hi = torch.randint(0, N + 1, (rows, 1), device="cuda", generator=g)
    cols = torch.arange(N, device="cuda")[None, :]
    x = torch.where((cols >= lo) & (cols < hi), x, torch.full_like(x, float("-inf")))
    x[3] = float("-inf")
    x[5] = torch.where(torch.isinf(x[5]), x[5], torch.round(x[5] * 2) / 2)   # ties
    x = x.to(dtype)
    sel = binding.indexer_topk(x, k)
    torch.cuda.synchronize()
    check_topk(x.float().double().cpu().numpy(), sel.cpu().numpy(), k)


@pytest.mark.parametrize("extra", [0, 1])
def test_topk_both_block_sizes(extra):
    """Calls with at most two rows per SM run 1024 threads per row, larger
    ones 512: the rows on either side of that line give the same answers."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, N, k = 2 * sms + extra, 8192, 512
    g = torch.Generator(device="cuda").manual_seed(7 + extra)
    x = torch.randn(rows, N, device="cuda", generator=g)
    lo = torch.randint(0, N, (rows, 1), device="cuda", generator=g)
    cols = torch.arange(N, device="cuda")[None, :]
    x = torch.where(cols >= lo // 2, x, torch.full_like(x, float("-inf")))
    sel = binding.indexer_topk(x, k)
    torch.cuda.synchronize()
    check_topk(x.double().cpu().numpy(), sel.cpu().numpy(), k)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,k", [(65536, 20000), (65536, 2048), (9000, 4500)])
def test_topk_tied_runs_overflow_the_boundary_bin(N, k, dtype):
    """A few distinct values only, with k falling inside a run of equal values
    far larger than the shared-memory candidate buffer: the boundary bin does
    not fit, so the low digits are resolved by sweeps over the row."""
    g = torch.Generator(device="cuda").manual_seed(N ^ k)
    rows = 9
    x = torch.randint(0, 4, (rows, N), device="cuda", generator=g).float() - 1.5
    x[1, : N // 3] = float("-inf")             # a tied row with a prefix outside the window
    x[2] = 0.25                                # one value only
    x = x.to(dtype)
    sel = binding.indexer_topk(x, k)
    torch.cuda.synchronize()
    check_topk(x.double().cpu().numpy(), sel.cpu().numpy(), k)


def test_topk_strided_rows_and_prefix_columns():
    x = torch.randn(20, 1000, device="cuda")
    sel = binding.indexer_topk(x, 64, n=900)               # only the first 900 columns
    torch.cuda.synchronize()
    s = sel.cpu().numpy()
    assert np.all((s >= 0) & (s < 900))
    check_topk(x[:, :900].double().cpu().numpy(), s, 64)


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4])
def test_topk_of_indexer_logits_against_oracle(fmt):
    case = synth.make_case(fmt, 1, 24, 3000, seed=200 + fmt, windows="irregular")
    t = binding.case_to_device(case)
    binding.run_case(case, t)
    k = 256
    sel = binding.indexer_topk(t["out"], k).view(-1, k).cpu().numpy()
    ref, den = oracle_rows(case)
    gpu = t["out"].view(-1, case.N).double().cpu().numpy()
    check_topk(gpu, sel, k)                                 # exact on the GPU's own values
    for r in range(ref.shape[0]):
        picked = sel[r][sel[r] >= 0]
        finite = np.flatnonzero(np.isfinite(ref[r]))
        if len(finite) <= k:
            assert set(picked.tolist()) == set(finite.tolist())
            continue
        thr = np.sort(ref[r, finite])[::-1][k - 1]
        slack = REL_TOL * (1e-6 + den[r, picked]) * 2
        assert np.all(ref[r, picked] >= thr - slack), f"row {r}"
        # and from above: a column whose oracle value beats the threshold by
        # more than twice the logits tolerance was picked
        sure = finite[ref[r, finite] > thr + 2 * REL_TOL * (1e-6 + den[r, finite])]
        assert set(sure.tolist()) <= set(picked.tolist()), f"row {r}: missed a clear top-k column"


def test_topk_full_size_mxfp8():
    case = synth.make_workload("mxfp8_8192x65536")
    t = binding.case_to_device(case, out_bf16=True)
    binding.run_case(case, t)
    sel = binding.indexer_topk(t["out"], 2048)
    torch.cuda.synchronize()
    rows = np.arange(0, case.S, 512)
    out = t["out"].view(-1, case.N)
    check_topk(out[torch.from_numpy(rows).cuda()].double().cpu().numpy(),
               sel.view(-1, 2048)[torch.from_numpy(rows).cuda()].cpu().numpy(), 2048)

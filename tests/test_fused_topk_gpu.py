"""indexer_logits_topk: the logits reduced straight to each row's top-k key
columns, without writing the logits.

The call computes every logit exactly as indexer_logits does (same tiles,
same arithmetic), so its selection must be a top-k of indexer_logits' FP32
output for the same inputs: check_topk on those values (ties at the
threshold may be resolved either way). Cases cover every input format,
ragged, empty, inverted and out-of-range windows, rows shorter than k, k
above N, a negative sm_scale, grouped rows, all-zero inputs (every in-window
logit ties), and the full-size MXFP8 workload against the float64 oracle on
sampled rows.
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import REL_TOL, check_topk, oracle_rows

pytestmark = pytest.mark.gpu

ALL = [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from infra_dsa_indexer_gb300 import build
    build.build()
    binding.load()
    yield
    assert binding.indexer_get_last_error() == binding.IDX_OK


def fused_vs_logits(case, k):
    """The fused selection and the FP32 logits of the same call."""
    t = binding.case_to_device(case)
    binding.run_case(case, t)
    sel = binding.topk_case(case, t, k)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    vals = t["out"].view(-1, case.N).double().cpu().numpy()
    return vals, sel.cpu().numpy()


def ragged_case(fmt, seed, B=2, S=40, N=3000, **kw):
    rng = np.random.default_rng(seed)
    ks = rng.integers(-50, N, size=(B, S))
    ke = ks + rng.integers(-100, N, size=(B, S))
    ks[0, :4] = 0
    ke[0, :4] = 0                          # an all-empty block
    ks[1, 8], ke[1, 8] = 900, 50           # inverted window
    ks[1, 9], ke[1, 9] = 100, 130          # shorter than most k below
    return synth.make_case(fmt, B, S, N, seed=seed, ks=ks, ke=ke, **kw)


@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("k", [1, 64, 700, 5000])
def test_fused_topk_ragged_windows(fmt, k):
    case = ragged_case(fmt, 300 + fmt)
    vals, sel = fused_vs_logits(case, k)
    check_topk(vals, sel, k)


@pytest.mark.parametrize("fmt", ALL)
def test_fused_topk_causal_several_tiles(fmt):
    case = synth.make_case(fmt, 1, 96, 4100, seed=310 + fmt, windows="causal")
    vals, sel = fused_vs_logits(case, 512)
    check_topk(vals, sel, 512)


@pytest.mark.parametrize("N", [1, 127, 129, 513, 999])
def test_fused_topk_ragged_key_tails(N):
    case = synth.make_case(synth.FMT_E4M3, 1, 12, N, seed=320 + N, windows="full")
    for k in (1, 100):
        vals, sel = fused_vs_logits(case, k)
        check_topk(vals, sel, k)


def test_fused_topk_negative_scale_mxfp4():
    case = synth.make_case(synth.FMT_MXFP4, 1, 24, 2000, seed=330, windows="irregular",
                           sm_scale=-0.0883883)
    vals, sel = fused_vs_logits(case, 256)
    check_topk(vals, sel, 256)


@pytest.mark.parametrize("fmt", [synth.FMT_E4M3, synth.FMT_MXFP4])
def test_fused_topk_grouped_rows(fmt):
    case = synth.make_case(fmt, 2, 64, 3000, seed=340 + fmt, windows="irregular",
                           group_rows=True)
    vals, sel = fused_vs_logits(case, 300)
    check_topk(vals, sel, 300)


def test_fused_topk_all_zero_inputs_tie_everywhere():
    case = synth.make_case(synth.FMT_MXFP8, 1, 16, 2500, seed=350, windows="causal", zero=True)
    vals, sel = fused_vs_logits(case, 600)
    check_topk(vals, sel, 600)


def test_fused_topk_workspace_too_small_is_refused():
    case = synth.make_case(synth.FMT_BF16, 1, 8, 300, seed=360, windows="causal")
    t = binding.case_to_device(case)
    shape = binding.make_shape(case.B, case.S, case.N, case.H, case.D, case.fmt, case.w_fmt)
    need = binding.indexer_logits_topk_workspace_bytes(shape)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    idx = torch.empty(case.S, 16, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.IndexerError) as e:
        binding.indexer_logits_topk(t["q"], None, t["k"], None, None, t["w"], t["ks"], t["ke"],
                                    case.sm_scale, shape, 16, idx, ws)
    assert e.value.status == 10


@pytest.mark.slow
def test_fused_topk_full_size_mxfp8_against_logits_and_oracle():
    case = synth.make_workload("mxfp8_8192x65536")
    k = 2048
    t = binding.case_to_device(case)
    binding.run_case(case, t)
    sel = binding.topk_case(case, t, k)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    rows = np.concatenate([np.arange(0, case.S, 257), [case.S - 1]])
    rt = torch.from_numpy(rows).cuda()
    picked = sel[rt].cpu().numpy()
    vals = t["out"].view(-1, case.N)[rt].double().cpu().numpy()
    check_topk(vals, picked, k)
    # against the float64 oracle on a few rows: the picked columns are a
    # top-k of the exact logits up to twice the logits tolerance
    few = rows[::8]
    ref, den = oracle_rows(case, rows=few)
    for i, r in enumerate(few):
        p = picked[list(rows).index(r)]
        p = p[p >= 0]
        fin = np.flatnonzero(np.isfinite(ref[i]))
        thr = np.sort(ref[i, fin])[::-1][k - 1]
        assert np.all(ref[i, p] >= thr - 2 * REL_TOL * (1e-6 + den[i, p])), f"row {r}"
        sure = fin[ref[i, fin] > thr + 2 * REL_TOL * (1e-6 + den[i, fin])]
        assert set(sure.tolist()) <= set(p.tolist()), f"row {r}"

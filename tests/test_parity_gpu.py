"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small cases span several 128-key tiles, several 4-row blocks and ragged tails;
the edge cases cover empty, inverted, out-of-range and nonzero-start windows,
N in {1, 127, 129, 999}, negative sm_scale, BF16 and FP32 W, padded output
rows, all-zero inputs and determinism. The full-size workloads are checked on
sampled rows against the oracle and on every row for the -inf pattern.
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, expected_mask, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from infra_dsa_indexer_gb300 import build
    build.build()
    binding.load()
    yield
    assert binding.indexer_get_last_error() == binding.IDX_OK


def gpu_run(case, out_row_stride=None, clean=None, sentinel=None):
    t = binding.case_to_device(case, out_row_stride=out_row_stride)
    if sentinel is not None:
        t["out"].fill_(sentinel)
    binding.run_case(case, t, clean=clean)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    return t["out"].cpu().numpy()


def check_full(case, **kw):
    out = gpu_run(case, **kw)
    ref, den, den_abs = oracle_rows(case, want_den_abs=True)
    return compare(out[..., :case.N].reshape(-1, case.N), ref, den, den_abs=den_abs,
                   label=f"{synth.FMT_NAMES[case.fmt]} B{case.B} S{case.S} N{case.N}")


PLAIN = [synth.FMT_BF16, synth.FMT_E4M3]
ALL = [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4]


@pytest.mark.parametrize("fmt", ALL)
def test_tiny_causal_workload(fmt):
    case = synth.make_workload("tiny_causal_bf16", fmt=fmt)
    check_full(case)


@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("w_fmt", [synth.W_F32, synth.W_BF16])
def test_random_windows_ragged(fmt, w_fmt):
    rng = np.random.default_rng(100 + fmt)
    B, S, N = 2, 40, 1000
    ks = rng.integers(-50, N, size=(B, S))
    ke = ks + rng.integers(-100, N, size=(B, S))
    ks[0, :4] = 0
    ke[0, :4] = 0                      # an all-empty 4-row block
    ks[1, 8], ke[1, 8] = 900, 50       # inverted window
    case = synth.make_case(fmt, B, S, N, seed=21 + fmt, ks=ks, ke=ke, w_fmt=w_fmt)
    check_full(case)


@pytest.mark.parametrize("fmt", ALL)
def test_grouped_rows_irregular_windows(fmt):
    """IDX_FLAG_GROUP_ROWS reorders rows into blocks of similar windows: parity
    with the oracle, and the same bits as the ungrouped call (every element's
    reduction is unchanged; only which rows share a block differs)."""
    rng = np.random.default_rng(200 + fmt)
    B, S, N = 2, 64, 3000
    ks = rng.integers(0, N // 2, size=(B, S))
    ke = ks + rng.integers(0, N // 2 + 1, size=(B, S))
    ke[0, 5] = ks[0, 5]                       # an empty row
    case = synth.make_case(fmt, B, S, N, seed=60 + fmt, ks=ks, ke=ke)
    plain = gpu_run(case)
    case.group_rows = True
    grouped = check_full(case) is not None and gpu_run(case)
    assert np.array_equal(plain.view(np.int32), grouped.view(np.int32))


def test_grouped_rows_beyond_16k_rows():
    # the counting sort has no row limit; grouped equals ungrouped bit for bit
    import dataclasses
    S, N = 16388, 700
    case = synth.make_case(synth.FMT_MXFP4, 1, S, N, seed=77, windows="irregular",
                           group_rows=True)
    tg = binding.case_to_device(case)
    tu = binding.case_to_device(dataclasses.replace(case, group_rows=False))
    binding.run_case(case, tg)
    binding.run_case(case, tu)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    assert torch.equal(tg["out"].view(torch.int32), tu["out"].view(torch.int32))
    rows = np.arange(0, S, 97)
    ref, den = oracle_rows(case, rows=rows)
    compare(tg["out"].view(-1, N)[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, den)


def test_grouped_scratch_grows_across_calls():
    """Grouped calls of growing size on one stream re-size the library's
    scratch; every result stays right, and so does an ungrouped call after."""
    for S in (8, 256, 1024):
        rng = np.random.default_rng(S)
        ks = rng.integers(0, 400, size=(1, S))
        ke = ks + rng.integers(0, 401, size=(1, S))
        case = synth.make_case(synth.FMT_E4M3, 1, S, 800, seed=S, ks=ks, ke=ke, group_rows=True)
        check_full(case)
    check_full(synth.make_case(synth.FMT_BF16, 1, 16, 300, seed=3, windows="causal"))


@pytest.mark.parametrize("N", [1, 127, 129, 999])
@pytest.mark.parametrize("fmt", ALL)
def test_ragged_key_tails(N, fmt):
    case = synth.make_case(fmt, 1, 16, N, seed=N + fmt, windows="full" if fmt % 2 else "causal")
    check_full(case)


def test_negative_and_zero_sm_scale():
    case = synth.make_case(synth.FMT_BF16, 1, 8, 300, seed=5, windows="full", sm_scale=-0.0625)
    check_full(case)
    case = synth.make_case(synth.FMT_E4M3, 1, 8, 300, seed=6, windows="full", sm_scale=0.0)
    check_full(case)
    case = synth.make_case(synth.FMT_E4M3, 2, 12, 700, seed=16, windows="causal",
                           sm_scale=-0.125, w_fmt=synth.W_BF16)
    check_full(case)
    for fmt in (synth.FMT_MXFP8, synth.FMT_MXFP4):
        case = synth.make_case(fmt, 1, 12, 400, seed=17 + fmt, windows="causal", sm_scale=-0.1)
        check_full(case)


def test_padded_output_rows_untouched_beyond_n():
    case = synth.make_case(synth.FMT_BF16, 2, 8, 200, seed=7, windows="causal")
    out = gpu_run(case, out_row_stride=264, sentinel=12345.0)
    assert np.all(out[..., 200:] == 12345.0)
    ref, den = oracle_rows(case)
    compare(out[..., :200].reshape(-1, 200), ref, den)


def test_clean_false_in_window_values():
    case = synth.make_case(synth.FMT_E4M3, 1, 16, 700, seed=8, windows="causal")
    case.clean = False
    out = gpu_run(case, sentinel=7.0)
    ref, den = oracle_rows(case)
    compare(out.reshape(-1, 700), ref, den, check_outside=False)


@pytest.mark.parametrize("fmt", ALL)
def test_all_zero_inputs_reproducer_property(fmt):
    """Zero Q/K/W, windows [0, N-S+row): -inf exactly off-window, 0 in-window."""
    m, n = 64, 1100
    case = synth.make_case(fmt, 1, m, n, zero=True, windows="causal_excl")
    out = gpu_run(case).reshape(m, n)
    valid = np.arange(n)[None, :] < (np.arange(m) + n - m)[:, None]
    assert np.array_equal(np.isneginf(out), ~valid)
    assert np.all(out[valid] == 0.0)


@pytest.mark.parametrize("fmt", ALL)
def test_bitwise_deterministic(fmt):
    case = synth.make_case(fmt, 2, 64, 2000, seed=9, windows="causal")
    t = binding.case_to_device(case)
    first = binding.run_case(case, t).clone()
    for _ in range(20):
        again = binding.run_case(case, t)
        assert torch.equal(again.view(torch.int32), first.view(torch.int32))


def test_consecutive_calls_different_shapes_same_stream():
    cases = [synth.make_case(synth.FMT_BF16, 1, 8, 129, seed=1, windows="causal"),
             synth.make_case(synth.FMT_E4M3, 1, 32, 4000, seed=2, windows="causal_excl"),
             synth.make_case(synth.FMT_BF16, 3, 12, 555, seed=3, windows="full")]
    tens = [binding.case_to_device(c) for c in cases]
    for c, t in zip(cases, tens):
        binding.run_case(c, t)
    torch.cuda.synchronize()
    for c, t in zip(cases, tens):
        ref, den = oracle_rows(c)
        compare(t["out"].cpu().numpy().reshape(-1, c.N), ref, den)


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP8, synth.FMT_MXFP4])
def test_mx_block_scales_are_applied(fmt):
    """Scale bytes spread over +-8 binades and differing per block, key and
    head: a wrong scale-factor layout or byte selection breaks parity."""
    case = synth.make_case(fmt, 1, 8, 600, seed=30 + fmt, windows="full")
    rng = np.random.default_rng(31)
    case.q_sf = (case.q_sf.astype(np.int32) + rng.integers(-8, 9, case.q_sf.shape)).astype(np.uint8)
    case.k_sf = (case.k_sf.astype(np.int32) + rng.integers(-8, 9, case.k_sf.shape)).astype(np.uint8)
    check_full(case)


def test_bf16_w_equals_f32_w_of_same_values():
    """W given as BF16, or as FP32 holding the same BF16 values: bitwise equal."""
    case = synth.make_case(synth.FMT_BF16, 1, 16, 900, seed=10, windows="causal",
                           w_fmt=synth.W_BF16)
    a = gpu_run(case)
    wf = (case.w.astype(np.uint32) << 16).view(np.float32)
    case.w, case.w_fmt = wf, synth.W_F32
    b = gpu_run(case)
    assert np.array_equal(a.view(np.int32), b.view(np.int32))


# ---------------------------------------------------------------------------
# full-size workloads: sampled rows vs the oracle, every row for the mask
# ---------------------------------------------------------------------------

def sample_rows(B, S, step):
    rows = set()
    for b in range(B):
        base = b * S
        rows.update(base + r for r in range(0, S, step))
        rows.update(base + r for r in range(min(4, S)))
        rows.update(base + S - 1 - r for r in range(min(4, S)))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("S", [1, 2, 3, 5, 7, 13, 130])
@pytest.mark.parametrize("fmt", ALL)
def test_partial_last_row_block(S, fmt):
    # S not a multiple of the 4-row block: the missing rows of the last block
    # are computed on valid addresses and never stored; extra rows of the
    # output buffer past B*S keep their sentinel.
    B, N = 2, 333
    case = synth.make_case(fmt, B, S, N, seed=100 + 7 * S + fmt, windows="irregular",
                           group_rows=(S % 2 == 1))
    t = binding.case_to_device(case)
    big = torch.full((B * S + 4, N), 5.0, dtype=torch.float32, device="cuda")
    t["out"] = big[: B * S].view(B, S, N)
    binding.run_case(case, t)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    assert torch.all(big[B * S:] == 5.0)
    ref, den = oracle_rows(case)
    compare(big[: B * S].cpu().numpy(), ref, den)


@pytest.mark.parametrize("fmt", ALL)
def test_thd_packed_sequences(fmt):
    lq, lk = (37, 64, 9), (100, 256, 40)
    case = synth.make_case(fmt, 1, sum(lq), sum(lk), seed=120 + fmt, windows="thd",
                           thd=(lq, lk))
    check_full(case)


@pytest.mark.parametrize("name,step", [("bf16_batched_causal_4096", 256),
                                       ("fp8_per_token_2048x32768", 256),
                                       ("mxfp8_8192x65536", 512),
                                       ("mxfp4_irregular_8192x65536", 512),
                                       ("mxfp8_2048x32768", 256),
                                       ("mxfp4_2048x32768", 256),
                                       ("mxfp4_8192x65536", 1024),
                                       ("thd_bf16_3seq_8192x32768", 256),
                                       ("paged_fp8_decode_64x2_32768", 8)])
def test_full_size_workload(name, step):
    case = synth.make_workload(name)
    t = binding.case_to_device(case)
    binding.run_case(case, t)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    out = t["out"].view(-1, case.N)
    # mask of every row, on the device
    ks = torch.from_numpy(case.ks.reshape(-1).astype(np.int64)).cuda().clamp(0, case.N)
    ke = torch.from_numpy(case.ke.reshape(-1).astype(np.int64)).cuda().clamp(0, case.N)
    cols = torch.arange(case.N, device="cuda")[None, :]
    for r0 in range(0, out.shape[0], 512):
        sl = slice(r0, r0 + 512)
        outside = (cols < ks[sl, None]) | (cols >= ke[sl, None])
        assert torch.equal(torch.isneginf(out[sl]), outside), f"mask rows {r0}+"
        assert torch.isfinite(out[sl][~outside]).all()
    rows = sample_rows(case.B, case.S, step)
    if name.startswith("mxfp4"):
        # the forced-empty rows and their neighbours
        rows = np.union1d(rows, np.array([r for r in synth.FORCED_EMPTY_ROWS if r < case.S]))
    ref, den = oracle_rows(case, rows=rows)
    compare(out[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, den)

"""Batches of at most two query rows (decode with one or two new tokens).

For BF16 and E4M3 keys such calls run in two-row blocks: N = 128 MMAs into
four 128-column accumulators, drained by two groups of epilogue warps that
take alternate tiles. Each logit is computed by the same per-element
arithmetic as in a four-row block, so the bars are:

- bit for bit, the logits of the same rows computed in four-row blocks (the
  rows placed first in a batch of three rows, whose third row differs);
- the float64 oracle on every row;

on contiguous and paged keys, FP32 and BF16 logits, FP32 and BF16 weights,
ragged, empty, inverted and decode windows, and many short units, so that the alternation of the two
groups crosses unit boundaries after odd and even tile counts.
"""
import dataclasses

import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, oracle_rows

pytestmark = pytest.mark.gpu

TWO_ROW = [synth.FMT_BF16, synth.FMT_E4M3]
BF16_OUT_ROUNDING = 2.0 ** -8  # half an ulp of a BF16 logit at the bottom of its binade


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from infra_dsa_indexer_gb300 import build
    build.build()
    binding.load()
    yield
    assert binding.indexer_get_last_error() == binding.IDX_OK


def first_rows(case, S):
    """The case restricted to its first S rows of every batch."""
    cut = lambda a: None if a is None else np.ascontiguousarray(a[:, :S])
    return dataclasses.replace(case, S=S, q=cut(case.q), w=cut(case.w), ks=cut(case.ks),
                               ke=cut(case.ke), q_sf=cut(case.q_sf))


def logits(case, out_bf16=False):
    t = binding.case_to_device(case, out_bf16=out_bf16)
    binding.run_case(case, t)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    return t["out"].view(case.B, case.S, case.N)


def ragged(B, S, N, seed):
    rng = np.random.default_rng(seed)
    ks = rng.integers(-40, N, size=(B, S)).astype(np.int32)
    ke = (ks + rng.integers(-60, N + 100, size=(B, S))).astype(np.int32)
    ks[0, :] = 0
    ke[0, :] = 0                     # an all-empty block: a unit without tiles
    ks[1, 0], ke[1, 0] = 700, 90     # inverted
    ke[2, -1] = N + 500              # past N
    return ks, ke


@pytest.mark.parametrize("out_bf16", [False, True])
@pytest.mark.parametrize("page_size", [0, 64])
@pytest.mark.parametrize("S", [1, 2])
@pytest.mark.parametrize("fmt", TWO_ROW)
def test_two_row_blocks_bitwise_and_oracle(fmt, S, page_size, out_bf16):
    # 40 batches of 2100 keys (17 tiles): about 8 units per SM of one or two
    # tiles each, so each group's share of a unit starts on either parity.
    B, N = 40, 2100
    ks, ke = ragged(B, 3, N, seed=700 + 10 * fmt + S)
    wide = synth.make_case(fmt, B, 3, N, seed=710 + fmt, ks=ks, ke=ke, page_size=page_size)
    case = first_rows(wide, S)
    two = logits(case, out_bf16)
    four = logits(wide, out_bf16)[:, :S]
    assert torch.equal(two.view(torch.int16 if out_bf16 else torch.int32),
                       four.contiguous().view(torch.int16 if out_bf16 else torch.int32))
    ref, den = oracle_rows(case)
    compare(two.reshape(-1, N).float().cpu().numpy(), ref, den,
            out_rounding=BF16_OUT_ROUNDING if out_bf16 else 0.0, label=f"S={S}")


@pytest.mark.parametrize("S", [1, 2])
@pytest.mark.parametrize("fmt", TWO_ROW)
def test_two_row_blocks_bf16_weights(fmt, S):
    # BF16 head weights: only the lanes that hold the block's rows store them.
    B, N = 30, 1500
    ks, ke = ragged(B, 3, N, seed=750 + 10 * fmt + S)
    wide = synth.make_case(fmt, B, 3, N, seed=760 + fmt, ks=ks, ke=ke, w_fmt=synth.W_BF16)
    case = first_rows(wide, S)
    two = logits(case)
    four = logits(wide)[:, :S]
    assert torch.equal(two.view(torch.int32), four.contiguous().view(torch.int32))
    ref, den = oracle_rows(case)
    compare(two.reshape(-1, N).cpu().numpy(), ref, den)


@pytest.mark.parametrize("page_size", [64, 256])
@pytest.mark.parametrize("fmt", TWO_ROW)
def test_two_row_blocks_decode_windows_long_units(fmt, page_size):
    # Few batches of long contexts: units of many tiles, odd and even counts.
    case = synth.make_case(fmt, 5, 2, 40000, seed=720 + fmt, windows="decode",
                           min_context=3000, page_size=page_size)
    out = logits(case)
    ref, den = oracle_rows(case)
    compare(out.reshape(-1, case.N).cpu().numpy(), ref, den)


@pytest.mark.parametrize("fmt", TWO_ROW)
def test_two_row_blocks_negative_scale_and_tail(fmt):
    # A negative sm_scale (the MMA's negated A operand) and a ragged key tail.
    case = synth.make_case(fmt, 7, 2, 1153, seed=730 + fmt, windows="full", sm_scale=-0.07)
    out = logits(case)
    ref, den = oracle_rows(case)
    compare(out.reshape(-1, case.N).cpu().numpy(), ref, den)


@pytest.mark.parametrize("fmt", TWO_ROW)
def test_two_row_blocks_deterministic(fmt):
    case = synth.make_case(fmt, 24, 2, 3000, seed=740 + fmt, windows="decode", page_size=64)
    first = logits(case).clone()
    for _ in range(5):
        assert torch.equal(logits(case).view(torch.int32), first.view(torch.int32))

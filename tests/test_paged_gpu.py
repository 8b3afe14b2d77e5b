"""Keys in a paged cache (indexer_paged_logits).

The keys of every batch are scattered into pages in random order, with spare
pages and the rows past N filled with random bytes. Two bars: the logits
equal, bit for bit, those of indexer_logits on the same keys stored
contiguously (only the addressing differs), and they match the float64
oracle on the logical keys.
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, oracle_rows

pytestmark = pytest.mark.gpu

ALL = [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4]


def _paged_and_contiguous(case):
    import dataclasses
    tp = binding.case_to_device(case)
    assert "block_table" in tp
    tc = binding.case_to_device(dataclasses.replace(case, page_size=0))
    binding.run_case(case, tp)
    binding.run_case(dataclasses.replace(case, page_size=0), tc)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    return tp["out"], tc["out"]


@pytest.mark.parametrize("page_size", [64, 128, 192, 256, 320, 1024])
@pytest.mark.parametrize("fmt", ALL)
def test_paged_equals_contiguous_and_oracle(fmt, page_size):
    case = synth.make_case(fmt, 3, 12, 1000, seed=140 + fmt, windows="irregular",
                           page_size=page_size)
    op, oc = _paged_and_contiguous(case)
    assert torch.equal(op.view(torch.int32), oc.view(torch.int32))
    ref, den = oracle_rows(case)
    compare(op.view(-1, case.N).cpu().numpy(), ref, den)


@pytest.mark.parametrize("S", [1, 2, 4])
@pytest.mark.parametrize("fmt", ALL)
def test_paged_decode_windows(fmt, S):
    case = synth.make_case(fmt, 6, S, 777, seed=150 + 4 * S + fmt, windows="decode",
                           min_context=1, page_size=64)
    op, oc = _paged_and_contiguous(case)
    assert torch.equal(op.view(torch.int32), oc.view(torch.int32))
    ref, den = oracle_rows(case)
    compare(op.view(-1, case.N).cpu().numpy(), ref, den)


@pytest.mark.parametrize("out_bf16", [False, True])
@pytest.mark.parametrize("S", [3, 5, 6, 7])
def test_paged_e4m3_partial_blocks(S, out_bf16):
    """Paged E4M3 four-row blocks (two epilogue groups on alternate tiles,
    each warp reducing two rows in turn) with a partial last block, several
    chunks per block and FP32 or BF16 logits: bit-equal to the contiguous
    call, and within the bound of the oracle."""
    import dataclasses
    case = synth.make_case(synth.FMT_E4M3, 2, S, 2600, seed=160 + S, windows="irregular",
                           page_size=64)
    flat = dataclasses.replace(case, page_size=0)
    tp = binding.case_to_device(case, out_bf16=out_bf16)
    tc = binding.case_to_device(flat, out_bf16=out_bf16)
    binding.run_case(case, tp)
    binding.run_case(flat, tc)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    assert torch.equal(tp["out"].view(torch.int16 if out_bf16 else torch.int32),
                       tc["out"].view(torch.int16 if out_bf16 else torch.int32))
    ref, den = oracle_rows(case)
    compare(tp["out"].float().view(-1, case.N).cpu().numpy(), ref, den,
            out_rounding=2.0 ** -8 if out_bf16 else 0.0)

"""BF16 logits output (IDX_FLAG_OUT_BF16).

Two bars. (1) Against the float64 oracle: the -inf pattern is exact and
in-window |gpu - ref| <= 2e-3 (1e-6 + den) + 2**-8 |ref|, the second term
being the rounding of a BF16 result (8-bit significand, half an ulp at the
bottom of a binade). (2) Against the same call with FP32 output: the BF16
logits are exactly the round-to-nearest-even of the FP32 ones (torch's
conversion), -inf included, since only the final store differs.
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, oracle_rows

pytestmark = pytest.mark.gpu

ALL = [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4]
BF16_ROUNDING = 2.0 ** -8


def _both(case, clean=None):
    t32 = binding.case_to_device(case)
    t16 = binding.case_to_device(case, out_bf16=True)
    t16["out"].fill_(7.0)
    binding.run_case(case, t32, clean=clean)
    binding.run_case(case, t16, clean=clean)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    return t32["out"], t16["out"]


@pytest.mark.parametrize("fmt", ALL)
def test_bf16_output_is_rounded_fp32_output(fmt):
    case = synth.make_case(fmt, 2, 64, 1000, seed=80 + fmt, windows="irregular")
    o32, o16 = _both(case)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("fmt", ALL)
def test_bf16_output_against_oracle(fmt):
    case = synth.make_case(fmt, 1, 96, 1500, seed=90 + fmt, windows="irregular")
    _, o16 = _both(case)
    ref, den = oracle_rows(case)
    compare(o16.float().view(-1, case.N).cpu().numpy(), ref, den, out_rounding=BF16_ROUNDING)


def test_bf16_output_padded_rows_untouched():
    case = synth.make_case(synth.FMT_E4M3, 1, 16, 300, seed=5, windows="causal")
    t = binding.case_to_device(case, out_row_stride=320, out_bf16=True)
    t["out"].fill_(3.0)
    binding.run_case(case, t)
    torch.cuda.synchronize()
    assert torch.all(t["out"][..., 300:] == 3.0)
    ref, den = oracle_rows(case)
    compare(t["out"][..., :300].float().reshape(-1, 300).cpu().numpy(), ref, den,
            out_rounding=BF16_ROUNDING)


def test_bf16_output_full_size_mxfp8():
    case = synth.make_workload("mxfp8_8192x65536")
    t = binding.case_to_device(case, out_bf16=True)
    binding.run_case(case, t)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    out = t["out"].view(-1, case.N)
    ks = torch.from_numpy(case.ks.reshape(-1).astype(np.int64)).cuda().clamp(0, case.N)
    ke = torch.from_numpy(case.ke.reshape(-1).astype(np.int64)).cuda().clamp(0, case.N)
    cols = torch.arange(case.N, device="cuda")[None, :]
    for r0 in range(0, out.shape[0], 512):
        sl = slice(r0, r0 + 512)
        outside = (cols < ks[sl, None]) | (cols >= ke[sl, None])
        assert torch.equal(torch.isneginf(out[sl]), outside), f"mask rows {r0}+"
    rows = np.array(sorted(set(range(0, case.S, 1024)) | {1, case.S - 1}), dtype=np.int64)
    ref, den = oracle_rows(case, rows=rows)
    compare(out[torch.from_numpy(rows).cuda()].float().cpu().numpy(), ref, den,
            out_rounding=BF16_ROUNDING)

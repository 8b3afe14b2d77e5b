"""Random combinations of the call's options against the float64 oracle.

Each seed draws a key format, W format, B, S, N, a window kind (random
windows with empty, inverted and out-of-range rows; causal; decode; full),
the sign and size of sm_scale, row grouping, FP32 or BF16 logits, contiguous
or paged keys (64-, 128- or 256-key pages), an output row stride above N,
and clean on or off. The call is checked on every row: the exact -inf
pattern (with clean), every in-window value within the bound, and the
padding columns past N left untouched. The targeted tests cover each option
on its own; this covers their combinations (two-row blocks with padded BF16
rows, paged keys with grouped rows, a negative scale with MXFP4 and clean
off, ...).
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, oracle_rows

pytestmark = pytest.mark.gpu

BF16_OUT_ROUNDING = 2.0 ** -8  # half an ulp of a BF16 logit at the bottom of its binade
SENTINEL = 12288.0             # padding columns must keep it (exact in FP32 and BF16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from infra_dsa_indexer_gb300 import build
    build.build()
    binding.load()
    yield
    assert binding.indexer_get_last_error() == binding.IDX_OK


def draw(seed):
    rng = np.random.default_rng(9000 + seed)
    fmt = int(rng.integers(0, 4))
    B = int(rng.integers(1, 4))
    S = int(rng.choice([1, 2, 3, 5, 8, 13]))
    N = int(rng.choice([1, 63, 127, 128, 129, 700, 1500, 2600]))
    kind = str(rng.choice(["random", "causal", "decode", "full"]))
    kw = dict(seed=9100 + seed,
              w_fmt=synth.W_BF16 if rng.random() < 0.3 else synth.W_F32,
              sm_scale=float((-1.0 if rng.random() < 0.3 else 1.0) * rng.uniform(0.02, 0.2)),
              page_size=int(rng.choice([0, 0, 64, 128, 192, 256])))
    if kind == "random":
        ks = rng.integers(-50, N + 50, size=(B, S))
        ke = ks + rng.integers(-100, N + 100, size=(B, S))
        kw.update(ks=ks.astype(np.int32), ke=ke.astype(np.int32),
                  group_rows=bool(rng.random() < 0.4))
    else:
        kw.update(windows=kind)
    case = synth.make_case(fmt, B, S, N, **kw)
    opts = dict(out_bf16=bool(rng.random() < 0.3), pad=int(rng.choice([0, 0, 8, 33])),
                clean=bool(rng.random() < 0.8))
    return case, opts


@pytest.mark.parametrize("seed", range(64))
def test_random_call_against_oracle(seed):
    case, o = draw(seed)
    t = binding.case_to_device(case, out_row_stride=case.N + o["pad"], out_bf16=o["out_bf16"])
    t["out"].fill_(SENTINEL)
    binding.run_case(case, t, clean=o["clean"])
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    out = t["out"].float()
    assert torch.all(out[..., case.N:] == SENTINEL), "a padding column was written"
    ref, den = oracle_rows(case)
    compare(out[..., :case.N].reshape(-1, case.N).cpu().numpy(), ref, den,
            check_outside=o["clean"],
            out_rounding=BF16_OUT_ROUNDING if o["out_bf16"] else 0.0,
            label=f"seed {seed}: fmt {case.fmt} B{case.B} S{case.S} N{case.N} {o}")

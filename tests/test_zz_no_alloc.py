"""indexer_logits_noalloc, the entry point for callers that may not allocate
device memory (code running inside a CUDA-graph capture, allocators that own
the memory pool, embedders with a fixed memory budget). It keeps its scratch
in a fixed device array inside the library instead of allocating it, and must
give the same logits as indexer_logits.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test. It also passes on its own in a
fresh process (the fixture builds and loads the library itself).
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from infra_dsa_indexer_gb300 import build
    build.build()
    binding.load()


def _call(fn, case, t, out):
    fn(t["q"], t["q_sf"], t["k"], t["k_sf"], t["k_scales"], t["w"], t["ks"], t["ke"],
       case.sm_scale, case.clean, out, t["shape"])


def test_noalloc_matches_indexer_logits_on_two_calls_in_a_row():
    # Two different problems back to back: the second call starts from the
    # words the first one left in the shared array.
    cases = [synth.make_case(synth.FMT_E4M3, 2, 48, 1500, seed=41, windows="causal"),
             synth.make_case(synth.FMT_BF16, 1, 64, 2100, seed=42, windows="causal_excl",
                             w_fmt=synth.W_BF16)]
    tens = [binding.case_to_device(c) for c in cases]
    refs = []
    for c, t in zip(cases, tens):
        out = torch.empty_like(t["out"])
        _call(binding.indexer_logits, c, t, out)
        refs.append(out)
    got = []
    for c, t in zip(cases, tens):
        out = torch.full_like(t["out"], 12345.0)
        _call(binding.indexer_logits_noalloc, c, t, out)
        got.append(out)
    torch.cuda.synchronize()
    assert binding.indexer_get_last_error() == binding.IDX_OK
    assert binding.indexer_noalloc_get_last_error() == binding.IDX_OK
    for c, ref_out, out in zip(cases, refs, got):
        # Same kernel, same grid and unit order, same inputs: the same bits.
        # A scratch-handling fault (a stale unit counter skipping or
        # repeating work) would show here even where values stay close.
        assert torch.equal(out.view(torch.int32), ref_out.view(torch.int32))
        a = out.cpu().numpy().reshape(-1, c.N)
        ref, den = oracle_rows(c)
        compare(a, ref, den)      # and both match the oracle within the parity bound

"""Failure detection on the device, without a GPU fault.

A device-side wait of the kind every role of the logits kernel uses is made
to run out on a barrier that nothing arrives on (a diagnostic entry point of
the library); the error word must report IDX_ERR_TIMEOUT, be cleared by the
read, and leave the context usable: a logits call right after on the same
stream matches the oracle.
"""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth
from parity import compare, oracle_rows

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_is_reported():
    binding.load()
    stream = torch.cuda.current_stream()
    binding.indexer_selftest_wait_timeout(2_000_000, stream)   # 2 ms
    assert binding.indexer_get_last_error(stream) == binding.IDX_ERR_TIMEOUT
    # the read cleared it
    assert binding.indexer_get_last_error(stream) == binding.IDX_OK


def test_context_usable_after_timeout():
    stream = torch.cuda.current_stream()
    binding.indexer_selftest_wait_timeout(1_000_000, stream)
    assert binding.indexer_get_last_error(stream) == binding.IDX_ERR_TIMEOUT
    case = synth.make_case(synth.FMT_MXFP8, 1, 64, 777, seed=31, windows="irregular")
    t = binding.case_to_device(case)
    binding.run_case(case, t, stream=stream)
    assert binding.indexer_get_last_error(stream) == binding.IDX_OK
    ref, den = oracle_rows(case)
    compare(t["out"].view(-1, case.N).cpu().numpy(), ref, den)


def test_selftest_rejects_out_of_range_limit():
    with pytest.raises(binding.IndexerError):
        binding.indexer_selftest_wait_timeout(10)
    with pytest.raises(binding.IndexerError):
        binding.indexer_selftest_wait_timeout(5_000_000_000)


def test_noalloc_wait_runs_out_and_is_reported():
    """The no-allocation entry point keeps its error word in its fixed device
    array; its own accessor reports a wait that ran out there, clears it, and
    the next no-allocation call on the stream is correct."""
    stream = torch.cuda.current_stream()
    binding.indexer_noalloc_selftest_wait_timeout(2_000_000, stream)
    assert binding.indexer_noalloc_get_last_error(stream) == binding.IDX_ERR_TIMEOUT
    assert binding.indexer_noalloc_get_last_error(stream) == binding.IDX_OK
    # the per-stream word of indexer_logits is a different word
    assert binding.indexer_get_last_error(stream) == binding.IDX_OK
    case = synth.make_case(synth.FMT_E4M3, 1, 40, 900, seed=33, windows="causal")
    t = binding.case_to_device(case)
    binding.indexer_logits_noalloc(t["q"], t["q_sf"], t["k"], t["k_sf"], t["k_scales"], t["w"],
                                   t["ks"], t["ke"], case.sm_scale, case.clean, t["out"],
                                   t["shape"], stream)
    assert binding.indexer_noalloc_get_last_error(stream) == binding.IDX_OK
    ref, den = oracle_rows(case)
    compare(t["out"].view(-1, case.N).cpu().numpy(), ref, den)


def test_stream_release_frees_and_later_calls_reallocate():
    s = torch.cuda.Stream()
    case = synth.make_case(synth.FMT_BF16, 1, 12, 300, seed=34, windows="causal")
    t = binding.case_to_device(case)
    with torch.cuda.stream(s):
        binding.run_case(case, t, stream=s)
        first = t["out"].clone()
        assert binding.indexer_stream_release(s) == binding.IDX_OK
        assert binding.indexer_get_last_error(s) == binding.IDX_OK   # no block: nothing to report
        binding.run_case(case, t, stream=s)                          # allocates again
        assert binding.indexer_get_last_error(s) == binding.IDX_OK
        assert torch.equal(t["out"].view(torch.int32), first.view(torch.int32))
        assert binding.indexer_stream_release(s) == binding.IDX_OK
    s.synchronize()

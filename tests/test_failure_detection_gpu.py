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

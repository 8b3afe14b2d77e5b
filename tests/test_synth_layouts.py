"""Input generators of the decode and paged workloads, on the CPU: the page
cache must hold exactly the logical keys (and key scales) at the rows its
block table names, and decode windows must end at each context."""
import dataclasses

import numpy as np
import pytest

from infra_dsa_indexer_gb300 import synth


def test_decode_windows_end_at_the_context():
    rng = np.random.Generator(np.random.PCG64(3))
    ks, ke = synth.decode_windows(rng, 5, 3, 1000, min_context=10)
    assert np.all(ks == 0)
    assert np.all(np.diff(ke, axis=1) == 1)                  # one more key per new token
    assert np.all(ke[:, -1] >= 10) and np.all(ke[:, -1] <= 1000)


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4])
@pytest.mark.parametrize("page_size", [64, 192])
def test_paged_layout_gathers_back_to_the_keys(fmt, page_size):
    case = synth.make_case(fmt, 3, 2, 500, seed=11, windows="decode", min_context=1,
                           page_size=page_size)
    pl = synth.paged_layout(case, page_size, seed=4)
    per = -(-case.N // page_size)
    table = pl["block_table"]
    assert table.shape == (case.B, pl["table_stride"]) and pl["table_stride"] >= per
    used = table[:, :per].reshape(-1)
    assert len(set(used.tolist())) == used.size                # distinct pages
    assert used.min() >= 0 and used.max() < pl["num_pages"]

    def gather(cache, b):
        rows = [cache[table[b, j // page_size], j % page_size] for j in range(case.N)]
        return np.stack(rows)

    kb = np.ascontiguousarray(case.k).view(np.uint8).reshape(case.B, case.N, -1)
    for b in range(case.B):
        assert np.array_equal(gather(pl["k_cache"], b), kb[b])
        if case.k_sf is not None:
            assert np.array_equal(gather(pl["k_sf_cache"], b), case.k_sf[b])
        if case.k_tok is not None:
            sc = np.array([pl["k_scales_cache"][table[b, j // page_size], j % page_size]
                           for j in range(case.N)])
            assert np.array_equal(sc, case.k_tok[b])


def test_paged_case_keeps_logical_keys_for_the_oracle():
    case = synth.make_case(synth.FMT_E4M3, 2, 1, 130, seed=2, windows="full", page_size=64)
    plain = dataclasses.replace(case, page_size=0)
    assert case.page_size == 64 and np.array_equal(case.k, plain.k)

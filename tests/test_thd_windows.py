"""Packed-sequence (THD) windows of the input generator, on the CPU."""
import numpy as np

from infra_dsa_indexer_gb300 import synth


def test_thd_windows_small_by_hand():
    ks, ke = synth.thd_windows([3, 2], [5, 4])
    assert ks.tolist() == [[0, 0, 0, 5, 5]]
    assert ke.tolist() == [[3, 4, 5, 8, 9]]


def test_thd_windows_stay_inside_their_sequence():
    lq, lk = (37, 64, 9, 1), (100, 256, 40, 7)
    ks, ke = synth.thd_windows(lq, lk)
    cq, ck = np.cumsum((0,) + lq), np.cumsum((0,) + lk)
    for s in range(len(lq)):
        rows = slice(cq[s], cq[s + 1])
        assert np.all(ks[0, rows] == ck[s])
        assert np.all(ke[0, rows] <= ck[s + 1]) and np.all(ke[0, rows] >= ck[s])
        assert ke[0, cq[s + 1] - 1] == ck[s + 1]            # last row sees all its keys
        assert np.all(np.diff(ke[0, rows]) == 1)             # one more key per row


def test_thd_windows_non_causal_and_short_keys():
    ks, ke = synth.thd_windows([4], [2], causal=False)
    assert ke.tolist() == [[2, 2, 2, 2]]
    ks, ke = synth.thd_windows([4], [2])
    assert ke.tolist() == [[0, 0, 1, 2]]                     # early rows see nothing

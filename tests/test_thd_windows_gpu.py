"""indexer_thd_windows: the packed-sequence (THD) windows built on the device
from cumulative lengths equal the input generator's windows (the same
definition written in numpy), causal and not, with empty sequences, keys
shorter than queries, and padding rows past the last sequence; a logits call
on windows built this way matches the call on the generator's windows."""
import numpy as np
import pytest
import torch

from infra_dsa_indexer_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def run(lq, lk, causal, pad=0):
    cq = torch.tensor(np.cumsum((0,) + tuple(lq)), dtype=torch.int32, device="cuda")
    ck = torch.tensor(np.cumsum((0,) + tuple(lk)), dtype=torch.int32, device="cuda")
    total = int(sum(lq)) + pad
    ks, ke = binding.indexer_thd_windows(cq, ck, total, causal=causal)
    torch.cuda.synchronize()
    return ks.cpu().numpy(), ke.cpu().numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lq,lk", [((3, 2), (5, 4)), ((37, 64, 9, 1), (100, 256, 40, 7)),
                                   ((4,), (2,)), ((5, 0, 7), (9, 3, 7)), ((1,) * 50, (3,) * 50)])
def test_device_windows_equal_the_definition(lq, lk, causal):
    ks, ke = run(lq, lk, causal)
    rks, rke = synth.thd_windows(lq, lk, causal=causal)
    assert np.array_equal(ks, rks) and np.array_equal(ke, rke)


def test_padding_rows_past_the_sequences_are_empty():
    ks, ke = run((3, 4), (6, 8), True, pad=5)
    assert np.all(ks[0, 7:] == 0) and np.all(ke[0, 7:] == 0)


def test_logits_on_device_built_windows():
    lq, lk = (100, 60, 40), (400, 240, 160)
    case = synth.make_case(synth.FMT_E4M3, 1, 200, 800, seed=77, windows="thd", thd=(lq, lk))
    t = binding.case_to_device(case)
    binding.run_case(case, t)
    ref = t["out"].clone()
    cq = torch.tensor(np.cumsum((0,) + lq), dtype=torch.int32, device="cuda")
    ck = torch.tensor(np.cumsum((0,) + lk), dtype=torch.int32, device="cuda")
    binding.indexer_thd_windows(cq, ck, case.S, causal=True, ks=t["ks"], ke=t["ke"])
    binding.run_case(case, t)
    torch.cuda.synchronize()
    assert torch.equal(t["out"].view(torch.int32), ref.view(torch.int32))

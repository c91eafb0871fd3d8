"""Failure detection without a GPU fault: a kernel's bounded barrier wait is made to run
out (nothing ever arrives; the CTA's abort flag goes up after a delay), the kernel
reports PISA_ERR_DEVICE_TIMEOUT in its status word, and the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
import pyramid_top_block_gb300 as pisa
from pyramid_top_block_gb300 import synth

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # PISA_ERR_DEVICE_TIMEOUT


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pisa.selftest_bounded_wait(ws, delay_cycles=2_000_000)  # about 1 ms
    assert pisa.check_device_status(ws) == TIMEOUT
    # the next call on the same context runs normally and reports no error
    q, k, w = synth.make("tiny-2k")
    pyr = pisa.build_pyramid(k.cuda())
    wsp = torch.empty(pisa.select_workspace_bytes(1, w["N"], w["Hq"], w["Hkv"], w["K"]), dtype=torch.uint8,
                      device="cuda")
    idx, _ = pisa.select_prefill(q.cuda(), pyr, w["K"], workspace=wsp, with_scores=False)
    torch.cuda.synchronize()
    assert pisa.check_device_status(wsp) == 0
    t = np.arange(0, w["N"], 61)
    orc = oracle.select(q[:, t].float().numpy(), k.float().numpy(), K=w["K"], t_list=t)
    ok = np.all(idx.cpu().numpy()[:, :, t] == orc["idx"], axis=-1) | (orc["min_gap"] < 1e-3)
    assert ok.all()


def test_a_zero_delay_still_times_out():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pisa.selftest_bounded_wait(ws, delay_cycles=0)
    assert pisa.check_device_status(ws) == TIMEOUT

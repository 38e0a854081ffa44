"""Failure detection of the executor's bounded waits, without a GPU fault.

MT_OPT_TEST_BARRIER_EXTRA makes every grid barrier of the runs started while
it is set wait for arrivals that never come (a flag nothing sets).  The
bounded wait must expire (~1 s), every CTA must return, the run must report
MT_ERR_TIMEOUT through mt_device_error(), and the context must stay usable:
a normal run afterwards gives the same result as before the failure.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_layers import DevLayer, plan_layer
from parity_util import dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def test_barrier_timeout_reports_and_recovers():
    import quantized_gemv_epilogues_gb300 as mt
    torch.cuda.set_device(0)
    wl = synth.TINY.with_(layers=2)
    layers = [plan_layer(DevLayer(mt, wl, l)) for l in range(2)]
    vals = dev_bf16(np.stack([synth.host_bf16(wl.d, synth.seed_for(wl.wid, l, synth.T_VALUES), synth.ACT)
                              for l in range(2)]))
    r0 = dev_bf16(synth.host_bf16(wl.d, synth.seed_for(wl.wid, 0, synth.T_RESIDUAL), synth.ACT))
    plan = mt.mt_mlp_plan_create(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps)
    try:
        mt.mt_device_error(True)
        y_ref = torch.empty(wl.d, dtype=torch.bfloat16, device="cuda")
        mt.mt_mlp_plan_run(plan, vals, r0, y_ref)
        torch.cuda.synchronize()
        assert mt.mt_device_error(False) == 0

        mt.mt_set_option(mt.MT_OPT_TEST_BARRIER_EXTRA, 1)
        try:
            y_bad = torch.empty(wl.d, dtype=torch.bfloat16, device="cuda")
            mt.mt_mlp_plan_run(plan, vals, r0, y_bad)
            torch.cuda.synchronize()  # returns: every CTA gave up and exited
        finally:
            mt.mt_set_option(mt.MT_OPT_TEST_BARRIER_EXTRA, 0)
        assert mt.mt_device_error(True) == mt.MT_ERR_TIMEOUT

        y = torch.empty(wl.d, dtype=torch.bfloat16, device="cuda")
        mt.mt_mlp_plan_run(plan, vals, r0, y)
        torch.cuda.synchronize()
        assert mt.mt_device_error(False) == 0
        assert np.array_equal(host_bits(y), host_bits(y_ref))
    finally:
        mt.mt_mlp_plan_destroy(plan)

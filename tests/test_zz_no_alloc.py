"""GPU test of mt_mlp_stack_run_noalloc, the stack pass whose scratch is the
library's static device array (no allocation in or around the call).

Collected last on purpose (file name), and also run alone in a fresh
process: the first call on the device does the one-time set-up either way.
Two calls in a row must both match the plan-based entry point
(mt_mlp_plan_run) on the same inputs: within the bf16 output tolerance, and in
fact bit for bit, since the kernel and its geometry are the same.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_layers import DevLayer, plan_layer
from parity_util import TOL_BF16, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    m.mt_device_error(True)
    return m


def _inputs(wl, n):
    vals = np.stack([synth.host_bf16(wl.d, synth.seed_for(wl.wid, l, synth.T_VALUES), synth.ACT)
                     for l in range(n)])
    r0 = synth.host_bf16(wl.d, synth.seed_for(wl.wid, 0, synth.T_RESIDUAL), synth.ACT)
    return dev_bf16(vals), dev_bf16(r0)


def _scaled_err(y, ref):
    y = y.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(y - ref)) / max(np.max(np.abs(ref)), 1e-30))


CASES = [
    synth.TINY.with_(layers=3),
    synth.TINY.with_(wid=11, name="stack d512 f1408 affine4 g32", d=512, f=1408,
                     fmt=synth.FMT_AFFINE4, group=32, layers=2),
    synth.TINY.with_(wid=12, name="stack d384 f1000 bf16", d=384, f=1000, fmt=synth.FMT_BF16,
                     group=0, eps=1e-6, layers=2),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name.replace(" ", "-"))
def test_noalloc_matches_plan(mt, wl):
    n = wl.layers
    layers = [plan_layer(DevLayer(mt, wl, l)) for l in range(n)]
    vals, r0 = _inputs(wl, n)
    ref = torch.empty(wl.d, dtype=torch.bfloat16, device="cuda")
    plan = mt.mt_mlp_plan_create(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps)
    try:
        mt.mt_mlp_plan_run(plan, vals, r0, ref)
        torch.cuda.synchronize()
    finally:
        mt.mt_mlp_plan_destroy(plan)
    for call in range(2):  # two calls in a row reuse the same static scratch
        y = torch.full((wl.d,), float("nan"), dtype=torch.bfloat16, device="cuda")
        mt.mt_mlp_stack_run_noalloc(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps, vals, r0, y)
        torch.cuda.synchronize()
        assert mt.mt_device_error(False) == 0
        err = _scaled_err(y, ref)
        assert err <= TOL_BF16, f"call {call}: max|y - y_plan| / max|y_plan| = {err:.3e}"
        assert np.array_equal(host_bits(y), host_bits(ref)), f"call {call}: not bit-identical to the plan"


def _plan_ref(mt, wl, layers, vals, r0):
    ref = torch.empty(wl.d, dtype=torch.bfloat16, device="cuda")
    plan = mt.mt_mlp_plan_create(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps)
    try:
        mt.mt_mlp_plan_run(plan, vals, r0, ref)
        torch.cuda.synchronize()
    finally:
        mt.mt_mlp_plan_destroy(plan)
    return ref


def test_noalloc_table_in_two_chunks(mt):
    """50 layers: the table reaches the device in two parameter blocks (48 + 2
    entries); the result is the plan's, bit for bit."""
    wl = synth.TINY.with_(layers=50)
    layers = [plan_layer(DevLayer(mt, wl, l)) for l in range(wl.layers)]
    vals, r0 = _inputs(wl, wl.layers)
    ref = _plan_ref(mt, wl, layers, vals, r0)
    y = torch.full((wl.d,), float("nan"), dtype=torch.bfloat16, device="cuda")
    mt.mt_mlp_stack_run_noalloc(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps, vals, r0, y)
    torch.cuda.synchronize()
    assert mt.mt_device_error(False) == 0
    assert np.array_equal(host_bits(y), host_bits(ref))


def test_noalloc_captured_in_a_graph(mt):
    """The call captured into a CUDA graph (after a first call outside any
    capture) and replayed on new contents of the same input buffers: each
    replay gives the plan's result on those contents, bit for bit."""
    wl = synth.TINY.with_(wid=13, layers=3)
    n = wl.layers
    layers = [plan_layer(DevLayer(mt, wl, l)) for l in range(n)]
    vals, r0 = _inputs(wl, n)
    y = torch.empty(wl.d, dtype=torch.bfloat16, device="cuda")
    mt.mt_mlp_stack_run_noalloc(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps, vals, r0, y)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mt.mt_mlp_stack_run_noalloc(layers, wl.d, wl.f, wl.group, wl.fmt, wl.eps, vals, r0, y)
    torch.cuda.synchronize()
    for trial in range(2):
        v = np.stack([synth.host_bf16(wl.d, 52000 + 10 * trial + l, synth.ACT) for l in range(n)])
        vals.copy_(dev_bf16(v))
        r0.copy_(dev_bf16(synth.host_bf16(wl.d, 52100 + trial, synth.ACT)))
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert mt.mt_device_error(False) == 0
        ref = _plan_ref(mt, wl, layers, vals, r0)
        assert np.array_equal(host_bits(y), host_bits(ref)), f"replay {trial}"


def test_noalloc_rejects_scratch_overflow(mt):
    """A layer table larger than the static scratch is refused before any
    device work (4096 layers x 80 bytes > MT_STACK_SCRATCH_BYTES)."""
    wl = synth.TINY
    ly = plan_layer(DevLayer(mt, wl, 0))
    L = 4096
    vals = torch.zeros(L, wl.d, dtype=torch.bfloat16, device="cuda")
    r0 = torch.zeros(wl.d, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(wl.d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mt.MTError) as e:
        mt.mt_mlp_stack_run_noalloc([ly] * L, wl.d, wl.f, wl.group, wl.fmt, wl.eps, vals, r0, y)
    assert e.value.status == mt.MT_ERR_SHAPE

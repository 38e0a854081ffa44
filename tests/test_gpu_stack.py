"""GPU parity of the warmed executor (mt_mlp_plan_create / run / destroy): L
one-row decode MLP layers run back to back by one persistent kernel.

Every layer's four tensors are traced and checked on the executor's own inputs
(the way each single-call kernel is checked): summed bit-exact against the
oracle's add, the normalised row, h and y within the bf16 tolerance of the
oracle fed the executor's previous tensor.  The executor must also agree bit
for bit with the single-call kernels on the same inputs (the same row
partition and reduction order), return the traced last y as out_y, and give
the same out_y with and without tracing.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_layers import DevLayer, plan_layer
from parity_util import assert_bf16_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    m.mt_set_option(m.MT_OPT_GEMV, 0)
    m.mt_set_option(m.MT_OPT_PDL, 1)
    assert m.mt_device_error(True) == 0
    return m


def _acts(wl, n_layers):
    vals = np.stack([synth.host_bf16(wl.d, synth.seed_for(wl.wid, l, synth.T_VALUES), synth.ACT)
                     for l in range(n_layers)])
    r0 = synth.host_bf16(wl.d, synth.seed_for(wl.wid, 0, synth.T_RESIDUAL), synth.ACT)
    return vals, r0


def _run(mt, plan, wl, n_layers, vals_d, r0_d, trace=True):
    d, f = wl.d, wl.f
    bf = torch.bfloat16
    out_y = torch.empty(d, dtype=bf, device="cuda")
    tr = None
    if trace:
        tr = dict(out_sum=torch.empty(n_layers, d, dtype=bf, device="cuda"),
                  out_norm=torch.empty(n_layers, d, dtype=bf, device="cuda"),
                  h=torch.empty(n_layers, f, dtype=bf, device="cuda"),
                  y=torch.empty(n_layers, d, dtype=bf, device="cuda"))
    mt.mt_mlp_plan_run(plan, vals_d, r0_d, out_y, tr)
    torch.cuda.synchronize()
    assert mt.mt_device_error(False) == 0
    return out_y, tr


def _single_call_check(mt, wl, L, tr, l):
    """h_l and y_l equal the single-call kernels' results on the traced inputs."""
    d, f = wl.d, wl.f
    h1 = torch.empty(1, f, dtype=torch.bfloat16, device="cuda")
    y1 = torch.empty(1, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_swiglu_gateup(tr["out_norm"][l:l + 1], L.Wg, L.Wu, L.sgu, L.bgu, wl.group, h1, fmt=wl.fmt)
    mt.mt_down_residual(tr["h"][l:l + 1], L.Wd, L.sdn, L.bdn, wl.group, tr["out_sum"][l:l + 1], y1,
                        fmt=wl.fmt)
    torch.cuda.synchronize()
    assert torch.equal(h1[0], tr["h"][l]), f"layer {l}: h differs from mt_swiglu_gateup"
    assert torch.equal(y1[0], tr["y"][l]), f"layer {l}: y differs from mt_down_residual"


SMALL = [
    synth.TINY.with_(layers=3),
    synth.TINY.with_(wid=11, name="stack d512 f1408 affine4 g32", d=512, f=1408,
                     fmt=synth.FMT_AFFINE4, group=32, layers=2),
    synth.TINY.with_(wid=12, name="stack d384 f1000 bf16", d=384, f=1000, fmt=synth.FMT_BF16,
                     group=0, eps=1e-6, layers=2),
    synth.TINY.with_(wid=13, name="stack d1024 f2816 affine8 g128", d=1024, f=2816, group=128,
                     eps=1e-6, layers=2),
    synth.TINY.with_(wid=14, name="stack d96 f224 affine8 g32", d=96, f=224, group=32, layers=2),
    # gate/up rows of 64 chunks (two rows per load stream), down rows of 32
    synth.TINY.with_(wid=15, name="stack d2048 f1024 affine4 g128", d=2048, f=1024,
                     fmt=synth.FMT_AFFINE4, group=128, eps=1e-6, layers=2),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name.replace(" ", "-"))
def test_stack_small(mt, wl):
    _check_stack(mt, wl)


@pytest.mark.parametrize("wl", [SMALL[1], SMALL[3]], ids=lambda w: w.name.replace(" ", "-"))
def test_stack_act_bits_24(mt, wl):
    """A plan created while MT_OPT_ACT_BITS is 24 stages x and h in 24-bit
    fixed point: parity, and bit-identity with the single calls made with the
    same option."""
    mt.mt_set_option(mt.MT_OPT_ACT_BITS, 24)
    try:
        _check_stack(mt, wl)
    finally:
        mt.mt_set_option(mt.MT_OPT_ACT_BITS, 16)


def _check_stack(mt, wl):
    n = wl.layers
    layers = [DevLayer(mt, wl, l) for l in range(n)]
    vals, r0 = _acts(wl, n)
    plan = mt.mt_mlp_plan_create([plan_layer(L) for L in layers], wl.d, wl.f, wl.group, wl.fmt, wl.eps)
    try:
        out_y, tr = _run(mt, plan, wl, n, dev_bf16(vals), dev_bf16(r0))
        out_y2, _ = _run(mt, plan, wl, n, dev_bf16(vals), dev_bf16(r0), trace=False)
    finally:
        mt.mt_mlp_plan_destroy(plan)
    assert torch.equal(out_y, tr["y"][n - 1]), "out_y is not the last traced y"
    assert torch.equal(out_y, out_y2), "tracing changed the result"
    r = r0
    for l, L in enumerate(layers):
        d, f = wl.d, wl.f
        w = synth.host_bf16(d, L.sd(synth.T_NORM_W), synth.NORM_W)
        s_ref, norm_x = oracle.add_rmsnorm(vals[l][None], r[None], w, wl.eps)
        s_gpu = host_bits(tr["out_sum"][l])
        assert np.array_equal(s_gpu, s_ref[0]), f"layer {l}: summed not bit-exact"
        assert_bf16_close(host_bits(tr["out_norm"][l]), norm_x[0], f"layer {l} out_norm")
        Wg = L.oracle_rows(synth.T_WG, range(f), f, d)
        Wu = L.oracle_rows(synth.T_WU, range(f), f, d)
        Wd = L.oracle_rows(synth.T_WD, range(d), d, f)
        h_ref = oracle.swiglu_gateup(host_bits(tr["out_norm"][l])[None], Wg, Wu)
        assert_bf16_close(host_bits(tr["h"][l]), h_ref[0], f"layer {l} h")
        y_ref = oracle.down_residual(host_bits(tr["h"][l])[None], Wd, s_gpu[None])
        assert_bf16_close(host_bits(tr["y"][l]), y_ref[0], f"layer {l} y")
        _single_call_check(mt, wl, L, tr, l)
        r = host_bits(tr["y"][l])


def test_stack_qwen3_8b(mt):
    """The 36-layer 4096 x 12288 affine INT8 g128 stack at full size, in the
    bench's launch configuration: all 36 layers bit-exact against the
    single-call kernels on the traced inputs, summed bit-exact against the
    oracle's add on every layer, and oracle parity of every output on layers
    0, 17 and 35 (sampled rows of h and y, the whole normalised row)."""
    wl = synth.QWEN8B
    n, d, f = wl.layers, wl.d, wl.f
    layers = [DevLayer(mt, wl, l) for l in range(n)]
    vals, r0 = _acts(wl, n)
    plan = mt.mt_mlp_plan_create([plan_layer(L) for L in layers], d, f, wl.group, wl.fmt, wl.eps)
    try:
        out_y, tr = _run(mt, plan, wl, n, dev_bf16(vals), dev_bf16(r0))
        out_y2, _ = _run(mt, plan, wl, n, dev_bf16(vals), dev_bf16(r0), trace=False)
    finally:
        mt.mt_mlp_plan_destroy(plan)
    assert torch.equal(out_y, tr["y"][n - 1])
    assert torch.equal(out_y, out_y2)
    rng = np.random.default_rng(3)
    r = r0
    for l, L in enumerate(layers):
        w = synth.host_bf16(d, L.sd(synth.T_NORM_W), synth.NORM_W)
        s_ref, norm_x = oracle.add_rmsnorm(vals[l][None], r[None], w, wl.eps)
        s_gpu = host_bits(tr["out_sum"][l])
        assert np.array_equal(s_gpu, s_ref[0]), f"layer {l}: summed not bit-exact"
        _single_call_check(mt, wl, L, tr, l)
        if l in (0, 17, 35):
            assert_bf16_close(host_bits(tr["out_norm"][l]), norm_x[0], f"layer {l} out_norm")
            rg = np.sort(rng.choice(f, 48, replace=False))
            rd = np.sort(rng.choice(d, 48, replace=False))
            h_ref = oracle.swiglu_gateup(host_bits(tr["out_norm"][l])[None],
                                         L.oracle_rows(synth.T_WG, rg, f, d),
                                         L.oracle_rows(synth.T_WU, rg, f, d))
            y_ref = oracle.down_residual(host_bits(tr["h"][l])[None], L.oracle_rows(synth.T_WD, rd, d, f),
                                         s_gpu[None, rd])
            # sampled rows are judged against the sample's own scale
            assert_bf16_close(host_bits(tr["h"][l])[rg], h_ref[0], f"layer {l} h (sampled)")
            assert_bf16_close(host_bits(tr["y"][l])[rd], y_ref[0], f"layer {l} y (sampled)")
        r = host_bits(tr["y"][l])
    del layers
    torch.cuda.empty_cache()


def test_plan_argument_errors(mt):
    """Invalid runs are refused before anything is launched."""
    wl = synth.TINY
    L = DevLayer(mt, wl, 0)
    plan = mt.mt_mlp_plan_create([plan_layer(L)], wl.d, wl.f, wl.group, wl.fmt, wl.eps)
    try:
        v = torch.zeros(1, wl.d, dtype=torch.bfloat16, device="cuda")
        y = torch.zeros(wl.d, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(mt.MTError) as e:
            mt.mt_mlp_plan_run(plan, v, y, v[0])  # out_y overlaps values
        assert e.value.status == mt.MT_ERR_ALIAS
        with pytest.raises(mt.MTError) as e:
            mt.mt_mlp_plan_run(plan, v, y, y.data_ptr() + 2)  # misaligned out_y
        assert e.value.status == mt.MT_ERR_ALIGN
        mt.mt_mlp_plan_run(plan, v, y, y)  # out_y may equal residual
        torch.cuda.synchronize()
    finally:
        mt.mt_mlp_plan_destroy(plan)

"""GPU parity at the measured workloads' full sizes, in the launch
configuration the bench uses (one-row warp-task kernel, programmatic dependent
launch on, weights generated and packed on the device).

The oracle never sees device data: it regenerates the rows it needs from the
seeded generator on the host and quantises them itself.  Where checking every
output is cheap the whole output is compared; for the 36-layer Qwen3-8B stack
one full layer is checked end to end and sampled rows of a second layer.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_layers import DevLayer, full_oracle_layer, host_acts, run_layer
from parity_util import assert_bf16_close, assert_f32_close, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    m.mt_set_option(m.MT_OPT_GEMV, 0)
    m.mt_set_option(m.MT_OPT_PDL, 1)
    return m


@pytest.mark.parametrize("wl", [synth.LLAMA1B, synth.QWEN15, synth.TINY], ids=lambda w: w.name.split()[0])
def test_layer_full(mt, wl):
    """Every output of one layer: the chained layer, and each kernel on the
    oracle's own inputs (so each kernel is judged on its own error)."""
    M = wl.M
    L = DevLayer(mt, wl, 0)
    v, r, w = host_acts(wl, 0, M)
    ref, (Wg, Wu, Wd) = full_oracle_layer(L, v, r, w)
    out_sum, out_norm, h, y = run_layer(mt, L, dev_bf16(v), dev_bf16(r), M)
    assert np.array_equal(host_bits(L.w), w), "device and host generators differ"
    assert np.array_equal(host_bits(out_sum), ref["out_sum"])
    assert_bf16_close(host_bits(out_norm), ref["norm_x"], "out_norm")
    assert_bf16_close(host_bits(y), ref["y_x"], "y (chained)")
    # gate/up and down on the oracle's own rounded inputs
    h2 = torch.empty(M, wl.f, dtype=torch.float32, device="cuda")
    mt.mt_swiglu_gateup(dev_bf16(ref["out_norm"]), L.Wg, L.Wu, L.sgu, L.bgu, wl.group, h2, fmt=wl.fmt)
    y2 = torch.empty(M, wl.d, dtype=torch.float32, device="cuda")
    mt.mt_down_residual(dev_bf16(ref["h"]), L.Wd, L.sdn, L.bdn, wl.group, dev_bf16(ref["out_sum"]), y2,
                        fmt=wl.fmt)
    torch.cuda.synchronize()
    assert_f32_close(host_f64(h2), ref["h_x"], "h (fp32 out, oracle input)")
    assert_f32_close(host_f64(y2), oracle.down_residual(ref["h"], Wd, ref["out_sum"]), "y (fp32 out, oracle input)")


def test_qwen3_8b_stack_layers(mt):
    """The 4096 x 12288 affine INT8 g128 layer at full size: layer 0 end to
    end (every output), layer 35 on sampled rows; packed bytes of sampled rows
    bit-exact."""
    wl = synth.QWEN8B
    d, f, M, g = wl.d, wl.f, wl.M, wl.group
    L0 = DevLayer(mt, wl, 0)
    v, r, w = host_acts(wl, 0, M)
    ref, (Wg, Wu, Wd) = full_oracle_layer(L0, v, r, w)
    out_sum, out_norm, h, y = run_layer(mt, L0, dev_bf16(v), dev_bf16(r), M)
    assert np.array_equal(host_bits(out_sum), ref["out_sum"])
    assert_bf16_close(host_bits(out_norm), ref["norm_x"], "out_norm")
    assert_bf16_close(host_bits(y), ref["y_x"], "y (chained)")
    h2 = torch.empty(M, f, dtype=torch.float32, device="cuda")
    mt.mt_swiglu_gateup(dev_bf16(ref["out_norm"]), L0.Wg, L0.Wu, L0.sgu, L0.bgu, g, h2, fmt=wl.fmt)
    torch.cuda.synchronize()
    assert_f32_close(host_f64(h2), ref["h_x"], "h (fp32 out, oracle input)")
    # packed layout of sampled rows, bit for bit
    rows = np.random.default_rng(0).choice(f, 24, replace=False)
    for n in rows:
        assert np.array_equal(L0.Wg[n].cpu().numpy(), oracle.pack_codes(Wg.W[n:n + 1], 8)[0])
        assert np.array_equal(host_bits(L0.sgu[0, n]), Wg.scales[n])
        assert np.array_equal(host_bits(L0.bgu[1, n]), Wu.biases[n])
    del L0
    torch.cuda.empty_cache()

    # the last layer of the stack: sampled outputs on generator inputs
    L = DevLayer(mt, wl, 35)
    x = synth.host_bf16(d, synth.seed_for(wl.wid, 35, synth.T_X), synth.ACT).reshape(1, d)
    hin = synth.host_bf16(f, synth.seed_for(wl.wid, 35, synth.T_H), synth.ACT).reshape(1, f)
    res = synth.host_bf16(d, synth.seed_for(wl.wid, 35, synth.T_RES3), synth.ACT).reshape(1, d)
    hg = torch.empty(1, f, dtype=torch.float32, device="cuda")
    yd = torch.empty(1, d, dtype=torch.float32, device="cuda")
    mt.mt_swiglu_gateup(dev_bf16(x), L.Wg, L.Wu, L.sgu, L.bgu, g, hg, fmt=wl.fmt)
    mt.mt_down_residual(dev_bf16(hin), L.Wd, L.sdn, L.bdn, g, dev_bf16(res), yd, fmt=wl.fmt)
    torch.cuda.synchronize()
    rg = np.sort(np.random.default_rng(1).choice(f, 64, replace=False))
    rd = np.sort(np.random.default_rng(2).choice(d, 64, replace=False))
    h_ref = oracle.swiglu_gateup(x, L.oracle_rows(synth.T_WG, rg, f, d), L.oracle_rows(synth.T_WU, rg, f, d))
    y_ref = oracle.down_residual(hin, L.oracle_rows(synth.T_WD, rd, d, f), res[:, rd])
    assert_f32_close(host_f64(hg)[:, rg], h_ref, "h sampled rows, layer 35")
    assert_f32_close(host_f64(yd)[:, rd], y_ref, "y sampled rows, layer 35")


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_sweep_point(mt, group, M):
    """d=2048, f=8192 affine INT8 with 1 % x20 outliers: every output of the
    gate/up and down kernels on generator inputs, bf16 and fp32 outputs."""
    wl = synth.sweep_point(group, M)
    d, f = wl.d, wl.f
    L = DevLayer(mt, wl, 0)
    x = synth.host_bf16(M * d, synth.seed_for(wl.wid, M, synth.T_X), synth.ACT).reshape(M, d)
    hin = synth.host_bf16(M * f, synth.seed_for(wl.wid, M, synth.T_H), synth.ACT).reshape(M, f)
    res = synth.host_bf16(M * d, synth.seed_for(wl.wid, M, synth.T_RES3), synth.ACT).reshape(M, d)
    Wg = L.oracle_rows(synth.T_WG, range(f), f, d)
    Wu = L.oracle_rows(synth.T_WU, range(f), f, d)
    Wd = L.oracle_rows(synth.T_WD, range(d), d, f)
    h_ref = oracle.swiglu_gateup(x, Wg, Wu)
    y_ref = oracle.down_residual(hin, Wd, res)
    for out_f32 in (False, True):
        dt = torch.float32 if out_f32 else torch.bfloat16
        h = torch.empty(M, f, dtype=dt, device="cuda")
        y = torch.empty(M, d, dtype=dt, device="cuda")
        mt.mt_swiglu_gateup(dev_bf16(x), L.Wg, L.Wu, L.sgu, L.bgu, group, h, fmt=wl.fmt)
        mt.mt_down_residual(dev_bf16(hin), L.Wd, L.sdn, L.bdn, group, dev_bf16(res), y, fmt=wl.fmt)
        torch.cuda.synchronize()
        if out_f32:
            assert_f32_close(host_f64(h), h_ref, "h")
            assert_f32_close(host_f64(y), y_ref, "y")
        else:
            assert_bf16_close(host_bits(h), h_ref, "h")
            assert_bf16_close(host_bits(y), y_ref, "y")

"""The seeded input generator: determinism, sub-range regeneration, the
distribution shapes the workloads ask for, and host == device bit equality."""
import numpy as np
import pytest
import torch

import synth


def test_deterministic_and_offsets():
    a = synth.host_f32(10000, 42, synth.ACT)
    b = synth.host_f32(10000, 42, synth.ACT)
    assert np.array_equal(a, b)
    c = synth.host_f32(3000, 42, synth.ACT, offset=5000)
    assert np.array_equal(a[5000:8000], c)
    assert not np.array_equal(a, synth.host_f32(10000, 43, synth.ACT))


def test_distributions():
    z = synth.host_f32(1 << 20, 7, synth.ACT).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    assert np.abs(z).max() <= 6.0
    # Irwin-Hall(12) is close to normal: tail mass beyond 3 sigma ~ 0.27%
    assert 0.0015 < np.mean(np.abs(z) > 3.0) < 0.0040
    w = synth.host_f32(1 << 20, 8, synth.WEIGHT).astype(np.float64)
    assert abs(w.std() - 0.02) < 2e-4
    nw = synth.host_f32(1 << 18, 9, synth.NORM_W).astype(np.float64)
    assert abs(nw.mean() - 1.0) < 2e-3 and abs(nw.std() - 0.1) < 2e-3
    wo = synth.host_f32(1 << 20, 8, synth.WEIGHT_OUTLIERS)
    frac = np.mean(wo != w.astype(np.float32))
    assert 0.009 < frac < 0.011
    sel = wo != w.astype(np.float32)
    assert np.allclose(wo[sel], w[sel].astype(np.float32) * np.float32(20.0))


def test_bf16_storage_is_round_to_nearest_even():
    f = synth.host_f32(100000, 11, synth.ACT)
    b = synth.host_bf16(100000, 11, synth.ACT)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)


def test_workload_byte_counts():
    # packed weights + scale/bias + activations of one layer
    assert synth.QWEN8B.layer_bytes() == 155_828_224
    assert synth.TINY.layer_bytes() == 633_856
    assert synth.LLAMA1B.layer_bytes() == 28_377_088
    assert synth.QWEN15.layer_bytes() == 82_635_776


@pytest.mark.gpu
@pytest.mark.parametrize("dist", [synth.ACT, synth.WEIGHT, synth.NORM_W, synth.WEIGHT_OUTLIERS])
def test_device_equals_host(dist):
    synth.build()
    n = 300_001
    t = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.device_f32(t, 1234, dist, offset=777)
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), synth.host_f32(n, 1234, dist, offset=777))
    tb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    synth.device_bf16(tb, 99, dist)
    torch.cuda.synchronize()
    assert np.array_equal(tb.cpu().view(torch.int16).numpy().view(np.uint16), synth.host_bf16(n, 99, dist))

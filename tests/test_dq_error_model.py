"""The error model of the dequantising prefill path, checked on the CPU
against the float64 oracle (no GPU, no CUDA code): a plain numpy model that
rounds each affine weight once to fp16 after a per-row power-of-two scale
(max over the row's groups of |s| (2^bits - 1) + |b| times 2^t in [2^14, 2^15))
and each activation once to fp16 after a per-row power-of-two scale
(max |x_m| 2^e in [2^14, 2^15)), then sums exactly.  Pins:
  * the row scale keeps every scaled weight below 2^15 (no fp16 overflow),
  * |y_model - y*| <= 2^-11 sum_k |w x| + 2^-11 sum_k |w x| (weights, then
    activations: each bf16 activation above 2^-28 of its row maximum is
    exact in fp16, so the second term is far looser than needed),
  * a weight matrix whose rows differ by 2^80 in magnitude keeps each row's
    relative precision (a single scale for all rows would not)."""
import numpy as np
import pytest

import oracle
import synth


def _pow2_scale(m, clamp=None):
    """t with m 2^t in [2^14, 2^15) (0 for m == 0); clamp: the kernel's
    range of t for the weight rows, [-126, 126] (2^t a normal fp32)."""
    m = np.asarray(m, dtype=np.float64)
    e = np.floor(np.log2(np.where(m > 0, m, 1.0)))
    t = np.where(m > 0, 14 - e, 0.0)
    return t if clamp is None else np.clip(t, -clamp, clamp)


def _model(x_bits, W: oracle.Weight, bits: int):
    w = W.dense()
    s = oracle.f64_from_bf16(W.scales)
    b = oracle.f64_from_bf16(W.biases)
    bound = (np.abs(s) * (2 ** bits - 1) + np.abs(b)).max(axis=1)
    t = _pow2_scale(bound, clamp=126)
    ws = w * np.exp2(t)[:, None]
    assert np.abs(ws).max() < 2.0 ** 15, "scaled weight beyond the fp16 plan"
    wq = ws.astype(np.float16).astype(np.float64) * np.exp2(-t)[:, None]
    x = oracle.f64_from_bf16(x_bits)
    ex = _pow2_scale(np.abs(x).max(axis=1))
    xq = (x * np.exp2(ex)[:, None]).astype(np.float16).astype(np.float64) * np.exp2(-ex)[:, None]
    return xq @ wq.T, np.abs(x) @ np.abs(w).T


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 128, 6, 512, 40), (8, 32, 5, 256, 33), (4, 64, 7, 384, 24)])
def test_dq_bound_holds(bits, group, M, K, N):
    seed = 41000 + bits + group + K
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    W = oracle.Weight.from_f32(synth.host_f32(N * K, seed + 1, synth.WEIGHT_OUTLIERS).reshape(N, K), bits, group)
    y, mag = _model(x, W, bits)
    ref = oracle.linear_bias(x, W)
    assert np.all(np.abs(y - ref) <= 2.0 ** -10 * mag + 1e-300)
    # and the model is not trivially exact: the fp16 rounding is visible
    assert np.abs(y - ref).max() > 0


def test_dq_rows_far_apart():
    bits, group, M, K, N = 8, 64, 4, 256, 48
    x = synth.host_bf16(M * K, 41900, synth.ACT).reshape(M, K)
    W32 = synth.host_f32(N * K, 41901, synth.WEIGHT).reshape(N, K)
    W32 = (W32 * np.exp2(np.linspace(-40, 40, N))[:, None]).astype(np.float32)
    W = oracle.Weight.from_f32(W32, bits, group)
    y, mag = _model(x, W, bits)
    ref = oracle.linear_bias(x, W)
    # each output column (one weight row) within 2^-10 of its own magnitude
    assert np.all(np.abs(y - ref) <= 2.0 ** -10 * mag)
    # one scale for the whole matrix (the largest row's) flushes the small rows
    w = W.dense()
    t_all = _pow2_scale(np.abs(w).max())
    wq = (w * 2.0 ** t_all).astype(np.float16).astype(np.float64) * 2.0 ** -t_all
    assert np.count_nonzero(wq[0]) == 0 and np.count_nonzero(w[0]) > 0


def test_dq_rows_near_the_bottom_of_the_range():
    """Rows scaled by 2^-120 (bf16 scales near the bottom of the normal range
    and below): t is clamped to 126, and each row still keeps its relative
    precision next to rows of ordinary and large magnitude."""
    bits, group, M, K, N = 8, 64, 3, 256, 24
    x = synth.host_bf16(M * K, 41950, synth.ACT).reshape(M, K)
    W32 = synth.host_f32(N * K, 41951, synth.WEIGHT).reshape(N, K).astype(np.float64)
    W32 = (W32 * np.exp2(np.linspace(-120, 60, N))[:, None]).astype(np.float32)
    W = oracle.Weight.from_f32(W32, bits, group)
    s = oracle.f64_from_bf16(W.scales)
    assert s[0].max() < 2.0 ** -120  # the smallest row's scales are bf16 subnormals
    y, mag = _model(x, W, bits)
    ref = oracle.linear_bias(x, W)
    assert np.all(np.abs(y - ref) <= 2.0 ** -10 * mag)

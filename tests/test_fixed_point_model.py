"""The error model of the one-row kernels' fixed-point activations, checked on
the CPU against the float64 oracle (no GPU, no CUDA code).  The kernels hold
x as X = round(x 2^e), nearest-even, with ONE power of two per vector chosen
from its largest |x| so that max|x| 2^e lies in [2^(8 PL - 3), 2^(8 PL - 2)),
PL = 2 bytes for bf16 outputs and PL = 3 for fp32 outputs, and every code.X
product and chunk sum is exact.  Pins:
  * |X| <= 2^(8 PL - 2): X fits the signed range of PL bytes,
  * every bf16 x within 2^(8 PL - 10) of the vector's maximum is represented
    exactly (2^6 for 16 bits, 2^14 for 24 bits),
  * the perturbation of y = x.W that the rounding of the smaller elements
    causes, as a scale-normalised max error, stays within a fraction of each
    output precision's bound on activations with 1 % x20 outliers, for INT8
    and INT4 weights of every group: half of 2e-3 for 16 bits (bf16 outputs;
    measured 3-6e-4 here, 1e-5 without outliers), a twentieth of 1e-5 for 24
    bits (fp32 outputs).  The 16-bit error grows with max|x| / rms(x), about
    (max|x| / rms(x)) 1.2e-5 in this model; that ratio is at most sqrt(K).
  * a vector with one channel 1000x the rest (max|x| / rms(x) near sqrt(K)):
    24 bits keep y within a twentieth of the bf16 bound, while 16 bits
    exceed the bound at K = 12288 (the limitation MT_OPT_ACT_BITS = 24 is
    for: the output row with the largest |y| is set by the other channels,
    whose fixed-point step is set by the large one)."""
import numpy as np
import pytest

import oracle
import synth


def _fixed_point(x, PL):
    """X and the exponent e as the kernels form them from bf16 values x (one
    vector): e = (8 PL - 3) - floor(log2 max|x|), clamped to [-126, 126]."""
    m = np.abs(x).max()
    e = 126 if m == 0 else int(np.clip((8 * PL - 3) - np.floor(np.log2(m)), -126, 126))
    X = np.rint(x * np.exp2(e))  # nearest-even, as the kernels' magic-number rounding
    return X, e


def _activations(K, seed, outliers):
    x = oracle.f64_from_bf16(synth.host_bf16(K, seed, synth.ACT))
    if outliers:  # 1 % of the elements x20, as the outlier weight distribution
        rng = np.random.default_rng(seed)
        idx = rng.choice(K, size=max(1, K // 100), replace=False)
        x[idx] *= 20.0
        x = oracle.f64_from_bf16(oracle.bf16_from_f64(x))
    return x


@pytest.mark.parametrize("PL", [2, 3])
@pytest.mark.parametrize("K,seed", [(2048, 1), (4096, 2), (12288, 3)])
@pytest.mark.parametrize("outliers", [False, True])
def test_range_and_exact_elements(PL, K, seed, outliers):
    x = _activations(K, seed, outliers)
    X, e = _fixed_point(x, PL)
    assert np.abs(X).max() <= 2.0 ** (8 * PL - 2)
    assert np.abs(X).max() >= 2.0 ** (8 * PL - 3)
    E = np.floor(np.log2(np.abs(x).max()))
    near = np.abs(x) >= 2.0 ** (E - (8 * PL - 10))
    xq = X * np.exp2(-e)
    assert np.array_equal(xq[near], x[near])
    # below that, the rounding is at most half a fixed-point step
    assert np.abs(xq - x).max() <= 0.5 * 2.0 ** -e


@pytest.mark.parametrize("bits,group", [(8, 128), (8, 64), (8, 32), (4, 128), (4, 64), (4, 32)])
@pytest.mark.parametrize("K", [2048, 12288])
def test_dot_product_perturbation(bits, group, K):
    N = 96
    W = oracle.Weight.from_f32(synth.host_f32(N * K, 700 + K + group + bits, synth.WEIGHT_OUTLIERS).reshape(N, K),
                               bits, group)
    x = _activations(K, K + group + bits, outliers=True)
    x_bits = oracle.bf16_from_f64(x)
    y = oracle.linear_bias(x_bits, W).reshape(-1)  # exact float64
    w = W.dense()
    scale = np.abs(y).max()
    for PL, frac in ((2, 2e-3 / 2), (3, 1e-5 / 20)):
        X, e = _fixed_point(x, PL)
        y_fx = (w @ X) * np.exp2(-e)  # exact sums in X, one scaling
        err = np.abs(y_fx - y).max() / scale
        assert err <= frac, (PL, err)


@pytest.mark.parametrize("K", [4096, 12288])
def test_massive_channel(K):
    N = 96
    W = oracle.Weight.from_f32(synth.host_f32(N * K, 900 + K, synth.WEIGHT_OUTLIERS).reshape(N, K), 8, 128)
    x = oracle.f64_from_bf16(synth.host_bf16(K, 901 + K, synth.ACT))
    x[17] = 1000.0
    x_bits = oracle.bf16_from_f64(x)
    y = oracle.linear_bias(x_bits, W).reshape(-1)
    assert np.abs(x).max() / np.sqrt((x * x).mean()) > 0.9 * np.sqrt(K) / np.sqrt(1 + K / 1e6)
    err = {}
    for PL in (2, 3):
        X, e = _fixed_point(x, PL)
        err[PL] = np.abs((W.dense() @ X) * np.exp2(-e) - y).max() / np.abs(y).max()
    assert err[3] <= 2e-3 / 20, err
    if K == 12288:
        assert err[2] > 2e-3, err

"""GPU parity of the dequantising prefill kernel (bf16 outputs over affine
weights: each weight rounded once to fp16 after a per-row power-of-two
scale, one fp32 tensor-memory sum over K) against the float64 oracle.

Beyond the bf16 tolerance shared with every test, these check the kernel's
own error model element by element,
    |y - y*| <= (2^-11 + K 2^-22) sum_k |w_nk x_mk| + ulp_bf16(y*) / 2,
(one fp16 rounding per weight, fp32 accumulation, the bf16 output rounding),
that rows whose weights differ by up to 2^80 in magnitude each keep their own
precision (the per-row scale; one scale for the tile would flush the small
rows to zero), and that all-zero weight rows give exactly the addend."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import TOL_BF16, dev_bf16, host_bits, ulp_bf16

pytestmark = pytest.mark.gpu

FMT_BITS = {1: 8, 2: 4}


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    yield m
    assert m.mt_device_error(clear=True) == 0, "a bounded device wait expired"


def _pack(mt, W32, fmt, group):
    N, K = W32.shape
    b = FMT_BITS[fmt]
    q = torch.empty(N, K * b // 8, dtype=torch.uint8, device="cuda")
    s = torch.empty(N, K // group, dtype=torch.bfloat16, device="cuda")
    bi = torch.empty_like(s)
    mt.mt_pack_affine(torch.from_numpy(np.ascontiguousarray(W32)).cuda(), N, K, group, b, q, s, bi)
    torch.cuda.synchronize()
    return q, s, bi


def _ws(mt, M, K, N, group):
    return torch.empty(mt.mt_prefill_workspace_bytes(M, K, N, group), dtype=torch.uint8, device="cuda")


def _oracle_weight(W32, fmt, group):
    """The oracle's own quantisation of the same fp32 weights (the library's
    packer is checked bit for bit against it elsewhere; nothing here is
    read back from the device)."""
    return oracle.Weight.from_f32(W32, FMT_BITS[fmt], group)


@pytest.mark.parametrize("fmt,group,M,K,N", [(1, 128, 70, 1024, 200), (1, 64, 257, 512, 384),
                                             (2, 32, 33, 256, 77), (2, 128, 130, 2048, 256)])
def test_dq_error_bound(mt, fmt, group, M, K, N):
    seed = 31000 + fmt * 7 + group + M + K + N
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    W32 = synth.host_f32(N * K, seed + 1, synth.WEIGHT_OUTLIERS).reshape(N, K)
    q, s, b = _pack(mt, W32, fmt, group)
    W = _oracle_weight(W32, fmt, group)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_prefill_linear_bias(dev_bf16(x), q, s, b, group, None, y, _ws(mt, M, K, N, group), fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.linear_bias(x, W)
    xa = np.abs(oracle.f64_from_bf16(x))
    bound = (2.0 ** -11 + K * 2.0 ** -22) * (xa @ np.abs(W.dense()).T) + 0.5 * ulp_bf16(ref)
    err = np.abs(oracle.f64_from_bf16(host_bits(y)) - ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"error {err[worst]:.3e} above the bound {bound[worst]:.3e} at {worst}"


@pytest.mark.parametrize("fmt,lo,hi", [(1, -40, 40), (2, -40, 40), (1, -120, 60)])
def test_dq_rows_of_any_magnitude(mt, fmt, lo, hi):
    """Rows scaled by 2^lo .. 2^hi (down to bf16-subnormal scales) each keep
    their own precision."""
    group, M, K, N = 64, 40, 512, 96
    seed = 32000 + fmt
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    W32 = synth.host_f32(N * K, seed + 1, synth.WEIGHT).reshape(N, K).astype(np.float64)
    W32 = (W32 * np.exp2(np.linspace(lo, hi, N))[:, None]).astype(np.float32)
    q, s, b = _pack(mt, W32, fmt, group)
    W = _oracle_weight(W32, fmt, group)
    res = np.zeros((M, N), dtype=np.uint16)  # zero addend: every row's own magnitude stays visible
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_prefill_down_residual(dev_bf16(x), q, s, b, group, dev_bf16(res), y, _ws(mt, M, K, N, group), fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.down_residual(x, W, res)
    got = oracle.f64_from_bf16(host_bits(y))
    excess = np.maximum(0.0, np.abs(got - ref) - 0.5 * ulp_bf16(ref))
    per_row = excess.max(axis=0) / np.maximum(np.abs(ref).max(axis=0), 1e-300)  # one weight row = one column
    assert per_row.max() <= TOL_BF16, f"row {int(per_row.argmax())}: {per_row.max():.3e}"


def test_dq_zero_rows(mt):
    fmt, group, M, K, N = 1, 128, 20, 256, 136
    seed = 33000
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    W32 = synth.host_f32(N * K, seed + 1, synth.WEIGHT).reshape(N, K)
    W32[::3] = 0.0
    q, s, b = _pack(mt, W32, fmt, group)
    res = synth.host_bf16(M * N, seed + 2, synth.ACT).reshape(M, N)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_prefill_down_residual(dev_bf16(x), q, s, b, group, dev_bf16(res), y, _ws(mt, M, K, N, group), fmt=fmt)
    torch.cuda.synchronize()
    got = host_bits(y)
    assert np.array_equal(got[:, ::3], res[:, ::3]), "a zero weight row must pass the residual through"
    ref = oracle.down_residual(x, _oracle_weight(W32, fmt, group), res)
    err = np.maximum(0.0, np.abs(oracle.f64_from_bf16(got) - ref) - 0.5 * ulp_bf16(ref)).max() / np.abs(ref).max()
    assert err <= TOL_BF16

"""GPU parity of the MX block-scaled weight formats (MXFP8: E4M3 elements,
MXFP4: E2M1 elements, one E8M0 scale per 32 along K) against the float64 CPU
oracle: the packer bit for bit, the three GEMV epilogues (SwiGLU, residual,
projection bias) for M in 1..8, an exact-arithmetic indexing case, and the
Qwen3-8B-shaped layer and a vocabulary-sized projection at full size."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_layers import DevLayer
from parity_util import assert_bf16_close, assert_f32_close, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu

MXF = {8: 3, 4: 4}  # bits -> mt_wfmt


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    m.mt_set_option(m.MT_OPT_GEMV, 0)
    yield m
    assert m.mt_device_error(clear=True) == 0


def gpu_pack_mx(mt, W32, bits):
    N, K = W32.shape
    q = torch.empty(N, K * bits // 8, dtype=torch.uint8, device="cuda")
    s = torch.empty(N, K // 32, dtype=torch.uint8, device="cuda")
    mt.mt_pack_mx(torch.from_numpy(np.ascontiguousarray(W32)).cuda(), N, K, bits, q, s)
    torch.cuda.synchronize()
    return q, s


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,K", [(37, 256), (5, 4096), (64, 96)])
def test_pack_mx_bit_exact(mt, bits, N, K):
    W = synth.host_f32(N * K, 9000 + N + K + bits, synth.WEIGHT_OUTLIERS).reshape(N, K)
    W[0, :32] = 0.0                                   # all-zero block: field 0
    W[1, :] = np.float32(0.25)                        # constant rows
    W[2, :32] = np.linspace(-448, 448, 32, dtype=np.float32) * np.float32(2.0 ** -10)
    W[3, :32] = np.float32(1.9) * np.float32(2.0 ** -3)  # above 1.75 * 2^emax after scaling: clamps
    W[4, :32] = -np.float32(2.0 ** -140)              # tiny negatives: negative zeros
    q, s = gpu_pack_mx(mt, W, bits)
    codes, rs = oracle.quantize_mx(W, bits)
    assert np.array_equal(s.cpu().numpy(), rs), "E8M0 scales differ"
    assert np.array_equal(q.cpu().numpy(), oracle.pack_codes(codes, bits)), "element codes differ"


SHAPES = [  # (bits, M, K, N)
    (8, 1, 256, 300), (8, 3, 1024, 129), (8, 8, 2048, 64), (8, 2, 4096, 1000), (8, 5, 96, 17),
    (4, 1, 512, 257), (4, 4, 2048, 100), (4, 8, 1024, 333), (4, 1, 4096, 2000), (4, 6, 160, 40),
]


def _ids(p):
    return f"mxfp{p[0]}-M{p[1]}-K{p[2]}-N{p[3]}"


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_f32", [False, True])
def test_mx_gemvs(mt, shape, out_f32):
    bits, M, K, N = shape
    fmt = MXF[bits]
    seed = 9100 + bits * 7 + M * 13 + K + N
    dt = torch.float32 if out_f32 else torch.bfloat16
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    Wg = synth.host_f32(N * K, seed + 1, synth.WEIGHT).reshape(N, K)
    Wu = synth.host_f32(N * K, seed + 2, synth.WEIGHT_OUTLIERS).reshape(N, K)
    qg, sg = gpu_pack_mx(mt, Wg, bits)
    qu, su = gpu_pack_mx(mt, Wu, bits)
    og, ou = oracle.Weight.from_f32_mx(Wg, bits), oracle.Weight.from_f32_mx(Wu, bits)
    xd = dev_bf16(x)
    check = assert_f32_close if out_f32 else assert_bf16_close
    get = host_f64 if out_f32 else host_bits
    # gate/up + SwiGLU
    h = torch.empty(M, N, dtype=dt, device="cuda")
    mt.mt_swiglu_gateup(xd, qg, qu, torch.stack([sg, su]).contiguous(), None, 32, h, fmt=fmt)
    # down + residual (the gate matrix as an [N][K] down projection)
    res = synth.host_bf16(M * N, seed + 3, synth.ACT).reshape(M, N)
    y = torch.empty(M, N, dtype=dt, device="cuda")
    mt.mt_down_residual(xd, qg, sg, None, 32, dev_bf16(res), y, fmt=fmt)
    # projection + bias
    bias = synth.host_bf16(N, seed + 4, synth.PROJ_BIAS)
    yb = torch.empty(M, N, dtype=dt, device="cuda")
    mt.mt_linear_bias(xd, qu, su, None, 32, dev_bf16(bias), yb, fmt=fmt)
    torch.cuda.synchronize()
    check(get(h), oracle.swiglu_gateup(x, og, ou), "h")
    check(get(y), oracle.down_residual(x, og, res), "y")
    check(get(yb), oracle.linear_bias(x, ou, bias), "y+bias")


@pytest.mark.parametrize("bits,M,K,N", [(8, 1, 256, 45), (8, 4, 512, 33), (4, 2, 512, 19), (4, 8, 256, 70)])
def test_mx_indexing_bit_exact(mt, bits, M, K, N):
    """Weights on a coarse grid (E4M3 values 1 .. 60 on a 2^-3 grid with scales
    1 .. 8; E2M1 values with scales 2^-3 .. 2^3) and small integer x: every
    product and sum stays within 24 significant bits, so the fp32 output
    equals the oracle bit for bit under any summation order."""
    rng = np.random.default_rng(bits * 101 + M + K + N)
    if bits == 8:
        # exponent fields 7..12 (1 .. 1.875 * 2^5), any fraction, either sign
        codes = (rng.integers(7, 13, size=(N, K)) << 3) | rng.integers(0, 8, size=(N, K))
        codes |= rng.integers(0, 2, size=(N, K)) << 7
        s = rng.integers(127, 131, size=(N, K // 32)).astype(np.uint8)
    else:
        codes = rng.integers(0, 16, size=(N, K))
        s = rng.integers(124, 131, size=(N, K // 32)).astype(np.uint8)
    codes = codes.astype(np.uint8)
    x = oracle.bf16_from_f64(rng.integers(-4, 5, size=(M, K)).astype(np.float64))
    res = oracle.bf16_from_f64(rng.integers(-8, 9, size=(M, N)).astype(np.float64))
    Wo = oracle.Weight(oracle.FMT_MXFP8 if bits == 8 else oracle.FMT_MXFP4, codes, s)
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    mt.mt_down_residual(dev_bf16(x), torch.from_numpy(oracle.pack_codes(codes, bits)).cuda(),
                        torch.from_numpy(s).cuda(), None, 32, dev_bf16(res), y, fmt=MXF[bits])
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().astype(np.float64), oracle.down_residual(x, Wo, res))


@pytest.mark.parametrize("wl", [synth.QWEN8B_MXFP8, synth.QWEN8B_MXFP4], ids=["mxfp8", "mxfp4"])
@pytest.mark.parametrize("M", [1, 4])
def test_mx_layer_full_size(mt, wl, M):
    """The 4096 x 12288 layer in MX formats: gate/up and down on every output."""
    d, f = wl.d, wl.f
    L = DevLayer(mt, wl, 0)
    x = synth.host_bf16(M * d, synth.seed_for(wl.wid, 0, synth.T_X), synth.ACT).reshape(M, d)
    hin = synth.host_bf16(M * f, synth.seed_for(wl.wid, 0, synth.T_H), synth.ACT).reshape(M, f)
    res = synth.host_bf16(M * d, synth.seed_for(wl.wid, 0, synth.T_RES3), synth.ACT).reshape(M, d)
    h = torch.empty(M, f, dtype=torch.float32, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_swiglu_gateup(dev_bf16(x), L.Wg, L.Wu, L.sgu, None, 32, h, fmt=wl.fmt)
    mt.mt_down_residual(dev_bf16(hin), L.Wd, L.sdn, None, 32, dev_bf16(res), y, fmt=wl.fmt)
    torch.cuda.synchronize()
    Wg = L.oracle_rows(synth.T_WG, range(f), f, d)
    Wu = L.oracle_rows(synth.T_WU, range(f), f, d)
    Wd = L.oracle_rows(synth.T_WD, range(d), d, f)
    # packed bytes of sampled rows, bit for bit
    for n in (0, 1, f // 2, f - 1):
        assert np.array_equal(L.Wg[n].cpu().numpy(), oracle.pack_codes(Wg.W[n:n + 1], wl.bits)[0])
        assert np.array_equal(L.sgu[0, n].cpu().numpy(), Wg.scales[n])
    assert_f32_close(host_f64(h), oracle.swiglu_gateup(x, Wg, Wu), "h")
    assert_bf16_close(host_bits(y), oracle.down_residual(hin, Wd, res), "y")


@pytest.mark.parametrize("bits", [8, 4])
def test_mx_vocab_projection(mt, bits):
    """A 4096 x 151936 vocabulary projection (more row ranges than SMs: the
    CTAs run in waves), M = 1 and 3, on 256 sampled outputs per row."""
    K, N = 4096, 151936
    wl = synth.QWEN8B_MXFP8 if bits == 8 else synth.QWEN8B_MXFP4
    seed = synth.seed_for(wl.wid, 0, synth.T_WVOCAB)
    tmp = torch.empty(N, K, dtype=torch.float32, device="cuda")
    synth.device_f32(tmp, seed, synth.WEIGHT)
    q = torch.empty(N, K * bits // 8, dtype=torch.uint8, device="cuda")
    s = torch.empty(N, K // 32, dtype=torch.uint8, device="cuda")
    mt.mt_pack_mx(tmp, N, K, bits, q, s)
    del tmp
    rows = np.sort(np.random.default_rng(bits).choice(N, 256, replace=False))
    rows[-1] = N - 1
    W32 = np.stack([synth.host_f32(K, seed, synth.WEIGHT, offset=int(n) * K) for n in rows])
    Wo = oracle.Weight.from_f32_mx(W32, bits)
    for M in (1, 3):
        x = synth.host_bf16(M * K, seed + M, synth.ACT).reshape(M, K)
        y = torch.empty(M, N, dtype=torch.float32, device="cuda")
        mt.mt_linear_bias(dev_bf16(x), q, s, None, 32, None, y, fmt=MXF[bits])
        torch.cuda.synchronize()
        assert_f32_close(host_f64(y)[:, rows], oracle.linear_bias(x, Wo), f"vocab M={M}")

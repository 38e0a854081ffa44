"""GPU parity of the projection GEMV with its bias epilogue (attention q/k/v/o
and the vocabulary projection) against the float64 CPU oracle, through the C
ABI: every kernel family, M in 1..8, bias present and absent, ragged row
tails, and the three model shapes at full size (every output of the attention
projections, sampled outputs of the vocabulary projection)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_layers import DevProj
from parity_util import assert_bf16_close, assert_f32_close, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu

FMT_BITS = {0: 16, 1: 8, 2: 4}


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.fixture(params=["default", "team", "mma"])
def gemv(request, mt):
    mt.mt_set_option(mt.MT_OPT_GEMV, {"default": 0, "team": 1, "mma": 2}[request.param])
    yield request.param
    mt.mt_set_option(mt.MT_OPT_GEMV, 0)
    assert mt.mt_device_error(clear=True) == 0, "a bounded device wait expired"


def _pack(mt, W32, fmt, group):
    N, K = W32.shape
    if fmt == 0:
        return dev_bf16(oracle.bf16_from_f64(W32.astype(np.float64))), None, None
    b = FMT_BITS[fmt]
    q = torch.empty(N, K * b // 8, dtype=torch.uint8, device="cuda")
    s = torch.empty(N, K // group, dtype=torch.bfloat16, device="cuda")
    bi = torch.empty_like(s)
    mt.mt_pack_affine(torch.from_numpy(np.ascontiguousarray(W32)).cuda(), N, K, group, b, q, s, bi)
    torch.cuda.synchronize()
    return q, s, bi


SHAPES = [  # (fmt, group, M, K, N)
    (1, 64, 1, 1536, 2048),     # stacked q/k/v of a 1536-wide model
    (1, 128, 1, 4096, 1000),
    (2, 32, 1, 2048, 3072),
    (0, 0, 1, 1536, 1536),
    (1, 32, 3, 1024, 700),
    (2, 64, 8, 2048, 333),
    (0, 0, 5, 512, 1201),
    (1, 128, 1, 512, 20000),    # long vocabulary-like row range per CTA
    (2, 128, 2, 768, 4999),
    (1, 64, 7, 256, 153),
    # one row: rows of 64 chunks, two rows per load stream (odd N: a last task with one row)
    (1, 64, 1, 1024, 1001),
    (2, 128, 1, 2048, 1337),
    (2, 32, 1, 2048, 153),
    (0, 0, 1, 512, 999),
]


def _ids(p):
    fmt, g, M, K, N = p
    return f"{['bf16', 'a8', 'a4'][fmt]}-g{g}-M{M}-K{K}-N{N}"


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("out_f32", [False, True])
def test_linear_bias(mt, gemv, shape, with_bias, out_f32):
    fmt, group, M, K, N = shape
    seed = 6000 + fmt * 97 + M * 13 + K + N
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    W32 = synth.host_f32(N * K, seed + 1, synth.WEIGHT).reshape(N, K)
    bias = synth.host_bf16(N, seed + 2, synth.PROJ_BIAS) if with_bias else None
    q, s, b = _pack(mt, W32, fmt, group)
    y = torch.empty(M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    mt.mt_linear_bias(dev_bf16(x), q, s, b, group, None if bias is None else dev_bf16(bias), y, fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.linear_bias(x, oracle.Weight.from_f32(W32, FMT_BITS[fmt], group), bias)
    if out_f32:
        assert_f32_close(host_f64(y), ref, "y f32")
    else:
        assert_bf16_close(host_bits(y), ref, "y bf16")


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 32, 1, 256, 45), (8, 128, 3, 512, 37),
                                              (4, 64, 8, 512, 19), (4, 32, 2, 256, 70)])
def test_linear_bias_bit_exact(mt, gemv, bits, group, M, K, N):
    """Codes, power-of-two scales, grid biases and an integer bias: every
    product and sum is exact in fp32, so the output equals the oracle bit for
    bit; M > 1 shows the bias is one row shared by every m."""
    rng = np.random.default_rng(bits * 31 + group + K + N + M)
    qmax = (1 << bits) - 1
    G = K // group
    codes = rng.integers(0, qmax + 1, size=(N, K)).astype(np.uint8)
    s = oracle.bf16_from_f64(np.ldexp(1.0, rng.integers(-8, -3, size=(N, G))))
    b = oracle.bf16_from_f64(rng.integers(-32, 32, size=(N, G)) * 2.0 ** -8)
    x = oracle.bf16_from_f64(rng.integers(-4, 5, size=(M, K)).astype(np.float64))
    bias = oracle.bf16_from_f64(rng.integers(-100, 101, size=N).astype(np.float64))
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    mt.mt_linear_bias(dev_bf16(x), torch.from_numpy(oracle.pack_codes(codes, bits)).cuda(), dev_bf16(s),
                      dev_bf16(b), group, dev_bf16(bias), y, fmt=1 if bits == 8 else 2)
    torch.cuda.synchronize()
    ref = oracle.linear_bias(x, oracle.Weight(oracle.FMT_CODES, codes, s, b, group), bias)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


def test_linear_bias_zero_weight_returns_bias(mt, gemv):
    M, K, N = 4, 1024, 300
    x = synth.host_bf16(M * K, 71, synth.ACT).reshape(M, K)
    bias = synth.host_bf16(N, 72, synth.PROJ_BIAS)
    W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_linear_bias(dev_bf16(x), W, None, None, 0, dev_bf16(bias), y, fmt=0)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y), np.broadcast_to(bias, (M, N)))


@pytest.mark.parametrize("wl", synth.PROJ_ALL, ids=lambda w: w.name.split()[0])
@pytest.mark.parametrize("M", [1, 4])
def test_projections_full_size(mt, wl, M):
    """The model's projections at full size, in the bench's launch
    configuration (default kernel choice, programmatic dependent launch on):
    the attention projections on every output, the vocabulary projection on
    256 sampled outputs per row."""
    mt.mt_set_option(mt.MT_OPT_GEMV, 0)
    mt.mt_set_option(mt.MT_OPT_PDL, 1)
    layer = wl.layers - 1
    for p in wl.projs:
        P = DevProj(mt, wl, p, layer if p.per_layer else 0)
        x = synth.host_bf16(M * p.K, synth.seed_for(wl.wid, layer, synth.T_X), synth.ACT).reshape(M, p.K)
        y = torch.empty(M, p.N, dtype=torch.float32, device="cuda")
        yb = torch.empty(M, p.N, dtype=torch.bfloat16, device="cuda")
        xd = dev_bf16(x)
        P.run(mt, xd, y)
        P.run(mt, xd, yb)
        torch.cuda.synchronize()
        if p.per_layer:
            rows = np.arange(p.N)
        else:
            rows = np.sort(np.random.default_rng(p.N + M).choice(p.N, 256, replace=False))
            rows[-1] = p.N - 1  # the last row of the last CTA
        Wo, bias = P.oracle_rows(rows)
        ref = oracle.linear_bias(x, Wo, bias)
        assert_f32_close(host_f64(y)[:, rows], ref, f"{p.name} f32")
        assert_bf16_close(host_bits(yb)[:, rows], ref, f"{p.name} bf16")
        del P
        torch.cuda.empty_cache()
    assert mt.mt_device_error(clear=True) == 0

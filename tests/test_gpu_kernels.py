"""GPU parity of each kernel against the float64 CPU oracle, through the C ABI.

Inputs come from the seeded generator (synth) on the host and are copied to
the device, so both sides see the same bytes.  Weights are quantised twice,
independently: by the library's packer on the GPU (the product path) and by
the oracle's quantiser on the CPU.  Shapes span several CTAs, ragged row
tails (N not a multiple of the row tile), ragged K (chunks not a multiple of
the team size) and M in 1..8.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (assert_bf16_close, assert_f32_close, dev_bf16, host_bits, host_f64)

pytestmark = pytest.mark.gpu

FMT_BITS = {0: 16, 1: 8, 2: 4}


@pytest.fixture(scope="module")
def mt():
    import quantized_gemv_epilogues_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.fixture(params=["default", "team", "mma"])
def gemv(request, mt):
    """Runs a test with each GEMV kernel family: the default choice (warp-task
    kernel for M = 1 and for M = 2 over affine INT8, tensor-core kernel for
    other M > 1), the team kernel for every M, and the tensor-core kernel for
    every M."""
    mt.mt_set_option(mt.MT_OPT_GEMV, {"default": 0, "team": 1, "mma": 2}[request.param])
    yield request.param
    mt.mt_set_option(mt.MT_OPT_GEMV, 0)
    assert mt.mt_device_error(clear=True) == 0, "a bounded device wait expired"


# ------------------------------------------------------------------ helpers
def gen_w32(N, K, seed, dist=synth.WEIGHT):
    return synth.host_f32(N * K, seed, dist).reshape(N, K)


def gpu_pack(mt, W32: np.ndarray, fmt: int, group: int):
    """Pack fp32 weights on the GPU with the library's packer.  Returns
    (W_dev, scales_dev, biases_dev); bf16 format rounds on the host generator
    side instead (dense weights are generated as bf16)."""
    N, K = W32.shape
    if fmt == 0:
        bits = oracle.bf16_from_f64(W32.astype(np.float64))  # generator-side storage rounding
        return dev_bf16(bits), None, None
    b = FMT_BITS[fmt]
    q = torch.empty(N, K * b // 8, dtype=torch.uint8, device="cuda")
    s = torch.empty(N, K // group, dtype=torch.bfloat16, device="cuda")
    bi = torch.empty_like(s)
    mt.mt_pack_affine(torch.from_numpy(np.ascontiguousarray(W32)).cuda(), N, K, group, b, q, s, bi)
    torch.cuda.synchronize()
    return q, s, bi


def orc_weight(W32, fmt, group):
    return oracle.Weight.from_f32(W32, FMT_BITS[fmt], group)


# ------------------------------------------------------------------ K1
@pytest.mark.parametrize("M,d", [(1, 256), (1, 1536), (1, 2048), (1, 4096), (3, 4096), (8, 2048),
                                 (2, 8), (5, 1000), (1, 12288), (1, 65536)])
@pytest.mark.parametrize("norm_f32", [False, True])
def test_add_rmsnorm(mt, M, d, norm_f32):
    seed = 1000 + M * 7 + d
    v = synth.host_bf16(M * d, seed, synth.ACT).reshape(M, d)
    r = synth.host_bf16(M * d, seed + 1, synth.ACT).reshape(M, d)
    w = synth.host_bf16(d, seed + 2, synth.NORM_W)
    eps = 1e-5 if d % 2 else 1e-6
    out_sum = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    out_norm = torch.empty(M, d, dtype=torch.float32 if norm_f32 else torch.bfloat16, device="cuda")
    mt.mt_add_rmsnorm(dev_bf16(v), dev_bf16(r), dev_bf16(w), eps, out_sum, out_norm)
    torch.cuda.synchronize()
    ref_sum, ref_norm = oracle.add_rmsnorm(v, r, w, eps)
    assert np.array_equal(host_bits(out_sum), ref_sum), "out_sum must equal bf16(values + residual)"
    if norm_f32:
        assert_f32_close(host_f64(out_norm), ref_norm, "out_norm f32")
    else:
        assert_bf16_close(host_bits(out_norm), ref_norm, "out_norm bf16")


def test_add_rmsnorm_in_place_residual(mt):
    M, d = 2, 4096
    v = synth.host_bf16(M * d, 77, synth.ACT).reshape(M, d)
    r = synth.host_bf16(M * d, 78, synth.ACT).reshape(M, d)
    w = synth.host_bf16(d, 79, synth.NORM_W)
    rd = dev_bf16(r)
    out_norm = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_add_rmsnorm(dev_bf16(v), rd, dev_bf16(w), 1e-6, rd, out_norm)
    torch.cuda.synchronize()
    ref_sum, ref_norm = oracle.add_rmsnorm(v, r, w, 1e-6)
    assert np.array_equal(host_bits(rd), ref_sum)
    assert_bf16_close(host_bits(out_norm), ref_norm, "out_norm")


# ------------------------------------------------------------------ packer
@pytest.mark.parametrize("N,K,group,bits", [(37, 256, 32, 8), (37, 256, 64, 4), (64, 4096, 128, 8),
                                            (16, 768, 64, 8), (20, 2048, 128, 4), (9, 96, 32, 4)])
def test_pack_affine_bit_exact(mt, N, K, group, bits):
    W = gen_w32(N, K, 2000 + N + K + group + bits, synth.WEIGHT_OUTLIERS)
    W[0, :] = 0.25                       # constant row: scale 0
    W[1, :group] = 0.0                   # zero group
    W[2, :] = np.arange(K, dtype=np.float32) * np.float32(2.0 ** -8)  # grid / tie values
    W[3, 5] = np.float32(3.0)            # outlier
    q, s, b = gpu_pack(mt, W, 1 if bits == 8 else 2, group)
    codes, rs, rb = oracle.quantize(W, group, bits)
    assert np.array_equal(q.cpu().numpy(), oracle.pack_codes(codes, bits)), "packed codes differ"
    assert np.array_equal(host_bits(s), rs), "scales differ"
    assert np.array_equal(host_bits(b), rb), "biases differ"
    Wd = torch.empty(N, K, dtype=torch.float32, device="cuda")
    mt.mt_unpack_affine(q, s, b, N, K, group, bits, Wd)
    torch.cuda.synchronize()
    exact = oracle.dequant(codes, rs, rb, group)
    assert np.array_equal(Wd.cpu().numpy(), exact.astype(np.float32)), "unpacked weights differ"


# ------------------------------------------------------------------ K2 / K3
SHAPES = [  # (fmt, group, M, d, f)
    (1, 64, 1, 256, 768),
    (1, 128, 1, 4096, 300),
    (1, 32, 2, 2048, 200),
    (1, 64, 3, 512, 333),
    (1, 128, 8, 1024, 130),
    (2, 64, 1, 2048, 257),
    (2, 32, 4, 512, 100),
    (2, 128, 8, 1024, 64),
    (0, 0, 1, 1536, 300),
    (0, 0, 2, 1000, 77),
    (0, 0, 8, 512, 40),
    (1, 128, 1, 12288, 161),   # 12 KB rows: split into pieces
    (1, 32, 1, 4096, 1000),    # many rows per CTA
    (2, 64, 1, 8192, 153),     # one more row than SMs
    (0, 0, 1, 8960, 40),       # 17.5 KB bf16 rows
    (1, 64, 1, 64, 7),         # rows shorter than a warp's stride
    (1, 32, 8, 2048, 1000),    # multi-row: several 16-row tiles per CTA
    (1, 64, 7, 768, 500),
    (2, 128, 5, 1024, 300),
    (2, 32, 2, 256, 170),
    (0, 0, 6, 1536, 350),
    (1, 64, 3, 512, 1300),     # row ranges shared by clusters of two CTAs (K halves)
    (1, 128, 8, 768, 1229),
    (2, 32, 5, 256, 1500),
    (0, 0, 4, 384, 1250),
    (1, 32, 6, 1024, 1400),    # clusters with 8-byte weight loads
    (2, 64, 7, 512, 1600),
]


def _ids(p):
    fmt, g, M, d, f = p
    return f"{['bf16', 'a8', 'a4'][fmt]}-g{g}-M{M}-d{d}-f{f}"


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_f32", [False, True])
def test_swiglu_gateup(mt, gemv, shape, out_f32):
    fmt, group, M, d, f = shape
    seed = 3000 + fmt * 97 + M * 13 + d + f
    x = synth.host_bf16(M * d, seed, synth.ACT).reshape(M, d)
    Wg = gen_w32(f, d, seed + 1)
    Wu = gen_w32(f, d, seed + 2)
    qg, sg, bg = gpu_pack(mt, Wg, fmt, group)
    qu, su, bu = gpu_pack(mt, Wu, fmt, group)
    if fmt:
        scales = torch.stack([sg, su]).contiguous()
        biases = torch.stack([bg, bu]).contiguous()
    else:
        scales = biases = None
    h = torch.empty(M, f, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    mt.mt_swiglu_gateup(dev_bf16(x), qg, qu, scales, biases, group, h, fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.swiglu_gateup(x, orc_weight(Wg, fmt, group), orc_weight(Wu, fmt, group))
    if out_f32:
        assert_f32_close(host_f64(h), ref, "h f32")
    else:
        assert_bf16_close(host_bits(h), ref, "h bf16")


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_f32", [False, True])
def test_down_residual(mt, gemv, shape, out_f32):
    fmt, group, M, d, f = shape
    # the down projection reads [M][f] and writes [M][d]; reuse the shape list
    # with the roles of d and f swapped so K = f covers the same K values
    K, N = d, f
    seed = 4000 + fmt * 97 + M * 13 + K + N
    hin = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    res = synth.host_bf16(M * N, seed + 1, synth.ACT).reshape(M, N)
    Wd = gen_w32(N, K, seed + 2)
    qd, sd, bd = gpu_pack(mt, Wd, fmt, group)
    y = torch.empty(M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    mt.mt_down_residual(dev_bf16(hin), qd, sd, bd, group, dev_bf16(res), y, fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.down_residual(hin, orc_weight(Wd, fmt, group), res)
    if out_f32:
        assert_f32_close(host_f64(y), ref, "y f32")
    else:
        assert_bf16_close(host_bits(y), ref, "y bf16")


@pytest.mark.parametrize("fmt,group", [(1, 128), (2, 64)])
def test_act_bits_24_massive_channel(mt, fmt, group):
    """An activation row with one channel 1000x the others (the case the
    16-bit fixed-point x cannot hold within the bf16 bound): with
    MT_OPT_ACT_BITS = 24 the one-row gate/up and down calls with bf16 outputs
    meet it, and 16 bits remain the default."""
    assert mt.mt_get_option(mt.MT_OPT_ACT_BITS) == 16
    d, f, N = 4096, 12288, 512
    seed = 71000 + fmt * 10 + group
    x = oracle.f64_from_bf16(synth.host_bf16(d, seed, synth.ACT))
    x[17] = 1000.0
    x = oracle.bf16_from_f64(x)[None]
    h = oracle.f64_from_bf16(synth.host_bf16(f, seed + 1, synth.ACT))
    h[4321] = 1000.0
    h = oracle.bf16_from_f64(h)[None]
    res = synth.host_bf16(N, seed + 2, synth.ACT)[None]
    Wg, Wu = gen_w32(N, d, seed + 3, synth.WEIGHT_OUTLIERS), gen_w32(N, d, seed + 4, synth.WEIGHT_OUTLIERS)
    Wd = gen_w32(N, f, seed + 5, synth.WEIGHT_OUTLIERS)
    qg, sg, bg = gpu_pack(mt, Wg, fmt, group)
    qu, su, bu = gpu_pack(mt, Wu, fmt, group)
    qd, sd, bd = gpu_pack(mt, Wd, fmt, group)
    sgu, bgu = torch.stack([sg, su]).contiguous(), torch.stack([bg, bu]).contiguous()
    hout = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    yout = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_set_option(mt.MT_OPT_ACT_BITS, 24)
    try:
        mt.mt_swiglu_gateup(dev_bf16(x), qg, qu, sgu, bgu, group, hout, fmt=fmt)
        mt.mt_down_residual(dev_bf16(h), qd, sd, bd, group, dev_bf16(res), yout, fmt=fmt)
        torch.cuda.synchronize()
    finally:
        mt.mt_set_option(mt.MT_OPT_ACT_BITS, 16)
    h_ref = oracle.swiglu_gateup(x, orc_weight(Wg, fmt, group), orc_weight(Wu, fmt, group))
    y_ref = oracle.down_residual(h, orc_weight(Wd, fmt, group), res)
    assert_bf16_close(host_bits(hout), h_ref, "h bf16, 24-bit x")
    assert_bf16_close(host_bits(yout), y_ref, "y bf16, 24-bit h")


@pytest.mark.parametrize("group,K,N", [(128, 4096, 1000), (64, 12288, 333), (32, 1024, 257)])
def test_two_rows_match_one_row_calls(mt, group, K, N):
    """Two activation rows over affine INT8 weights (one kernel reading each
    weight once): every output row equals the one-row call on that row alone,
    bit for bit, for gate/up + SwiGLU, down + residual and a projection with
    bias (each row keeps its own fixed-point scale and summation order)."""
    seed = 61000 + K + N + group
    x = synth.host_bf16(2 * K, seed, synth.ACT).reshape(2, K)
    res = synth.host_bf16(2 * N, seed + 1, synth.ACT).reshape(2, N)
    bias = synth.host_bf16(N, seed + 2, synth.PROJ_BIAS)
    qg, sg, bg = gpu_pack(mt, gen_w32(N, K, seed + 3), 1, group)
    qu, su, bu = gpu_pack(mt, gen_w32(N, K, seed + 4), 1, group)
    sgu, bgu = torch.stack([sg, su]).contiguous(), torch.stack([bg, bu]).contiguous()
    xd, rd, bd = dev_bf16(x), dev_bf16(res), dev_bf16(bias)
    calls = {
        "h": lambda xx, rr, out: mt.mt_swiglu_gateup(xx, qg, qu, sgu, bgu, group, out, fmt=1),
        "y": lambda xx, rr, out: mt.mt_down_residual(xx, qg, sg, bg, group, rr, out, fmt=1),
        "y + bias": lambda xx, rr, out: mt.mt_linear_bias(xx, qu, su, bu, group, bd, out, fmt=1),
    }
    for name, call in calls.items():
        two = torch.empty(2, N, dtype=torch.bfloat16, device="cuda")
        call(xd, rd, two)
        ones = []
        for r in range(2):
            one = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
            call(xd[r:r + 1].clone(), rd[r:r + 1].clone(), one)  # fresh 16-byte aligned rows
            ones.append(one)
        torch.cuda.synchronize()
        for r in range(2):
            assert torch.equal(two[r], ones[r][0]), f"{name}: row {r} differs from the one-row call"


def test_down_residual_in_place(mt, gemv):
    M, K, N, g = 1, 4096, 1024, 128
    hin = synth.host_bf16(M * K, 91, synth.ACT).reshape(M, K)
    res = synth.host_bf16(M * N, 92, synth.ACT).reshape(M, N)
    Wd = gen_w32(N, K, 93)
    qd, sd, bd = gpu_pack(mt, Wd, 1, g)
    rd = dev_bf16(res)
    mt.mt_down_residual(dev_bf16(hin), qd, sd, bd, g, rd, rd, fmt=1)
    torch.cuda.synchronize()
    ref = oracle.down_residual(hin, orc_weight(Wd, 1, g), res)
    assert_bf16_close(host_bits(rd), ref, "in-place y")


# ------------------------------------------- exact-arithmetic indexing cases
def _exact_affine(N, K, group, bits, rng, bias_lo=-32, bias_hi=32):
    """Codes, power-of-two scales and biases on a 2^-8 grid: every product and
    partial sum of the GEMV is exact in fp32."""
    qmax = (1 << bits) - 1
    G = K // group
    codes = rng.integers(0, qmax + 1, size=(N, K)).astype(np.uint8)
    s = oracle.bf16_from_f64(np.ldexp(1.0, rng.integers(-8, -3, size=(N, G))))
    b = oracle.bf16_from_f64(rng.integers(bias_lo, bias_hi, size=(N, G)) * 2.0 ** -8)
    return codes, s, b


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 32, 1, 128, 45), (8, 64, 2, 512, 33),
                                              (8, 128, 8, 384, 17), (4, 32, 1, 256, 23),
                                              (4, 64, 3, 512, 16), (4, 128, 1, 384, 9)])
def test_indexing_down_bit_exact(mt, gemv, bits, group, M, K, N):
    rng = np.random.default_rng(bits * 1000 + group + K + N + M)
    codes, s, b = _exact_affine(N, K, group, bits, rng)
    x = oracle.bf16_from_f64(rng.integers(-4, 5, size=(M, K)).astype(np.float64))
    res = oracle.bf16_from_f64(rng.integers(-8, 9, size=(M, N)).astype(np.float64))
    packed = oracle.pack_codes(codes, bits)
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    mt.mt_down_residual(dev_bf16(x), torch.from_numpy(packed).cuda(), dev_bf16(s), dev_bf16(b), group,
                        dev_bf16(res), y, fmt=1 if bits == 8 else 2)
    torch.cuda.synchronize()
    ref = oracle.down_residual(x, oracle.Weight(oracle.FMT_CODES, codes, s, b, group), res)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 32, 1, 256, 31), (8, 128, 2, 512, 20),
                                              (4, 64, 1, 512, 12), (4, 32, 8, 256, 10)])
def test_indexing_gateup_bit_exact(mt, gemv, bits, group, M, K, N):
    # gate rows give g >= 40, where silu(g) == g in both binary64 and fp32, so
    # h = g * u is one rounding of an exact product on both sides
    rng = np.random.default_rng(bits * 77 + group + K + N + M)
    cg, sgb, bgb = _exact_affine(N, K, group, bits, rng, bias_lo=128, bias_hi=256)
    cu, sub, bub = _exact_affine(N, K, group, bits, rng)
    x = oracle.bf16_from_f64(rng.integers(1, 5, size=(M, K)).astype(np.float64))
    Wg = oracle.Weight(oracle.FMT_CODES, cg, sgb, bgb, group)
    Wu = oracle.Weight(oracle.FMT_CODES, cu, sub, bub, group)
    h_ref, g_ref, u_ref = oracle.swiglu_gateup(x, Wg, Wu, return_gu=True)
    assert np.all(g_ref >= 40.0)
    h = torch.empty(M, N, dtype=torch.float32, device="cuda")
    scales = dev_bf16(np.stack([sgb, sub]))
    biases = dev_bf16(np.stack([bgb, bub]))
    mt.mt_swiglu_gateup(dev_bf16(x), torch.from_numpy(oracle.pack_codes(cg, bits)).cuda(),
                        torch.from_numpy(oracle.pack_codes(cu, bits)).cuda(), scales, biases, group, h,
                        fmt=1 if bits == 8 else 2)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), (g_ref * u_ref).astype(np.float32))


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 32, 1, 128, 45), (8, 64, 2, 512, 33), (8, 64, 1, 1024, 40),
                                              (4, 32, 1, 256, 23), (4, 64, 1, 2048, 20), (4, 128, 2, 384, 9)])
def test_indexing_down_bf16_out_bit_exact(mt, gemv, bits, group, M, K, N):
    """bf16 outputs, which the one-row kernels compute from a 16-bit
    fixed-point x: in the exact case every sum is exact in fp32, so each
    output is the one nearest-even bf16 rounding of the exact value.  (K = 1024
    INT8 and K = 2048 INT4 rows are 64 chunks: two rows per load stream.)"""
    rng = np.random.default_rng(bits * 3000 + group + K + N + M)
    codes, s, b = _exact_affine(N, K, group, bits, rng)
    x = oracle.bf16_from_f64(rng.integers(-4, 5, size=(M, K)).astype(np.float64))
    res = oracle.bf16_from_f64(rng.integers(-8, 9, size=(M, N)).astype(np.float64))
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_down_residual(dev_bf16(x), torch.from_numpy(oracle.pack_codes(codes, bits)).cuda(), dev_bf16(s),
                        dev_bf16(b), group, dev_bf16(res), y, fmt=1 if bits == 8 else 2)
    torch.cuda.synchronize()
    ref = oracle.down_residual(x, oracle.Weight(oracle.FMT_CODES, codes, s, b, group), res)
    assert np.array_equal(host_bits(y), oracle.bf16_from_f64(ref))


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 32, 1, 256, 31), (8, 128, 2, 512, 20), (8, 64, 1, 1024, 16),
                                              (4, 64, 1, 512, 12), (4, 32, 1, 2048, 10)])
def test_indexing_gateup_bf16_out_bit_exact(mt, gemv, bits, group, M, K, N):
    # as the fp32 case (g >= 40, silu(g) == g in fp32); the kernel rounds the
    # product g * u to fp32 and then to bf16
    rng = np.random.default_rng(bits * 91 + group + K + N + M)
    cg, sgb, bgb = _exact_affine(N, K, group, bits, rng, bias_lo=128, bias_hi=256)
    cu, sub, bub = _exact_affine(N, K, group, bits, rng)
    x = oracle.bf16_from_f64(rng.integers(1, 5, size=(M, K)).astype(np.float64))
    Wg = oracle.Weight(oracle.FMT_CODES, cg, sgb, bgb, group)
    Wu = oracle.Weight(oracle.FMT_CODES, cu, sub, bub, group)
    _, g_ref, u_ref = oracle.swiglu_gateup(x, Wg, Wu, return_gu=True)
    assert np.all(g_ref >= 40.0)
    h = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    mt.mt_swiglu_gateup(dev_bf16(x), torch.from_numpy(oracle.pack_codes(cg, bits)).cuda(),
                        torch.from_numpy(oracle.pack_codes(cu, bits)).cuda(), dev_bf16(np.stack([sgb, sub])),
                        dev_bf16(np.stack([bgb, bub])), group, h, fmt=1 if bits == 8 else 2)
    torch.cuda.synchronize()
    want = oracle.bf16_from_f64((g_ref * u_ref).astype(np.float32).astype(np.float64))
    assert np.array_equal(host_bits(h), want)


def test_indexing_bf16_weights_bit_exact(mt, gemv):
    rng = np.random.default_rng(5)
    M, K, N = 2, 1000, 37
    W = oracle.bf16_from_f64(rng.integers(-64, 65, size=(N, K)) * 2.0 ** -6)
    x = oracle.bf16_from_f64(rng.integers(-4, 5, size=(M, K)).astype(np.float64))
    res = oracle.bf16_from_f64(rng.integers(-8, 9, size=(M, N)).astype(np.float64))
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    mt.mt_down_residual(dev_bf16(x), dev_bf16(W), None, None, 0, dev_bf16(res), y, fmt=0)
    torch.cuda.synchronize()
    ref = oracle.down_residual(x, oracle.Weight(oracle.FMT_BF16, W), res)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


# ------------------------------------------------------------------ layer
def test_tiny_layer_chained(mt, gemv):
    wl = synth.TINY
    d, f, M, g = wl.d, wl.f, wl.M, wl.group
    sd = lambda t: synth.seed_for(wl.wid, 0, t)
    v = synth.host_bf16(M * d, sd(synth.T_VALUES), synth.ACT).reshape(M, d)
    r = synth.host_bf16(M * d, sd(synth.T_RESIDUAL), synth.ACT).reshape(M, d)
    w = synth.host_bf16(d, sd(synth.T_NORM_W), synth.NORM_W)
    Wg, Wu = gen_w32(f, d, sd(synth.T_WG)), gen_w32(f, d, sd(synth.T_WU))
    Wd = gen_w32(d, f, sd(synth.T_WD))
    qg, sg, bg = gpu_pack(mt, Wg, 1, g)
    qu, su, bu = gpu_pack(mt, Wu, 1, g)
    qd, s3, b3 = gpu_pack(mt, Wd, 1, g)
    out_sum = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    out_norm = torch.empty_like(out_sum)
    h = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_add_rmsnorm(dev_bf16(v), dev_bf16(r), dev_bf16(w), wl.eps, out_sum, out_norm)
    mt.mt_swiglu_gateup(out_norm, qg, qu, torch.stack([sg, su]), torch.stack([bg, bu]), g, h, fmt=1)
    mt.mt_down_residual(h, qd, s3, b3, g, out_sum, y, fmt=1)
    torch.cuda.synchronize()
    ref = oracle.mlp_layer(v, r, w, wl.eps, orc_weight(Wg, 1, g), orc_weight(Wu, 1, g),
                           orc_weight(Wd, 1, g))
    assert np.array_equal(host_bits(out_sum), ref["out_sum"])
    assert_bf16_close(host_bits(out_norm), ref["norm_x"], "out_norm")
    # each later step is compared on the oracle's chain; the GPU chain differs
    # only through 1-ulp bf16 rounding differences of out_norm and h
    assert_bf16_close(host_bits(y), ref["y_x"], "y (chained)")

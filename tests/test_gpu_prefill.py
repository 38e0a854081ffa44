"""GPU parity of the multi-row prefill GEMMs (tcgen05 tensor cores, M > 8)
against the float64 CPU oracle, through the C ABI: gate/up + SwiGLU, down +
residual and projection + bias over affine INT8 / INT4 weights, groups
32/64/128, ragged tiles on both sides (M and N not multiples of the 64 x 128
tile), an exact-arithmetic indexing case, and the Qwen3-8B layer at M = 256."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_layers import DevLayer
from parity_util import assert_bf16_close, assert_f32_close, dev_bf16, host_bits, host_f64

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
    n = mt.mt_prefill_workspace_bytes(M, K, N, group)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


SHAPES = [  # (fmt, group, M, K, N)
    (1, 64, 1, 64, 5),        # one row, one K block, a tiny tile
    (1, 128, 9, 256, 200),
    (1, 64, 64, 512, 128),    # exact tiles
    (1, 32, 100, 256, 300),   # two groups per K block
    (2, 64, 70, 512, 129),
    (2, 128, 130, 1024, 256),
    (1, 128, 257, 1024, 384),
    (2, 32, 33, 128, 77),
]


def _ids(p):
    fmt, g, M, K, N = p
    return f"{['', 'a8', 'a4'][fmt]}-g{g}-M{M}-K{K}-N{N}"


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
def test_prefill_epilogues(mt, shape):
    fmt, group, M, K, N = shape
    seed = 12000 + fmt * 97 + M * 13 + K + N + group
    bits = FMT_BITS[fmt]
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    Wg = synth.host_f32(N * K, seed + 1, synth.WEIGHT).reshape(N, K)
    Wu = synth.host_f32(N * K, seed + 2, synth.WEIGHT_OUTLIERS).reshape(N, K)
    qg, sg, bg = _pack(mt, Wg, fmt, group)
    qu, su, bu = _pack(mt, Wu, fmt, group)
    og, ou = oracle.Weight.from_f32(Wg, bits, group), oracle.Weight.from_f32(Wu, bits, group)
    res = synth.host_bf16(M * N, seed + 3, synth.ACT).reshape(M, N)
    bias = synth.host_bf16(N, seed + 4, synth.PROJ_BIAS)
    refs = {"h": oracle.swiglu_gateup(x, og, ou), "y": oracle.down_residual(x, og, res),
            "y + bias": oracle.linear_bias(x, ou, bias), "y, no bias": oracle.linear_bias(x, og)}
    ws = _ws(mt, M, K, N, group)
    xd = dev_bf16(x)
    sgu, bgu = torch.stack([sg, su]).contiguous(), torch.stack([bg, bu]).contiguous()
    for out_f32 in (False, True):
        dt = torch.float32 if out_f32 else torch.bfloat16
        check = assert_f32_close if out_f32 else assert_bf16_close
        get = host_f64 if out_f32 else host_bits
        outs = {k: torch.empty(M, N, dtype=dt, device="cuda") for k in refs}
        mt.mt_prefill_swiglu_gateup(xd, qg, qu, sgu, bgu, group, outs["h"], ws, fmt=fmt)
        mt.mt_prefill_down_residual(xd, qg, sg, bg, group, dev_bf16(res), outs["y"], ws, fmt=fmt)
        mt.mt_prefill_linear_bias(xd, qu, su, bu, group, dev_bf16(bias), outs["y + bias"], ws, fmt=fmt)
        mt.mt_prefill_linear_bias(xd, qg, sg, bg, group, None, outs["y, no bias"], ws, fmt=fmt)
        torch.cuda.synchronize()
        for k, ref in refs.items():
            check(get(outs[k]), ref, f"{k} ({'f32' if out_f32 else 'bf16'})")


@pytest.mark.parametrize("bits,group,M,K,N", [(8, 64, 70, 256, 150), (8, 128, 65, 256, 129),
                                              (4, 32, 40, 256, 100), (4, 64, 128, 192, 64)])
def test_prefill_indexing_bit_exact(mt, bits, group, M, K, N):
    """Codes, power-of-two scales, biases on a 2^-8 grid and small integer x:
    every product and partial sum is exact in fp32, so the output equals the
    oracle bit for bit whatever the tile, group and summation order."""
    rng = np.random.default_rng(bits * 11 + group + M + K + N)
    qmax = (1 << bits) - 1
    G = K // group
    codes = rng.integers(0, qmax + 1, size=(N, K)).astype(np.uint8)
    s = oracle.bf16_from_f64(np.ldexp(1.0, rng.integers(-8, -3, size=(N, G))))
    b = oracle.bf16_from_f64(rng.integers(-32, 32, size=(N, G)) * 2.0 ** -8)
    x = oracle.bf16_from_f64(rng.integers(-4, 5, size=(M, K)).astype(np.float64))
    res = oracle.bf16_from_f64(rng.integers(-8, 9, size=(M, N)).astype(np.float64))
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    fmt = 1 if bits == 8 else 2
    mt.mt_prefill_down_residual(dev_bf16(x), torch.from_numpy(oracle.pack_codes(codes, bits)).cuda(), dev_bf16(s),
                                dev_bf16(b), group, dev_bf16(res), y, _ws(mt, M, K, N, group), fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.down_residual(x, oracle.Weight(oracle.FMT_CODES, codes, s, b, group), res)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


def test_prefill_in_place_residual(mt):
    M, K, N, g = 80, 512, 256, 64
    x = synth.host_bf16(M * K, 12501, synth.ACT).reshape(M, K)
    res = synth.host_bf16(M * N, 12502, synth.ACT).reshape(M, N)
    W = synth.host_f32(N * K, 12503, synth.WEIGHT).reshape(N, K)
    q, s, b = _pack(mt, W, 1, g)
    rd = dev_bf16(res)
    mt.mt_prefill_down_residual(dev_bf16(x), q, s, b, g, rd, rd, _ws(mt, M, K, N, g), fmt=1)
    torch.cuda.synchronize()
    assert_bf16_close(host_bits(rd), oracle.down_residual(x, oracle.Weight.from_f32(W, 8, g), res), "in place")


@pytest.mark.parametrize("M", [256])
def test_prefill_qwen3_8b_layer(mt, M):
    """The 4096 x 12288 affine INT8 g128 layer at M = 256: gate/up and down on
    64 sampled output features each, every activation row."""
    wl = synth.QWEN8B
    d, f, g = wl.d, wl.f, wl.group
    L = DevLayer(mt, wl, 0)
    x = synth.host_bf16(M * d, synth.seed_for(wl.wid, 0, synth.T_X) + M, synth.ACT).reshape(M, d)
    hin = synth.host_bf16(M * f, synth.seed_for(wl.wid, 0, synth.T_H) + M, synth.ACT).reshape(M, f)
    res = synth.host_bf16(M * d, synth.seed_for(wl.wid, 0, synth.T_RES3) + M, synth.ACT).reshape(M, d)
    h = torch.empty(M, f, dtype=torch.float32, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_prefill_swiglu_gateup(dev_bf16(x), L.Wg, L.Wu, L.sgu, L.bgu, g, h, _ws(mt, M, d, f, g), fmt=wl.fmt)
    mt.mt_prefill_down_residual(dev_bf16(hin), L.Wd, L.sdn, L.bdn, g, dev_bf16(res), y, _ws(mt, M, f, d, g),
                                fmt=wl.fmt)
    torch.cuda.synchronize()
    rg = np.sort(np.random.default_rng(21).choice(f, 64, replace=False))
    rg[-1] = f - 1
    rd = np.sort(np.random.default_rng(22).choice(d, 64, replace=False))
    h_ref = oracle.swiglu_gateup(x, L.oracle_rows(synth.T_WG, rg, f, d), L.oracle_rows(synth.T_WU, rg, f, d))
    y_ref = oracle.down_residual(hin, L.oracle_rows(synth.T_WD, rd, d, f), res[:, rd])
    assert_f32_close(host_f64(h)[:, rg], h_ref, "h sampled")
    assert_bf16_close(host_bits(y)[:, rd], y_ref, "y sampled")


@pytest.mark.parametrize("M", [40, 300])
def test_prefill_llama_layer_int4(mt, M):
    """The Llama-3.2-1B-shaped layer (d=2048, f=8192, affine INT4 g64) at M = 40
    (narrow tile, split K) and M = 300 (two 256-row tiles): gate/up and down on
    every activation row, 48 sampled output features each, bf16 outputs."""
    wl = synth.LLAMA1B
    d, f, g = wl.d, wl.f, wl.group
    L = DevLayer(mt, wl, 0)
    x = synth.host_bf16(M * d, synth.seed_for(wl.wid, 0, synth.T_X) + M, synth.ACT).reshape(M, d)
    hin = synth.host_bf16(M * f, synth.seed_for(wl.wid, 0, synth.T_H) + M, synth.ACT).reshape(M, f)
    res = synth.host_bf16(M * d, synth.seed_for(wl.wid, 0, synth.T_RES3) + M, synth.ACT).reshape(M, d)
    h = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_prefill_swiglu_gateup(dev_bf16(x), L.Wg, L.Wu, L.sgu, L.bgu, g, h, _ws(mt, M, d, f, g), fmt=wl.fmt)
    mt.mt_prefill_down_residual(dev_bf16(hin), L.Wd, L.sdn, L.bdn, g, dev_bf16(res), y, _ws(mt, M, f, d, g),
                                fmt=wl.fmt)
    torch.cuda.synchronize()
    rg = np.sort(np.random.default_rng(31).choice(f, 48, replace=False))
    rd = np.sort(np.random.default_rng(32).choice(d, 48, replace=False))
    h_ref = oracle.swiglu_gateup(x, L.oracle_rows(synth.T_WG, rg, f, d), L.oracle_rows(synth.T_WU, rg, f, d))
    y_ref = oracle.down_residual(hin, L.oracle_rows(synth.T_WD, rd, d, f), res[:, rd])
    assert_bf16_close(host_bits(h)[:, rg], h_ref, "h sampled")
    assert_bf16_close(host_bits(y)[:, rd], y_ref, "y sampled")


@pytest.mark.parametrize("bits,M,K,N", [(8, 40, 512, 200), (8, 300, 1024, 136), (4, 70, 512, 129),
                                        (4, 257, 256, 96)])
def test_prefill_mx(mt, bits, M, K, N):
    """MXFP8 / MXFP4 weights (E8M0 block scales per 32) on the prefill GEMMs:
    gate/up, down and projection against the oracle, bf16 and fp32 outputs."""
    fmt = 3 if bits == 8 else 4
    seed = 13000 + bits + M + K + N
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    Wg = synth.host_f32(N * K, seed + 1, synth.WEIGHT).reshape(N, K)
    Wu = synth.host_f32(N * K, seed + 2, synth.WEIGHT_OUTLIERS).reshape(N, K)

    def pack(W):
        q = torch.empty(N, K * bits // 8, dtype=torch.uint8, device="cuda")
        s = torch.empty(N, K // 32, dtype=torch.uint8, device="cuda")
        mt.mt_pack_mx(torch.from_numpy(np.ascontiguousarray(W)).cuda(), N, K, bits, q, s)
        return q, s

    (qg, sg), (qu, su) = pack(Wg), pack(Wu)
    torch.cuda.synchronize()
    og, ou = oracle.Weight.from_f32_mx(Wg, bits), oracle.Weight.from_f32_mx(Wu, bits)
    res = synth.host_bf16(M * N, seed + 3, synth.ACT).reshape(M, N)
    bias = synth.host_bf16(N, seed + 4, synth.PROJ_BIAS)
    refs = {"h": oracle.swiglu_gateup(x, og, ou), "y": oracle.down_residual(x, og, res),
            "y + bias": oracle.linear_bias(x, ou, bias)}
    ws = _ws(mt, M, K, N, 32)
    xd = dev_bf16(x)
    sgu = torch.stack([sg, su]).contiguous()
    for out_f32 in (False, True):
        dt = torch.float32 if out_f32 else torch.bfloat16
        check = assert_f32_close if out_f32 else assert_bf16_close
        get = host_f64 if out_f32 else host_bits
        outs = {k: torch.empty(M, N, dtype=dt, device="cuda") for k in refs}
        mt.mt_prefill_swiglu_gateup(xd, qg, qu, sgu, None, 32, outs["h"], ws, fmt=fmt)
        mt.mt_prefill_down_residual(xd, qg, sg, None, 32, dev_bf16(res), outs["y"], ws, fmt=fmt)
        mt.mt_prefill_linear_bias(xd, qu, su, None, 32, dev_bf16(bias), outs["y + bias"], ws, fmt=fmt)
        torch.cuda.synchronize()
        for k, ref in refs.items():
            check(get(outs[k]), ref, f"{k} ({'f32' if out_f32 else 'bf16'})")


@pytest.mark.parametrize("M,K,N", [(40, 512, 200), (130, 1536, 136), (300, 768, 64), (9, 64, 77)])
def test_prefill_bf16_weights(mt, M, K, N):
    """Dense bf16 weights on the prefill GEMMs (bf16 MMA operands, x as
    stored): gate/up, down and projection against the oracle."""
    seed = 14000 + M + K + N
    x = synth.host_bf16(M * K, seed, synth.ACT).reshape(M, K)
    Wg = synth.host_bf16(N * K, seed + 1, synth.WEIGHT).reshape(N, K)
    Wu = synth.host_bf16(N * K, seed + 2, synth.WEIGHT).reshape(N, K)
    og, ou = oracle.Weight(oracle.FMT_BF16, Wg), oracle.Weight(oracle.FMT_BF16, Wu)
    res = synth.host_bf16(M * N, seed + 3, synth.ACT).reshape(M, N)
    bias = synth.host_bf16(N, seed + 4, synth.PROJ_BIAS)
    refs = {"h": oracle.swiglu_gateup(x, og, ou), "y": oracle.down_residual(x, og, res),
            "y + bias": oracle.linear_bias(x, ou, bias)}
    ws = _ws(mt, M, K, N, 0)
    xd, gd, ud = dev_bf16(x), dev_bf16(Wg), dev_bf16(Wu)
    for out_f32 in (False, True):
        dt = torch.float32 if out_f32 else torch.bfloat16
        check = assert_f32_close if out_f32 else assert_bf16_close
        get = host_f64 if out_f32 else host_bits
        outs = {k: torch.empty(M, N, dtype=dt, device="cuda") for k in refs}
        mt.mt_prefill_swiglu_gateup(xd, gd, ud, None, None, 0, outs["h"], ws, fmt=0)
        mt.mt_prefill_down_residual(xd, gd, None, None, 0, dev_bf16(res), outs["y"], ws, fmt=0)
        mt.mt_prefill_linear_bias(xd, ud, None, None, 0, dev_bf16(bias), outs["y + bias"], ws, fmt=0)
        torch.cuda.synchronize()
        for k, ref in refs.items():
            check(get(outs[k]), ref, f"{k} ({'f32' if out_f32 else 'bf16'})")

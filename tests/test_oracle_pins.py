"""Pins of the float64 CPU oracle to facts that do not come from the oracle.

Each oracle function is tied to at least one of: hand-derived fixtures
(tests/golden), IEEE-754 textbook cases, a library routine on the special case
where it applies (torch's fp32 -> bf16 conversion), exact rational brute force
(fractions.Fraction) on tiny shapes, closed forms and invariants.  Shapes are
non-square and M > 1 where it matters, so a transposed operand, a swapped gate
and up, a wrong group index or a dropped term fails a test.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- helpers
def torch_bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    """Library conversion fp32 -> bf16 (round to nearest even) as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def torch_f64_from_bf16(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def frac_bf16(bits: int) -> Fraction:
    return Fraction(float(torch_f64_from_bf16(np.array([bits], dtype=np.uint16))[0]))


def bf16_neighbours_nearest(value: Fraction, bits: int) -> bool:
    """True if bf16 `bits` is a nearest bf16 to the exact `value` (checks the
    two adjacent bf16 patterns of the same sign)."""
    c = frac_bf16(bits)
    d = abs(c - value)
    for nb in (bits - 1, bits + 1):
        if 0 <= nb < 0x10000 and (nb & 0x7F80) != 0x7F80:
            if abs(frac_bf16(nb) - value) < d:
                return False
    return True


def gen_bf16(n, seed, dist=synth.ACT):
    return synth.host_bf16(n, seed, dist)


# ------------------------------------------------------------------ bf16
def _read_bf16_cases():
    rows = []
    with open(os.path.join(GOLD, "bf16_cases.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            a, b = line.split()[:2]
            rows.append((float.fromhex(a) if a not in ("inf", "-inf", "nan") else float(a), int(b, 16)))
    return rows


@pytest.mark.parametrize("x,expect", _read_bf16_cases())
def test_bf16_textbook_cases(x, expect):
    got = int(oracle.bf16_from_f64(np.array([x]))[0])
    assert got == expect, f"{x!r}: {got:04x} != {expect:04x}"


def test_bf16_matches_library_on_fp32_values():
    # For inputs that are binary32 values a single rounding from binary64 and
    # torch's fp32 -> bf16 conversion must agree bit for bit.
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    x32 = u.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    # add exact ties and near-ties around bf16 rounding boundaries
    base = rng.integers(0, 2**16, size=20000, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    near = (base | 0x7FFF).view(np.float32)
    x32 = np.concatenate([x32, ties[np.isfinite(ties)], near[np.isfinite(near)]])
    got = oracle.bf16_from_f64(x32.astype(np.float64))
    exp = torch_bf16_bits_from_f32(x32)
    assert np.array_equal(got, exp)


def test_bf16_decode_matches_library_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f64_from_bf16(bits)
    exp = torch_f64_from_bf16(bits)
    nan = np.isnan(exp)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], exp[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(exp[~nan]))


def test_bf16_round_trip_identity():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.f64_from_bf16(bits)
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.bf16_from_f64(vals[ok]), bits[ok])


# ------------------------------------------------------------- quantiser
def _read_quant_groups():
    groups, cur = [], None
    with open(os.path.join(GOLD, "quant_groups.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "group":
                cur = dict(name=tok[1], bits=int(tok[2].split("=")[1]), vals=[], codes=[])
                groups.append(cur)
            elif tok[0] in ("scale", "bias"):
                cur[tok[0]] = int(tok[1], 16)
            else:
                cur["vals"].append(float.fromhex(tok[0]))
                cur["codes"].append(int(tok[1]))
    return groups


@pytest.mark.parametrize("grp", _read_quant_groups(), ids=lambda g: g["name"])
def test_quantizer_hand_built_groups(grp):
    g = 32
    vals = grp["vals"] + [grp["vals"][0]] * (g - len(grp["vals"]))
    codes_exp = grp["codes"] + [grp["codes"][0]] * (g - len(grp["codes"]))
    W = np.array([vals], dtype=np.float32)
    assert np.array_equal(W.astype(np.float64)[0], np.array(vals))  # all exact in fp32
    codes, s, b = oracle.quantize(W, g, grp["bits"])
    assert list(codes[0]) == codes_exp
    assert int(s[0, 0]) == grp["scale"]
    assert int(b[0, 0]) == grp["bias"]


def test_quantizer_grid_round_trip_exact():
    # scale 2^-8 / 2^-4 exactly: dequantised values reproduce the inputs
    for bits, step in ((8, 2.0 ** -8), (4, 2.0 ** -4)):
        qmax = (1 << bits) - 1
        k = np.arange(64) % (qmax + 1)
        k[0], k[1] = 0, qmax
        W = (k * step).astype(np.float32)[None, :].repeat(3, 0)
        codes, s, b = oracle.quantize(W, 64, bits)
        assert np.array_equal(codes[0], k)
        wd = oracle.dequant(codes, s, b, 64)
        assert np.array_equal(wd, W.astype(np.float64))


def test_quantizer_against_brute_force_argmin():
    rng = np.random.default_rng(7)
    for bits, group in ((8, 32), (4, 32), (8, 64), (4, 128)):
        qmax = (1 << bits) - 1
        N, K = 3, 2 * group
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        W[1, 5] *= 20.0  # an outlier inside one group
        codes, s, b = oracle.quantize(W, group, bits)
        assert codes.shape == (N, K) and s.shape == (N, K // group)
        for n in range(N):
            for gi in range(K // group):
                seg = W[n, gi * group:(gi + 1) * group].astype(np.float64)
                mn, mx = Fraction(float(seg.min())), Fraction(float(seg.max()))
                # bias: nearest bf16 to min (library conversion of an fp32 value)
                assert int(b[n, gi]) == int(torch_bf16_bits_from_f32(np.array([seg.min()], np.float32))[0])
                # scale: a nearest bf16 to (max - min) / qmax
                assert bf16_neighbours_nearest((mx - mn) / qmax, int(s[n, gi]))
                sc, bi = frac_bf16(int(s[n, gi])), frac_bf16(int(b[n, gi]))
                for k in range(group):
                    w = Fraction(float(seg[k]))
                    errs = [abs(w - (sc * c + bi)) for c in range(qmax + 1)]
                    best = min(errs)
                    cands = [c for c in range(qmax + 1) if errs[c] == best]
                    exp_c = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
                    assert codes[n, gi * group + k] == exp_c


def test_quantizer_error_bound():
    # |w - w'| <= scale/2 + |bias - min| + qmax*|scale - (max-min)/qmax| (closed form)
    W = synth.host_f32(16 * 256, 99, synth.WEIGHT_OUTLIERS).reshape(16, 256)
    for bits in (8, 4):
        qmax = (1 << bits) - 1
        codes, s, b = oracle.quantize(W, 64, bits)
        wd = oracle.dequant(codes, s, b, 64)
        sv = oracle.f64_from_bf16(s).repeat(64, axis=1)
        bv = oracle.f64_from_bf16(b).repeat(64, axis=1)
        Wg = W.astype(np.float64).reshape(16, 4, 64)
        mn = Wg.min(-1).repeat(64, axis=1)
        mx = Wg.max(-1).repeat(64, axis=1)
        bound = sv / 2 + np.abs(bv - mn) + qmax * np.abs(sv - (mx - mn) / qmax)
        assert np.all(np.abs(W - wd) <= bound * (1 + 1e-12))


def test_quantizer_constant_and_zero_groups():
    W = np.zeros((2, 64), dtype=np.float32)
    W[1, :] = -0.75
    codes, s, b = oracle.quantize(W, 32, 8)
    assert not codes.any() and not s.any()
    assert list(b[0]) == [0, 0] and list(b[1]) == [0xBF40, 0xBF40]
    assert np.array_equal(oracle.dequant(codes, s, b, 32), W.astype(np.float64))


def test_zero_minimum_gives_positive_zero_bias():
    W = np.full((1, 32), 0.5, dtype=np.float32)
    W[0, 3] = -0.0
    W[0, 7] = 0.0
    _, _, b = oracle.quantize(W, 32, 8)
    assert int(b[0, 0]) == 0x0000


def test_groups_run_along_k_not_n():
    # Row 0 uses a small range, row 1 a large one, and the two halves of each
    # row differ: scales must be indexed [n][k / group].
    W = np.zeros((2, 64), dtype=np.float32)
    W[0, :32] = np.linspace(0, 1, 32)
    W[0, 32:] = np.linspace(0, 2, 32)
    W[1, :32] = np.linspace(0, 4, 32)
    W[1, 32:] = np.linspace(0, 8, 32)
    _, s, _ = oracle.quantize(W, 32, 8)
    vals = oracle.f64_from_bf16(s)
    assert vals[0, 0] < vals[0, 1] < vals[1, 0] < vals[1, 1]


def test_pack_codes_layout():
    codes = np.array([[1, 2, 3, 4, 15, 0], [0, 15, 7, 8, 9, 10]], dtype=np.uint8)
    p4 = oracle.pack_codes(codes, 4)
    assert p4.tolist() == [[0x21, 0x43, 0x0F], [0xF0, 0x87, 0xA9]]
    p8 = oracle.pack_codes(codes, 8)
    assert np.array_equal(p8, codes)
    with pytest.raises(ValueError):
        oracle.pack_codes(np.array([[16, 0]], dtype=np.uint8), 4)


def test_dequant_exact_rational():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(3, 64)).astype(np.uint8)
    s = torch_bf16_bits_from_f32(rng.uniform(1e-4, 1e-2, size=(3, 2)).astype(np.float32))
    b = torch_bf16_bits_from_f32(rng.uniform(-0.1, 0.0, size=(3, 2)).astype(np.float32))
    wd = oracle.dequant(codes, s, b, 32)
    for n in range(3):
        for k in range(64):
            exp = frac_bf16(int(s[n, k // 32])) * int(codes[n, k]) + frac_bf16(int(b[n, k // 32]))
            assert Fraction(float(wd[n, k])) == exp


# --------------------------------------------------------------- RMSNorm
def _read_rms_cases():
    rows = []
    with open(os.path.join(GOLD, "rmsnorm_worked.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, eps, v, r, w, exp = line.split()
            hx = lambda t: np.array([int(x, 16) for x in t.split(",")], dtype=np.uint16)
            rows.append((name, float(eps), hx(v), hx(r), hx(w), np.array([float(x) for x in exp.split(",")])))
    return rows


@pytest.mark.parametrize("case", _read_rms_cases(), ids=lambda c: c[0])
def test_rmsnorm_worked_vectors(case):
    _, eps, v, r, w, exp = case
    out_sum, norm = oracle.add_rmsnorm(v, r, w, eps)
    np.testing.assert_allclose(norm[0], exp, rtol=2e-16 * 8, atol=0)
    assert np.array_equal(out_sum[0], oracle.bf16_from_f64(oracle.f64_from_bf16(v) + oracle.f64_from_bf16(r)))


def test_rmsnorm_constant_vector_closed_form():
    for c_bits, eps in ((0x4040, 1e-5), (0x3C00, 1e-6), (0xC2C8, 1e-5)):
        d = 96
        v = np.full(d, c_bits, dtype=np.uint16)
        r = np.zeros(d, dtype=np.uint16)
        w = gen_bf16(d, 5, synth.NORM_W)
        _, norm = oracle.add_rmsnorm(v, r, w, eps)
        c = float(oracle.f64_from_bf16(np.array([c_bits]))[0])
        exp = c * oracle.f64_from_bf16(w) / math.sqrt(c * c + eps)
        np.testing.assert_allclose(norm[0], exp, rtol=1e-14)


def test_add_rmsnorm_brute_force_and_fusion_invariance():
    M, d = 3, 40
    v = gen_bf16(M * d, 11).reshape(M, d)
    r = gen_bf16(M * d, 12).reshape(M, d)
    w = gen_bf16(d, 13, synth.NORM_W)
    eps = 1e-5
    out_sum, norm = oracle.add_rmsnorm(v, r, w, eps)
    vf, rf, wf = torch_f64_from_bf16(v), torch_f64_from_bf16(r), torch_f64_from_bf16(w)
    # summed output = bf16(values + residual); for these operands the fp32 sum
    # is exact, so the library conversion of it is the reference
    assert np.array_equal(out_sum, torch_bf16_bits_from_f32((vf + rf).astype(np.float32)))
    sf = torch_f64_from_bf16(out_sum)
    for m in range(M):
        ms = sum(Fraction(float(x)) ** 2 for x in sf[m]) / d
        den = math.sqrt(float(ms) + eps)
        exp = [float(sf[m, i]) * float(wf[i]) / den for i in range(d)]
        np.testing.assert_allclose(norm[m], exp, rtol=1e-14)
    # rows are independent: permuting rows permutes both outputs
    perm = [2, 0, 1]
    s2, n2 = oracle.add_rmsnorm(v[perm], r[perm], w, eps)
    assert np.array_equal(s2, out_sum[perm]) and np.array_equal(n2, norm[perm])


def test_rmsnorm_scale_invariance():
    d = 64
    v = gen_bf16(d, 21)
    r = np.zeros(d, dtype=np.uint16)
    w = gen_bf16(d, 22, synth.NORM_W)
    v4 = oracle.bf16_from_f64(oracle.f64_from_bf16(v) * 4.0)  # exact power-of-two scaling
    _, n1 = oracle.add_rmsnorm(v, r, w, 1e-12)
    _, n4 = oracle.add_rmsnorm(v4, r, w, 1e-12)
    np.testing.assert_allclose(n1, n4, rtol=1e-10)


# ---------------------------------------------------------------- SwiGLU
def _weight(fmt_bits, N, K, group, seed, dist=synth.WEIGHT):
    W32 = synth.host_f32(N * K, seed, dist).reshape(N, K)
    return oracle.Weight.from_f32(W32, fmt_bits, group)


def _frac_dense(w: oracle.Weight):
    if w.fmt == oracle.FMT_BF16:
        return [[Fraction(float(x)) for x in row] for row in torch_f64_from_bf16(w.W)]
    out = []
    G = w.W.shape[1] // w.group
    for n in range(w.W.shape[0]):
        row = []
        for k in range(w.W.shape[1]):
            sc = frac_bf16(int(w.scales[n, k // w.group]))
            bi = frac_bf16(int(w.biases[n, k // w.group]))
            row.append(sc * int(w.W[n, k]) + bi)
        out.append(row)
    return out


@pytest.mark.parametrize("fmt_bits,group", [(8, 32), (4, 64), (16, 0)])
def test_swiglu_gateup_brute_force(fmt_bits, group):
    M, K, N = 2, 128, 5
    x = gen_bf16(M * K, 31).reshape(M, K)
    Wg = _weight(fmt_bits, N, K, group, 32)
    Wu = _weight(fmt_bits, N, K, group, 33)
    h, g, u = oracle.swiglu_gateup(x, Wg, Wu, return_gu=True)
    xf = [[Fraction(float(t)) for t in row] for row in torch_f64_from_bf16(x)]
    Gd, Ud = _frac_dense(Wg), _frac_dense(Wu)
    for m in range(M):
        for n in range(N):
            ge = sum(a * b for a, b in zip(xf[m], Gd[n]))
            ue = sum(a * b for a, b in zip(xf[m], Ud[n]))
            scale = float(sum(abs(a * b) for a, b in zip(xf[m], Gd[n])))
            assert abs(g[m, n] - float(ge)) <= 1e-14 * scale
            assert abs(u[m, n] - float(ue)) <= 1e-14 * float(sum(abs(a * b) for a, b in zip(xf[m], Ud[n])))
            hb = float(ge) / (1.0 + math.exp(-float(ge))) * float(ue)
            assert abs(h[m, n] - hb) <= 1e-13 * max(1.0, abs(hb))
    # gate and up are not interchangeable
    h_swapped = oracle.swiglu_gateup(x, Wu, Wg)
    assert not np.allclose(h, h_swapped)


def _const_weight(N, K, group, scale_bits, bias_bits, code):
    G = K // group
    return oracle.Weight(oracle.FMT_CODES, np.full((N, K), code, np.uint8),
                         np.full((N, G), scale_bits, np.uint16), np.full((N, G), bias_bits, np.uint16),
                         group)


def test_silu_special_cases():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(20.0) - 20.0) <= 20.0 * 2.1e-9
    assert 0 > oracle.silu(-20.0) > -20.0 * math.exp(-20.0) * 1.0000001
    K, N = 64, 3
    x = gen_bf16(K, 41)[None, :]
    zero = _const_weight(N, K, 32, 0, 0, 0)                 # all-zero gate rows
    Wu = _weight(8, N, K, 32, 42)
    h = oracle.swiglu_gateup(x, zero, Wu)
    assert np.all(h == 0.0)
    # g = 20 exactly: x = 1 everywhere (bf16 0x3F80), gate weights 20/64 = 0.3125
    ones = np.full((1, K), 0x3F80, np.uint16)
    gate20 = _const_weight(N, K, 32, 0x3EA0, 0, 1)           # scale 0.3125 * q(=1)
    h, g, u = oracle.swiglu_gateup(ones, gate20, Wu, return_gu=True)
    assert np.all(g == 20.0)
    np.testing.assert_allclose(h, 20.0 * u, rtol=2.1e-9)
    gate_m20 = _const_weight(N, K, 32, 0, 0xBEA0, 0)         # bias -0.3125
    h, g, u = oracle.swiglu_gateup(ones, gate_m20, Wu, return_gu=True)
    assert np.all(g == -20.0)
    assert np.all(np.abs(h) <= 20.0 * math.exp(-20.0) * np.abs(u) * 1.0000001)


# ------------------------------------------------------------ down + res
@pytest.mark.parametrize("fmt_bits,group", [(8, 64), (4, 32), (16, 0)])
def test_down_residual_brute_force(fmt_bits, group):
    M, K, N = 2, 192, 7
    h = gen_bf16(M * K, 51).reshape(M, K)
    res = gen_bf16(M * N, 52).reshape(M, N)
    Wd = _weight(fmt_bits, N, K, group, 53)
    y = oracle.down_residual(h, Wd, res)
    hf = [[Fraction(float(t)) for t in row] for row in torch_f64_from_bf16(h)]
    rf = torch_f64_from_bf16(res)
    D = _frac_dense(Wd)
    for m in range(M):
        for n in range(N):
            exact = sum(a * b for a, b in zip(hf[m], D[n])) + Fraction(float(rf[m, n]))
            scale = float(sum(abs(a * b) for a, b in zip(hf[m], D[n]))) + abs(float(rf[m, n]))
            assert abs(y[m, n] - float(exact)) <= 1e-14 * scale


def test_down_residual_zero_weights_and_identity():
    M, K = 2, 64
    h = gen_bf16(M * K, 61).reshape(M, K)
    res = gen_bf16(M * K, 62).reshape(M, K)
    zero = _const_weight(K, K, 32, 0, 0, 0)
    y = oracle.down_residual(h, zero, res)
    assert np.array_equal(y, torch_f64_from_bf16(res))
    eye = oracle.Weight(oracle.FMT_BF16, np.where(np.eye(K, dtype=bool), 0x3F80, 0).astype(np.uint16))
    y = oracle.down_residual(h, eye, res)
    assert np.array_equal(y, torch_f64_from_bf16(h) + torch_f64_from_bf16(res))
    # a non-square projection with one non-zero column per row picks h[:, k]
    N = 5
    sel = np.zeros((N, K), np.uint16)
    for n in range(N):
        sel[n, 3 * n + 1] = 0x4000  # weight 2.0
    y = oracle.down_residual(h, oracle.Weight(oracle.FMT_BF16, sel), np.zeros((M, N), np.uint16))
    hf = torch_f64_from_bf16(h)
    assert np.array_equal(y, 2.0 * hf[:, [3 * n + 1 for n in range(N)]])


# ------------------------------------------------------------ projection
@pytest.mark.parametrize("fmt_bits,group,with_bias", [(8, 32, True), (4, 128, True), (16, 0, True),
                                                      (8, 64, False)])
def test_linear_bias_brute_force(fmt_bits, group, with_bias):
    M, K, N = 3, 256, 9
    x = gen_bf16(M * K, 111).reshape(M, K)
    W = _weight(fmt_bits, N, K, group, 112)
    bias = gen_bf16(N, 113) if with_bias else None
    y = oracle.linear_bias(x, W, bias)
    xf = [[Fraction(float(t)) for t in row] for row in torch_f64_from_bf16(x)]
    bf = torch_f64_from_bf16(bias) if with_bias else np.zeros(N)
    D = _frac_dense(W)
    for m in range(M):
        for n in range(N):
            exact = sum(a * b for a, b in zip(xf[m], D[n])) + Fraction(float(bf[n]))
            scale = float(sum(abs(a * b) for a, b in zip(xf[m], D[n]))) + abs(float(bf[n]))
            assert abs(y[m, n] - float(exact)) <= 1e-14 * scale
    if with_bias:
        # the bias is indexed by the output column, not by the row
        assert not np.allclose(y, oracle.linear_bias(x, W, bias[::-1].copy()))


def test_linear_bias_zero_weights_and_selection():
    M, K, N = 2, 128, 6
    x = gen_bf16(M * K, 121).reshape(M, K)
    bias = gen_bf16(N, 122)
    zero = _const_weight(N, K, 64, 0, 0, 0)
    y = oracle.linear_bias(x, zero, bias)
    assert np.array_equal(y, np.broadcast_to(torch_f64_from_bf16(bias), (M, N)))
    assert np.array_equal(oracle.linear_bias(x, zero), np.zeros((M, N)))
    # one non-zero column per row: row n of W picks x[:, 5n + 2] times 0.5
    sel = np.zeros((N, K), np.uint16)
    for n in range(N):
        sel[n, 5 * n + 2] = 0x3F00  # weight 0.5
    y = oracle.linear_bias(x, oracle.Weight(oracle.FMT_BF16, sel), bias)
    xf = torch_f64_from_bf16(x)
    expect = 0.5 * xf[:, [5 * n + 2 for n in range(N)]] + torch_f64_from_bf16(bias)[None, :]
    assert np.array_equal(y, expect)


def test_linear_bias_tied_embedding_reading():
    # A tied embedding used as the vocabulary projection: E [V, d] is the weight
    # as stored ([N, K] = [V, d]), so a one-hot activation e_j returns column j
    # of E for every vocabulary row, and the logit of row v is x . E[v].
    V, d = 11, 64
    E = _weight(8, V, d, 32, 131)
    Ed = E.dense()
    for j in (0, 17, d - 1):
        x = np.zeros((1, d), np.uint16)
        x[0, j] = 0x3F80  # 1.0
        assert np.array_equal(oracle.linear_bias(x, E)[0], Ed[:, j])


# ------------------------------------------------------------- MX formats
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX v1.0, FP4 E2M1 values of codes 0..7


def _read_mx_cases():
    rows = []
    with open(os.path.join(GOLD, "mx_cases.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            kind, v, code = line.split()[:3]
            rows.append((kind, float.fromhex(v), int(code, 16)))
    return rows


@pytest.mark.parametrize("kind,v,expect", _read_mx_cases())
def test_mx_textbook_cases(kind, v, expect):
    if kind == "e4m3":
        assert oracle.e4m3_from_f64(v) == expect
    elif kind == "e2m1":
        assert oracle.e2m1_from_f64(v) == expect
    else:
        bits = 8 if kind == "scale8" else 4
        W = np.zeros((1, 64), np.float32)
        W[0, 5] = np.float32(v)          # block 0 holds the maximum
        W[0, 40] = np.float32(-v) * 0.5  # block 1: half of it, negative
        codes, s = oracle.quantize_mx(W, bits)
        assert int(s[0, 0]) == expect
        if v > 0:
            # the second block's maximum is half: one field lower, unless clamped
            assert int(s[0, 1]) == max(0, expect - 1) or expect == 0


def test_e4m3_decode_matches_library_all_codes():
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(ours[ok], lib[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(lib[ok]))


def test_e2m1_decode_table():
    for c in range(16):
        mag = E2M1_TABLE[c & 7]
        v = oracle.e2m1_value(c)
        assert abs(v) == mag and (math.copysign(1.0, v) < 0) == bool(c & 8)


def test_e4m3_encode_matches_library_in_range():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.normal(0, 1, 4000) * 2.0 ** rng.integers(-12, 8, 4000),
        # every midpoint between neighbouring finite codes (ties)
        [(oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)) / 2 for c in range(0, 126)],
    ]).astype(np.float32)
    lib = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_from_f64(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(ours, lib)


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(12)
    vals = list(rng.uniform(-7, 7, 3000)) + [m / 4 for m in range(-28, 29)]
    for v in vals:
        c = oracle.e2m1_from_f64(v)
        a = min(abs(v), 6.0)
        dist = [abs(a - t) for t in E2M1_TABLE]
        best = min(dist)
        cands = [i for i, dd in enumerate(dist) if dd == best]
        want = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        assert c & 7 == want, (v, c)
        assert bool(c & 8) == (math.copysign(1.0, v) < 0)


def test_quantize_mx_round_trip_and_bound():
    rng = np.random.default_rng(13)
    # blocks whose values are all representable at scale 2^(E-127): exact
    for bits, table in ((8, [oracle.e4m3_value(c) for c in range(0x7F)]), (4, E2M1_TABLE)):
        E = 120
        vals = np.array(table)[rng.integers(0, len(table), size=(4, 64))] * rng.choice([-1, 1], (4, 64))
        vals[:, 0] = table[-1]  # each block's maximum is the largest finite element
        vals[:, 32] = table[-1]
        W = (vals * 2.0 ** (E - 127)).astype(np.float32)
        codes, s = oracle.quantize_mx(W, bits)
        emax = 8 if bits == 8 else 2
        assert np.all(s == int(math.floor(math.log2(table[-1]))) - emax + 127 + (E - 127))
        assert np.array_equal(oracle.dequant_mx(codes, s, bits), W.astype(np.float64))
    # random blocks: error within half a spacing of the element format at the
    # scaled value, or the clamp of values above the largest finite element
    W = synth.host_f32(8 * 256, 14, synth.WEIGHT_OUTLIERS).reshape(8, 256)
    for bits, mbits, lo_exp, maxv in ((8, 3, -6, 448.0), (4, 1, 0, 6.0)):
        codes, s = oracle.quantize_mx(W, bits)
        X = np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)
        v = W.astype(np.float64) / X
        back = oracle.dequant_mx(codes, s, bits) / X
        a = np.minimum(np.abs(v), maxv)
        e = np.floor(np.log2(np.maximum(a, 2.0 ** lo_exp)))
        half = np.ldexp(0.5, (e - mbits).astype(int))
        assert np.all(np.abs(np.sign(v) * a - back) <= half)


@pytest.mark.parametrize("bits", [8, 4])
def test_mx_gemvs_brute_force(bits):
    M, K, N = 2, 96, 5
    x = gen_bf16(M * K, 141).reshape(M, K)
    W32 = synth.host_f32(N * K, 142, synth.WEIGHT).reshape(N, K)
    W = oracle.Weight.from_f32_mx(W32, bits)
    # exact weight values from the library decode (E4M3) or the E2M1 table
    if bits == 8:
        dec = torch.from_numpy(W.W).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        dec = np.array([[math.copysign(E2M1_TABLE[c & 7], -1.0 if c & 8 else 1.0) for c in row]
                        for row in W.W])
    D = [[Fraction(float(dec[n, k])) * Fraction(2) ** (int(W.scales[n, k // 32]) - 127) for k in range(K)]
         for n in range(N)]
    xf = [[Fraction(float(t)) for t in row] for row in torch_f64_from_bf16(x)]
    bias = gen_bf16(N, 143)
    y = oracle.linear_bias(x, W, bias)
    res = gen_bf16(M * N, 144).reshape(M, N)
    yd = oracle.down_residual(x, W, res)
    for m in range(M):
        for n in range(N):
            dot = sum(a * b for a, b in zip(xf[m], D[n]))
            scale = float(sum(abs(a * b) for a, b in zip(xf[m], D[n])))
            exact = dot + Fraction(float(torch_f64_from_bf16(bias[n:n + 1])[0]))
            assert abs(y[m, n] - float(exact)) <= 1e-14 * (scale + 1)
            exact_d = dot + Fraction(float(torch_f64_from_bf16(res[m, n:n + 1])[0]))
            assert abs(yd[m, n] - float(exact_d)) <= 1e-14 * (scale + 1)
    # gate/up with two MX matrices
    W2 = oracle.Weight.from_f32_mx(synth.host_f32(N * K, 145, synth.WEIGHT).reshape(N, K), bits)
    h, g, u = oracle.swiglu_gateup(x, W, W2, return_gu=True)
    for m in range(M):
        for n in range(N):
            ge = float(sum(a * b for a, b in zip(xf[m], D[n])))
            assert abs(g[m, n] - ge) <= 1e-14 * (abs(ge) + float(sum(abs(a * b) for a, b in zip(xf[m], D[n]))))


# ----------------------------------------------------------- composition
def test_mlp_layer_and_stack_composition():
    d, f, M, g = 64, 96, 2, 32
    rng_seed = 70
    v = [gen_bf16(M * d, rng_seed + i).reshape(M, d) for i in range(2)]
    r0 = gen_bf16(M * d, rng_seed + 5).reshape(M, d)
    layers = []
    for l in range(2):
        layers.append((gen_bf16(d, 80 + l, synth.NORM_W), _weight(8, f, d, g, 90 + l),
                       _weight(8, f, d, g, 95 + l), _weight(8, d, f, g, 99 + l)))
    out = oracle.mlp_stack(v, r0, layers, 1e-5)
    r = r0
    for l in range(2):
        w, Wg, Wu, Wd = layers[l]
        s, nx = oracle.add_rmsnorm(v[l], r, w, 1e-5)
        hx = oracle.swiglu_gateup(oracle.bf16_from_f64(nx), Wg, Wu)
        yx = oracle.down_residual(oracle.bf16_from_f64(hx), Wd, s)
        assert np.array_equal(out[l]["out_sum"], s)
        assert np.array_equal(out[l]["h"], oracle.bf16_from_f64(hx))
        assert np.array_equal(out[l]["y_x"], yx)
        r = oracle.bf16_from_f64(yx)
    assert not np.array_equal(out[0]["y"], out[1]["y"])


# ------------------------------------------------- composition, closed forms
# "Compute-Graph Fusion", Automatic Gated Epilogues: the down projection adds
# the transformer residual (the layer's own summed row) in its epilogue, and
# each tensor handed to the next call is bf16.  These cases fix the answer
# without the oracle: dense bf16 weights with zeros or one non-zero entry
# reduce every dot product to at most one exact product.

def _dense(bits):
    return oracle.Weight(oracle.FMT_BF16, np.ascontiguousarray(bits, dtype=np.uint16))


def _torch_bf16_add(a_bits, b_bits):
    """bf16(a + b) by torch (bf16 tensors on the CPU)."""
    ta = torch.from_numpy(np.ascontiguousarray(a_bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(np.ascontiguousarray(b_bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return (ta + tb).view(torch.int16).numpy().view(np.uint16)


def test_mlp_layer_zero_down_returns_summed():
    """Wd = 0: y == out_sum bit for bit, and out_sum == torch's bf16(v + r),
    so the residual of the down projection is the layer's own summed row
    (not r, not the normalised row) and y is rounded once from it."""
    d, f, M = 48, 80, 3
    v = gen_bf16(M * d, 301).reshape(M, d)
    r = gen_bf16(M * d, 302).reshape(M, d)
    w = gen_bf16(d, 303, synth.NORM_W)
    Wg = _dense(gen_bf16(f * d, 304, synth.WEIGHT).reshape(f, d))
    Wu = _dense(gen_bf16(f * d, 305, synth.WEIGHT).reshape(f, d))
    Wd = _dense(np.zeros((d, f), dtype=np.uint16))
    out = oracle.mlp_layer(v, r, w, 1e-5, Wg, Wu, Wd)
    assert np.array_equal(out["out_sum"], _torch_bf16_add(v, r))
    assert np.array_equal(out["y"], out["out_sum"])
    assert not np.array_equal(out["y"], r) and np.any(out["h"] != 0)


@pytest.mark.parametrize("zero", ["gate", "up"])
def test_mlp_layer_zero_gate_or_up_gives_zero_h(zero):
    """Wg = 0 (silu(0) = 0) or Wu = 0: every h is zero and y == out_sum."""
    d, f, M = 40, 56, 2
    v = gen_bf16(M * d, 311).reshape(M, d)
    r = gen_bf16(M * d, 312).reshape(M, d)
    w = gen_bf16(d, 313, synth.NORM_W)
    rnd = _dense(gen_bf16(f * d, 314, synth.WEIGHT).reshape(f, d))
    zero_w = _dense(np.zeros((f, d), dtype=np.uint16))
    Wg, Wu = (zero_w, rnd) if zero == "gate" else (rnd, zero_w)
    Wd = _dense(gen_bf16(d * f, 315, synth.WEIGHT).reshape(d, f))
    out = oracle.mlp_layer(v, r, w, 1e-5, Wg, Wu, Wd)
    assert np.all(oracle.f64_from_bf16(out["h"]) == 0.0)
    assert np.array_equal(out["y"], out["out_sum"])


def test_mlp_stack_chains_y_into_the_next_residual():
    """Two layers with Wg = Wd = 0: y_l = out_sum_l, so
    y_1 = bf16(v_1 + bf16(v_0 + r_0)) (torch bf16 adds)."""
    d, f, M = 32, 64, 2
    v0 = gen_bf16(M * d, 321).reshape(M, d)
    v1 = gen_bf16(M * d, 322).reshape(M, d)
    r0 = gen_bf16(M * d, 323).reshape(M, d)
    zg = _dense(np.zeros((f, d), dtype=np.uint16))
    zd = _dense(np.zeros((d, f), dtype=np.uint16))
    up = _dense(gen_bf16(f * d, 324, synth.WEIGHT).reshape(f, d))
    layer = (gen_bf16(d, 325, synth.NORM_W), zg, up, zd)
    out = oracle.mlp_stack([v0, v1], r0, [layer, layer], 1e-6)
    y0 = _torch_bf16_add(v0, r0)
    assert np.array_equal(out[0]["y"], y0)
    assert np.array_equal(out[1]["y"], _torch_bf16_add(v1, y0))
    assert not np.array_equal(out[1]["y"], _torch_bf16_add(v1, r0))


def _one_hot_case(s0_bits, w0_bits, a_bits, b_bits, c_bits, d=8, f=4, n0=2, eps=1e-5):
    """summed = (s0, 0, ..., 0); Wg[n][0] = a, Wu[n][0] = b for every n;
    Wd[0][n0] = c, other weights 0.  Returns the oracle layer and the closed
    form with Python floats: x0 = bf16(s0 w0 / sqrt(s0^2 / d + eps)),
    h = bf16(silu(x0 a) * x0 b), y0 = bf16(h c + s0), and the variants that
    skip the rounding of x0 or of h."""
    f64 = lambda b: float(torch_f64_from_bf16(np.array([b], dtype=np.uint16))[0])
    v = np.zeros((1, d), dtype=np.uint16)
    v[0, 0] = s0_bits
    r = np.zeros((1, d), dtype=np.uint16)  # summed = v + 0 = v exactly
    w = np.full(d, 0x3F80, dtype=np.uint16)  # 1.0
    w[0] = w0_bits
    Wg = np.zeros((f, d), dtype=np.uint16)
    Wu = np.zeros((f, d), dtype=np.uint16)
    Wg[:, 0] = a_bits
    Wu[:, 0] = b_bits
    Wd = np.zeros((d, f), dtype=np.uint16)
    Wd[0, n0] = c_bits
    out = oracle.mlp_layer(v, r, w, eps, _dense(Wg), _dense(Wu), _dense(Wd))
    s0, w0, a, b, c = (f64(t) for t in (s0_bits, w0_bits, a_bits, b_bits, c_bits))
    bf = lambda x: int(oracle.bf16_from_f64(np.array([x]))[0])
    nx = s0 * w0 / math.sqrt(s0 * s0 / d + eps)
    silu = lambda g: g / (1.0 + math.exp(-g))
    x0 = f64(bf(nx))
    h = f64(bf(silu(x0 * a) * (x0 * b)))
    y0 = bf(h * c + s0)
    h_unrounded_x = f64(bf(silu(nx * a) * (nx * b)))
    y_unrounded_h = bf(silu(x0 * a) * (x0 * b) * c + s0)
    return out, bf(nx), h, y0, h_unrounded_x, y_unrounded_h


def test_mlp_layer_one_hot_closed_form_rounds_each_handoff():
    """One non-zero summed element and one-hot weights: out_norm, h and y
    follow from a single bf16 element in closed form (math.sqrt and
    math.exp in Python).  The case is chosen so that feeding the unrounded
    normalised value into gate/up, or the unrounded h into down, gives a
    different bf16 result: the oracle rounds both hand-offs."""
    found = 0
    for s0, w0, a, b, c in [(0x3FA0, 0x3F9A, 0x4040, 0x3FC8, 0x4120), (0x3F80, 0x3F8D, 0x40A3, 0x3FB1, 0x41F0),
                            (0x4010, 0x3FB7, 0x3FD3, 0x4003, 0x4250), (0xBF90, 0x3FA9, 0x4071, 0x3F93, 0x4305)]:
        out, x0_bits, h, y0, h_alt, y_alt = _one_hot_case(s0, w0, a, b, c)
        assert out["out_norm"][0, 0] == x0_bits
        assert np.all(oracle.f64_from_bf16(out["h"][0]) == h)
        assert out["y"][0, 0] == y0
        assert np.array_equal(out["y"][0, 1:], out["out_sum"][0, 1:])  # rows with no weights: the residual
        if h_alt != h and y_alt != y0:
            found += 1
    assert found >= 1, "no case separates the rounded from the unrounded hand-offs"

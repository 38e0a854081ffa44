"""float64 CPU oracle of the one-row decode MLP -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code with the CUDA library: the arithmetic lives in ``orc.c`` (plain
C loops in IEEE binary64, its own bf16 rounding and quantiser), compiled with
gcc on first use; this module only marshals numpy arrays.

What each function follows (meTile docs unless stated):

* :func:`bf16_from_f64` -- round-to-nearest-even to bf16 from binary64 in one
  step (the storage type of every activation, "MLX-LM Backend", Dispatch Policy
  and Block-Scaled MLX Primitive: BF16 inputs and outputs, FP32 accumulation).
* :func:`quantize`, :func:`pack_codes`, :func:`dequant` -- affine group
  quantisation w = scale*q + bias along K with groups of 32/64/128 in INT8 or
  4-bit nibbles ("MLX-LM Backend", prepare/autotune section and Dispatch
  Policy: "affine nibbles, scales, and biases").
* :func:`add_rmsnorm` -- summed = values + residual and
  normalized = rms_norm(summed, weight, eps), both kept as outputs
  ("Compute-Graph Fusion", opening example).
* :func:`swiglu_gateup` -- two projections sharing one activation, then
  silu(gate) * up ("Compute-Graph Fusion", Automatic Gated Epilogues).
* :func:`down_residual` -- values @ weight.T + residual, the down projection
  with the residual added in its epilogue ("Compute-Graph Fusion", Automatic
  Gated Epilogues; "MLX-LM Backend", Dispatch Policy).
* :func:`quantize_mx`, :func:`e4m3_value`, :func:`e2m1_value`,
  :meth:`Weight.from_f32_mx` -- MXFP8 / MXFP4 block-scaled weights: E4M3 or
  E2M1 elements with one E8M0 scale per 32 elements along K ("MLX-LM
  Backend", Block-Scaled MLX Primitive; encodings and block size as in the
  OCP Microscaling Formats (MX) v1.0 specification named by the format).
  Every GEMV above accepts them.
* :func:`linear_bias` -- values @ weight.T + bias for the attention
  projections (q/k/v/o, bias kept) and the vocabulary projection, which run
  the same one-row GEMV ("MLX-LM Backend", the attention-projection and
  vocabulary compression passages before Dispatch Policy).
* :func:`mlp_layer`, :func:`mlp_stack` -- the three steps composed; a stack
  layer takes the previous layer's output as its residual.

Pinned by ``tests/test_oracle_pins.py`` (closed forms, textbook IEEE cases,
exact rational brute force, library routines for special cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orc.c")
_SO = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

FMT_BF16 = 0     # dense bf16 weights [N][K]
FMT_CODES = 1    # affine codes [N][K], one code per byte, + scales/biases
FMT_MXFP8 = 2    # E4M3 codes [N][K], one per byte, + E8M0 scales [N][K/32]
FMT_MXFP4 = 3    # E2M1 codes [N][K], one per byte, + E8M0 scales [N][K/32]
MX_BLOCK = 32


def build(force: bool = False) -> str:
    """Compile ``orc.c`` into ``liborc.so`` (gcc, binary64, no FMA contraction)."""
    if force or not (os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"], cwd=_HERE)
        os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            P, L, I, D = ctypes.c_void_p, ctypes.c_long, ctypes.c_int, ctypes.c_double
            sig = {
                "orc_bf16_from_f64": (ctypes.c_uint16, [D]),
                "orc_f64_from_bf16": (D, [ctypes.c_uint16]),
                "orc_bf16_from_f64_array": (None, [P, P, L]),
                "orc_f64_from_bf16_array": (None, [P, P, L]),
                "orc_quantize": (I, [P, L, L, I, I, P, P, P]),
                "orc_pack_codes": (I, [P, L, L, I, P]),
                "orc_dequant": (I, [P, P, P, L, L, I, P]),
                "orc_add_rmsnorm": (I, [P, P, P, D, L, L, P, P]),
                "orc_silu": (D, [D]),
                "orc_swiglu_gateup": (I, [P, L, L, L, I, P, P, P, P, P, P, I, P, P, P]),
                "orc_down_residual": (I, [P, L, L, L, I, P, P, P, I, P, P]),
                "orc_linear_bias": (I, [P, L, L, L, I, P, P, P, I, P, P]),
                "orc_e4m3_value": (D, [ctypes.c_uint8]),
                "orc_e2m1_value": (D, [ctypes.c_uint8]),
                "orc_e4m3_from_f64": (ctypes.c_uint8, [D]),
                "orc_e2m1_from_f64": (ctypes.c_uint8, [D]),
                "orc_quantize_mx": (I, [P, L, L, I, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data


# ------------------------------------------------------------------ bf16
def bf16_from_f64(x) -> np.ndarray:
    """binary64 -> bf16 bit patterns (uint16), nearest-even, one rounding."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().orc_bf16_from_f64_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def f64_from_bf16(h) -> np.ndarray:
    """bf16 bit patterns -> their exact binary64 values."""
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _L().orc_f64_from_bf16_array(h.ctypes.data, out.ctypes.data, h.size)
    return out


def silu(g: float) -> float:
    return _L().orc_silu(float(g))


# ------------------------------------------------------------- quantiser
def quantize(W, group: int, bits: int):
    """Affine group quantisation of fp32 W [N, K] along K.

    Returns (codes uint8 [N, K], scales uint16 [N, K/group], biases uint16 [N, K/group]).
    """
    W = _c(W, np.float32)
    N, K = W.shape
    G = K // group
    codes = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N, G), dtype=np.uint16)
    b = np.empty((N, G), dtype=np.uint16)
    rc = _L().orc_quantize(W.ctypes.data, N, K, group, bits, codes.ctypes.data, s.ctypes.data,
                           b.ctypes.data)
    if rc:
        raise ValueError("orc_quantize: bad arguments")
    return codes, s, b


def pack_codes(codes, bits: int) -> np.ndarray:
    """Stored byte layout: INT8 one byte per code; INT4 code 2j low nibble, 2j+1 high."""
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    out = np.empty((N, K if bits == 8 else K // 2), dtype=np.uint8)
    if _L().orc_pack_codes(codes.ctypes.data, N, K, bits, out.ctypes.data):
        raise ValueError("orc_pack_codes: bad arguments")
    return out


def e4m3_value(code: int) -> float:
    """Value of an OCP FP8 E4M3 code (NaN for S.1111.111)."""
    return _L().orc_e4m3_value(int(code))


def e2m1_value(code: int) -> float:
    """Value of an OCP FP4 E2M1 code (low four bits)."""
    return _L().orc_e2m1_value(int(code))


def e4m3_from_f64(v: float) -> int:
    """Nearest E4M3 code (ties to even, saturating at 448, sign kept)."""
    return int(_L().orc_e4m3_from_f64(float(v)))


def e2m1_from_f64(v: float) -> int:
    """Nearest E2M1 code (ties to even, saturating at 6, sign kept)."""
    return int(_L().orc_e2m1_from_f64(float(v)))


def quantize_mx(W, bits: int):
    """MX quantisation of fp32 W [N, K] along K in blocks of 32: bits 8 =
    MXFP8 (E4M3), bits 4 = MXFP4 (E2M1).  Returns (codes uint8 [N, K] one code
    per byte, scales uint8 [N, K/32] E8M0 fields)."""
    W = _c(W, np.float32)
    N, K = W.shape
    codes = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N, K // MX_BLOCK), dtype=np.uint8)
    if _L().orc_quantize_mx(W.ctypes.data, N, K, bits, codes.ctypes.data, s.ctypes.data):
        raise ValueError("orc_quantize_mx: bad arguments")
    return codes, s


def dequant_mx(codes, scales, bits: int) -> np.ndarray:
    """Exact values of MX weights [N, K]: element value * 2^(E - 127)."""
    W = Weight(FMT_MXFP8 if bits == 8 else FMT_MXFP4, codes, scales, None, MX_BLOCK)
    return W.dense()


def dequant(codes, scales, biases, group: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    out = np.empty((N, K), dtype=np.float64)
    if _L().orc_dequant(codes.ctypes.data, _p(_c(scales, np.uint16)), _p(_c(biases, np.uint16)),
                        N, K, group, out.ctypes.data):
        raise ValueError("orc_dequant: bad arguments")
    return out


# ------------------------------------------------------------------- K1
def add_rmsnorm(v, r, w, eps: float):
    """Returns (out_sum bf16 bits [M, d], out_norm exact float64 [M, d])."""
    v = _c(np.atleast_2d(v), np.uint16)
    r = _c(np.atleast_2d(r), np.uint16)
    w = _c(w, np.uint16)
    M, d = v.shape
    out_sum = np.empty((M, d), dtype=np.uint16)
    out_norm = np.empty((M, d), dtype=np.float64)
    if _L().orc_add_rmsnorm(v.ctypes.data, r.ctypes.data, w.ctypes.data, float(eps), M, d,
                            out_sum.ctypes.data, out_norm.ctypes.data):
        raise ValueError("orc_add_rmsnorm: bad arguments")
    return out_sum, out_norm


# ---------------------------------------------------------------- weights
class Weight:
    """One projection as the oracle consumes it: dense bf16 [N, K], or affine
    codes [N, K] (one code per byte) with bf16 scales/biases [N, K/group]."""

    def __init__(self, fmt, W, scales=None, biases=None, group=0):
        self.fmt = fmt
        self.W = _c(W, np.uint16 if fmt == FMT_BF16 else np.uint8)
        mx = fmt in (FMT_MXFP8, FMT_MXFP4)
        self.scales = None if scales is None else _c(scales, np.uint8 if mx else np.uint16)
        self.biases = None if (biases is None or mx) else _c(biases, np.uint16)
        self.group = MX_BLOCK if mx else int(group)

    @property
    def shape(self):
        return self.W.shape

    @classmethod
    def from_f32(cls, W32, fmt_bits: int, group: int):
        """Quantise fp32 weights with the oracle's own quantiser (bits 8 or 4);
        bits 16 rounds them to bf16."""
        if fmt_bits == 16:
            return cls(FMT_BF16, bf16_from_f64(np.asarray(W32, dtype=np.float64)))
        codes, s, b = quantize(W32, group, fmt_bits)
        return cls(FMT_CODES, codes, s, b, group)

    @classmethod
    def from_f32_mx(cls, W32, bits: int):
        """MX-quantise fp32 weights with the oracle's own quantiser (bits 8:
        MXFP8, bits 4: MXFP4)."""
        codes, s = quantize_mx(W32, bits)
        return cls(FMT_MXFP8 if bits == 8 else FMT_MXFP4, codes, s, None, MX_BLOCK)

    def dense(self) -> np.ndarray:
        if self.fmt == FMT_BF16:
            return f64_from_bf16(self.W)
        if self.fmt in (FMT_MXFP8, FMT_MXFP4):
            val = e4m3_value if self.fmt == FMT_MXFP8 else e2m1_value
            table = np.array([val(c) for c in range(256 if self.fmt == FMT_MXFP8 else 16)])
            codes = self.W if self.fmt == FMT_MXFP8 else (self.W & 0xF)
            scale = np.ldexp(1.0, self.scales.astype(np.int64) - 127)
            return table[codes] * np.repeat(scale, MX_BLOCK, axis=1)
        return dequant(self.W, self.scales, self.biases, self.group)


# ------------------------------------------------------------------- K2
def swiglu_gateup(x, Wg: Weight, Wu: Weight, return_gu: bool = False):
    """h[m, n] = silu(x . Wg[n]) * (x . Wu[n]), exact float64 [M, N]."""
    x = _c(np.atleast_2d(x), np.uint16)
    M, K = x.shape
    N, K2 = Wg.shape
    assert K2 == K and Wu.shape == Wg.shape and Wg.fmt == Wu.fmt
    h = np.empty((M, N), dtype=np.float64)
    g = np.empty((M, N), dtype=np.float64) if return_gu else None
    u = np.empty((M, N), dtype=np.float64) if return_gu else None
    rc = _L().orc_swiglu_gateup(x.ctypes.data, M, K, N, Wg.fmt, Wg.W.ctypes.data, Wu.W.ctypes.data,
                                _p(Wg.scales), _p(Wg.biases), _p(Wu.scales), _p(Wu.biases),
                                Wg.group, h.ctypes.data, _p(g), _p(u))
    if rc:
        raise ValueError("orc_swiglu_gateup: bad arguments")
    return (h, g, u) if return_gu else h


# ------------------------------------------------------------------- K3
def down_residual(h, Wd: Weight, res):
    """y[m, n] = h[m] . Wd[n] + res[m, n], exact float64 [M, N]."""
    h = _c(np.atleast_2d(h), np.uint16)
    res = _c(np.atleast_2d(res), np.uint16)
    M, K = h.shape
    N, K2 = Wd.shape
    assert K2 == K and res.shape == (M, N)
    y = np.empty((M, N), dtype=np.float64)
    rc = _L().orc_down_residual(h.ctypes.data, M, K, N, Wd.fmt, Wd.W.ctypes.data, _p(Wd.scales),
                                _p(Wd.biases), Wd.group, res.ctypes.data, y.ctypes.data)
    if rc:
        raise ValueError("orc_down_residual: bad arguments")
    return y


# ----------------------------------------------------------- projection
def linear_bias(x, W: Weight, bias=None):
    """y[m, n] = x[m] . W[n] + bias[n] (bias bf16 [N], or None for none),
    exact float64 [M, N]."""
    x = _c(np.atleast_2d(x), np.uint16)
    M, K = x.shape
    N, K2 = W.shape
    assert K2 == K
    if bias is not None:
        bias = _c(bias, np.uint16).reshape(-1)
        assert bias.shape == (N,)
    y = np.empty((M, N), dtype=np.float64)
    rc = _L().orc_linear_bias(x.ctypes.data, M, K, N, W.fmt, W.W.ctypes.data, _p(W.scales),
                              _p(W.biases), W.group, _p(bias), y.ctypes.data)
    if rc:
        raise ValueError("orc_linear_bias: bad arguments")
    return y


# ------------------------------------------------------------- composed
def mlp_layer(v, r, w_norm, eps, Wg: Weight, Wu: Weight, Wd: Weight):
    """One decode MLP layer; each tensor that crosses a call boundary is rounded
    to bf16.  Returns dict of out_sum, out_norm, h, y (bf16 bits) and the exact
    pre-rounding values (norm_x, h_x, y_x)."""
    out_sum, norm_x = add_rmsnorm(v, r, w_norm, eps)
    out_norm = bf16_from_f64(norm_x)
    h_x = swiglu_gateup(out_norm, Wg, Wu)
    h = bf16_from_f64(h_x)
    y_x = down_residual(h, Wd, out_sum)
    y = bf16_from_f64(y_x)
    return dict(out_sum=out_sum, out_norm=out_norm, h=h, y=y, norm_x=norm_x, h_x=h_x, y_x=y_x)


def mlp_stack(values_per_layer, r0, layers, eps):
    """Layers run back to back: layer l takes values_per_layer[l] as its values
    and the previous layer's y as its residual.  ``layers`` is a list of
    (w_norm, Wg, Wu, Wd).  Returns the list of per-layer result dicts."""
    out = []
    r = r0
    for v, (w_norm, Wg, Wu, Wd) in zip(values_per_layer, layers):
        res = mlp_layer(v, r, w_norm, eps, Wg, Wu, Wd)
        out.append(res)
        r = res["y"]
    return out

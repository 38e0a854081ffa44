"""Seeded synthetic inputs shared by the tests, the bench and the oracle's callers.

The generator is defined once in ``synth_core.h`` (SplitMix64 counter stream ->
Irwin-Hall twelve-uniform normal approximation -> one IEEE rounding per
operation -> optional Bernoulli outlier scaling -> bf16 round-to-nearest-even
for activations).  ``libmtsynth_host.so`` evaluates it on the host and
``libmtsynth_dev.so`` on the GPU; both give the same bits for the same element
index.  Nothing here computes any part of the decode MLP itself.

The workloads below stand in for the Llama/Qwen-shaped layers the meTile
"MLX-LM Backend" page measures (no checkpoints are used or needed): every
tensor is drawn from the generator with the distribution stated per workload.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libmtsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libmtsynth_dev.so")
_lock = threading.Lock()
_host = None
_dev = None

# tensor ids inside one layer's seed space
T_VALUES, T_RESIDUAL, T_NORM_W, T_WG, T_WU, T_WD, T_X, T_H, T_RES3 = range(9)
# projections: stacked q/k/v weight and bias, o weight, vocabulary weight
T_WQKV, T_BQKV, T_WO, T_WVOCAB = range(9, 13)

OUTLIER_P32_1PCT = 42949673  # round(0.01 * 2**32)


def seed_for(workload_id: int, layer: int, tensor: int) -> int:
    """Seed of one tensor: 0x5EED0000 + 16*workload + tensor, layer in the high word."""
    return (0x5EED0000 + 16 * workload_id + tensor + (layer << 32)) & 0xFFFFFFFFFFFFFFFF


def _newer(dst: str, srcs) -> bool:
    return os.path.exists(dst) and all(os.path.getmtime(dst) >= os.path.getmtime(s) for s in srcs)


def build(force: bool = False, device: bool = True) -> None:
    """Compile the host (gcc) and device (nvcc, sm_103a) generator libraries."""
    hdr = os.path.join(_HERE, "synth_core.h")
    hsrc = os.path.join(_HERE, "synth_host.c")
    if force or not _newer(_HOST_SO, [hdr, hsrc]):
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", _HOST_SO, hsrc],
            cwd=_HERE)
    if device:
        dsrc = os.path.join(_HERE, "synth_dev.cu")
        if force or not _newer(_DEV_SO, [hdr, dsrc]):
            subprocess.check_call(
                ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                 "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_SO, dsrc],
                cwd=_HERE)


def _host_lib():
    global _host
    with _lock:
        if _host is None:
            build(device=False)
            lib = ctypes.CDLL(_HOST_SO)
            for name, ptr_t in (("syn_fill_f32_host", ctypes.c_void_p),
                                ("syn_fill_bf16_host", ctypes.c_void_p)):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = [ptr_t, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                               ctypes.c_float, ctypes.c_float, ctypes.c_uint32, ctypes.c_float]
            _host = lib
    return _host


def _dev_lib():
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(_DEV_SO):
                raise RuntimeError("synth device library missing: run synth.build()")
            lib = ctypes.CDLL(_DEV_SO)
            for name in ("syn_fill_f32_device", "syn_fill_bf16_device"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                               ctypes.c_float, ctypes.c_float, ctypes.c_uint32, ctypes.c_float,
                               ctypes.c_void_p]
            _dev = lib
    return _dev


@dataclass(frozen=True)
class Dist:
    """Distribution of one tensor: normal(mean, std) with optional outliers."""
    mean: float = 0.0
    std: float = 1.0
    outlier_p32: int = 0
    outlier_scale: float = 1.0

    def args(self):
        return (float(np.float32(self.mean)), float(np.float32(self.std)),
                int(self.outlier_p32), float(np.float32(self.outlier_scale)))


ACT = Dist(0.0, 1.0)
PROJ_BIAS = Dist(0.0, 0.5)
NORM_W = Dist(1.0, 0.1)
WEIGHT = Dist(0.0, 0.02)
WEIGHT_OUTLIERS = Dist(0.0, 0.02, OUTLIER_P32_1PCT, 20.0)


def host_f32(n: int, seed: int, dist: Dist, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _host_lib().syn_fill_f32_host(out.ctypes.data, n, seed, offset, *dist.args())
    return out


def host_bf16(n: int, seed: int, dist: Dist, offset: int = 0) -> np.ndarray:
    """bf16 values as their uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    _host_lib().syn_fill_bf16_host(out.ctypes.data, n, seed, offset, *dist.args())
    return out


def device_f32(tensor, seed: int, dist: Dist, offset: int = 0, stream=None) -> None:
    """Fill a contiguous float32 CUDA tensor in place."""
    import torch
    assert tensor.is_cuda and tensor.dtype == torch.float32 and tensor.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _dev_lib().syn_fill_f32_device(tensor.data_ptr(), tensor.numel(), seed, offset,
                                        *dist.args(), s)
    if rc != 0:
        raise RuntimeError(f"syn_fill_f32_device failed: cudaError {rc}")


def device_bf16(tensor, seed: int, dist: Dist, offset: int = 0, stream=None) -> None:
    """Fill a contiguous bfloat16 (or int16/uint16) CUDA tensor in place."""
    import torch
    assert tensor.is_cuda and tensor.element_size() == 2 and tensor.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _dev_lib().syn_fill_bf16_device(tensor.data_ptr(), tensor.numel(), seed, offset,
                                         *dist.args(), s)
    if rc != 0:
        raise RuntimeError(f"syn_fill_bf16_device failed: cudaError {rc}")


# ---------------------------------------------------------------------------
# Workloads (shapes and distributions of the five measured layer shapes)
# ---------------------------------------------------------------------------
FMT_BF16, FMT_AFFINE8, FMT_AFFINE4, FMT_MXFP8, FMT_MXFP4 = 0, 1, 2, 3, 4
FMT_NAMES = {FMT_BF16: "bf16", FMT_AFFINE8: "affine8", FMT_AFFINE4: "affine4", FMT_MXFP8: "mxfp8",
             FMT_MXFP4: "mxfp4"}
_FMT_BITS = {FMT_BF16: 16, FMT_AFFINE8: 8, FMT_AFFINE4: 4, FMT_MXFP8: 8, FMT_MXFP4: 4}


def is_mx(fmt: int) -> bool:
    return fmt in (FMT_MXFP8, FMT_MXFP4)


def scale_bytes(fmt: int, n_weights: int, group: int) -> int:
    """Scale (and bias) bytes of n_weights weights: affine 2 bf16 per group,
    MX one E8M0 byte per 32, bf16 none."""
    if fmt == FMT_BF16:
        return 0
    if is_mx(fmt):
        return n_weights // 32
    return 2 * 2 * (n_weights // group)


@dataclass(frozen=True)
class Workload:
    wid: int            # seed-space id
    name: str
    d: int              # hidden size
    f: int              # intermediate size
    M: int              # rows
    fmt: int            # weight format
    group: int          # affine group along K (0 for bf16)
    eps: float
    layers: int = 1
    weight_dist: Dist = WEIGHT
    out_f32: bool = False

    @property
    def bits(self) -> int:
        return _FMT_BITS[self.fmt]

    def weight_bytes(self) -> int:
        """Packed weight + scale/bias bytes of one layer (gate, up, down)."""
        n_w = 3 * self.d * self.f
        return n_w * self.bits // 8 + scale_bytes(self.fmt, n_w, self.group)

    def act_bytes(self) -> int:
        """Activation bytes of one layer: K1 reads v, r (2*M*d bf16) and the norm
        weight (d), writes out_sum and out_norm (2*M*d); K2 reads x (M*d), writes
        h (M*f); K3 reads h (M*f) and the residual (M*d), writes y (M*d)."""
        M, d, f = self.M, self.d, self.f
        return 2 * (7 * M * d + 2 * M * f + d)

    def layer_bytes(self) -> int:
        return self.weight_bytes() + self.act_bytes()

    def with_(self, **kw) -> "Workload":
        from dataclasses import replace
        return replace(self, **kw)


TINY = Workload(1, "tiny d256 f768 affine8 g64", 256, 768, 1, FMT_AFFINE8, 64, 1e-5)
LLAMA1B = Workload(2, "llama3.2-1b layer d2048 f8192 affine4 g64", 2048, 8192, 1, FMT_AFFINE4, 64, 1e-5)
QWEN15 = Workload(3, "qwen2.5-1.5b layer d1536 f8960 bf16", 1536, 8960, 1, FMT_BF16, 0, 1e-6)
QWEN8B = Workload(4, "qwen3-8b stack d4096 f12288 affine8 g128 x36", 4096, 12288, 1, FMT_AFFINE8, 128,
                  1e-6, layers=36)


# the Qwen3-8B layer with MX block-scaled weights (OCP MXFP8 / MXFP4, E8M0
# scales per 32): a stack of distinct layers, timed through the single calls
QWEN8B_MXFP8 = Workload(11, "qwen3-8b layer d4096 f12288 mxfp8", 4096, 12288, 1, FMT_MXFP8, 32, 1e-6,
                        layers=8)
QWEN8B_MXFP4 = Workload(12, "qwen3-8b layer d4096 f12288 mxfp4", 4096, 12288, 1, FMT_MXFP4, 32, 1e-6,
                        layers=8)


def sweep_point(group: int, M: int) -> Workload:
    return Workload(5, f"sweep d2048 f8192 affine8 g{group} M{M} outliers", 2048, 8192, M,
                    FMT_AFFINE8, group, 1e-5, weight_dist=WEIGHT_OUTLIERS)


SWEEP = [sweep_point(g, m) for g in (32, 64, 128) for m in (1, 2, 4, 8)]
ALL = [TINY, LLAMA1B, QWEN15, QWEN8B] + SWEEP


# ---------------------------------------------------------------------------
# Projection workloads: the attention projections of a decode step (q, k and v
# stacked into one weight, as they share the activation, then o) and the
# vocabulary projection, with the shapes of the models named.
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Projection:
    name: str
    tensor: int                 # seed-space id of the weight
    K: int
    N: int
    bias: Optional[int] = None  # seed-space id of the bias, None without one
    per_layer: bool = True      # False: once per step (the vocabulary projection)


@dataclass(frozen=True)
class ProjWorkload:
    wid: int
    name: str
    M: int
    fmt: int
    group: int
    projs: tuple
    layers: int = 1
    weight_dist: Dist = WEIGHT

    @property
    def bits(self) -> int:
        return _FMT_BITS[self.fmt]

    def proj_weight_bytes(self, p: Projection) -> int:
        wb = p.N * p.K * self.bits // 8
        sb = scale_bytes(self.fmt, p.N * p.K, self.group)
        return wb + sb + (2 * p.N if p.bias is not None else 0)

    def proj_act_bytes(self, p: Projection) -> int:
        """x read (M*K bf16) and y written (M*N bf16)."""
        return 2 * self.M * (p.K + p.N)

    def step_bytes(self) -> int:
        """Bytes one decode step's projections must move: per-layer projections
        once per layer, the vocabulary projection once."""
        tot = 0
        for p in self.projs:
            n = self.layers if p.per_layer else 1
            tot += n * (self.proj_weight_bytes(p) + self.proj_act_bytes(p))
        return tot


QWEN8B_PROJ = ProjWorkload(
    8, "qwen3-8b projections qkv 4096x6144 + o 4096x4096 x36, lm_head 4096x151936 affine8 g128",
    1, FMT_AFFINE8, 128,
    (Projection("qkv", T_WQKV, 4096, 6144), Projection("o", T_WO, 4096, 4096),
     Projection("lm_head", T_WVOCAB, 4096, 151936, per_layer=False)), layers=36)
QWEN15_PROJ = ProjWorkload(
    9, "qwen2.5-1.5b projections qkv+bias 1536x2048 + o 1536x1536, tied vocab 1536x151936 bf16",
    1, FMT_BF16, 0,
    (Projection("qkv", T_WQKV, 1536, 2048, bias=T_BQKV), Projection("o", T_WO, 1536, 1536),
     Projection("vocab", T_WVOCAB, 1536, 151936, per_layer=False)), layers=28)
LLAMA1B_PROJ = ProjWorkload(
    10, "llama3.2-1b projections qkv 2048x3072 + o 2048x2048, tied vocab 2048x128256 affine4 g64",
    1, FMT_AFFINE4, 64,
    (Projection("qkv", T_WQKV, 2048, 3072), Projection("o", T_WO, 2048, 2048),
     Projection("vocab", T_WVOCAB, 2048, 128256, per_layer=False)), layers=16)
PROJ_ALL = [QWEN8B_PROJ, QWEN15_PROJ, LLAMA1B_PROJ]

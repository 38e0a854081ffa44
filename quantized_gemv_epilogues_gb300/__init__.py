"""Python binding of the GB300 (sm_103a) decode-MLP library ``libmt.so``.

Argument marshalling only: every call forwards device pointers, sizes and the
current CUDA stream to the C ABI declared in ``include/mt.h``; all work runs in
the library's CUDA kernels.  There is no CPU fallback: importing this package
fails with ImportError when ``libmt.so`` has not been built (build it with
``python -c "import __graft_entry__ as g; g.build()"``).

Calls (same names as the C ABI):

* :func:`mt_add_rmsnorm` -- residual add + RMSNorm, both outputs written.
* :func:`mt_swiglu_gateup` -- gate/up GEMV with the silu(gate) * up epilogue.
* :func:`mt_down_residual` -- down GEMV with the residual added in its epilogue.
* :func:`mt_linear_bias` -- projection GEMV with an optional bias (attention
  q/k/v/o, vocabulary projection).
* :func:`mt_prefill_swiglu_gateup`, :func:`mt_prefill_down_residual`,
  :func:`mt_prefill_linear_bias` -- the same epilogues for many activation
  rows (prefill) on the tcgen05 tensor cores, with a caller-owned workspace
  of :func:`mt_prefill_workspace_bytes` bytes.
* :func:`mt_pack_affine` / :func:`mt_unpack_affine` -- affine group packer.
* :func:`mt_pack_mx` -- MXFP8 / MXFP4 block-scaled packer (E8M0 scales).
* :func:`mt_mlp_plan_create` / :func:`mt_mlp_plan_run` / :func:`mt_mlp_plan_destroy`
  -- the warmed executor: L one-row layers as one persistent kernel.
* :func:`mt_mlp_stack_run_noalloc` -- the same pass without any allocation.

Tensors are ``torch.Tensor`` on the current CUDA device (bf16 activations,
uint8 packed codes, bf16 scales/biases); raw integer device pointers are also
accepted, in which case the sizes given are trusted.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmt.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: the CUDA library has not been built "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

MT_OK, MT_ERR_NULL, MT_ERR_SHAPE, MT_ERR_GROUP, MT_ERR_ALIGN = 0, 1, 2, 3, 4
MT_ERR_FORMAT, MT_ERR_ALIAS, MT_ERR_CUDA, MT_ERR_TIMEOUT = 5, 6, 7, 8
MT_BF16, MT_F32 = 0, 1
MT_W_BF16, MT_W_AFFINE8, MT_W_AFFINE4, MT_W_MXFP8, MT_W_MXFP4 = 0, 1, 2, 3, 4
MT_OPT_PDL, MT_OPT_GEMV, MT_OPT_TEST_BARRIER_EXTRA, MT_OPT_ACT_BITS = 0, 1, 2, 3

_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_SIGS = {
    "mt_add_rmsnorm": (_I, [_P, _P, _P, _F, _P, _P, _I, _I, _I, _P]),
    "mt_swiglu_gateup": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "mt_down_residual": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "mt_linear_bias": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "mt_pack_affine": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "mt_unpack_affine": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "mt_pack_mx": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "mt_prefill_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "mt_prefill_swiglu_gateup": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "mt_prefill_down_residual": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "mt_prefill_linear_bias": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "mt_set_option": (_I, [_I, _I]),
    "mt_get_option": (_I, [_I]),
    "mt_status_string": (ctypes.c_char_p, [_I]),
    "mt_last_cuda_error": (_I, []),
    "mt_device_error": (_I, [_I]),
    "mt_version": (_I, []),
    "mt_mlp_plan_create": (_I, [_P, _I, _I, _I, _I, _I, _F, _P]),
    "mt_mlp_plan_run": (_I, [_P, _P, _P, _P, _P, _P]),
    "mt_mlp_plan_destroy": (_I, [_P]),
    "mt_mlp_stack_run_noalloc": (_I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class MlpLayer(ctypes.Structure):
    """``mt_mlp_layer``: one layer's device pointers."""
    _fields_ = [(n, _P) for n in ("norm_weight", "Wg", "Wu", "gu_scales", "gu_biases", "Wd",
                                  "d_scales", "d_biases")]


class MlpTrace(ctypes.Structure):
    """``mt_mlp_trace``: optional per-layer outputs (device pointers or NULL)."""
    _fields_ = [(n, _P) for n in ("out_sum", "out_norm", "h", "y")]


class MTError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = _lib.mt_status_string(status).decode()
        if status == MT_ERR_CUDA:
            msg += f" (cudaError {_lib.mt_last_cuda_error()})"
        super().__init__(f"{call}: {msg}")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, call: str) -> None:
    if st != MT_OK:
        raise MTError(st, call)


def _rows_cols(t, cols_hint=None):
    if isinstance(t, int):
        raise TypeError("shape arguments are required with raw pointers")
    if t.dim() == 1:
        return 1, t.shape[0]
    return t.shape[0], t.shape[1]


def _odt(t, explicit):
    if explicit is not None:
        return explicit
    import torch
    return MT_F32 if t.dtype == torch.float32 else MT_BF16


def mt_add_rmsnorm(values, residual, weight, eps, out_sum, out_norm, M=None, d=None,
                   norm_dtype=None, stream=None):
    if M is None or d is None:
        M, d = _rows_cols(values)
    nd = _odt(out_norm, norm_dtype) if not isinstance(out_norm, int) else (norm_dtype or MT_BF16)
    _check(_lib.mt_add_rmsnorm(_ptr(values), _ptr(residual), _ptr(weight), float(eps),
                               _ptr(out_sum), _ptr(out_norm), M, d, nd, _stream(stream)),
           "mt_add_rmsnorm")


def mt_swiglu_gateup(x, Wg, Wu, scales, biases, group, out_h, M=None, d=None, f=None, fmt=None,
                     out_dtype=None, stream=None):
    if M is None or d is None:
        M, d = _rows_cols(x)
    if f is None:
        f = _rows_cols(out_h)[1]
    if fmt is None:
        raise TypeError("fmt (MT_W_BF16 / MT_W_AFFINE8 / MT_W_AFFINE4) is required")
    od = _odt(out_h, out_dtype) if not isinstance(out_h, int) else (out_dtype or MT_BF16)
    _check(_lib.mt_swiglu_gateup(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(scales), _ptr(biases),
                                 int(group), _ptr(out_h), M, d, f, int(fmt), od, _stream(stream)),
           "mt_swiglu_gateup")


def mt_down_residual(h, Wd, scales, biases, group, residual, out_y, M=None, f=None, d=None,
                     fmt=None, out_dtype=None, stream=None):
    if M is None or f is None:
        M, f = _rows_cols(h)
    if d is None:
        d = _rows_cols(out_y)[1]
    if fmt is None:
        raise TypeError("fmt (MT_W_BF16 / MT_W_AFFINE8 / MT_W_AFFINE4) is required")
    od = _odt(out_y, out_dtype) if not isinstance(out_y, int) else (out_dtype or MT_BF16)
    _check(_lib.mt_down_residual(_ptr(h), _ptr(Wd), _ptr(scales), _ptr(biases), int(group),
                                 _ptr(residual), _ptr(out_y), M, f, d, int(fmt), od,
                                 _stream(stream)),
           "mt_down_residual")


def mt_linear_bias(x, W, scales, biases, group, bias, out_y, M=None, K=None, N=None, fmt=None,
                   out_dtype=None, stream=None):
    if M is None or K is None:
        M, K = _rows_cols(x)
    if N is None:
        N = _rows_cols(out_y)[1]
    if fmt is None:
        raise TypeError("fmt (MT_W_BF16 / MT_W_AFFINE8 / MT_W_AFFINE4) is required")
    od = _odt(out_y, out_dtype) if not isinstance(out_y, int) else (out_dtype or MT_BF16)
    _check(_lib.mt_linear_bias(_ptr(x), _ptr(W), _ptr(scales), _ptr(biases), int(group),
                               _ptr(bias), _ptr(out_y), M, K, N, int(fmt), od, _stream(stream)),
           "mt_linear_bias")


def mt_prefill_workspace_bytes(M, K, N, group):
    return int(_lib.mt_prefill_workspace_bytes(int(M), int(K), int(N), int(group)))


def _ws(workspace, M, K, N, group):
    need = mt_prefill_workspace_bytes(M, K, N, group)
    if workspace is None:
        raise TypeError(f"a device workspace of at least {need} bytes is required")
    nbytes = workspace.numel() * workspace.element_size() if not isinstance(workspace, int) else need
    return _ptr(workspace), nbytes


def mt_prefill_swiglu_gateup(x, Wg, Wu, scales, biases, group, out_h, workspace, M=None, d=None, f=None,
                             fmt=None, out_dtype=None, workspace_bytes=None, stream=None):
    if M is None or d is None:
        M, d = _rows_cols(x)
    if f is None:
        f = _rows_cols(out_h)[1]
    if fmt is None:
        raise TypeError("fmt (MT_W_AFFINE8 / MT_W_AFFINE4) is required")
    od = _odt(out_h, out_dtype) if not isinstance(out_h, int) else (out_dtype or MT_BF16)
    wp, wb = _ws(workspace, M, d, f, group)
    _check(_lib.mt_prefill_swiglu_gateup(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(scales), _ptr(biases), int(group),
                                         _ptr(out_h), M, d, f, int(fmt), od, wp,
                                         workspace_bytes if workspace_bytes is not None else wb, _stream(stream)),
           "mt_prefill_swiglu_gateup")


def mt_prefill_down_residual(h, Wd, scales, biases, group, residual, out_y, workspace, M=None, f=None, d=None,
                             fmt=None, out_dtype=None, workspace_bytes=None, stream=None):
    if M is None or f is None:
        M, f = _rows_cols(h)
    if d is None:
        d = _rows_cols(out_y)[1]
    if fmt is None:
        raise TypeError("fmt (MT_W_AFFINE8 / MT_W_AFFINE4) is required")
    od = _odt(out_y, out_dtype) if not isinstance(out_y, int) else (out_dtype or MT_BF16)
    wp, wb = _ws(workspace, M, f, d, group)
    _check(_lib.mt_prefill_down_residual(_ptr(h), _ptr(Wd), _ptr(scales), _ptr(biases), int(group),
                                         _ptr(residual), _ptr(out_y), M, f, d, int(fmt), od, wp,
                                         workspace_bytes if workspace_bytes is not None else wb, _stream(stream)),
           "mt_prefill_down_residual")


def mt_prefill_linear_bias(x, W, scales, biases, group, bias, out_y, workspace, M=None, K=None, N=None, fmt=None,
                           out_dtype=None, workspace_bytes=None, stream=None):
    if M is None or K is None:
        M, K = _rows_cols(x)
    if N is None:
        N = _rows_cols(out_y)[1]
    if fmt is None:
        raise TypeError("fmt (MT_W_AFFINE8 / MT_W_AFFINE4) is required")
    od = _odt(out_y, out_dtype) if not isinstance(out_y, int) else (out_dtype or MT_BF16)
    wp, wb = _ws(workspace, M, K, N, group)
    _check(_lib.mt_prefill_linear_bias(_ptr(x), _ptr(W), _ptr(scales), _ptr(biases), int(group), _ptr(bias),
                                       _ptr(out_y), M, K, N, int(fmt), od, wp,
                                       workspace_bytes if workspace_bytes is not None else wb, _stream(stream)),
           "mt_prefill_linear_bias")


def mt_pack_affine(W, N, K, group, bits, q, scales, biases, stream=None):
    _check(_lib.mt_pack_affine(_ptr(W), int(N), int(K), int(group), int(bits), _ptr(q),
                               _ptr(scales), _ptr(biases), _stream(stream)), "mt_pack_affine")


def mt_pack_mx(W, N, K, bits, q, scales, stream=None):
    _check(_lib.mt_pack_mx(_ptr(W), int(N), int(K), int(bits), _ptr(q), _ptr(scales), _stream(stream)),
           "mt_pack_mx")


def mt_unpack_affine(q, scales, biases, N, K, group, bits, W, stream=None):
    _check(_lib.mt_unpack_affine(_ptr(q), _ptr(scales), _ptr(biases), int(N), int(K), int(group),
                                 int(bits), _ptr(W), _stream(stream)), "mt_unpack_affine")


def mt_mlp_plan_create(layers, d, f, group, fmt, eps) -> int:
    """Binds L layers (each a mapping with the ``mt_mlp_layer`` field names to
    tensors or device pointers; scale/bias fields may be None for bf16) and
    returns the plan handle (an int)."""
    arr = (MlpLayer * len(layers))()
    for i, ly in enumerate(layers):
        for name, _ in MlpLayer._fields_:
            setattr(arr[i], name, _ptr(ly.get(name)))
    plan = ctypes.c_void_p()
    _check(_lib.mt_mlp_plan_create(arr, len(layers), int(d), int(f), int(group), int(fmt),
                                   float(eps), ctypes.byref(plan)), "mt_mlp_plan_create")
    return plan.value


def mt_mlp_plan_run(plan, values, residual, out_y, trace=None, stream=None) -> None:
    """One pass over the plan's layers.  trace: None or a mapping with some of
    out_sum / out_norm / h / y (tensors [L][.] or device pointers)."""
    tr = None
    if trace is not None:
        tr = MlpTrace(*[_ptr(trace.get(n)) for n, _ in MlpTrace._fields_])
    _check(_lib.mt_mlp_plan_run(plan, _ptr(values), _ptr(residual), _ptr(out_y),
                                ctypes.byref(tr) if tr is not None else None, _stream(stream)),
           "mt_mlp_plan_run")


def mt_mlp_plan_destroy(plan) -> None:
    _check(_lib.mt_mlp_plan_destroy(plan), "mt_mlp_plan_destroy")


def mt_mlp_stack_run_noalloc(layers, d, f, group, fmt, eps, values, residual, out_y,
                             stream=None) -> None:
    """The stack pass with the library's static scratch instead of a plan's
    memory (see include/mt.h)."""
    arr = (MlpLayer * len(layers))()
    for i, ly in enumerate(layers):
        for name, _ in MlpLayer._fields_:
            setattr(arr[i], name, _ptr(ly.get(name)))
    _check(_lib.mt_mlp_stack_run_noalloc(arr, len(layers), int(d), int(f), int(group), int(fmt),
                                         float(eps), _ptr(values), _ptr(residual), _ptr(out_y),
                                         _stream(stream)), "mt_mlp_stack_run_noalloc")


def mt_set_option(opt: int, value: int) -> None:
    _check(_lib.mt_set_option(int(opt), int(value)), "mt_set_option")


def mt_get_option(opt: int) -> int:
    return _lib.mt_get_option(int(opt))


def mt_status_string(status: int) -> str:
    return _lib.mt_status_string(int(status)).decode()


def mt_last_cuda_error() -> int:
    return _lib.mt_last_cuda_error()


def mt_device_error(clear: bool = False) -> int:
    return _lib.mt_device_error(1 if clear else 0)


def mt_version() -> int:
    return _lib.mt_version()


def raw(name: str):
    """The ctypes function of a C-ABI entry point (for tests that call the ABI
    directly with raw pointers)."""
    return getattr(_lib, name)

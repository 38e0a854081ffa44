"""Host-side checks of the C-ABI library: it builds, loads, exports every
function include/mt.h declares, and rejects invalid arguments with the
documented status before touching the GPU (no device is needed: validation
happens before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._libbuild().build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(mt_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("mt_add_rmsnorm", "mt_swiglu_gateup", "mt_down_residual", "mt_linear_bias",
              "mt_pack_affine"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mt_[a-z0-9_]+)", out))
    assert set(declared_functions()) <= exported


def test_header_compiles_as_c():
    src = '#include "mt.h"\nint main(void){ return (int)MT_OK; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", HEADER_DIR, "-x", "c", "-",
                        "-o", os.devnull], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


# fake, 16-byte aligned, non-overlapping "device" addresses: never dereferenced,
# because every case below fails validation first
A = [0x10000000 * (i + 1) for i in range(12)]
P = ctypes.c_void_p


def _rms(lib, *a):
    f = lib.mt_add_rmsnorm
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, ctypes.c_float, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    return f(*a)


def _gu(lib, *a):
    f = lib.mt_swiglu_gateup
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, P, ctypes.c_int, P] + [ctypes.c_int] * 5 + [P]
    return f(*a)


def _dn(lib, *a):
    f = lib.mt_down_residual
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, ctypes.c_int, P, P] + [ctypes.c_int] * 5 + [P]
    return f(*a)


def _lb(lib, *a):
    f = lib.mt_linear_bias
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, ctypes.c_int, P, P] + [ctypes.c_int] * 5 + [P]
    return f(*a)


def _pk(lib, *a):
    f = lib.mt_pack_affine
    f.restype = ctypes.c_int
    f.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P]
    return f(*a)


NULL, SHAPE, GROUP, ALIGN, FORMAT, ALIAS = 1, 2, 3, 4, 5, 6


def test_add_rmsnorm_validation(lib):
    v, r, w, s, n = A[:5]
    assert _rms(lib, None, r, w, 1e-5, s, n, 1, 256, 0, None) == NULL
    assert _rms(lib, v, r, w, 1e-5, s, n, 0, 256, 0, None) == SHAPE
    assert _rms(lib, v, r, w, 1e-5, s, n, 9, 256, 0, None) == SHAPE
    assert _rms(lib, v, r, w, 1e-5, s, n, 1, 260, 0, None) == SHAPE
    assert _rms(lib, v, r, w, -1.0, s, n, 1, 256, 0, None) == SHAPE
    assert _rms(lib, v, r, w, float("nan"), s, n, 1, 256, 0, None) == SHAPE
    assert _rms(lib, v, r, w, 1e-5, s, n, 1, 256, 7, None) == FORMAT
    assert _rms(lib, v + 2, r, w, 1e-5, s, n, 1, 256, 0, None) == ALIGN
    assert _rms(lib, v, r, w, 1e-5, v, n, 1, 256, 0, None) == ALIAS     # out_sum == values
    assert _rms(lib, v, r, w, 1e-5, s, r, 1, 256, 0, None) == ALIAS     # out_norm == residual
    assert _rms(lib, v, r, w, 1e-5, s, s + 16, 1, 256, 0, None) == ALIAS  # outputs overlap


def test_swiglu_gateup_validation(lib):
    x, wg, wu, sc, bi, h = A[:6]
    ok = dict(M=1, d=256, f=768, fmt=1, od=0)

    def call(x=x, wg=wg, wu=wu, sc=sc, bi=bi, g=64, h=h, M=1, d=256, f=768, fmt=1, od=0):
        return _gu(lib, x, wg, wu, sc, bi, g, h, M, d, f, fmt, od, None)

    assert call(x=None) == NULL
    assert call(sc=None) == NULL
    assert call(g=48) == GROUP
    assert call(fmt=0, g=64, sc=None, bi=None) == GROUP      # bf16 takes group 0
    assert call(d=200) == SHAPE                              # 200 % 64 != 0
    assert call(M=0) == SHAPE
    assert call(M=9) == SHAPE
    assert call(f=0) == SHAPE
    assert call(fmt=3) == FORMAT
    assert call(od=2) == FORMAT
    assert call(wu=wu + 8) == ALIGN
    assert call(h=x) == ALIAS
    assert call(h=sc) == ALIAS
    assert call(fmt=0, g=0, sc=None, bi=None, d=260) == SHAPE  # bf16 needs d % 8 == 0


def test_down_residual_validation(lib):
    h, wd, sc, bi, res, y = A[:6]

    def call(h=h, wd=wd, sc=sc, bi=bi, g=128, res=res, y=y, M=1, f=12288, d=4096, fmt=1, od=0):
        return _dn(lib, h, wd, sc, bi, g, res, y, M, f, d, fmt, od, None)

    assert call(res=None) == NULL
    assert call(g=16) == GROUP
    assert call(f=1000) == SHAPE
    assert call(f=40000) == SHAPE
    assert call(fmt=-1) == FORMAT
    assert call(y=y + 4) == ALIGN
    assert call(y=h) == ALIAS
    assert call(y=res + 16) == ALIAS          # partial overlap with the residual
    assert call(y=res, od=1) == ALIAS         # in place only with the same element size


def test_linear_bias_validation(lib):
    x, w, sc, bi, bias, y = A[:6]

    def call(x=x, w=w, sc=sc, bi=bi, g=64, bias=bias, y=y, M=1, K=1536, N=2048, fmt=2, od=0):
        return _lb(lib, x, w, sc, bi, g, bias, y, M, K, N, fmt, od, None)

    assert call(x=None) == NULL
    assert call(w=None) == NULL
    assert call(bi=None) == NULL
    assert call(g=96) == GROUP
    assert call(fmt=0, g=64, sc=None, bi=None) == GROUP      # bf16 takes group 0
    assert call(K=1000) == SHAPE                             # 1000 % 64 != 0
    assert call(K=32832) == SHAPE                            # above 32768
    assert call(N=0) == SHAPE
    assert call(N=(1 << 20) + 1) == SHAPE
    assert call(M=9) == SHAPE
    assert call(fmt=3) == FORMAT
    assert call(od=5) == FORMAT
    assert call(bias=bias + 2) == ALIGN
    assert call(y=y + 8) == ALIGN
    assert call(y=x) == ALIAS
    assert call(y=w + 64) == ALIAS
    assert call(y=bias) == ALIAS
    assert call(y=bi + 32) == ALIAS
    # MX formats: group 32, scales only
    assert call(fmt=3, g=64, bi=None) == GROUP
    assert call(fmt=4, g=32) == FORMAT                      # biases must be NULL
    assert call(fmt=4, g=32, sc=None, bi=None) == NULL
    assert call(fmt=5, g=32, bi=None) == FORMAT
    assert call(fmt=3, g=32, bi=None, K=1000) == SHAPE      # 1000 % 32 != 0
    assert call(fmt=3, g=32, bi=None, y=sc + 16) == ALIAS   # E8M0 scales: N * K/32 bytes


def test_prefill_validation(lib):
    wsb = lib.mt_prefill_workspace_bytes
    wsb.restype = ctypes.c_size_t
    wsb.argtypes = [ctypes.c_int] * 4
    assert wsb(100, 512, 256, 64) > 100 * 512 * 2      # at least the fp16 activations
    assert wsb(0, 512, 256, 64) == 0 and wsb(10, 512, 256, 48) == 0 and wsb(10, 32, 256, 32) == 0
    # the documented parts: fp16 activations, group sums [K/g][Mp], 2^-e_m [Mp] and the
    # dequantised weight rows' 2^t_n and 2^-t_n [2][2][N] (Mp: M rounded up to 256)
    for M, K, N, g in ((100, 512, 256, 64), (4096, 4096, 12288, 128), (9, 256, 200, 32), (1, 64, 5, 0)):
        Mp = -(-M // 256) * 256
        gb = g or max(v for v in (64, 128, 256, 512) if K % v == 0)  # dense bf16: its accumulation group
        G = K // gb
        assert wsb(M, K, N, g) >= 2 * M * K + 4 * G * Mp + 4 * Mp + 16 * N, (M, K, N, g)
    f = lib.mt_prefill_linear_bias
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, ctypes.c_int, P, P] + [ctypes.c_int] * 5 + [P, ctypes.c_size_t, P]
    x, w, sc, bi, bias, y, ws = A[:7]
    need = wsb(100, 512, 256, 64)

    def call(x=x, w=w, sc=sc, bi=bi, g=64, bias=bias, y=y, M=100, K=512, N=256, fmt=1, od=0, ws=ws, wb=need):
        return f(x, w, sc, bi, g, bias, y, M, K, N, fmt, od, ws, wb, None)

    assert call(ws=None) == NULL
    assert call(bi=None) == NULL
    assert call(fmt=0, g=64, sc=None, bi=None) == GROUP     # bf16 weights take group 0
    assert call(fmt=0, g=0, bi=None) == FORMAT              # and no scales
    assert call(fmt=3, g=32) == FORMAT                      # MX weights take no biases
    assert call(fmt=4, g=64, bi=None) == GROUP               # MX blocks are 32
    assert call(g=96) == GROUP
    assert call(K=480) == SHAPE                             # K % 64 != 0
    assert call(M=0) == SHAPE
    assert call(wb=need - 1) == SHAPE                       # workspace too small
    assert call(ws=ws + 8) == ALIGN
    assert call(y=ws + 64) == ALIAS                         # output inside the workspace
    assert call(ws=x) == ALIAS                              # workspace over the activations
    g = lib.mt_prefill_down_residual
    g.restype = ctypes.c_int
    g.argtypes = [P, P, P, P, ctypes.c_int, P, P] + [ctypes.c_int] * 5 + [P, ctypes.c_size_t, P]
    assert g(x, w, sc, bi, 64, None, y, 100, 512, 256, 1, 0, ws, need, None) == NULL  # residual required


def test_pack_mx_validation(lib):
    f = lib.mt_pack_mx
    f.restype = ctypes.c_int
    f.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P]
    W, q, s = A[:3]
    assert f(None, 4, 256, 8, q, s, None) == NULL
    assert f(W, 4, 256, 8, q, None, None) == NULL
    assert f(W, 4, 256, 6, q, s, None) == FORMAT
    assert f(W, 4, 100, 8, q, s, None) == SHAPE
    assert f(W, 4, 256, 8, q + 4, s, None) == ALIGN
    assert f(W, 4, 256, 8, q, q + 256, None) == ALIAS


def test_pack_validation(lib):
    W, q, s, b = A[:4]
    assert _pk(lib, None, 4, 256, 64, 8, q, s, b, None) == NULL
    assert _pk(lib, W, 4, 256, 64, 5, q, s, b, None) == FORMAT
    assert _pk(lib, W, 4, 256, 100, 8, q, s, b, None) == GROUP
    assert _pk(lib, W, 4, 250, 64, 8, q, s, b, None) == SHAPE
    assert _pk(lib, W, 4, 256, 64, 8, q, q, b, None) == ALIAS
    assert _pk(lib, W + 4, 4, 256, 64, 8, q, s, b, None) == ALIGN


def test_status_strings_and_options(lib):
    f = lib.mt_status_string
    f.restype = ctypes.c_char_p
    for s in range(9):
        assert f(s)
    assert f(99) == b"unknown mt_status"
    lib.mt_set_option.restype = ctypes.c_int
    lib.mt_get_option.restype = ctypes.c_int
    assert lib.mt_set_option(0, 0) == 0 and lib.mt_get_option(0) == 0
    assert lib.mt_set_option(0, 1) == 0 and lib.mt_get_option(0) == 1
    assert lib.mt_set_option(5, 1) == FORMAT
    assert lib.mt_set_option(1, 2) == 0 and lib.mt_get_option(1) == 2
    assert lib.mt_set_option(1, 3) == FORMAT and lib.mt_get_option(1) == 2
    assert lib.mt_set_option(1, 0) == 0
    assert lib.mt_set_option(2, 9) == FORMAT and lib.mt_set_option(2, -1) == FORMAT
    assert lib.mt_set_option(2, 0) == 0 and lib.mt_get_option(2) == 0
    assert lib.mt_get_option(3) == 16  # fixed-point activation bits, default
    assert lib.mt_set_option(3, 20) == FORMAT and lib.mt_get_option(3) == 16
    assert lib.mt_set_option(3, 24) == 0 and lib.mt_get_option(3) == 24
    assert lib.mt_set_option(3, 16) == 0 and lib.mt_get_option(3) == 16
    assert lib.mt_version() >> 16 == 1


class _Layer(ctypes.Structure):
    _fields_ = [(n, P) for n in ("norm_weight", "Wg", "Wu", "gu_scales", "gu_biases", "Wd",
                                 "d_scales", "d_biases")]


def _create(lib, layers, L, d=256, f=768, g=64, fmt=1, eps=1e-5, plan=True):
    fn = lib.mt_mlp_plan_create
    fn.restype = ctypes.c_int
    fn.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_float, P]
    out = P()
    return fn(layers, L, d, f, g, fmt, eps, ctypes.byref(out) if plan else None)


def test_mlp_plan_validation(lib):
    """mt_mlp_plan_create / run / destroy refuse invalid arguments before any
    CUDA call (so these run without a device)."""
    arr = (_Layer * 2)()
    for i in range(2):
        for j, (name, _) in enumerate(_Layer._fields_):
            setattr(arr[i], name, A[j] + 0x1000 * i)
    assert _create(lib, arr, 2, plan=False) == NULL
    assert _create(lib, None, 2) == NULL
    assert _create(lib, arr, 0) == SHAPE
    assert _create(lib, arr, 2, d=260) == SHAPE          # d % 8 != 0
    assert _create(lib, arr, 2, f=40000) == SHAPE
    assert _create(lib, arr, 2, d=96) == SHAPE           # d % group != 0
    assert _create(lib, arr, 2, eps=-1.0) == SHAPE
    assert _create(lib, arr, 2, g=48) == GROUP
    assert _create(lib, arr, 2, fmt=0) == GROUP          # bf16 takes group 0
    assert _create(lib, arr, 2, fmt=4) == FORMAT
    arr[1].Wd = None
    assert _create(lib, arr, 2) == NULL
    arr[1].Wd = A[5] + 0x1000
    arr[1].d_scales = None
    assert _create(lib, arr, 2) == NULL
    arr[1].d_scales = A[6] + 0x1008                        # misaligned scales
    assert _create(lib, arr, 2) == ALIGN
    run = lib.mt_mlp_plan_run
    run.restype = ctypes.c_int
    run.argtypes = [P, P, P, P, P, P]
    assert run(None, A[0], A[1], A[2], None, None) == NULL
    lib.mt_mlp_plan_destroy.restype = ctypes.c_int
    lib.mt_mlp_plan_destroy.argtypes = [P]
    assert lib.mt_mlp_plan_destroy(None) == NULL


def test_noalloc_validation(lib):
    """mt_mlp_stack_run_noalloc refuses invalid arguments before any CUDA call."""
    fn = lib.mt_mlp_stack_run_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_float, P, P, P, P]
    arr = (_Layer * 2)()
    for i in range(2):
        for j, (name, _) in enumerate(_Layer._fields_):
            setattr(arr[i], name, A[j] + 0x1000 * i)
    v, r, y = A[9], A[10], A[11]

    def call(layers=arr, L=2, d=256, f=768, g=64, fmt=1, eps=1e-5, v=v, r=r, y=y):
        return fn(layers, L, d, f, g, fmt, eps, v, r, y, None)

    assert call(layers=None) == NULL
    assert call(v=None) == NULL
    assert call(L=0) == SHAPE
    assert call(d=260) == SHAPE
    assert call(g=48) == GROUP
    assert call(fmt=7) == FORMAT
    assert call(y=y + 8) == ALIGN
    assert call(y=v) == ALIAS                 # out_y inside values
    assert call(y=r + 16) == ALIAS           # partial overlap with the residual

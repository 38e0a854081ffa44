// mt_api.cu - the extern "C" entry points declared in include/mt.h: argument
// validation (before anything is launched), aliasing checks, per-device
// facts and dispatch to the kernels.
#include <math.h>

#include <atomic>
#include <mutex>

#include "mt_internal.h"

namespace mt {

static thread_local int g_last_cuda_error = 0;
static std::atomic<int> g_opt_pdl{1};
static std::atomic<int> g_opt_gemv{0};
static std::atomic<int> g_opt_barrier_extra{0};
static std::atomic<int> g_opt_act_bits{16};

// Device error word: kernels with bounded waits record MT_ERR_TIMEOUT here.
__device__ int g_device_error;

// Looked up on every call (no allocation, no synchronisation): a cached
// address would dangle after a cudaDeviceReset reloads the module.
int* device_error_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

int gemv_choice() { return g_opt_gemv.load(); }
int test_barrier_extra() { return g_opt_barrier_extra.load(); }
int act_bits() { return g_opt_act_bits.load(); }

mt_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return MT_ERR_CUDA;
}

const DeviceInfo* device_info(int* err) {
  static std::mutex mu;
  static DeviceInfo info[64];
  static bool have[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = (int)e; g_last_cuda_error = (int)e; return nullptr; }
  if (dev < 0 || dev >= 64) { *err = (int)cudaErrorInvalidDevice; return nullptr; }
  std::lock_guard<std::mutex> g(mu);
  if (!have[dev]) {
    int sms = 0, smem = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) { *err = (int)e; g_last_cuda_error = (int)e; return nullptr; }
    info[dev].sm_count = sms;
    info[dev].max_smem_optin = smem;
    have[dev] = true;
  }
  return &info[dev];
}

mt_status launch_gemv_bf16(const GemvProblem& p, const Launch& l);
mt_status launch_gemv_a8(const GemvProblem& p, const Launch& l);
mt_status launch_gemv_a4(const GemvProblem& p, const Launch& l);
mt_status launch_gemv_mx8(const GemvProblem& p, const Launch& l);
mt_status launch_gemv_mx4(const GemvProblem& p, const Launch& l);

mt_status launch_gemv(const GemvProblem& p, const Launch& l) {
  switch (p.fmt) {
    case MT_W_BF16: return launch_gemv_bf16(p, l);
    case MT_W_AFFINE8: return launch_gemv_a8(p, l);
    case MT_W_AFFINE4: return launch_gemv_a4(p, l);
    case MT_W_MXFP8: return launch_gemv_mx8(p, l);
    case MT_W_MXFP4: return launch_gemv_mx4(p, l);
    default: return MT_ERR_FORMAT;
  }
}

}  // namespace mt

using namespace mt;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Byte range [p, p + n).
struct Range {
  uintptr_t lo, hi;
};
Range rng(const void* p, size_t n) { return Range{(uintptr_t)p, (uintptr_t)p + n}; }
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool is_mx(int fmt) { return fmt == MT_W_MXFP8 || fmt == MT_W_MXFP4; }
bool valid_wfmt(int fmt) { return fmt >= MT_W_BF16 && fmt <= MT_W_MXFP4; }

size_t weight_bytes(int fmt, long N, long K) {
  if (fmt == MT_W_BF16) return (size_t)N * K * 2;
  if (fmt == MT_W_AFFINE8 || fmt == MT_W_MXFP8) return (size_t)N * K;
  return (size_t)N * K / 2;
}

// Bytes of the scales of one [N][K] weight (and of its biases, affine).
size_t sb_bytes(int fmt, long N, long K, int group) {
  if (fmt == MT_W_BF16) return 0;
  return (size_t)N * (K / group) * (is_mx(fmt) ? 1 : 2);
}

// Which of scales / biases a format takes: affine both, MX scales only (biases
// must be NULL), bf16 neither.
mt_status check_sb(int fmt, const void* scales, const void* biases) {
  if (fmt == MT_W_BF16) return MT_OK;
  if (!scales) return MT_ERR_NULL;
  if (is_mx(fmt)) return biases ? MT_ERR_FORMAT : MT_OK;
  return biases ? MT_OK : MT_ERR_NULL;
}

bool valid_group(int fmt, int group, long K, mt_status* st) {
  if (fmt == MT_W_BF16) {
    if (group != 0) { *st = MT_ERR_GROUP; return false; }
    if (K % 8 != 0) { *st = MT_ERR_SHAPE; return false; }
    return true;
  }
  if (is_mx(fmt) && group != 32) { *st = MT_ERR_GROUP; return false; }
  if (group != 32 && group != 64 && group != 128) { *st = MT_ERR_GROUP; return false; }
  if (K % group != 0) { *st = MT_ERR_SHAPE; return false; }
  return true;
}

Launch make_launch(void* stream) { return Launch{(cudaStream_t)stream, g_opt_pdl.load() != 0}; }

}  // namespace

extern "C" {

mt_status mt_add_rmsnorm(const void* values, const void* residual, const void* weight, float eps,
                         void* out_sum, void* out_norm, int M, int d, mt_dtype norm_dtype,
                         void* stream) {
  if (!values || !residual || !weight || !out_sum || !out_norm) return MT_ERR_NULL;
  if (M < 1 || M > 8 || d < 8 || d > 65536 || d % 8 != 0) return MT_ERR_SHAPE;
  if (norm_dtype != MT_BF16 && norm_dtype != MT_F32) return MT_ERR_FORMAT;
  if (!(eps >= 0.0f) || eps == INFINITY) return MT_ERR_SHAPE;
  if (!aligned16(values) || !aligned16(residual) || !aligned16(weight) || !aligned16(out_sum) ||
      !aligned16(out_norm))
    return MT_ERR_ALIGN;
  const size_t act = (size_t)M * d * 2;
  const size_t nb = (size_t)M * d * (norm_dtype == MT_F32 ? 4 : 2);
  const Range rs = rng(out_sum, act), rn = rng(out_norm, nb);
  const Range iv = rng(values, act), ir = rng(residual, act), iw = rng(weight, (size_t)d * 2);
  if (overlap(rs, rn) || overlap(rs, iv) || overlap(rs, iw) || overlap(rn, iv) || overlap(rn, ir) ||
      overlap(rn, iw))
    return MT_ERR_ALIAS;
  if (overlap(rs, ir) && out_sum != residual) return MT_ERR_ALIAS;
  return launch_add_rmsnorm((const uint16_t*)values, (const uint16_t*)residual,
                            (const uint16_t*)weight, eps, (uint16_t*)out_sum, out_norm, M, d,
                            norm_dtype == MT_F32, make_launch(stream));
}

mt_status mt_swiglu_gateup(const void* x, const void* Wg, const void* Wu, const void* scales,
                           const void* biases, int group, void* out_h, int M, int d, int f,
                           mt_wfmt fmt, mt_dtype out_dtype, void* stream) {
  if (!valid_wfmt(fmt)) return MT_ERR_FORMAT;
  if (out_dtype != MT_BF16 && out_dtype != MT_F32) return MT_ERR_FORMAT;
  if (!x || !Wg || !Wu || !out_h) return MT_ERR_NULL;
  if (const mt_status sbst = check_sb(fmt, scales, biases)) return sbst;
  if (M < 1 || M > 8 || d < 1 || d > 32768 || f < 1) return MT_ERR_SHAPE;
  mt_status st = MT_OK;
  if (!valid_group(fmt, group, d, &st)) return st;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(out_h) ||
      (fmt != MT_W_BF16 && (!aligned16(scales) || !aligned16(biases))))
    return MT_ERR_ALIGN;
  const size_t wb = weight_bytes(fmt, f, d);
  const size_t sbb = 2 * sb_bytes(fmt, f, d, group);  // two planes
  const Range ro = rng(out_h, (size_t)M * f * (out_dtype == MT_F32 ? 4 : 2));
  if (overlap(ro, rng(x, (size_t)M * d * 2)) || overlap(ro, rng(Wg, wb)) ||
      overlap(ro, rng(Wu, wb)) ||
      (sbb && (overlap(ro, rng(scales, sbb)) || (biases && overlap(ro, rng(biases, sbb))))))
    return MT_ERR_ALIAS;
  GemvProblem p = {};
  p.kind = Kind::GateUp;
  p.fmt = fmt;
  p.M = M; p.K = d; p.N = f;
  p.group = fmt == MT_W_BF16 ? 0 : group;
  p.x = (const uint16_t*)x;
  p.W0 = Wg; p.W1 = Wu;
  if (fmt != MT_W_BF16) {
    const size_t plane = sb_bytes(fmt, f, d, group);  // bytes of one plane
    p.s0 = (const uint16_t*)scales;
    p.s1 = (const uint16_t*)((const char*)scales + plane);
    if (biases) {
      p.b0 = (const uint16_t*)biases;
      p.b1 = (const uint16_t*)((const char*)biases + plane);
    }
  }
  p.out = out_h;
  p.out_f32 = out_dtype == MT_F32;
  return launch_gemv(p, make_launch(stream));
}

mt_status mt_down_residual(const void* h, const void* Wd, const void* scales, const void* biases,
                           int group, const void* residual, void* out_y, int M, int f, int d,
                           mt_wfmt fmt, mt_dtype out_dtype, void* stream) {
  if (!valid_wfmt(fmt)) return MT_ERR_FORMAT;
  if (out_dtype != MT_BF16 && out_dtype != MT_F32) return MT_ERR_FORMAT;
  if (!h || !Wd || !residual || !out_y) return MT_ERR_NULL;
  if (const mt_status sbst = check_sb(fmt, scales, biases)) return sbst;
  if (M < 1 || M > 8 || f < 1 || f > 32768 || d < 1) return MT_ERR_SHAPE;
  mt_status st = MT_OK;
  if (!valid_group(fmt, group, f, &st)) return st;
  if (!aligned16(h) || !aligned16(Wd) || !aligned16(residual) || !aligned16(out_y) ||
      (fmt != MT_W_BF16 && (!aligned16(scales) || !aligned16(biases))))
    return MT_ERR_ALIGN;
  const size_t wb = weight_bytes(fmt, d, f);
  const size_t sbb = sb_bytes(fmt, d, f, group);
  const Range ro = rng(out_y, (size_t)M * d * (out_dtype == MT_F32 ? 4 : 2));
  const Range rr = rng(residual, (size_t)M * d * 2);
  if (overlap(ro, rng(h, (size_t)M * f * 2)) || overlap(ro, rng(Wd, wb)) ||
      (sbb && (overlap(ro, rng(scales, sbb)) || (biases && overlap(ro, rng(biases, sbb))))))
    return MT_ERR_ALIAS;
  if (overlap(ro, rr) && !(out_y == residual && out_dtype == MT_BF16)) return MT_ERR_ALIAS;
  GemvProblem p = {};
  p.kind = Kind::Down;
  p.fmt = fmt;
  p.M = M; p.K = f; p.N = d;
  p.group = fmt == MT_W_BF16 ? 0 : group;
  p.x = (const uint16_t*)h;
  p.W0 = Wd; p.W1 = nullptr;
  p.s0 = (const uint16_t*)scales;
  p.b0 = (const uint16_t*)biases;
  p.res = (const uint16_t*)residual;
  p.res_ld = d;
  p.out = out_y;
  p.out_f32 = out_dtype == MT_F32;
  return launch_gemv(p, make_launch(stream));
}

mt_status mt_linear_bias(const void* x, const void* W, const void* scales, const void* biases,
                         int group, const void* bias, void* out_y, int M, int K, int N,
                         mt_wfmt fmt, mt_dtype out_dtype, void* stream) {
  if (!valid_wfmt(fmt)) return MT_ERR_FORMAT;
  if (out_dtype != MT_BF16 && out_dtype != MT_F32) return MT_ERR_FORMAT;
  if (!x || !W || !out_y) return MT_ERR_NULL;
  if (const mt_status sbst = check_sb(fmt, scales, biases)) return sbst;
  if (M < 1 || M > 8 || K < 1 || K > 32768 || N < 1 || N > (1 << 20)) return MT_ERR_SHAPE;
  mt_status st = MT_OK;
  if (!valid_group(fmt, group, K, &st)) return st;
  if (!aligned16(x) || !aligned16(W) || !aligned16(out_y) || (bias && !aligned16(bias)) ||
      (fmt != MT_W_BF16 && (!aligned16(scales) || !aligned16(biases))))
    return MT_ERR_ALIGN;
  const size_t wb = weight_bytes(fmt, N, K);
  const size_t sbb = sb_bytes(fmt, N, K, group);
  const Range ro = rng(out_y, (size_t)M * N * (out_dtype == MT_F32 ? 4 : 2));
  if (overlap(ro, rng(x, (size_t)M * K * 2)) || overlap(ro, rng(W, wb)) ||
      (bias && overlap(ro, rng(bias, (size_t)N * 2))) ||
      (sbb && (overlap(ro, rng(scales, sbb)) || (biases && overlap(ro, rng(biases, sbb))))))
    return MT_ERR_ALIAS;
  GemvProblem p = {};
  p.kind = Kind::Down;
  p.fmt = fmt;
  p.M = M; p.K = K; p.N = N;
  p.group = fmt == MT_W_BF16 ? 0 : group;
  p.x = (const uint16_t*)x;
  p.W0 = W; p.W1 = nullptr;
  p.s0 = (const uint16_t*)scales;
  p.b0 = (const uint16_t*)biases;
  p.res = (const uint16_t*)bias;  // nullable; one row broadcast over M
  p.res_ld = 0;
  p.out = out_y;
  p.out_f32 = out_dtype == MT_F32;
  return launch_gemv(p, make_launch(stream));
}

mt_status mt_pack_affine(const float* W, int N, int K, int group, int bits, void* q, void* scales,
                         void* biases, void* stream) {
  if (!W || !q || !scales || !biases) return MT_ERR_NULL;
  if (bits != 8 && bits != 4) return MT_ERR_FORMAT;
  if (group != 32 && group != 64 && group != 128) return MT_ERR_GROUP;
  if (N < 0 || K < 0 || K % group != 0) return MT_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(q) || !aligned16(scales) || !aligned16(biases))
    return MT_ERR_ALIGN;
  const size_t qb = (size_t)N * K * bits / 8, sb = (size_t)N * (K / group) * 2;
  const Range rq = rng(q, qb), rs = rng(scales, sb), rb = rng(biases, sb),
              rw = rng(W, (size_t)N * K * 4);
  if (overlap(rq, rs) || overlap(rq, rb) || overlap(rs, rb) || overlap(rw, rq) ||
      overlap(rw, rs) || overlap(rw, rb))
    return MT_ERR_ALIAS;
  return launch_pack_affine(W, N, K, group, bits, (uint8_t*)q, (uint16_t*)scales,
                            (uint16_t*)biases, Launch{(cudaStream_t)stream, false});
}

mt_status mt_pack_mx(const float* W, int N, int K, int bits, void* q, void* scales, void* stream) {
  if (!W || !q || !scales) return MT_ERR_NULL;
  if (bits != 8 && bits != 4) return MT_ERR_FORMAT;
  if (N < 0 || K < 0 || K % 32 != 0) return MT_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(q) || !aligned16(scales)) return MT_ERR_ALIGN;
  const size_t qb = (size_t)N * K * bits / 8, sb = (size_t)N * (K / 32);
  const Range rq = rng(q, qb), rs = rng(scales, sb), rw = rng(W, (size_t)N * K * 4);
  if (overlap(rq, rs) || overlap(rw, rq) || overlap(rw, rs)) return MT_ERR_ALIAS;
  return launch_pack_mx(W, N, K, bits, (uint8_t*)q, (uint8_t*)scales,
                        Launch{(cudaStream_t)stream, false});
}

mt_status mt_unpack_affine(const void* q, const void* scales, const void* biases, int N, int K,
                           int group, int bits, float* W, void* stream) {
  if (!W || !q || !scales || !biases) return MT_ERR_NULL;
  if (bits != 8 && bits != 4) return MT_ERR_FORMAT;
  if (group != 32 && group != 64 && group != 128) return MT_ERR_GROUP;
  if (N < 0 || K < 0 || K % group != 0) return MT_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(q) || !aligned16(scales) || !aligned16(biases))
    return MT_ERR_ALIGN;
  const size_t qb = (size_t)N * K * bits / 8, sb = (size_t)N * (K / group) * 2;
  const Range rw = rng(W, (size_t)N * K * 4);
  if (overlap(rw, rng(q, qb)) || overlap(rw, rng(scales, sb)) || overlap(rw, rng(biases, sb)))
    return MT_ERR_ALIAS;
  return launch_unpack_affine((const uint8_t*)q, (const uint16_t*)scales,
                              (const uint16_t*)biases, N, K, group, bits, W,
                              Launch{(cudaStream_t)stream, false});
}

mt_status mt_set_option(mt_option opt, int value) {
  if (opt == MT_OPT_PDL) {
    g_opt_pdl.store(value ? 1 : 0);
    return MT_OK;
  }
  if (opt == MT_OPT_GEMV) {
    if (value < 0 || value > 2) return MT_ERR_FORMAT;
    g_opt_gemv.store(value);
    return MT_OK;
  }
  if (opt == MT_OPT_TEST_BARRIER_EXTRA) {
    if (value < 0 || value > 8) return MT_ERR_FORMAT;
    g_opt_barrier_extra.store(value);
    return MT_OK;
  }
  if (opt == MT_OPT_ACT_BITS) {
    if (value != 16 && value != 24) return MT_ERR_FORMAT;
    g_opt_act_bits.store(value);
    return MT_OK;
  }
  return MT_ERR_FORMAT;
}

int mt_get_option(mt_option opt) {
  if (opt == MT_OPT_PDL) return g_opt_pdl.load();
  if (opt == MT_OPT_GEMV) return g_opt_gemv.load();
  if (opt == MT_OPT_TEST_BARRIER_EXTRA) return g_opt_barrier_extra.load();
  if (opt == MT_OPT_ACT_BITS) return g_opt_act_bits.load();
  return -1;
}

int mt_device_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

const char* mt_status_string(mt_status s) {
  switch (s) {
    case MT_OK: return "MT_OK";
    case MT_ERR_NULL: return "MT_ERR_NULL: a required pointer is NULL";
    case MT_ERR_SHAPE: return "MT_ERR_SHAPE: a size is out of range or not divisible";
    case MT_ERR_GROUP: return "MT_ERR_GROUP: group must be 32, 64 or 128 (0 for bf16)";
    case MT_ERR_ALIGN: return "MT_ERR_ALIGN: pointer not 16-byte aligned";
    case MT_ERR_FORMAT: return "MT_ERR_FORMAT: unknown format, dtype, bit width or option";
    case MT_ERR_ALIAS: return "MT_ERR_ALIAS: output overlaps an input";
    case MT_ERR_CUDA: return "MT_ERR_CUDA: a CUDA runtime call failed";
    case MT_ERR_TIMEOUT: return "MT_ERR_TIMEOUT: a bounded device wait expired";
    default: return "unknown mt_status";
  }
}

int mt_last_cuda_error(void) { return g_last_cuda_error; }

int mt_version(void) { return (1 << 16) | 0; }

}  // extern "C"

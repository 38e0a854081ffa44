// k_prefill.cu - the prefill GEMMs for affine INT8/INT4 and dense bf16
// weights (exact-operand kernel, k_prefill.cuh; single-accumulator kernel
// for bf16 outputs, k_prefill_dq.cuh), the dispatch over weight formats and
// output types, and the C ABI of the prefill calls.
#include "k_prefill.cuh"
#include "k_prefill_dq.cuh"

namespace mt {

mt_status launch_prefill_mx(const GemvProblem& p, void* ws, const Launch& l);

__global__ void __launch_bounds__(256) prefill_x_kernel(const uint16_t* __restrict__ x, int M, int K, int group,
                                                        __half* __restrict__ x16, float* __restrict__ XgT,
                                                        float* __restrict__ einv) {
  const int m = blockIdx.x;  // rows M .. Mp-1 only zero their group sums and scale
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = K / group, Mp = gridDim.x;
  if (m >= M) {
    for (int g = tid; g < G; g += 256) XgT[(size_t)g * Mp + m] = 0.f;
    if (tid == 0) einv[m] = 0.f;
    return;
  }
  const uint16_t* row = x + (size_t)m * K;
  __shared__ uint32_t wmax[8];
  uint32_t mx = 0;  // bf16 magnitude bits order like the magnitudes
  for (int k = tid; k < K; k += 256) mx = max(mx, (uint32_t)(row[k] & 0x7FFFu));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) wmax[warp] = mx;
  __syncthreads();
  mx = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) mx = max(mx, wmax[w]);
  // max in [2^(E-127), 2^(E-126)) for bf16 exponent field E: e = 14 - (E - 127)
  const int E = (int)(mx >> 7);
  const int e = (mx == 0 || E == 0xFF) ? 0 : max(-100, min(100, 14 - (E - 127)));
  const float sc = exp2i(e);
  for (int k = tid; k < K; k += 256) x16[(size_t)m * K + k] = __float2half_rn(bf16f(row[k]) * sc);
  for (int g = warp; g < G; g += 8) {
    float s = 0.f;
    for (int j = lane; j < group; j += 32) s += bf16f(row[g * group + j]) * sc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) XgT[(size_t)g * Mp + m] = s;
  }
  if (tid == 0) einv[m] = exp2i(-e);
}


mt_status launch_prefill(const GemvProblem& p, void* ws, const Launch& l) {
  // bf16 outputs: weights dequantised to fp16 tiles, one accumulator over K;
  // fp32 outputs: exact operands, one tensor-memory sum per group
  if (p.fmt == MT_W_AFFINE8 && !p.out_f32)
    return p.kind == Kind::GateUp ? run_prefill_dq_nt<FMT_A8, 0>(p, ws, l) : run_prefill_dq_nt<FMT_A8, 1>(p, ws, l);
  if (p.fmt == MT_W_AFFINE4 && !p.out_f32)
    return p.kind == Kind::GateUp ? run_prefill_dq_nt<FMT_A4, 0>(p, ws, l) : run_prefill_dq_nt<FMT_A4, 1>(p, ws, l);
  if (p.fmt == MT_W_AFFINE8)
    return p.kind == Kind::GateUp ? run_prefill_nt<FMT_A8, 0>(p, ws, l) : run_prefill_nt<FMT_A8, 1>(p, ws, l);
  if (p.fmt == MT_W_AFFINE4)
    return p.kind == Kind::GateUp ? run_prefill_nt<FMT_A4, 0>(p, ws, l) : run_prefill_nt<FMT_A4, 1>(p, ws, l);
  if (p.fmt == MT_W_MXFP8 || p.fmt == MT_W_MXFP4) return launch_prefill_mx(p, ws, l);
  if (p.fmt == MT_W_BF16 && !p.out_f32)  // one accumulator over K (the operands are exact either way)
    return p.kind == Kind::GateUp ? run_prefill_dq_nt<FMT_BF16, 0>(p, ws, l) : run_prefill_dq_nt<FMT_BF16, 1>(p, ws, l);
  if (p.fmt == MT_W_BF16)
    return p.kind == Kind::GateUp ? run_prefill_nt<FMT_BF16, 0>(p, ws, l) : run_prefill_nt<FMT_BF16, 1>(p, ws, l);
  return MT_ERR_FORMAT;
}

}  // namespace mt

// ------------------------------------------------------------------ C ABI

using namespace mt;

namespace {

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
struct Rg {
  uintptr_t lo, hi;
};
Rg rg(const void* p, size_t n) { return Rg{(uintptr_t)p, (uintptr_t)p + n}; }
bool ovl(Rg a, Rg b) { return a.lo < b.hi && b.lo < a.hi; }

// Shared validation and dispatch of the three prefill calls.  W1 is the up
// matrix (gate/up) or nullptr; the addend is the residual (ld = N) or the
// bias (ld = 0) or nullptr.
mt_status prefill_call(Kind kind, const void* x, const void* W0, const void* W1, const void* scales,
                       const void* biases, int group, const void* addend, int addend_ld, void* out, int M,
                       int K, int N, mt_wfmt fmt, mt_dtype out_dtype, void* ws, size_t ws_bytes, void* stream) {
  const bool mx = fmt == MT_W_MXFP8 || fmt == MT_W_MXFP4, bf = fmt == MT_W_BF16;
  if (fmt != MT_W_AFFINE8 && fmt != MT_W_AFFINE4 && !mx && !bf) return MT_ERR_FORMAT;
  if (out_dtype != MT_BF16 && out_dtype != MT_F32) return MT_ERR_FORMAT;
  if (!x || !W0 || (kind == Kind::GateUp && !W1) || (!bf && !scales) || (!mx && !bf && !biases) || !out || !ws)
    return MT_ERR_NULL;
  if ((mx || bf) && biases) return MT_ERR_FORMAT;  // MX and bf16 weights have no biases
  if (bf && scales) return MT_ERR_FORMAT;           // nor bf16 weights scales
  if (bf) {
    if (group != 0) return MT_ERR_GROUP;
  } else {
    if (group != 32 && group != 64 && group != 128) return MT_ERR_GROUP;
    if (mx && group != 32) return MT_ERR_GROUP;
  }
  if (M < 1 || M > (1 << 20) || K < PF_KB || K > 65536 || K % PF_KB || (group && K % group) || N < 1 ||
      N > (1 << 20))
    return MT_ERR_SHAPE;
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  const size_t need = prefill_ws_bytes(M, K, N, group, di ? di->sm_count : 1);
  if (ws_bytes < need) return MT_ERR_SHAPE;
  if (!al16(x) || !al16(W0) || !al16(W1) || !al16(scales) || !al16(biases) || !al16(out) || !al16(ws) ||
      !al16(addend))
    return MT_ERR_ALIGN;
  const int NW = kind == Kind::GateUp ? 2 : 1;
  const size_t wb = bf ? (size_t)N * K * 2 : (size_t)N * K / (fmt == MT_W_AFFINE8 || fmt == MT_W_MXFP8 ? 1 : 2);
  const size_t sbb = bf ? 0 : (size_t)NW * N * (K / group) * (mx ? 1 : 2);  // scale (and bias) bytes
  const Rg ro = rg(out, (size_t)M * N * (out_dtype == MT_F32 ? 4 : 2));
  const Rg rw = rg(ws, need);
  const Rg rx = rg(x, (size_t)M * K * 2), rw0 = rg(W0, wb), rw1 = rg(W1, W1 ? wb : 0);
  const Rg rs = rg(scales, sbb), rb = rg(biases, biases ? sbb : 0);
  const Rg ra = rg(addend, !addend ? 0 : (addend_ld ? (size_t)M * N * 2 : (size_t)N * 2));
  if (ovl(ro, rx) || ovl(ro, rw0) || ovl(ro, rw1) || ovl(ro, rs) || ovl(ro, rb) || ovl(ro, rw)) return MT_ERR_ALIAS;
  if (ovl(rw, rx) || ovl(rw, rw0) || ovl(rw, rw1) || ovl(rw, rs) || ovl(rw, rb) || ovl(rw, ra)) return MT_ERR_ALIAS;
  // the residual may be the output itself (each element read, then written, by one thread)
  if (ovl(ro, ra) && !(addend_ld && addend == out && out_dtype == MT_BF16)) return MT_ERR_ALIAS;
  GemvProblem p = {};
  p.kind = kind;
  p.fmt = fmt;
  p.M = M; p.K = K; p.N = N; p.group = group;
  p.x = (const uint16_t*)x;
  p.W0 = W0; p.W1 = W1;
  const size_t plane = bf ? 0 : (size_t)N * (K / group) * (mx ? 1 : 2);  // bytes of one scale plane
  p.s0 = (const uint16_t*)scales;
  p.b0 = (const uint16_t*)biases;
  if (kind == Kind::GateUp && !bf) {
    p.s1 = (const uint16_t*)((const char*)scales + plane);
    p.b1 = biases ? (const uint16_t*)((const char*)biases + plane) : nullptr;
  }
  p.res = (const uint16_t*)addend;
  p.res_ld = addend_ld;
  p.out = out;
  p.out_f32 = out_dtype == MT_F32;
  return launch_prefill(p, ws, Launch{(cudaStream_t)stream, false});
}

}  // namespace

extern "C" {

size_t mt_prefill_workspace_bytes(int M, int K, int N, int group) {
  if (M < 1 || K < PF_KB || N < 1 || (group != 0 && group != 32 && group != 64 && group != 128)) return 0;
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  return prefill_ws_bytes(M, K, N, group, di ? di->sm_count : 1);
}

mt_status mt_prefill_swiglu_gateup(const void* x, const void* Wg, const void* Wu, const void* scales,
                                   const void* biases, int group, void* out_h, int M, int d, int f,
                                   mt_wfmt fmt, mt_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  return prefill_call(Kind::GateUp, x, Wg, Wu, scales, biases, group, nullptr, 0, out_h, M, d, f, fmt, out_dtype,
                      workspace, workspace_bytes, stream);
}

mt_status mt_prefill_down_residual(const void* h, const void* Wd, const void* scales, const void* biases,
                                   int group, const void* residual, void* out_y, int M, int f, int d,
                                   mt_wfmt fmt, mt_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  if (!residual) return MT_ERR_NULL;
  return prefill_call(Kind::Down, h, Wd, nullptr, scales, biases, group, residual, d, out_y, M, f, d, fmt,
                      out_dtype, workspace, workspace_bytes, stream);
}

mt_status mt_prefill_linear_bias(const void* x, const void* W, const void* scales, const void* biases, int group,
                                 const void* bias, void* out_y, int M, int K, int N, mt_wfmt fmt,
                                 mt_dtype out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_call(Kind::Down, x, W, nullptr, scales, biases, group, bias, 0, out_y, M, K, N, fmt, out_dtype,
                      workspace, workspace_bytes, stream);
}

}  // extern "C"

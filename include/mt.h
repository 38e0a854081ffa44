/*
 * mt.h - C ABI of the GB300 (sm_103a) one-row decode-MLP library.
 *
 * One decode MLP layer is three stream-ordered calls:
 *
 *   mt_add_rmsnorm    summed = values + residual, normalized = rms_norm(summed,
 *                     weight, eps); both are outputs (one multi-output kernel).
 *                     meTile docs, "Compute-Graph Fusion", opening example.
 *   mt_swiglu_gateup  g = x @ Wg^T, u = x @ Wu^T over group-wise affine weights
 *                     (or dense bf16), h = silu(g) * u applied on-chip before
 *                     the only store.  meTile docs, "Compute-Graph Fusion",
 *                     Automatic Gated Epilogues; "MLX-LM Backend", Dispatch
 *                     Policy (affine INT8/4-bit groups 32/64/128, dense BF16
 *                     paired gate/up QMV).
 *   mt_down_residual  y = h @ Wd^T + residual with the residual added in the
 *                     GEMV's epilogue.  meTile docs, "Compute-Graph Fusion",
 *                     Automatic Gated Epilogues ("a second composable
 *                     epilogue adds the transformer residual to the down
 *                     projection"); "MLX-LM Backend", Dispatch Policy
 *                     ("values @ weight.T + residual").
 *
 * and, for the rest of a decode step, the same GEMV as a projection:
 *
 *   mt_linear_bias    y = x @ W^T (+ bias): the attention projections q/k/v/o
 *                     (bias kept where the model has one) and the vocabulary
 *                     projection (untied lm_head, or a tied embedding table
 *                     used as the weight).  meTile docs, "MLX-LM Backend", the
 *                     attention-projection and vocabulary compression passages
 *                     before Dispatch Policy.
 *
 * plus the offline packer mt_pack_affine (affine group quantisation of fp32
 * weights into the stored layout), and the warmed executor mt_mlp_plan_*
 * that runs L such layers back to back as one persistent kernel.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Layouts.  Activations are row-major [M][.] bf16 (M = rows, 1..8).  A
 *   weight is stored output-major [N][K] with K contiguous ("x[.., K] @ W[N, K]
 *   stored transposed", ANEForge docs, "The optimizer and the cost model", The
 *   roofline).  Gate/up: N = f, K = d.  Down: N = d, K = f.
 *   MT_W_BF16    : W is bf16 [N][K].
 *   MT_W_AFFINE8 : W is uint8 [N][K], one code q per byte.
 *   MT_W_AFFINE4 : W is uint8 [N][K/2], byte j of a row holds code 2j in bits
 *                  0..3 and code 2j+1 in bits 4..7.
 *   Affine weights are w[n][k] = scale[n][k/group] * q[n][k] + bias[n][k/group]
 *   with bf16 scales and biases [N][K/group], row-major.
 *   MT_W_MXFP8   : W is uint8 [N][K], one OCP FP8 E4M3 code per byte.
 *   MT_W_MXFP4   : W is uint8 [N][K/2], OCP FP4 E2M1 codes, nibble order as
 *                  MT_W_AFFINE4.
 *   MX weights are w[n][k] = value(code[n][k]) * 2^(E[n][k/32] - 127) with
 *   uint8 E8M0 scale fields E [N][K/32] passed as `scales`, `biases` NULL
 *   and group 32 (meTile docs, "MLX-LM Backend", Block-Scaled MLX Primitive;
 *   encodings of the OCP Microscaling Formats v1.0).  They run on the
 *   tensor-core kernel for every M; the executor (mt_mlp_plan_*) does not
 *   take them.
 *   For mt_swiglu_gateup one scales array and one biases array hold two
 *   planes [2][f][d/group]: plane 0 belongs to Wg, plane 1 to Wu.
 * - Pointers.  Every tensor pointer is a DEVICE pointer (cudaMalloc, or memory
 *   the device can address), 16-byte aligned.  The caller owns every buffer;
 *   the hot calls allocate nothing and never synchronise.
 * - Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream).  All work is enqueued on it in call order.
 * - Errors.  Arguments are validated before anything is launched; on an
 *   invalid argument nothing is launched and the matching MT_ERR_* is
 *   returned.  A failed launch returns MT_ERR_CUDA (mt_last_cuda_error()
 *   gives the cudaError_t).  Faults during execution surface at the caller's
 *   next synchronisation, as for any CUDA kernel.
 * - Aliasing.  Outputs must not overlap inputs, except: out_sum may equal
 *   residual in mt_add_rmsnorm, and out_y may equal residual in
 *   mt_down_residual (each element is read and then written by the same
 *   thread).  Other overlaps return MT_ERR_ALIAS.
 * - Programmatic dependent launch.  By default the three hot calls are
 *   launched so that each kernel may start while the previous kernel on the
 *   stream finishes; before waiting for that kernel a call reads only its
 *   weights, scales, biases and RMSNorm weight.  Those must therefore not be
 *   written by work still running on the stream (upload or pack them, then
 *   synchronise or record an event, before the first call that reads them).
 *   mt_set_option(MT_OPT_PDL, 0) turns this off.
 * - Device reset.  The first launch of a kernel that uses more than 48 KB of
 *   shared memory on a device sets its limit once per process.  A
 *   cudaDeviceReset may drop that limit, and such a launch then returns
 *   MT_ERR_CUDA (cudaErrorInvalidValue) instead of running; plans made
 *   before the reset hold freed memory.  mt_mlp_stack_run_noalloc and
 *   mt_device_error look everything up on each call and stay valid.
 */
#ifndef MT_H
#define MT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mt_status {
  MT_OK = 0,
  MT_ERR_NULL = 1,    /* a required pointer is NULL */
  MT_ERR_SHAPE = 2,   /* a size is out of range or not divisible as required */
  MT_ERR_GROUP = 3,   /* group not in {32, 64, 128} for affine, not 0 for bf16 */
  MT_ERR_ALIGN = 4,   /* a pointer is not 16-byte aligned */
  MT_ERR_FORMAT = 5,  /* unknown weight format, dtype, bit width or option */
  MT_ERR_ALIAS = 6,   /* an output overlaps an input it may not overlap */
  MT_ERR_CUDA = 7,    /* a CUDA runtime call failed (see mt_last_cuda_error) */
  MT_ERR_TIMEOUT = 8  /* a bounded device-side wait expired (mt_device_error) */
} mt_status;

/* Output element type of a call.  Inputs are always bf16. */
typedef enum mt_dtype { MT_BF16 = 0, MT_F32 = 1 } mt_dtype;

/* Weight storage format. */
typedef enum mt_wfmt { MT_W_BF16 = 0, MT_W_AFFINE8 = 1, MT_W_AFFINE4 = 2,
                       MT_W_MXFP8 = 3, MT_W_MXFP4 = 4 } mt_wfmt;

/* Library options (mt_set_option / mt_get_option). */
typedef enum mt_option {
  MT_OPT_PDL = 0, /* 1 (default): launch with programmatic stream serialization */
  MT_OPT_GEMV = 1, /* GEMV kernel family: 0 (default) warp-task kernel for
                      M = 1 and tensor-core kernel for M > 1; 1 team kernel
                      for every M; 2 tensor-core kernel for every M (shapes
                      a kernel cannot hold fall back to the team kernel) */
  MT_OPT_TEST_BARRIER_EXTRA = 2, /* test hook for failure detection, 0 (default)
                      to 8: executor runs started while it is n > 0 make
                      every grid barrier wait for n arrivals that never come,
                      so the bounded wait expires (~1 s) and the run ends with
                      MT_ERR_TIMEOUT in mt_device_error() */
  MT_OPT_ACT_BITS = 3 /* bits of the fixed-point activation x = X 2^-e (one
                      power of two per activation row) with which the one-row
                      affine GEMVs with bf16 outputs and the executor compute
                      their dot products: 16 (default) or 24.  fp32 outputs
                      always use 24.  With 16 bits, elements more than 2^6
                      below the row's largest |x| are rounded to 2^-14 of it:
                      within the 2e-3 bf16 bound on activations whose
                      max|x| / rms(x) stays below ~30, but a row with a channel
                      ~1000x the others (one weight row's output dominated by
                      the other channels) can exceed it; 24 bits keep such
                      rows within the bound at ~1.5 us more per executor layer
                      (Qwen3-8B shape).  A plan takes the value set when it is
                      created; mt_mlp_stack_run_noalloc the value set when it
                      is called. */
} mt_option;

/*
 * Residual add + RMSNorm as one multi-output kernel.
 *   values, residual : bf16 [M][d]
 *   weight           : bf16 [d] (RMSNorm gain)
 *   out_sum          : bf16 [M][d], out_sum = bf16(values + residual)
 *   out_norm         : [M][d] of norm_dtype,
 *                      out_norm = out_sum * weight / sqrt(mean(out_sum^2) + eps)
 *                      computed from the rounded out_sum with fp32 accumulation.
 * Limits: 1 <= M <= 8, 8 <= d <= 65536, d % 8 == 0, eps >= 0.
 * meTile docs, "Compute-Graph Fusion" (opening example: the residual value
 * remains a graph output); "MLX-LM Backend", Dispatch Policy (RMSNorm with FP32
 * accumulation, residual-add followed by RMSNorm kept as two outputs).
 */
mt_status mt_add_rmsnorm(const void* values, const void* residual, const void* weight,
                         float eps, void* out_sum, void* out_norm, int M, int d,
                         mt_dtype norm_dtype, void* stream);

/*
 * Gate/up GEMV with the SwiGLU epilogue.
 *   x        : bf16 [M][d]
 *   Wg, Wu   : [f][d] in format fmt (see Layouts)
 *   scales   : bf16 [2][f][d/group] (NULL for MT_W_BF16; uint8 E8M0 for MX)
 *   biases   : bf16 [2][f][d/group] (NULL for MT_W_BF16 and MX)
 *   group    : 32, 64 or 128 for affine formats, 0 for MT_W_BF16
 *   out_h    : [M][f] of out_dtype, h = silu(g) * u, silu(g) = g / (1 + e^-g),
 *              g = x . Wg[n], u = x . Wu[n], fp32 accumulation, one rounding.
 * Limits: 1 <= M <= 8; d % group == 0 (affine; group 32 for MX), d % 8 == 0 (bf16);
 *         1 <= f; d <= 32768.
 * meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (two matmuls
 * sharing the activation, silu(gate) * up applied on-chip); "MLX-LM Backend",
 * Dispatch Policy (gate and up dot products share each activation load and
 * apply the SwiGLU epilogue before the only output write).
 */
mt_status mt_swiglu_gateup(const void* x, const void* Wg, const void* Wu,
                           const void* scales, const void* biases, int group,
                           void* out_h, int M, int d, int f,
                           mt_wfmt fmt, mt_dtype out_dtype, void* stream);

/*
 * Down GEMV with the residual epilogue.
 *   h        : bf16 [M][f]
 *   Wd       : [d][f] in format fmt
 *   scales   : bf16 [d][f/group] (NULL for MT_W_BF16; uint8 E8M0 for MX)
 *   biases   : bf16 [d][f/group] (NULL for MT_W_BF16 and MX)
 *   residual : bf16 [M][d]
 *   out_y    : [M][d] of out_dtype, y = h . Wd[n] + residual[n], fp32
 *              accumulation, one rounding.  out_y may equal residual.
 * Limits: 1 <= M <= 8; f % group == 0 (affine; group 32 for MX), f % 8 == 0 (bf16);
 *         1 <= d; f <= 32768.
 * meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (residual
 * added to the down projection in the same kernel); "MLX-LM Backend",
 * Dispatch Policy (typed store adds the transformer residual without
 * materialising the unfused projection).
 */
mt_status mt_down_residual(const void* h, const void* Wd, const void* scales,
                           const void* biases, int group, const void* residual,
                           void* out_y, int M, int f, int d,
                           mt_wfmt fmt, mt_dtype out_dtype, void* stream);

/*
 * Projection GEMV with an optional bias epilogue.
 *   x        : bf16 [M][K]
 *   W        : [N][K] in format fmt.  q, k and v of one layer share x, so a
 *              caller may stack their rows into one [Nq + Nk + Nv][K] weight
 *              (and one bias) and make one call.  A tied embedding table
 *              [vocab][K] is used as W unchanged.
 *   scales   : bf16 [N][K/group] (NULL for MT_W_BF16; uint8 E8M0 for MX)
 *   biases   : bf16 [N][K/group] (NULL for MT_W_BF16 and MX)
 *   bias     : bf16 [N], added to every row, or NULL for a projection without
 *              bias
 *   out_y    : [M][N] of out_dtype, y = x . W[n] (+ bias[n]), fp32
 *              accumulation, one rounding.
 * Limits: 1 <= M <= 8; K % group == 0 (affine; group 32 for MX), K % 8 == 0 (bf16);
 *         K <= 32768; 1 <= N <= 1048576.
 * Aliasing: out_y overlaps no input.
 * meTile docs, "MLX-LM Backend", the attention-projection compression passage
 * (q_proj, k_proj, v_proj and o_proj per layer, projection biases preserved,
 * one-row decode only) and the vocabulary compression passage (tied
 * embedding's linear projection or untied lm_head, one-row decode only).
 */
mt_status mt_linear_bias(const void* x, const void* W, const void* scales,
                         const void* biases, int group, const void* bias,
                         void* out_y, int M, int K, int N,
                         mt_wfmt fmt, mt_dtype out_dtype, void* stream);

/*
 * Multi-row prefill (M > 8 activation rows, any M >= 1) of the same three
 * GEMV epilogues as tensor-core GEMMs (tcgen05 with tensor-memory
 * accumulators, TMA-fed activation tiles): a tile of 128 weight rows x 64,
 * 128 or 256 activation rows per CTA, the gate and up rows of a feature range
 * in one tile and the SwiGLU applied before the only store.  meTile docs, "MLX-LM Backend", Dispatch
 * Policy (multi-row shapes: a row-tiled dual GEMM with the SwiGLU in
 * registers); "Compute-Graph Fusion", Automatic Gated Epilogues.
 *   Arguments, layouts and results as mt_swiglu_gateup / mt_down_residual /
 *   mt_linear_bias, plus a caller-owned device workspace of at least
 *   mt_prefill_workspace_bytes(M, K, N, group) bytes (16-byte aligned; K, N
 *   are d, f for gate/up and f, d for down) that holds the activations
 *   converted for the tensor cores and, when the output tiles do not fill
 *   the GPU, the partial sums of K slices (added in a fixed order by a second
 *   kernel); it must not overlap any argument.  The call allocates nothing
 *   and never synchronises.
 * Formats: MT_W_AFFINE8, MT_W_AFFINE4 (group 32, 64 or 128), MT_W_MXFP8,
 *          MT_W_MXFP4 (group 32, biases NULL), MT_W_BF16 (group 0, scales
 *          and biases NULL; x enters the MMA as stored).
 * Limits: 1 <= M <= 2^20; K % 64 == 0 and K % group == 0; 64 <= K <= 65536;
 *         1 <= N <= 2^20.  A workspace below the required size is
 *         MT_ERR_SHAPE.  out_y may equal residual (bf16 output).
 * Accumulation, fp32 outputs (and MX or bf16 weights): each quantisation
 * group's code . x sum is exact products with fp32 accumulation on the
 * tensor cores (codes as fp16 q * 2^-24; x as fp16 scaled per activation row
 * by a power of two, exact for every bf16 value above 2^-28 of the row's
 * maximum); scales, biases and the total are fp32.
 * Accumulation, bf16 outputs over affine weights (the pages' multi-row path
 * dequantises weight tiles into the activations' type before the matmul):
 * each weight w = s q + b is formed in fp32 times a power of two 2^t_n per
 * weight row (max |w| 2^t_n < 2^15) and rounded once to fp16 (relative error
 * at most 2^-11), and the whole K range accumulates in fp32 on the tensor
 * cores; the workspace also holds the rows' 2^t_n.  Dense bf16 weights with
 * bf16 outputs accumulate the whole K range the same way (exact operands).
 */
size_t mt_prefill_workspace_bytes(int M, int K, int N, int group);
mt_status mt_prefill_swiglu_gateup(const void* x, const void* Wg, const void* Wu,
                                   const void* scales, const void* biases, int group,
                                   void* out_h, int M, int d, int f, mt_wfmt fmt,
                                   mt_dtype out_dtype, void* workspace,
                                   size_t workspace_bytes, void* stream);
mt_status mt_prefill_down_residual(const void* h, const void* Wd, const void* scales,
                                   const void* biases, int group, const void* residual,
                                   void* out_y, int M, int f, int d, mt_wfmt fmt,
                                   mt_dtype out_dtype, void* workspace,
                                   size_t workspace_bytes, void* stream);
mt_status mt_prefill_linear_bias(const void* x, const void* W, const void* scales,
                                 const void* biases, int group, const void* bias,
                                 void* out_y, int M, int K, int N, mt_wfmt fmt,
                                 mt_dtype out_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Affine group quantiser and packer (offline preparation; stream-ordered).
 *   W        : fp32 [N][K], device
 *   bits     : 8 or 4;  group : 32, 64 or 128;  K % group == 0
 *   q        : uint8 [N][K] (bits 8) or [N][K/2] (bits 4), device
 *   scales   : bf16 [N][K/group], biases : bf16 [N][K/group], device
 * Per group of `group` consecutive elements along K, in binary64:
 *   bias  = bf16(min),  scale = bf16((max - min) / (2^bits - 1)),
 *   q     = clamp(round_half_even((w - bias) / scale), 0, 2^bits - 1),
 *   and q = 0 when scale == 0.  bf16() rounds to nearest even.
 * meTile docs, "MLX-LM Backend": affine INT8 and 4-bit "affine nibbles,
 * scales, and biases" with group sizes 32, 64 and 128 prepared ahead of time.
 * The formula itself is not printed there; this is the min/max reading.
 */
mt_status mt_pack_affine(const float* W, int N, int K, int group, int bits,
                         void* q, void* scales, void* biases, void* stream);

/*
 * MX block-scaled quantiser and packer (offline preparation; stream-ordered).
 *   W        : fp32 [N][K], device;  K % 32 == 0
 *   bits     : 8 (MXFP8, E4M3 elements) or 4 (MXFP4, E2M1 elements)
 *   q        : uint8 [N][K] (bits 8) or [N][K/2] (bits 4, code 2j in bits
 *              0..3 of byte j, 2j+1 in bits 4..7), device
 *   scales   : uint8 [N][K/32] E8M0 fields, device
 * Per block of 32 consecutive elements along K: E = clamp(floor(log2(amax))
 * - emax + 127, 0, 254) with emax = 8 (E4M3) or 2 (E2M1), E = 0 for an
 * all-zero block; each element is w / 2^(E - 127) rounded to nearest-even
 * in the element format, magnitudes above its largest finite value (448,
 * 6) clamped to it, the sign kept.  Deterministic; bit-identical to the CPU
 * oracle's quantiser.  meTile docs, "MLX-LM Backend", Block-Scaled MLX
 * Primitive (MXFP8 / MXFP4 weights quantised ahead of time); the shared-scale
 * rule and encodings are those of the OCP Microscaling Formats v1.0.
 */
mt_status mt_pack_mx(const float* W, int N, int K, int bits, void* q, void* scales,
                     void* stream);

/*
 * Dequantise packed affine weights to fp32 [N][K] (w = scale * q + bias,
 * rounded once to fp32).  Stream-ordered, device pointers.  For layout checks.
 */
mt_status mt_unpack_affine(const void* q, const void* scales, const void* biases,
                           int N, int K, int group, int bits, float* W, void* stream);

/*
 * Warmed decode-MLP executor (one row, M = 1): L layers run back to back by
 * one persistent kernel.  Layer l (l = 0 .. L-1) computes, with r_0 = residual:
 *   summed_l = bf16(values[l] + r_l)
 *   x_l      = bf16(summed_l * norm_weight_l / sqrt(mean(summed_l^2) + eps))
 *   h_l      = bf16(silu(x_l . Wg_l[n]) * (x_l . Wu_l[n]))      n < f
 *   y_l      = bf16(h_l . Wd_l[n] + summed_l[n])                 n < d
 *   r_{l+1}  = y_l
 * i.e. exactly the tensors of L rounds of mt_add_rmsnorm, mt_swiglu_gateup and
 * mt_down_residual with bf16 outputs (fp32 accumulation, each tensor rounded
 * once where it crosses a call boundary); out_y = y_{L-1}.
 * meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (the selected
 * gate/up and down/residual stages are bound once into a warmed MLP executor);
 * "MLX-LM Backend", Dispatch Policy (residual add + RMSNorm keeps the residual
 * as a second output; steady-state decode does not go through a per-call
 * wrapper).
 *
 * mt_mlp_plan_create binds the layers' weights (device pointers, layouts as
 * for the single calls; one format and group size for all layers) and plans
 * the kernel for the CURRENT device.  It allocates the plan's device memory
 * (a layer table of 80 * L bytes and a workspace of about 2 * (d + f) bytes
 * plus 1 KB) with cudaMalloc, uploads the table synchronously and returns the
 * plan in *plan.
 * The weights stay owned by the caller and must outlive the plan; they must
 * not be written while a run that reads them may execute.
 *   layers : host array of L layer descriptions (copied; may be freed after)
 *   d, f   : hidden and intermediate sizes, 8 <= d, f <= 32768, multiples of 8
 *            and (affine) of group
 *   Limits : 1 <= L <= 4096; the kernel's shared-memory layout must fit one SM
 *            (MT_ERR_SHAPE otherwise; d = 4096, f = 12288 fits).
 * mt_mlp_plan_run enqueues one pass over the L layers on `stream` (a 128-byte
 * memset of the plan's barrier line and one cooperative kernel launch).  It allocates
 * nothing and does not synchronise.
 *   values   : bf16 [L][d], values[l] is layer l's addend (device)
 *   residual : bf16 [d], r_0 (device)
 *   out_y    : bf16 [d], y_{L-1} (device); may equal residual
 *   trace    : NULL, or per-layer copies of the intermediate tensors, each
 *              NULL or a device buffer: out_sum [L][d] (summed_l), out_norm
 *              [L][d] (x_l), h [L][f], y [L][d].
 *   The device current at the call must be the plan's (else MT_ERR_CUDA with
 *   cudaErrorInvalidDevice).  Runs of one plan share its workspace: they must
 *   not execute concurrently (enqueue them on one stream, or order them with
 *   events); different plans are independent.  The run's kernel keeps one
 *   CTA resident on every SM for its whole duration (cooperative launch);
 *   kernels running concurrently on other streams can delay its CTAs.
 *   A grid-wide wait that expires (bounded at about one second) makes every
 *   CTA return: mt_device_error() then reports MT_ERR_TIMEOUT and out_y is
 *   undefined.
 * mt_mlp_plan_destroy frees the plan's device memory (cudaFree, which
 * synchronises the device) and the plan.
 */
typedef struct mt_mlp_layer {
  const void* norm_weight; /* bf16 [d] RMSNorm gain */
  const void* Wg;          /* [f][d] in the plan's format */
  const void* Wu;          /* [f][d] */
  const void* gu_scales;   /* bf16 [2][f][d/group] (plane 0 Wg, 1 Wu); NULL for MT_W_BF16 */
  const void* gu_biases;   /* bf16 [2][f][d/group]; NULL for MT_W_BF16 */
  const void* Wd;          /* [d][f] */
  const void* d_scales;    /* bf16 [d][f/group]; NULL for MT_W_BF16 */
  const void* d_biases;    /* bf16 [d][f/group]; NULL for MT_W_BF16 */
} mt_mlp_layer;

typedef struct mt_mlp_trace {
  void* out_sum;  /* bf16 [L][d] or NULL */
  void* out_norm; /* bf16 [L][d] or NULL */
  void* h;        /* bf16 [L][f] or NULL */
  void* y;        /* bf16 [L][d] or NULL */
} mt_mlp_trace;

typedef struct mt_mlp_plan mt_mlp_plan;

mt_status mt_mlp_plan_create(const mt_mlp_layer* layers, int L, int d, int f, int group,
                             mt_wfmt fmt, float eps, mt_mlp_plan** plan);
mt_status mt_mlp_plan_run(const mt_mlp_plan* plan, const void* values, const void* residual,
                          void* out_y, const mt_mlp_trace* trace, void* stream);
mt_status mt_mlp_plan_destroy(mt_mlp_plan* plan);

/*
 * The same L-layer pass as mt_mlp_plan_run, for callers that cannot let the
 * library allocate device memory: engines that reserve the device's memory up
 * front for their own pool (an allocation by the library would fail or take
 * memory the engine has already planned) and code that must not synchronise
 * the device (cudaMalloc and cudaFree may).  The meTile pages have no
 * counterpart to this call: their executor is built once together with its
 * memory.
 *   layers, L, d, f, group, fmt, eps : as for mt_mlp_plan_create (layers is a
 *            host array, read during the call; it may be freed afterwards)
 *   values, residual, out_y, stream  : as for mt_mlp_plan_run (no trace)
 * Scratch.  The layer table and the hand-off words live in one static device
 * array of MT_STACK_SCRATCH_BYTES bytes per device:
 *   128*ceil(80 L / 128) + 128 + 2*128*ceil(4 S / 128)
 *     + 128*ceil(2 d / 128) + 128*ceil(2 f / 128)      bytes, S = SM count
 * (37,120 bytes for 36 layers of d = 4096, f = 12288 on 152 SMs).  Larger
 * problems return MT_ERR_SHAPE.
 * Launches.  Each call launches a one-block kernel per 48 layers that takes
 * the table as kernel parameters, writes it to the array and zeroes the
 * barrier line, then the stack kernel, all on `stream`.  It makes no copy
 * from host memory and calls no allocating or synchronising routine, so the
 * call can be captured into a CUDA graph; the graph then replays the table
 * and the pointers of the captured call.
 * Set-up.  Every call looks up the array's device address
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit
 * (cudaFuncSetAttribute), so the call stays valid across a cudaDeviceReset.
 * The first call in a process may load the library's device code: make it
 * before any stream capture.
 * Concurrency.  Every call on a device uses the same array: calls that can
 * overlap in time (other streams, or calls not ordered by the caller) race
 * and give undefined results.
 * Errors.  As for mt_mlp_plan_create and mt_mlp_plan_run.
 */
#define MT_STACK_SCRATCH_BYTES 262144
mt_status mt_mlp_stack_run_noalloc(const mt_mlp_layer* layers, int L, int d, int f, int group,
                                   mt_wfmt fmt, float eps, const void* values,
                                   const void* residual, void* out_y, void* stream);

/* Library options.  Returns MT_ERR_FORMAT for an unknown option. */
mt_status mt_set_option(mt_option opt, int value);
int mt_get_option(mt_option opt);

/* Device error word: MT_ERR_TIMEOUT if a kernel's bounded wait expired since
 * the word was last cleared, 0 otherwise, -1 if it cannot be read.  Reading it
 * synchronises with the device (cudaMemcpyFromSymbol); clear != 0 resets it. */
int mt_device_error(int clear);

/* Static description of a status code (never NULL). */
const char* mt_status_string(mt_status s);

/* cudaError_t of the last failed CUDA call made by the library in this
 * thread (0 if none). */
int mt_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
int mt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MT_H */

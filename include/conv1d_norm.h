/*
 * conv1d_norm.h — C ABI of the fused Conv1d (implicit GEMM) + normalization operator for GB300 (sm_103a).
 *
 * What it computes (web pages on the subject "gemm_groupnorm_accelerator"):
 *   [p1] Kimi-K2.6 l2_p35 page — Conv1d followed by GroupNorm: convolution sum, output length,
 *        GroupNorm statistics over (channels of a group x all time steps) of one sample,
 *        population variance, eps inside the square root, per-channel affine.
 *   [p2] Kimi-K2.6 l2_p75 page — Linear + GroupNorm on [rows, channels], then the minimum over
 *        channels of every row and a broadcast add of a per-channel bias.
 *   [p3] Kimi-K2.6 l1_p5 page — causal Conv1d: left padding (k-1)*dilation, tap 0 is the oldest
 *        input; the convolution viewed as a GEMM with M = N*T_out, N = C_out, K = C_in*k.
 *   [p4] Kimi-K2.6 l2_p3 page — LayerNorm with affine and the exact-erf GELU; its model's
 *        ConvTranspose3d, scalar add, LayerNorm over the last dimension, AvgPool3d and GELU
 *        (conv_transpose3d_run, ln_avgpool3d_gelu_run and the one-pass
 *        conv_transpose3d_ln_avgpool3d_gelu_run below).
 *
 *   c[n][co][t] = b[co] + sum_ci sum_kk w[co][ci][kk] * x[n][ci][t*stride + kk*dilation - pad_left]
 *                 (x = 0 outside [0, T));  T_out = (T + pad_left + pad_right - dilation*(k-1) - 1)/stride + 1
 *   norm  GROUP:          z = (c - mean_{n,g}) / sqrt(var_{n,g} + eps) * gamma[co] + beta[co]
 *         CHANNEL_LAYER:  the same with the statistics of all C_out channels at one (n, t)
 *   post  GELU_ERF:       y = 0.5 z (1 + erf(z / sqrt 2))
 *         ROWMIN_BIAS:    m[n][t] = min_co z[n][co][t]; y[n][co][t] = m[n][t] + bias2[co]
 *
 * Layouts (all dense, row-major, no padding between rows):
 *   x [N][C_in][T], w [C_out][C_in][k], y [N][C_out][T_out] in the descriptor's dtype (fp32 or bf16);
 *   b, gamma, beta, bias2 [C_out] fp32; argmin [N][T_out] int32.
 *   A Linear layer is the case T = 1, k = 1, no padding: x = X[rows][in], w = W[out][in], y = Y[rows][out].
 *
 * Ownership: the caller owns every device buffer, the workspace and the stream. The library owns only
 * the descriptor (host memory). The library never allocates device memory and never synchronises inside
 * run(); all work is enqueued on the caller's stream.
 *
 * Errors: every entry point returns a c1n_status; nothing throws across this boundary.
 *   Argument errors are reported by desc_create; pointer alignment and workspace errors by run.
 *   Device-side failures (a bounded wait that ran out) set a status word in the workspace that
 *   conv1d_norm_check() reads. conv1d_norm_last_error() gives a message for the calling thread.
 *
 * Thread safety: a descriptor may be used by one host thread at a time (run() caches encoded TMA
 * descriptors inside it). Distinct descriptors are independent.
 */
#ifndef CONV1D_NORM_H
#define CONV1D_NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* c1n_stream_t;

typedef enum {
    C1N_OK = 0,
    C1N_ERR_INVALID_ARG = 1,  /* a parameter or pointer is out of range / missing */
    C1N_ERR_UNSUPPORTED = 2,  /* valid operator, but the requested math path cannot run it */
    C1N_ERR_ALIGNMENT = 3,    /* a device pointer is not 16-byte aligned where the tensor path needs it */
    C1N_ERR_WORKSPACE = 4,    /* workspace missing or smaller than conv1d_norm_workspace_size() */
    C1N_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch error, no device, ...) */
    C1N_ERR_TIMEOUT = 6,      /* a device-side bounded wait ran out (reported by conv1d_norm_check) */
    C1N_ERR_DEVICE = 7        /* another device-side consistency check failed (reported by check) */
} c1n_status;

typedef enum { C1N_NORM_NONE = 0, C1N_NORM_GROUP = 1, C1N_NORM_CHANNEL_LAYER = 2 } c1n_norm;
typedef enum { C1N_POST_NONE = 0, C1N_POST_GELU_ERF = 1, C1N_POST_ROWMIN_BIAS = 2 } c1n_post;
typedef enum { C1N_F32 = 0, C1N_BF16 = 1 } c1n_dtype;

/* Arithmetic used for the contraction. AUTO and TENSOR take the tensor-core path (TF32 tensor
 * cores for fp32 data, BF16 for bf16 data); a shape that path cannot take (stride > 1, T not a
 * multiple of 16 bytes of elements, more than 16 taps, ...) makes desc_create return
 * C1N_ERR_UNSUPPORTED: there is no silent fallback to another kind of arithmetic. SIMT (the fp32
 * FMA CUDA-core path, which takes every valid shape) runs only when the caller asks for it.
 * TENSOR_X3 (fp32 data, convolution plans): fp32-accurate tensor cores. Each operand is split into
 * a TF32 head and a TF32 tail (x = hi + lo, hi = x rounded to TF32, lo = x - hi) and the products
 * are accumulated in fp32 as hi*hi + hi*lo + lo*hi (three MMAs per step; lo*lo, ~2^-22 of the
 * product, is dropped), which meets fp32-level tolerances at about a third of the TF32 rate.
 * Unsupported (C1N_ERR_UNSUPPORTED) for bf16 data and for the Linear plan. */
typedef enum { C1N_MATH_AUTO = 0, C1N_MATH_SIMT = 1, C1N_MATH_TENSOR = 2, C1N_MATH_TENSOR_X3 = 3 } c1n_math;

/* Execution plans (reported by conv1d_norm_plan_info; forceable for testing and measurement). */
typedef enum {
    C1N_PATH_AUTO = -1,
    C1N_PATH_SIMT = 0,            /* SIMT conv kernel + statistics + normalize/post-op kernels */
    C1N_PATH_TC_DIRECT = 1,       /* tcgen05 conv, bias (and GELU) in the epilogue, no normalization */
    C1N_PATH_TC_FUSED_GN = 2,     /* tcgen05 conv with GroupNorm fused: the CTAs covering one sample
                                     exchange partial statistics (through global memory across a
                                     cooperative grid when the whole grid fits on the GPU at once,
                                     else through distributed shared memory inside a thread-block
                                     cluster), then normalize their tiles in place and store once */
    C1N_PATH_TC_TWO_PASS = 3,     /* tcgen05 conv writes raw tiles and their partial statistics
                                     (mean, M2 per tile), a small kernel merges the partials, then one
                                     normalize pass; GroupNorm whose groups straddle a channel block
                                     reads the raw output in a statistics pass instead */
    C1N_PATH_TC_LINEAR = 4,       /* T = 1, k = 1: tcgen05 GEMM (rows x out); GroupNorm over groups of
                                     8/16/32 channels, affine, GELU or row-min fused in the epilogue
                                     (row-min then needs one finisher kernel); other shapes use the
                                     statistics / normalize / row-min passes */
    C1N_PATH_TC_FUSED_GN_DSMEM = 5, /* as TC_FUSED_GN, always through a thread-block cluster (DSMEM) */
    C1N_PATH_TC_FUSED_LN = 6      /* tcgen05 conv with channel LayerNorm (+ GELU) fused: one CTA holds
                                     all C_out <= 512 channels of a 128-step tile in TMEM */
} c1n_path;

/* Tensor-core mainloop. PAIR: two CTAs on neighbouring SMs (a thread-block cluster of two)
 * compute one 256-row x BN tile with tcgen05.mma.cta_group::2; each CTA stages its own 128 rows of
 * A and half of the BN columns of B, so every SM streams a third less operand data per MMA.
 * SINGLE: one CTA per 128-row tile. AUTO takes PAIR for the Linear plan and for convolution plans
 * with at least 148 units of 256 rows (about two per pair of SMs), SINGLE for
 * smaller convolutions (more tiles to spread over the SMs). PAIR fails with C1N_ERR_UNSUPPORTED
 * where the plan cannot use pairs (fused GroupNorm, SIMT, MMA N not a multiple of 32). */
typedef enum { C1N_MAINLOOP_AUTO = 0, C1N_MAINLOOP_SINGLE = 1, C1N_MAINLOOP_PAIR = 2 } c1n_mainloop;

typedef struct {
    int32_t N, C_in, C_out, T, k;
    int32_t stride, pad_left, pad_right, dilation;
    int32_t norm;        /* c1n_norm */
    int32_t groups;      /* GroupNorm group count; C_out % groups == 0 */
    float eps;           /* > 0 when norm != NONE */
    int32_t post;        /* c1n_post */
    int32_t dtype;       /* c1n_dtype of x, w and y */
    int32_t math;        /* c1n_math */
    int32_t force_path;  /* c1n_path; C1N_PATH_AUTO (-1) lets the planner choose */
    int32_t mainloop;    /* c1n_mainloop; 0 = AUTO */
} c1n_params;

typedef struct c1n_desc c1n_desc;

typedef struct {
    int32_t path;            /* c1n_path chosen */
    int32_t T_out;
    int32_t tile_t;          /* output time steps per tile (tensor paths) */
    int32_t tile_co;         /* output channels per tile */
    int32_t mma_n;           /* tcgen05 N extent per MMA */
    int32_t cluster;         /* CTAs per thread-block cluster (1 = none) */
    int32_t n_tiles;
    int32_t grid;            /* CTAs of the main kernel */
    int32_t kernels;         /* kernels one run() enqueues */
    int32_t cta_pair;        /* 1 when the tensor-core mainloop runs on CTA pairs (tile_t = 256) */
    int64_t workspace_bytes;
} c1n_plan_info;

/* Validate `params`, choose an execution plan and return a host-side descriptor in *out.
 * No device memory is touched; the call works without a GPU. */
c1n_status conv1d_norm_desc_create(const c1n_params* params, c1n_desc** out);

/* Bytes of device scratch that run() needs (status word, packed weights, statistics, raw tiles). */
c1n_status conv1d_norm_workspace_size(const c1n_desc* desc, size_t* bytes);

/* Attach caller-owned device scratch of at least conv1d_norm_workspace_size() bytes (256-byte
 * aligned) for use by conv1d_norm_run(). The library never frees it. */
c1n_status conv1d_norm_set_workspace(c1n_desc* desc, void* workspace, size_t bytes);

c1n_status conv1d_norm_plan_info(const c1n_desc* desc, c1n_plan_info* info);

/* Enqueue the operator on `stream`, using the attached workspace. x, w, y are device pointers in
 * the descriptor's dtype; b, gamma, beta are device fp32 pointers or NULL (no bias; gamma = 1,
 * beta = 0). Needs post != ROWMIN_BIAS (use run_ex for bias2/argmin). Asynchronous. The tensor-core
 * kernels release programmatic dependents once their MMAs are done: a kernel the caller launches
 * next on `stream` with programmatic stream serialization must, as that launch mode requires, wait
 * (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads y. Ordinary launches, copies
 * and events are ordered as usual. */
c1n_status conv1d_norm_run(c1n_desc* desc, const void* x, const void* w, const float* b,
                           const float* gamma, const float* beta, void* y, c1n_stream_t stream);

typedef struct {
    const void* x;
    const void* w;
    const float* b;          /* nullable */
    const float* gamma;      /* nullable */
    const float* beta;       /* nullable */
    const float* bias2;      /* required iff post == ROWMIN_BIAS */
    void* y;
    int32_t* argmin;         /* nullable; [N][T_out] when post == ROWMIN_BIAS */
    void* workspace;         /* NULL: use the workspace attached with conv1d_norm_set_workspace */
    size_t workspace_bytes;
    uint32_t flags;          /* C1N_FLAG_* */
} c1n_args;

/* The weights were already packed into this workspace by conv1d_norm_pack_weights (same w, same
 * workspace); run_ex then skips its own packing step. */
#define C1N_FLAG_WEIGHTS_PACKED 1u
/* Testing aid for the device failure path (no counterpart on the pages): on the fused GroupNorm
 * plan whose CTAs exchange statistics through global memory, the first CTA withholds its partial
 * statistics, so the bounded waits of the CTAs of its sample run out (after about one second). The
 * kernel then records C1N_ERR_TIMEOUT (site 10, the grid exchange) in the workspace status word and
 * returns; y is unspecified. Nothing faults or hangs. Other plans refuse the flag with
 * C1N_ERR_INVALID_ARG. conv1d_norm_check reports the timeout and resets the exchange state. */
#define C1N_FLAG_TEST_STALL_EXCHANGE 2u

c1n_status conv1d_norm_run_ex(c1n_desc* desc, const c1n_args* args, c1n_stream_t stream);

/* The weight-packing step alone (the first kernel run()/run_ex() enqueue on the tensor-core conv
 * paths): w[co][ci][kk] -> wp[kk][co][ci_pad] inside the workspace, rounded to tf32 for fp32 data.
 * On paths that read w directly (SIMT, Linear) it enqueues nothing and returns C1N_OK.
 * workspace NULL: the attached one. Asynchronous. */
c1n_status conv1d_norm_pack_weights(c1n_desc* desc, const void* w, void* workspace, size_t workspace_bytes,
                                    c1n_stream_t stream);

/* Synchronise `stream`, read and clear the device status word of the given workspace (NULL: the
 * attached one) and return C1N_OK, C1N_ERR_TIMEOUT or C1N_ERR_DEVICE (the message from
 * conv1d_norm_last_error names the wait site, the CTA and the pipeline's progress counters). After
 * a device failure it also resets the fused GroupNorm exchange words of that workspace, so the next
 * run (weights packed or not) starts from a consistent state. */
c1n_status conv1d_norm_check(const c1n_desc* desc, void* workspace, c1n_stream_t stream);

/* Operator run for callers that cannot allocate device memory (no counterpart on the pages; this is
 * an interface of this library only). Some callers may not call cudaMalloc or any other allocator
 * where they run the operator: code inside a host framework that owns all device allocations, a
 * plugin whose host forbids allocating after start-up, a real-time loop that must not block on an
 * allocator. This entry point allocates nothing. Its scratch is one array of
 * C1N_STATIC_SCRATCH_BYTES bytes in device global memory, part of the library's device image: every
 * GPU that loads the library holds it until the process exits.
 *
 *   - args->x, w, b, gamma, beta, bias2, y, argmin as for conv1d_norm_run_ex; args->workspace must
 *     be NULL (the array is the workspace).
 *   - args->flags must not hold C1N_FLAG_WEIGHTS_PACKED (C1N_ERR_INVALID_ARG): the array is shared
 *     by every descriptor, so the packed weights in it may be another operator's; every call packs.
 *   - Returns C1N_ERR_WORKSPACE if conv1d_norm_workspace_size(desc) exceeds C1N_STATIC_SCRATCH_BYTES.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture.
 *   - Every call clears the status word at the start of the array (stream-ordered) and attaches the
 *     array to `desc` as its workspace, replacing any workspace attached before, so that
 *     conv1d_norm_check(desc, NULL, stream) reads this call's device status.
 *   - All calls, from every descriptor and stream, share the one array and it keeps the last call's
 *     contents: calls that overlap on the GPU (different streams, no ordering between them) race.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine. Asynchronous like run_ex. */
#define C1N_STATIC_SCRATCH_BYTES (4u << 20)
c1n_status conv1d_norm_run_static_scratch(c1n_desc* desc, const c1n_args* args, c1n_stream_t stream);

void conv1d_norm_destroy(c1n_desc* desc);

const char* conv1d_norm_status_string(c1n_status status);

/* Message describing the last failure on the calling host thread ("" if none). */
const char* conv1d_norm_last_error(void);

/* Kernel timing. With profiling enabled, every run records a CUDA event on its stream before each
 * kernel it launches and one after the last (event creation happens on the first such run).
 * conv1d_norm_kernel_times() waits for the last run's final event and reports, in launch order,
 * each kernel's name and the time between its event and the next (milliseconds, that kernel's
 * device time when the stream runs nothing else). *count = number of kernels of the last run (0
 * before any profiled run); at most `capacity` entries are written. Not thread-safe against a
 * concurrent run() on the same descriptor. No counterpart on the pages: a measurement aid. */
typedef struct {
    char name[32];
    float ms;
} c1n_kernel_time;
c1n_status conv1d_norm_set_profiling(c1n_desc* desc, int32_t enable);
c1n_status conv1d_norm_kernel_times(c1n_desc* desc, c1n_kernel_time* out, int32_t capacity, int32_t* count);

/* [p4]'s second operator (Kimi-K2.6 l2_p3 page, the model's steps after its ConvTranspose3d: a
 * scalar added, LayerNorm over the last dimension, AvgPool3d with kernel 2, GELU):
 *
 *   s[n][c][d][h][w] = z[n][c][d][h][w] + sum_weight
 *   l = (s - mean_w s) / sqrt(var_w s + eps) * gamma[w] + beta[w]   (statistics over the W values of
 *        one (n, c, d, h) row, population variance)
 *   out[n][c][d'][h'][w'] = GELU(mean of l over d in {2d', 2d'+1}, h in {2h', 2h'+1}, w in {2w', 2w'+1})
 *
 *   - z [N][C][D][H][W] fp32, out [N][C][D/2][H/2][W/2] fp32 (floor: a trailing odd plane, row or
 *     column belongs to no window), both dense and 16-byte aligned, caller-owned, not overlapping.
 *   - gamma, beta [W] fp32 or NULL (1 and 0).
 *   - W must be 64, 128, 256 or 512 (a row is spread over the lanes of one warp or half-warp);
 *     N, C, D, H >= 1; eps > 0. Otherwise C1N_ERR_INVALID_ARG (bad values) or C1N_ERR_UNSUPPORTED
 *     (another W), and nothing is launched. D < 2 or H < 2 leaves an empty output (C1N_OK).
 *   - One kernel on `stream`, asynchronous; no workspace, no allocation, no synchronisation.
 *   - GELU and the statistics as in the fused operator; memory-bound: z is read once and the pooled
 *     output written once. */
typedef struct {
    int32_t N, C, D, H, W;
    float eps;
} c1n_lnpool_params;
c1n_status ln_avgpool3d_gelu_run(const c1n_lnpool_params* p, const float* z, float sum_weight, const float* gamma,
                                 const float* beta, float* out, c1n_stream_t stream);

/* [p4]'s transposed 3-D convolution (Kimi-K2.6 l2_p3 page, ConvTranspose3d with bias, dilation 1),
 * whose output the pass above takes as z:
 *
 *   y[n][co][od][oh][ow] = b[co] + sum_{ci, kd, kh, kw} x[n][ci][id][ih][iw] * w[ci][co][kd][kh][kw]
 *   over the taps with od = id*stride - pad + kd (likewise h, w) and the input index inside the input;
 *   output extent per axis (in - 1)*stride - 2*pad + (k - 1) + out_pad + 1.
 *
 *   - x [N][C_in][D][H][W], w [C_in][C_out][k][k][k] (the library's transposed-convolution weight
 *     layout), b [C_out] or NULL, y [N][C_out][Do][Ho][Wo]; fp32, dense, caller-owned.
 *   - Taken: k = 3, stride = 2, pad = 1, out_pad 0 or 1, C_out a multiple of 32, all extents >= 1;
 *     other values: C1N_ERR_UNSUPPORTED (or C1N_ERR_INVALID_ARG for non-positive extents).
 *   - math: 0 auto, 1 CUDA cores (fp32 FMA), 2 tensor cores (TF32 operands, fp32 accumulation; takes
 *     C_in = 32, C_out = 64, Wo a multiple of 4, x and y 16-byte aligned, an sm_103a device —
 *     C1N_ERR_UNSUPPORTED otherwise). Auto picks the tensor cores when they take the shape.
 *   - The tensor-core plan needs a workspace (channels-last x, packed weights, a status word) of
 *     conv_transpose3d_workspace_size() bytes, 256-byte aligned, caller-owned; the CUDA-core plan
 *     needs none (0 bytes; workspace may be NULL). Asynchronous on `stream`; no allocation. */
typedef struct {
    int32_t N, C_in, C_out, D, H, W, k, stride, pad, out_pad;
    int32_t math;
} c1n_convt3d_params;
c1n_status conv_transpose3d_workspace_size(const c1n_convt3d_params* p, size_t* bytes);
c1n_status conv_transpose3d_run(const c1n_convt3d_params* p, const float* x, const float* w, const float* b, float* y,
                                void* workspace, size_t workspace_bytes, c1n_stream_t stream);

/* [p4]'s whole model after its weights in one pass (Kimi-K2.6 l2_p3 page: ConvTranspose3d, then
 * + sum_weight, LayerNorm over the last dimension, AvgPool3d(kernel 2, stride 2), exact GELU):
 *
 *   y   = ConvTranspose3d(x; w, b)                     as conv_transpose3d_run defines it
 *   out[n][c][i][j][l] = GELU( mean over a, b2, e in {0,1} of
 *                              LN(y + sum_weight)[n][c][2i+a][2j+b2][2l+e] )
 *   LN over the last dimension (W_out = 64 values): (v - mean) / sqrt(var + eps) * gamma[w] + beta[w],
 *   population variance; gamma, beta [64] (NULL: 1 and 0).
 *
 *   - x [N][32][D][H][32], w [32][64][3][3][3], b [64] or NULL; out [N][64][D][H][32] (the pooled
 *     output has the input's spatial extent); fp32, dense, caller-owned; x and out 16-byte aligned.
 *   - Taken: C_in 32, C_out 64, W 32, k 3, stride 2, pad 1, output pad 1 (the page's model), D, H,
 *     N >= 1, eps > 0; other shapes C1N_ERR_UNSUPPORTED (run conv_transpose3d_run, then
 *     ln_avgpool3d_gelu_run). `math` is ignored (tensor cores: TF32 operands, fp32 accumulation and
 *     statistics). Needs an sm_103a device.
 *   - The convolution's output stays on chip: x is read once (after a channels-last copy into the
 *     workspace) and out written once. b and sum_weight are constant along every LayerNorm row and
 *     cancel in it (LN(v + const) = LN(v)); they are accepted for the model's definition and do not
 *     change the result.
 *   - workspace: conv_transpose3d_ln_avgpool3d_gelu_workspace_size() bytes, 256-byte aligned,
 *     caller-owned (status word, channels-last x, packed weights). Asynchronous on `stream`; no
 *     allocation; three kernels. */
c1n_status conv_transpose3d_ln_avgpool3d_gelu_workspace_size(const c1n_convt3d_params* p, size_t* bytes);
c1n_status conv_transpose3d_ln_avgpool3d_gelu_run(const c1n_convt3d_params* p, float eps, float sum_weight,
                                                  const float* x, const float* w, const float* b,
                                                  const float* gamma, const float* beta, float* out,
                                                  void* workspace, size_t workspace_bytes, c1n_stream_t stream);

/* Library version: major*10000 + minor*100 + patch. */
int32_t conv1d_norm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONV1D_NORM_H */

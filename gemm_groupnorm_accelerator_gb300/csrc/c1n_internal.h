// Internal plan, kernel-argument structures and launcher declarations of the conv1d_norm library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "conv1d_norm.h"

namespace c1n {

constexpr int kMaxTaps = 16;
constexpr int kWsStatusBytes = 256;

// Everything the planner decides once per descriptor.
struct Plan {
    int path = C1N_PATH_SIMT;
    long long T_out = 0;
    int bf16 = 0;         // x/w/y are bf16
    int esize = 4;        // bytes per x/w/y element
    int align = 4;        // elements per 16 bytes
    // tensor-core geometry: tiles of 128 output rows (time steps, or Linear rows) x BN channels
    int BK = 32;          // input channels per pipeline stage (one 128-byte row)
    int R = 128;          // rows of one A tile (128 + tap halo, multiple of 8)
    int RS = 0;           // time steps of one staged x box (R + alignment shift, multiple of 16 bytes)
    int t_shift = 0;      // staged index of A row 0 (pad_left rounded up to 16 bytes, minus pad_left)
    int BN = 0;           // output channels per MMA (<= 256)
    int n_cb = 0;         // channel blocks
    int cb_per_unit = 1;  // channel blocks accumulated by one work unit
    int n_ci_chunks = 0;
    int ci_pad = 0;       // packed-weight row length (multiple of BK)
    int n_t_tiles = 0;    // row tiles along time (conv) or rows (Linear): 128 rows, 256 with a CTA pair
    int n_units = 0;
    int n_acc = 2;        // accumulators per CTA (2: epilogue overlaps the next mainloop)
    int tmem_cols = 512;  // TMEM columns allocated per CTA
    int cluster = 1;
    int pair = 0;         // CTA-pair mainloop (cta_group::2): units of 256 rows, each CTA loads half of B
    int x3 = 0;           // 3xTF32: A and B split into TF32 head + tail, three MMAs per step
    int grid = 0;
    int stages_a = 0, stages_b = 0, stages_s = 0;
    int a_slot_bytes = 0, b_slot_bytes = 0, s_slot_bytes = 0;
    int o_bytes = 0;      // output staging (fused LayerNorm: 4 warps x 2 tiles of 32 x 32 elements)
    int smem_bytes = 0;
    int kernels = 0;
    // workspace layout (byte offsets)
    size_t ws_wp = 0, ws_stats = 0, ws_raw = 0, ws_rowmin = 0, ws_total = 0;
    size_t ws_gx = 0;                   // fused GroupNorm across a cooperative grid: exchange words
    size_t ws_rowpart = 0;              // fused row-min partials
    int row_epilogue = 0;               // Linear plan with the fused row epilogue
    size_t ws_part = 0;                 // two-pass plan: partial statistics from the conv epilogue
    int part_kind = 0;                  // 0: statistics pass over the raw output; 1 / 2: see TcArgs
    int part_tiles = 0;                 // 128-row tiles along T_out
    int gx_words = 0;   // 32-bit words of the exchange area (zeroed by the weight pack)
    int gstride = 0;    // groups per channel block (exchange words per tile / 2)
};

// Shared memory beyond the operand rings: barriers, flags and epilogue scratch.
constexpr int kTcMiscBytes = 16384;

// Arguments of the tensor-core kernel (passed by value as a __grid_constant__).
struct TcArgs {
    int N, C_in, C_out, T, T_out, k, dil, pad_left;
    int BK, R, BN, n_cb, cb_per_unit, n_ci_chunks, n_t_tiles, n_units;
    int n_acc, tmem_cols, stages_a, stages_b, a_slot_bytes, b_slot_bytes;
    int RS, t_shift, stages_s, s_slot_bytes;  // x staging ring (conv mode)
    int groups, cpg;
    int sub;        // channels per partial-sum run in the GroupNorm statistics (4, 8, 16; 0 = per column)
    int tma_store;  // fused GroupNorm / LayerNorm: store the output through TMA bulk stores
    int x3;         // 3xTF32 mainloop (A slots hold the head tile then the tail tile; B stages alternate)
    int o_off;      // LayerNorm: byte offset of the per-warp output staging tiles in shared memory
    int o_bytes;    // ... and their size (shared memory between the operand rings and the barriers)
    float eps;
    int gelu;
    uint32_t idesc;
    const void* x;
    const float* bias;
    const float* gamma;
    const float* beta;
    void* y;
    int* status;
    // per (sample, channel block, time tile, group) two 64-bit words: (mean | epoch), (M2 | epoch)
    unsigned long long* gx;
    int gstride;       // groups per (sample, channel block, time tile) in gx
    int early_inputs;  // the preceding launch is this library's weight pack, which released this
                       // kernel after its own wait for all earlier work: x may be read before
                       // griddepcontrol.wait
    int row_cpg;       // row epilogue: GroupNorm over runs of row_cpg channels (8, 16, 32; 0 = none)
    int rowmin;        // row epilogue: keep (min, argmin) per row instead of storing y
    float2* rowpart;   // row epilogue: per (row, channel block) minimum and its channel (int bits)
    // Two-pass plans (kEpiDirectStats): the epilogue stores the raw tile and its partial statistics
    // (mean, M2) about the partial's own mean. GroupNorm (part_kind 1): per (sample, group, 128-row
    // tile), at part[(n * groups + g) * part_tiles + row0 / 128]; channel LayerNorm (part_kind 2):
    // per (sample, channel block, time step), at part[(n * n_cb + cb) * T_out + t].
    int part_kind;
    int part_tiles;
    float2* part;
    int test_stall;  // C1N_FLAG_TEST_STALL_EXCHANGE: the first CTA withholds its exchange words
};

// Sets the calling thread's message returned by conv1d_norm_last_error().
void set_last_error(const char* msg);

// Launchers (each enqueues on `stream`, returns cudaGetLastError()).
cudaError_t launch_simt_conv(const c1n_params& p, const Plan& pl, const void* x, const void* w, const float* b,
                             void* out, bool out_is_raw_f32, cudaStream_t stream);
cudaError_t launch_gn_stats(const c1n_params& p, const Plan& pl, const float* raw, float2* stats, cudaStream_t stream);
// Statistics from the tensor-core epilogue's partials (TcArgs::part): Chan's merge over the
// 128-row tiles of each (sample, group), or over the channel blocks of each (sample, time step).
cudaError_t launch_gn_merge(const c1n_params& p, const Plan& pl, const float2* part, float2* stats,
                            cudaStream_t stream);
cudaError_t launch_ln_merge(const c1n_params& p, const Plan& pl, const float2* part, float2* stats,
                            cudaStream_t stream);
cudaError_t launch_ln_stats(const c1n_params& p, const Plan& pl, const float* raw, float2* stats, cudaStream_t stream);
cudaError_t launch_normalize(const c1n_params& p, const Plan& pl, const float* raw, const float2* stats,
                             const float* gamma, const float* beta, void* y, cudaStream_t stream);
cudaError_t launch_rowmin(const c1n_params& p, const Plan& pl, const float* raw, const float2* stats,
                          const float* gamma, const float* beta, float* rowmin, int32_t* argmin,
                          cudaStream_t stream);
cudaError_t launch_broadcast(const c1n_params& p, const Plan& pl, const float* rowmin, const float* bias2, void* y,
                             cudaStream_t stream);
// Row-min finisher: per row, the minimum (lowest channel on ties) over the per-block partials,
// then y[row][c] = min + bias2[c]; argmin optional.
cudaError_t launch_rowmin_finish(const c1n_params& p, const Plan& pl, const float2* part, const float* bias2, void* y,
                                 int32_t* argmin, cudaStream_t stream);
// Also zeroes `nzero` words at `zero` (the fused-GroupNorm arrival counters) when given.
// fp32 weights are rounded to TF32; with pl.x3 the TF32 tail w - tf32(w) follows as taps k..2k-1.
cudaError_t launch_pack_weights(const c1n_params& p, const Plan& pl, const void* w, void* wp, cudaStream_t stream,
                                unsigned* zero = nullptr, int nzero = 0, bool release_first = false);

// [p4]'s LayerNorm(last dim) + AvgPool3d + GELU pass; p already validated (W in 64, 128, 256, 512).
cudaError_t launch_ln_avgpool3d_gelu(const c1n_lnpool_params& p, const float* z, float sum_weight,
                                     const float* gamma, const float* beta, float* out, int num_sms,
                                     cudaStream_t stream);

// [p4]'s ConvTranspose3d (k 3, stride 2, pad 1; p already validated): CUDA-core kernel, and the
// tensor-core plan (C_in 32, C_out 64) with its workspace (status word, channels-last x, packed weights).
cudaError_t launch_conv_transpose3d(const c1n_convt3d_params& p, const float* x, const float* w, const float* b,
                                    float* y, cudaStream_t stream);
size_t convt3d_tc_workspace_bytes(const c1n_convt3d_params& p);
// [p4]'s model in one tensor-core kernel (C_in 32, C_out 64, W 32, output pad 1; p validated):
// ConvTranspose3d with + sum_weight, LayerNorm over W_out = 64, AvgPool3d(2) and GELU in the
// epilogue; workspace: status word, channels-last x, the two channel halves' packed weights.
size_t convt3d_lnpool_fused_workspace_bytes(const c1n_convt3d_params& p);
cudaError_t launch_convt3d_lnpool_fused(const c1n_convt3d_params& p, float eps, float sum_weight, const float* x,
                                        const float* w, const float* b, const float* gamma, const float* beta,
                                        float* out, void* workspace, int num_sms, cudaStream_t stream);
cudaError_t launch_conv_transpose3d_tc(const c1n_convt3d_params& p, const float* x, const float* w, const float* b,
                                       float* y, void* workspace, int num_sms, cudaStream_t stream);

// Tensor-core kernels. `tm_a`: x (conv mode, staged time-contiguous boxes) or X (Linear mode);
// `tm_b`: packed weights (conv mode) or W (Linear mode).
// kEpiLNX: channel LayerNorm over the two channel halves held by the two CTAs of a cluster.
// kEpiDirectStats: the direct epilogue plus the partial statistics of a two-pass plan.
enum TcEpilogue {
    kEpiDirect = 0, kEpiClusterGN = 1, kEpiGridGN = 2, kEpiRowGN = 3, kEpiLN = 4, kEpiLNX = 5, kEpiDirectStats = 6
};
cudaError_t launch_tc(const Plan& pl, const TcArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                      const CUtensorMap& tm_y, bool linear, int epilogue, bool out_bf16, int num_sms,
                      cudaStream_t stream);

}  // namespace c1n

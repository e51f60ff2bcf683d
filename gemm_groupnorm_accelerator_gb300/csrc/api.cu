// C ABI, validation and planning of the fused Conv1d + normalization operator.
// The operator is defined on the Kimi-K2.6 l2_p35 (Conv1d + GroupNorm), l2_p75 (Linear +
// GroupNorm + row-min + bias), l1_p5 (causal Conv1d as a GEMM) and l2_p3 (LayerNorm, exact GELU)
// pages; the output length is the padded-window count of the l2_p35 page's output-length check
// with separate left/right padding.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "c1n_internal.h"
#include "sm100_ptx.cuh"

using namespace c1n;

struct c1n_desc {
    c1n_params p;
    Plan plan;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    // cached TMA descriptors (re-encoded when a pointer changes)
    const void* tm_x_ptr = nullptr;
    const void* tm_w_ptr = nullptr;
    const void* tm_y_ptr = nullptr;
    CUtensorMap tm_a;  // A operand map
    CUtensorMap tm_b;  // B operand map
    CUtensorMap tm_y;  // output map (TMA store of the fused GroupNorm tile)
    int device = -1;
    int num_sms = 0;
    // kernel timing (conv1d_norm_set_profiling): one event before each launch of a run, one after
    static constexpr int kMaxMarks = 8;
    int profiling = 0;
    int events_ready = 0;
    int n_marks = 0;
    cudaEvent_t ev[kMaxMarks] = {};
    const char* ev_name[kMaxMarks] = {};
};

namespace {

thread_local std::string g_last_error;

c1n_status fail(c1n_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
c1n_status fail(c1n_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

c1n_status cuda_fail(cudaError_t e, const char* what) {
    return fail(C1N_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// SM count assumed when planning without a device (the smallest Blackwell part); the cooperative
// exchange is re-checked against the real device at run time.
constexpr int kMinSmCount = 148;
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

long long t_out_of(const c1n_params& p) {
    long long span = (long long)p.T + p.pad_left + p.pad_right - (long long)p.dilation * (p.k - 1) - 1;
    if (span < 0) return 0;
    return span / p.stride + 1;
}

// Why the tensor-core conv path cannot take this shape ("" when it can).
const char* tc_conv_blocker(const c1n_params& p, const Plan& pl) {
    if (p.stride != 1) return "stride > 1";
    if (p.T % pl.align != 0) return "T is not a multiple of 16 bytes of elements (TMA row stride of x)";
    if ((long long)p.C_in * p.k > 32768) return "C_in * k above 32768 (one weight row per packing CTA)";
    if (p.k > kMaxTaps) return "more than 16 taps";
    if (p.N > 65535) return "N above 65535";
    return "";
}

void plan_workspace(const c1n_params& p, Plan& pl, bool conv_tc, bool need_raw, bool need_stats) {
    size_t off = kWsStatusBytes;
    if (conv_tc) {
        pl.ws_wp = off;
        off = round_up(off + (size_t)(pl.x3 ? 2 : 1) * p.k * p.C_out * pl.ci_pad * pl.esize, 256);
    }
    if (need_stats) {
        pl.ws_stats = off;
        size_t n = p.norm == C1N_NORM_GROUP ? (size_t)p.N * p.groups : (size_t)p.N * pl.T_out;
        off = round_up(off + n * sizeof(float2), 256);
    }
    if (p.post == C1N_POST_ROWMIN_BIAS) {
        pl.ws_rowmin = off;
        off = round_up(off + (size_t)p.N * pl.T_out * sizeof(float), 256);
    }
    if (need_raw) {
        pl.ws_raw = off;
        off = round_up(off + (size_t)p.N * p.C_out * pl.T_out * sizeof(float), 256);
    }
    pl.ws_total = off;
}

// Channel blocks of at most 256 (MMA N), balanced and rounded to 16.
void plan_channel_blocks(const c1n_params& p, Plan& pl) {
    pl.n_cb = (int)ceil_div(p.C_out, 256);
    pl.BN = (int)round_up(ceil_div(p.C_out, pl.n_cb), 16);
    pl.b_slot_bytes = pl.BN * 128;
}

// Ring depths from the shared-memory budget (one CTA per SM), after the output staging area. The
// x-staging ring gives way first (down to two slots: its boxes are small and prefetched to L2),
// then the weight ring (whose 16-32 KB stages come from L2 with ~1 us of latency and feed every
// MMA), then the A ring. (bf16 LayerNorm, 5 taps: 3 weight stages instead of 2 took a short burst
// of calls from 266 to 250 us each; under seconds of load the power cap holds both near 267 us.)
void plan_stages(Plan& pl, int max_a, int max_b, int max_s) {
    const int budget = 227 * 1024 - 1024 - kTcMiscBytes;
    pl.stages_a = max_a;
    pl.stages_b = max_b;
    pl.stages_s = pl.s_slot_bytes > 0 ? max_s : 0;
    auto total = [&]() {
        return pl.stages_a * pl.a_slot_bytes + pl.stages_b * pl.b_slot_bytes + pl.stages_s * pl.s_slot_bytes +
               pl.o_bytes;
    };
    while (total() > budget && pl.stages_s > 2) --pl.stages_s;
    while (total() > budget && pl.stages_b > 2) --pl.stages_b;
    while (total() > budget && pl.stages_a > 2) --pl.stages_a;
    pl.smem_bytes = 1024 + total() + kTcMiscBytes;
}

// The weight pack releases the fused-GroupNorm conv kernel that follows before it waits for the
// preceding kernel when the grid is large: the conv CTAs then take the SMs as the preceding
// kernel's leave, instead of launching once the pack has waited (conv_gn, 128 CTAs: 17.75 vs
// 18.06 us per step). The conv kernel then waits for the pack before it loads x; with few CTAs the
// early x loads matter more (2 CTAs: 8.0 vs 8.2 us), and the pack releases after its wait.
bool pack_releases_first(const Plan& pl) { return pl.path == C1N_PATH_TC_FUSED_GN && pl.n_units >= 32; }

// CTA pairs (cta_group::2) need an MMA N that splits into two halves of whole 16-row groups. Each
// CTA of a pair streams half of the weight tile through its shared memory. AUTO uses them for the
// Linear GEMM (0.88 vs 0.70 of tensor peak on 1024x8192x8192) and for convolutions with at least
// two 256-row units per pair of SMs (causal 32x256x8192 k4: 200 vs 209 us with four A slots per
// CTA); smaller convolutions keep one CTA per 128-row tile (more tiles to spread over the SMs).
bool pair_ok(const c1n_params& p, const Plan& pl, bool linear) {
    if (pl.BN % 32 != 0 || p.mainloop == C1N_MAINLOOP_SINGLE || pl.x3) return false;
    if (linear || p.mainloop == C1N_MAINLOOP_PAIR) return true;
    const long long pair_units = (long long)p.N * ceil_div(pl.T_out, 256) * pl.n_cb;
    return pair_units >= kMinSmCount;
}

// Geometry of the tensor-core conv tiles: 128 output time steps x BN channels per tile (256 steps
// for a CTA pair, 128 per CTA); the A tile carries the (k-1)*dilation halo rows. `cluster` selects
// one CTA per tile with single-buffered TMEM (cluster GroupNorm) instead of the persistent
// double-buffered layout; `o_bytes` reserves output staging.
bool plan_tc_geometry(const c1n_params& p, Plan& pl, bool cluster, bool pair = false, int o_bytes = 0) {
    pl.o_bytes = o_bytes;
    pl.BK = pl.bf16 ? 64 : 32;
    const long long halo = (long long)(p.k - 1) * p.dilation;
    pl.R = (int)round_up(128 + halo, 8);
    // x is staged by TMA from a 16-byte aligned time coordinate: pad_left rounded up to the
    // alignment, so A row r is staged index r + t_shift.
    const long long pl_al = (long long)round_up(p.pad_left, pl.align);
    pl.t_shift = (int)(pl_al - p.pad_left);
    pl.RS = (int)round_up(pl.R + pl.t_shift, pl.align);
    // bf16: the transposer's ldmatrix reads 8 channel rows of 16 bytes at the row pitch RS; an odd
    // multiple of 16 bytes puts them in 8 different bank groups
    if (pl.bf16) {
        pl.RS = (int)round_up(pl.R + pl.t_shift, 8);
        if (pl.RS % 16 != 8) pl.RS += 8;
    }
    if (pl.RS > 256) return false;  // one TMA box per (chunk, tile)
    pl.a_slot_bytes = pl.R * 128 * (pl.x3 ? 2 : 1);  // 3xTF32: head tile then tail tile
    pl.s_slot_bytes = (int)round_up((size_t)pl.BK * pl.RS * pl.esize, 1024);
    pl.n_ci_chunks = (int)ceil_div(p.C_in, pl.BK);
    pl.ci_pad = pl.n_ci_chunks * pl.BK;
    plan_channel_blocks(p, pl);
    pl.pair = (pair && !cluster && pair_ok(p, pl, false)) ? 1 : 0;
    if (pl.pair) pl.b_slot_bytes = pl.BN / 2 * 128;
    pl.cb_per_unit = 1;
    pl.n_t_tiles = (int)ceil_div(pl.T_out, pl.pair ? 256 : 128);
    pl.n_units = p.N * pl.n_t_tiles * pl.n_cb;
    if (cluster) {
        pl.n_acc = 1;
        pl.tmem_cols = 256;
    } else {
        pl.n_acc = 2;
        pl.tmem_cols = 512;
    }
    if (pl.pair) plan_stages(pl, 4, 8, 2);  // half-size B slots: a deeper weight ring; A slots for 4 chunks
    else if (cluster) plan_stages(pl, std::max(2, std::min(pl.n_ci_chunks, 4)), 4, 2);  // one tile per CTA: A
                                                                                        // slots for up to 4
                                                                                        // chunks, so x staging
                                                                                        // runs ahead of the MMA
    else plan_stages(pl, 2, 4, 4);
    return pl.smem_bytes <= 227 * 1024;
}

bool plan_tc_linear(const c1n_params& p, Plan& pl) {
    pl.BK = pl.bf16 ? 64 : 32;
    pl.R = 128;
    pl.a_slot_bytes = 128 * 128;
    pl.n_ci_chunks = (int)ceil_div(p.C_in, pl.BK);
    pl.ci_pad = 0;
    plan_channel_blocks(p, pl);
    pl.pair = pair_ok(p, pl, true) ? 1 : 0;
    if (pl.pair) pl.b_slot_bytes = pl.BN / 2 * 128;
    pl.cb_per_unit = 1;
    pl.n_t_tiles = (int)ceil_div(p.N, pl.pair ? 256 : 128);  // row tiles
    pl.n_units = pl.n_t_tiles * pl.n_cb;
    pl.n_acc = 2;
    pl.tmem_cols = 512;
    pl.s_slot_bytes = 0;
    // one ring: stage i holds A chunk i and B chunk i (one full / empty barrier pair)
    const int budget = 227 * 1024 - 1024 - kTcMiscBytes;
    const int stages = std::min(8, budget / (pl.a_slot_bytes + pl.b_slot_bytes));
    pl.stages_a = pl.stages_b = stages;
    pl.stages_s = 0;
    pl.smem_bytes = 1024 + stages * (pl.a_slot_bytes + pl.b_slot_bytes) + kTcMiscBytes;
    return stages >= 2 && pl.smem_bytes <= 227 * 1024;
}

c1n_status make_plan(const c1n_params& p, Plan& pl) {
    pl = Plan();
    pl.T_out = t_out_of(p);
    pl.bf16 = p.dtype == C1N_BF16;
    pl.esize = pl.bf16 ? 2 : 4;
    pl.x3 = p.math == C1N_MATH_TENSOR_X3 ? 1 : 0;
    if (pl.x3 && pl.bf16) return fail(C1N_ERR_UNSUPPORTED, "3xTF32 math needs fp32 data");
    pl.align = 16 / pl.esize;
    const bool is_linear = p.T == 1 && p.k == 1 && p.pad_left == 0 && p.pad_right == 0 && p.stride == 1;
    const bool out_needs_second_pass = p.norm != C1N_NORM_NONE || p.post == C1N_POST_ROWMIN_BIAS;
    int want = p.force_path;

    auto choose_simt = [&]() {
        pl.path = C1N_PATH_SIMT;
        const bool need_stats = p.norm != C1N_NORM_NONE;
        const bool need_raw = out_needs_second_pass && pl.bf16;
        plan_workspace(p, pl, false, need_raw, need_stats);
        pl.kernels = 1 + (need_stats ? 2 : 0) + (p.post == C1N_POST_ROWMIN_BIAS ? (need_stats ? 1 : 2) : 0);
        pl.grid = (int)(ceil_div(pl.T_out, 64) * ceil_div(p.C_out, 64) * p.N);
        pl.n_units = pl.grid;
        return C1N_OK;
    };

    if (p.math == C1N_MATH_SIMT) {
        if (want != C1N_PATH_AUTO && want != C1N_PATH_SIMT)
            return fail(C1N_ERR_INVALID_ARG, "force_path %d conflicts with math=SIMT", want);
        return choose_simt();
    }
    if (want == C1N_PATH_SIMT) return choose_simt();

    // ---------------------------------------------------------------- tensor-core plans
    const char* why = "";
    if (is_linear && pl.x3) {
        why = "3xTF32 math is built for the convolution plans, not the Linear GEMM";
    } else if (is_linear && (want == C1N_PATH_AUTO || want == C1N_PATH_TC_LINEAR)) {
        if (p.C_in % pl.align != 0) {
            why = "Linear: input features not a multiple of 16 bytes of elements";
        } else if (plan_tc_linear(p, pl)) {
            pl.path = C1N_PATH_TC_LINEAR;
            pl.cluster = 1;
            // Fused row epilogue: GroupNorm groups of 8/16/32 channels inside one channel block
            // (or no normalization), any post-op.
            const int cpg = p.norm == C1N_NORM_GROUP ? p.C_out / p.groups : 0;
            const bool row_ok = p.norm == C1N_NORM_NONE ||
                                (p.norm == C1N_NORM_GROUP && (cpg == 8 || cpg == 16 || cpg == 32) && pl.BN % cpg == 0);
            if (row_ok && (p.norm != C1N_NORM_NONE || p.post == C1N_POST_ROWMIN_BIAS)) {
                pl.row_epilogue = 1;
                plan_workspace(p, pl, false, false, false);
                if (p.post == C1N_POST_ROWMIN_BIAS) {
                    pl.ws_rowpart = pl.ws_total;
                    pl.ws_total = round_up(pl.ws_total + (size_t)p.N * pl.n_cb * sizeof(float2), 256);
                }
                pl.kernels = p.post == C1N_POST_ROWMIN_BIAS ? 2 : 1;
                return C1N_OK;
            }
            const bool need_stats = p.norm != C1N_NORM_NONE;
            const bool need_raw = out_needs_second_pass && pl.bf16;
            plan_workspace(p, pl, false, need_raw, need_stats);
            pl.kernels = 1 + (need_stats ? 1 : 0) + (p.post == C1N_POST_ROWMIN_BIAS ? 2 : (need_stats ? 1 : 0));
            return C1N_OK;
        }
    } else if (want == C1N_PATH_TC_LINEAR) {
        why = "TC_LINEAR needs T = 1, k = 1, stride 1 and no padding";
    } else {
        why = tc_conv_blocker(p, pl);
        if (!*why) {
            const int cpg = p.norm == C1N_NORM_GROUP ? p.C_out / p.groups : 0;
            // 1. GroupNorm fused into the conv kernel: one CTA per (sample, time tile, channel
            //    block); groups must not straddle a channel block. The CTAs of a sample exchange
            //    partial statistics across a cooperative grid (whole grid resident at once) or a
            //    thread-block cluster of at most 8 CTAs.
            Plan trial = pl;
            const bool geom_ok = plan_tc_geometry(p, trial, true);
            const bool groups_ok = p.norm == C1N_NORM_GROUP && p.post != C1N_POST_ROWMIN_BIAS && geom_ok &&
                                   (trial.n_cb == 1 || trial.BN % cpg == 0);
            const bool cluster_ok = groups_ok && trial.n_t_tiles <= 8;
            const bool grid_ok = groups_ok && trial.n_units <= kMinSmCount;
            const bool fused_ok = want == C1N_PATH_TC_FUSED_GN_DSMEM ? cluster_ok : (cluster_ok || grid_ok);
            if ((want == C1N_PATH_AUTO || want == C1N_PATH_TC_FUSED_GN || want == C1N_PATH_TC_FUSED_GN_DSMEM) &&
                fused_ok) {
                pl = trial;
                pl.path = want == C1N_PATH_TC_FUSED_GN_DSMEM ? C1N_PATH_TC_FUSED_GN_DSMEM : C1N_PATH_TC_FUSED_GN;
                pl.cluster = pl.n_t_tiles;
                pl.grid = pl.n_units;
                plan_workspace(p, pl, true, false, false);
                // grid exchange: per (sample, channel block, time tile, group) two 64-bit words
                pl.gstride = (std::min(pl.BN, p.C_out) + cpg - 1) / cpg;
                pl.gx_words = pl.n_units * pl.gstride * 4;
                pl.ws_gx = pl.ws_total;
                pl.ws_total = round_up(pl.ws_gx + (size_t)pl.gx_words * 4, 256);
                pl.kernels = 2;
                return C1N_OK;
            }
            if (want == C1N_PATH_TC_FUSED_GN || want == C1N_PATH_TC_FUSED_GN_DSMEM)
                why = "fused GroupNorm needs groups inside a channel block, no row-min, and the CTAs of a sample "
                      "in one cluster (<= 8) or the whole grid resident at once";
            // 1b. Channel LayerNorm fused. C_out <= 256: one CTA holds every channel of its tile.
            //     256 < C_out <= 512: the two CTAs of a cluster hold one channel half each of the
            //     same 128 time steps and exchange per-step partial sums through distributed shared
            //     memory. Either way each CTA keeps two accumulators, so the epilogue of one tile
            //     overlaps the mainloop of the next.
            if (!*why && p.norm == C1N_NORM_CHANNEL_LAYER && p.post != C1N_POST_ROWMIN_BIAS && p.C_out <= 512 &&
                (want == C1N_PATH_AUTO || want == C1N_PATH_TC_FUSED_LN)) {
                Plan ln = pl;
                const bool two = p.C_out > 256;
                // output staging: 2 tiles of 32 x 32 per epilogue warp (8 warps for bf16, else 4)
                if (plan_tc_geometry(p, ln, false, !two, (ln.bf16 ? 8 : 4) * 2 * 32 * 32 * ln.esize)) {
                    ln.cb_per_unit = two ? 1 : ln.n_cb;
                    ln.n_units = p.N * ln.n_t_tiles;
                    ln.n_acc = 2;
                    ln.tmem_cols = 512;
                    ln.cluster = two ? 2 : 1;
                    pl = ln;
                    pl.path = C1N_PATH_TC_FUSED_LN;
                    plan_workspace(p, pl, true, false, false);
                    pl.kernels = 2;
                    return C1N_OK;
                }
            }
            if (want == C1N_PATH_TC_FUSED_LN && !*why)
                why = "TC_FUSED_LN needs channel LayerNorm, no row-min and C_out <= 512";
            // 2. Direct epilogue (no normalization).
            if (!*why && p.norm == C1N_NORM_NONE && p.post != C1N_POST_ROWMIN_BIAS &&
                (want == C1N_PATH_AUTO || want == C1N_PATH_TC_DIRECT)) {
                if (plan_tc_geometry(p, pl, false, true)) {
                    pl.path = C1N_PATH_TC_DIRECT;
                    plan_workspace(p, pl, true, false, false);
                    pl.kernels = 2;
                    return C1N_OK;
                }
                why = "tap span too wide for one A tile";
            } else if (want == C1N_PATH_TC_DIRECT) {
                why = "TC_DIRECT needs norm NONE and no row-min";
            }
            // 3. Two passes: raw tiles, then statistics and normalize / row-min passes.
            if (!*why && (want == C1N_PATH_AUTO || want == C1N_PATH_TC_TWO_PASS)) {
                if (plan_tc_geometry(p, pl, false, true)) {
                    pl.path = C1N_PATH_TC_TWO_PASS;
                    const bool need_stats = p.norm != C1N_NORM_NONE;
                    const bool need_raw = out_needs_second_pass && pl.bf16;
                    plan_workspace(p, pl, true, need_raw, need_stats);
                    // The conv epilogue writes partial statistics with the raw tiles (GroupNorm:
                    // when no group straddles a channel block), so no pass re-reads the raw output
                    // for them; a small kernel merges the partials.
                    size_t n_part = 0;
                    if (p.norm == C1N_NORM_GROUP && (pl.n_cb == 1 || pl.BN % (p.C_out / p.groups) == 0)) {
                        pl.part_kind = 1;
                        pl.part_tiles = (int)ceil_div(pl.T_out, 128);
                        n_part = (size_t)p.N * p.groups * pl.part_tiles;
                    } else if (p.norm == C1N_NORM_CHANNEL_LAYER) {
                        pl.part_kind = 2;
                        n_part = (size_t)p.N * pl.n_cb * pl.T_out;
                    }
                    if (n_part) {
                        pl.ws_part = pl.ws_total;
                        pl.ws_total = round_up(pl.ws_part + n_part * sizeof(float2), 256);
                    }
                    pl.kernels = 2 + (need_stats ? 1 : 0) + (p.post == C1N_POST_ROWMIN_BIAS ? 2 : 1);
                    return C1N_OK;
                }
                why = "tap span too wide for one A tile";
            }
        }
    }
    // No silent fallback: a shape the tensor-core path cannot take is refused; the SIMT fp32 CUDA
    // path runs only when the caller asks for it (math = SIMT).
    if (want != C1N_PATH_AUTO)
        return fail(C1N_ERR_UNSUPPORTED, "tensor-core path unavailable: %s", *why ? why : "forced path not applicable");
    return fail(C1N_ERR_UNSUPPORTED, "tensor-core path unavailable: %s (math = SIMT runs the fp32 CUDA-core path)",
                *why ? why : "no tensor-core plan takes this operator");
}

c1n_status validate(const c1n_params* p) {
    if (!p) return fail(C1N_ERR_INVALID_ARG, "params is NULL");
    if (p->N < 1 || p->C_in < 1 || p->C_out < 1 || p->T < 1 || p->k < 1)
        return fail(C1N_ERR_INVALID_ARG, "N, C_in, C_out, T and k must be >= 1");
    if (p->stride < 1 || p->dilation < 1) return fail(C1N_ERR_INVALID_ARG, "stride and dilation must be >= 1");
    if (p->pad_left < 0 || p->pad_right < 0) return fail(C1N_ERR_INVALID_ARG, "padding must be >= 0");
    if (p->norm < 0 || p->norm > 2) return fail(C1N_ERR_INVALID_ARG, "unknown norm %d", p->norm);
    if (p->post < 0 || p->post > 2) return fail(C1N_ERR_INVALID_ARG, "unknown post-op %d", p->post);
    if (p->dtype < 0 || p->dtype > 1) return fail(C1N_ERR_INVALID_ARG, "unknown dtype %d", p->dtype);
    if (p->math < 0 || p->math > 3) return fail(C1N_ERR_INVALID_ARG, "unknown math %d", p->math);
    if (p->force_path < -1 || p->force_path > 6) return fail(C1N_ERR_INVALID_ARG, "unknown path %d", p->force_path);
    if (p->mainloop < 0 || p->mainloop > 2) return fail(C1N_ERR_INVALID_ARG, "unknown mainloop %d", p->mainloop);
    if (p->norm == C1N_NORM_GROUP && (p->groups < 1 || p->C_out % p->groups != 0))
        return fail(C1N_ERR_INVALID_ARG, "GroupNorm needs groups >= 1 dividing C_out (%d %% %d)", p->C_out, p->groups);
    if (p->norm != C1N_NORM_NONE && !(std::isfinite(p->eps) && p->eps > 0.f))
        return fail(C1N_ERR_INVALID_ARG, "eps must be finite and > 0");
    const long long T_out = t_out_of(*p);
    if (T_out < 1) return fail(C1N_ERR_INVALID_ARG, "empty output: T_out = %lld", T_out);
    const long long elems_y = (long long)p->N * p->C_out * T_out;
    const long long elems_x = (long long)p->N * p->C_in * p->T;
    if (elems_y > (1LL << 40) || elems_x > (1LL << 40)) return fail(C1N_ERR_INVALID_ARG, "tensor too large");
    if (T_out > (1LL << 31) - 1 || (long long)p->T + p->pad_left + p->pad_right > (1LL << 31) - 1)
        return fail(C1N_ERR_INVALID_ARG, "time axis too long");
    return C1N_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

c1n_status encode(CUtensorMap* m, const void* ptr, bool bf16, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides_bytes, const cuuint32_t* box,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = encode_fn();
    if (!fn) return fail(C1N_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank,
                    const_cast<void*>(ptr), dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(C1N_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return C1N_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

c1n_status ensure_device(c1n_desc* d) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != d->device) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (d->plan.path != C1N_PATH_SIMT && !(major == 10 && minor == 3))
            return fail(C1N_ERR_UNSUPPORTED, "tensor-core path is built for sm_103a; device is sm_%d%d", major, minor);
        d->device = dev;
        d->num_sms = sms;
        d->tm_x_ptr = d->tm_w_ptr = nullptr;
    }
    return C1N_OK;
}

// Records a timing event before the launch of kernel `name` (nullptr: after the last one).
// Under stream capture the record becomes an event-record node of the graph (external), so a
// replay of the graph times its kernels too.
void mark(c1n_desc* d, cudaStream_t s, const char* name) {
    if (!d->profiling || !d->events_ready || d->n_marks >= c1n_desc::kMaxMarks) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        e = cudaEventRecordWithFlags(d->ev[d->n_marks], s, cudaEventRecordExternal);
    else if (e == cudaSuccess)
        e = cudaEventRecord(d->ev[d->n_marks], s);
    if (e == cudaSuccess) d->ev_name[d->n_marks++] = name;
    else cudaGetLastError();  // timing is best effort: leave no error behind for the launches
}

c1n_status run_body(c1n_desc* d, const c1n_args* a, cudaStream_t s);

c1n_status run_impl(c1n_desc* d, const c1n_args* a, cudaStream_t s) {
    d->n_marks = 0;
    if (d->profiling && !d->events_ready) {
        for (int i = 0; i < c1n_desc::kMaxMarks; ++i) {
            cudaError_t e = cudaEventCreate(&d->ev[i]);
            if (e != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(d->ev[j]);
                return cuda_fail(e, "cudaEventCreate (profiling)");
            }
        }
        d->events_ready = 1;
    }
    c1n_status st = run_body(d, a, s);
    if (st == C1N_OK) mark(d, s, nullptr);
    else d->n_marks = 0;
    return st;
}

c1n_status run_body(c1n_desc* d, const c1n_args* a, cudaStream_t s) {
    const c1n_params& p = d->p;
    const Plan& pl = d->plan;
    if (!a->x || !a->w || !a->y) return fail(C1N_ERR_INVALID_ARG, "x, w and y must be non-NULL");
    if (p.post == C1N_POST_ROWMIN_BIAS && !a->bias2) return fail(C1N_ERR_INVALID_ARG, "row-min post-op needs bias2");
    void* ws = a->workspace ? a->workspace : d->ws;
    size_t ws_bytes = a->workspace ? a->workspace_bytes : d->ws_bytes;
    if (!ws || ws_bytes < pl.ws_total)
        return fail(C1N_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", pl.ws_total, ws ? ws_bytes : 0);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(C1N_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    c1n_status st = ensure_device(d);
    if (st != C1N_OK) return st;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    int* status = reinterpret_cast<int*>(wsb);
    float2* stats = reinterpret_cast<float2*>(wsb + pl.ws_stats);
    float* rowmin = reinterpret_cast<float*>(wsb + pl.ws_rowmin);
    const bool need_stats = p.norm != C1N_NORM_NONE;
    const bool second = need_stats || p.post == C1N_POST_ROWMIN_BIAS;
    // Raw conv values (fp32) for the statistics / normalize passes: y itself when y is fp32.
    float* raw = pl.bf16 ? reinterpret_cast<float*>(wsb + pl.ws_raw) : static_cast<float*>(a->y);
    cudaError_t e;

    if (pl.path == C1N_PATH_SIMT) {
        mark(d, s, "simt_conv");
        e = launch_simt_conv(p, pl, a->x, a->w, a->b, second ? static_cast<void*>(raw) : a->y, second, s);
        if (e != cudaSuccess) return cuda_fail(e, "SIMT conv launch");
    } else {
        const bool linear = pl.path == C1N_PATH_TC_LINEAR;
        if (!aligned16(a->x) || (linear && !aligned16(a->w)))
            return fail(C1N_ERR_ALIGNMENT, "x (and w on the Linear path) must be 16-byte aligned for TMA");
        const void* wsrc = a->w;
        if (!linear) {
            void* wp = wsb + pl.ws_wp;
            if (!(a->flags & C1N_FLAG_WEIGHTS_PACKED)) {
                unsigned* zero = pl.gx_words ? reinterpret_cast<unsigned*>(wsb + pl.ws_gx) : nullptr;
                mark(d, s, "pack_weights");
                e = launch_pack_weights(p, pl, a->w, wp, s, zero, pl.gx_words, pack_releases_first(pl));
                if (e != cudaSuccess) return cuda_fail(e, "weight pack launch");
            }
            wsrc = wp;
        }
        if (d->tm_x_ptr != a->x || d->tm_w_ptr != wsrc) {
            const cuuint64_t es = (cuuint64_t)pl.esize;
            if (linear) {
                // A: X[rows][in], box = BK channels x 128 rows; B: W[out][in], box = BK x BN.
                cuuint64_t dx[2] = {(cuuint64_t)p.C_in, (cuuint64_t)p.N};
                cuuint64_t sx[1] = {(cuuint64_t)p.C_in * es};
                cuuint32_t bx[2] = {(cuuint32_t)pl.BK, 128u};
                st = encode(&d->tm_a, a->x, pl.bf16, 2, dx, sx, bx);
                if (st != C1N_OK) return st;
                cuuint64_t dw[2] = {(cuuint64_t)p.C_in, (cuuint64_t)p.C_out};
                cuuint64_t sw[1] = {(cuuint64_t)p.C_in * es};
                // (a CTA pair: each CTA loads BN/2 of the BN rows)
                cuuint32_t bw[2] = {(cuuint32_t)pl.BK, (cuuint32_t)(pl.pair ? pl.BN / 2 : pl.BN)};
                st = encode(&d->tm_b, wsrc, pl.bf16, 2, dw, sw, bw);
                if (st != C1N_OK) return st;
            } else {
                // B: packed weights wp[kk][co][ci_pad], box = BK channels x BN outputs x 1 tap.
                // (A is written by the kernel's transposer warps; its map slot repeats B's.)
                // (3xTF32: the TF32 tails follow as taps k..2k-1)
                cuuint64_t dw[3] = {(cuuint64_t)pl.ci_pad, (cuuint64_t)p.C_out, (cuuint64_t)p.k * (pl.x3 ? 2 : 1)};
                cuuint64_t sw[2] = {(cuuint64_t)pl.ci_pad * es, (cuuint64_t)pl.ci_pad * p.C_out * es};
                cuuint32_t bw[3] = {(cuuint32_t)pl.BK, (cuuint32_t)(pl.pair ? pl.BN / 2 : pl.BN), 1};
                st = encode(&d->tm_b, wsrc, pl.bf16, 3, dw, sw, bw);
                if (st != C1N_OK) return st;
                // A source: x[n][ci][t], box = RS time steps x BK channels x 1 sample, unswizzled
                // (the kernel transposes it in shared memory).
                cuuint64_t dx[3] = {(cuuint64_t)p.T, (cuuint64_t)p.C_in, (cuuint64_t)p.N};
                cuuint64_t sx[2] = {(cuuint64_t)p.T * es, (cuuint64_t)p.T * p.C_in * es};
                cuuint32_t bx[3] = {(cuuint32_t)pl.RS, (cuuint32_t)pl.BK, 1};
                st = encode(&d->tm_a, a->x, pl.bf16, 3, dx, sx, bx, CU_TENSOR_MAP_SWIZZLE_NONE);
                if (st != C1N_OK) return st;
            }
            d->tm_x_ptr = a->x;
            d->tm_w_ptr = wsrc;
        }
        const bool fused_gn = pl.path == C1N_PATH_TC_FUSED_GN || pl.path == C1N_PATH_TC_FUSED_GN_DSMEM;
        const bool fused_ln_path = pl.path == C1N_PATH_TC_FUSED_LN;
        // The fused LayerNorm stores 32 x 32 tiles staged per warp by TMA bulk stores when y's rows
        // are 16-byte multiples; their 32-channel boxes must not reach into the other CTA's channel
        // half (BN a multiple of 32 when the channels are split). (The fused GroupNorm epilogue
        // stores straight from registers.)
        const bool y_tma_ok = aligned16(a->y) && (pl.T_out * pl.esize) % 16 == 0;
        const bool box_ok = pl.n_cb == 1 || pl.BN % 32 == 0;  // 32-channel boxes stay in this CTA's block
        const bool tma_store = y_tma_ok && box_ok && fused_ln_path && pl.o_bytes > 0;
        if (tma_store && d->tm_y_ptr != a->y) {
            const cuuint64_t es = (cuuint64_t)pl.esize;
            cuuint64_t dy[3] = {(cuuint64_t)pl.T_out, (cuuint64_t)p.C_out, (cuuint64_t)p.N};
            cuuint64_t sy[2] = {(cuuint64_t)pl.T_out * es, (cuuint64_t)pl.T_out * p.C_out * es};
            cuuint32_t by[3] = {32u, 32u, 1};  // one warp's 32 steps x 32 channels
            st = encode(&d->tm_y, a->y, pl.bf16, 3, dy, sy, by, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != C1N_OK) return st;
            d->tm_y_ptr = a->y;
        }
        TcArgs t;
        std::memset(&t, 0, sizeof(t));
        t.N = p.N; t.C_in = p.C_in; t.C_out = p.C_out; t.T = p.T; t.T_out = (int)pl.T_out; t.k = p.k;
        t.dil = p.dilation; t.pad_left = p.pad_left;
        t.BK = pl.BK; t.R = pl.R; t.BN = pl.BN; t.n_cb = pl.n_cb; t.cb_per_unit = pl.cb_per_unit;
        t.n_ci_chunks = pl.n_ci_chunks; t.n_t_tiles = pl.n_t_tiles; t.n_units = pl.n_units;
        t.n_acc = pl.n_acc; t.tmem_cols = pl.tmem_cols; t.stages_a = pl.stages_a; t.stages_b = pl.stages_b;
        t.a_slot_bytes = pl.a_slot_bytes; t.b_slot_bytes = pl.b_slot_bytes;
        t.RS = pl.RS; t.t_shift = pl.t_shift; t.stages_s = pl.stages_s; t.s_slot_bytes = pl.s_slot_bytes;
        t.groups = p.norm == C1N_NORM_GROUP ? p.groups : 1;
        t.cpg = p.C_out / t.groups;
        t.sub = (t.cpg == 4 || t.cpg == 8) ? t.cpg : (t.cpg % 16 == 0 ? 16 : 0);
        t.tma_store = tma_store ? 1 : 0;
        t.x3 = pl.x3;
        t.o_bytes = pl.o_bytes;
        t.o_off = pl.stages_a * pl.a_slot_bytes + pl.stages_b * pl.b_slot_bytes + pl.stages_s * pl.s_slot_bytes;
        t.gx = reinterpret_cast<unsigned long long*>(wsb + pl.ws_gx);
        t.gstride = pl.gstride;
        // x may be read before the kernel waits on its predecessor only when that predecessor is
        // the weight pack launched just above and it releases this kernel only after its own wait
        // for all earlier work
        t.early_inputs = (!linear && !(a->flags & C1N_FLAG_WEIGHTS_PACKED) && !pack_releases_first(pl)) ? 1 : 0;
        t.row_cpg = (pl.row_epilogue && p.norm == C1N_NORM_GROUP) ? p.C_out / p.groups : 0;
        t.rowmin = (pl.row_epilogue && p.post == C1N_POST_ROWMIN_BIAS) ? 1 : 0;
        t.rowpart = reinterpret_cast<float2*>(wsb + pl.ws_rowpart);
        t.part_kind = pl.part_kind;
        t.part_tiles = pl.part_tiles;
        t.part = reinterpret_cast<float2*>(wsb + pl.ws_part);
        t.eps = p.eps;
        const bool fused_ln = pl.path == C1N_PATH_TC_FUSED_LN;
        // GELU in the kernel whenever no later pass sees the values (the normalize pass applies it
        // otherwise).
        const bool last_pass = pl.path == C1N_PATH_TC_DIRECT || fused_gn || fused_ln || pl.row_epilogue || !second;
        t.gelu = (p.post == C1N_POST_GELU_ERF && last_pass) ? 1 : 0;
        const uint32_t fmt = pl.bf16 ? 1u : 2u;
        t.idesc = make_idesc(fmt, fmt, 0u, 0u, pl.pair ? 256u : 128u, (uint32_t)pl.BN);
        t.x = a->x;
        t.bias = a->b;
        t.gamma = a->gamma;
        t.beta = a->beta;
        const bool fused_out = pl.path == C1N_PATH_TC_DIRECT || fused_gn || fused_ln || pl.row_epilogue;
        t.y = fused_out ? a->y : (second ? static_cast<void*>(raw) : a->y);
        t.status = status;
        const bool out_bf16 = pl.bf16 && (fused_out || !second);
        int epi = kEpiDirect;
        if (fused_ln) epi = pl.cluster == 2 ? kEpiLNX : kEpiLN;
        if (pl.row_epilogue) epi = kEpiRowGN;
        if (pl.part_kind) epi = kEpiDirectStats;
        if (fused_gn) {
            // Cooperative grid when every CTA fits on the device at once (one per SM), else a cluster.
            const bool grid_fits = pl.path == C1N_PATH_TC_FUSED_GN && pl.n_units <= d->num_sms;
            if (grid_fits) epi = kEpiGridGN;
            else if (pl.n_t_tiles <= 8) epi = kEpiClusterGN;
            else return fail(C1N_ERR_UNSUPPORTED, "fused GroupNorm grid of %d CTAs exceeds the %d SMs of this device",
                             pl.n_units, d->num_sms);
        }
        if (a->flags & C1N_FLAG_TEST_STALL_EXCHANGE) {
            if (epi != kEpiGridGN)
                return fail(C1N_ERR_INVALID_ARG, "C1N_FLAG_TEST_STALL_EXCHANGE needs the fused GroupNorm plan that "
                                                 "exchanges statistics through global memory");
            t.test_stall = 1;
        }
        mark(d, s, "tc_conv");
        e = launch_tc(pl, t, d->tm_a, d->tm_b, tma_store ? d->tm_y : d->tm_b, linear, epi, out_bf16, d->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
        if (pl.row_epilogue && p.post == C1N_POST_ROWMIN_BIAS) {
            mark(d, s, "rowmin_finish");
            e = launch_rowmin_finish(p, pl, t.rowpart, a->bias2, a->y, a->argmin, s);
            if (e != cudaSuccess) return cuda_fail(e, "row-min finisher launch");
        }
        if (fused_out) return C1N_OK;
    }
    if (!second) return C1N_OK;
    if (need_stats && pl.part_kind) {
        const float2* part = reinterpret_cast<const float2*>(wsb + pl.ws_part);
        mark(d, s, pl.part_kind == 1 ? "gn_merge" : "ln_merge");
        e = pl.part_kind == 1 ? launch_gn_merge(p, pl, part, stats, s) : launch_ln_merge(p, pl, part, stats, s);
        if (e != cudaSuccess) return cuda_fail(e, "statistics merge launch");
    } else if (need_stats) {
        mark(d, s, p.norm == C1N_NORM_GROUP ? "gn_stats" : "ln_stats");
        e = p.norm == C1N_NORM_GROUP ? launch_gn_stats(p, pl, raw, stats, s) : launch_ln_stats(p, pl, raw, stats, s);
        if (e != cudaSuccess) return cuda_fail(e, "statistics launch");
    }
    if (p.post == C1N_POST_ROWMIN_BIAS) {
        mark(d, s, "rowmin");
        e = launch_rowmin(p, pl, raw, stats, need_stats ? a->gamma : nullptr, need_stats ? a->beta : nullptr, rowmin,
                          a->argmin, s);
        if (e != cudaSuccess) return cuda_fail(e, "row-min launch");
        mark(d, s, "broadcast");
        e = launch_broadcast(p, pl, rowmin, a->bias2, a->y, s);
        if (e != cudaSuccess) return cuda_fail(e, "broadcast launch");
    } else {
        mark(d, s, "normalize");
        e = launch_normalize(p, pl, raw, stats, a->gamma, a->beta, a->y, s);
        if (e != cudaSuccess) return cuda_fail(e, "normalize launch");
    }
    return C1N_OK;
}

}  // namespace

namespace c1n {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace c1n

namespace {
// Validates p; *tc tells whether the tensor-core plan runs (math 0 picks it when it takes the shape).
c1n_status convt3d_plan(const c1n_convt3d_params* p, bool* tc) {
    if (!p) return fail(C1N_ERR_INVALID_ARG, "params must be non-NULL");
    if (p->N < 1 || p->C_in < 1 || p->C_out < 1 || p->D < 1 || p->H < 1 || p->W < 1)
        return fail(C1N_ERR_INVALID_ARG, "N, C_in, C_out, D, H, W must be >= 1");
    if (p->math < 0 || p->math > 2) return fail(C1N_ERR_INVALID_ARG, "math must be 0, 1 or 2");
    if (p->k != 3 || p->stride != 2 || p->pad != 1 || (p->out_pad != 0 && p->out_pad != 1))
        return fail(C1N_ERR_UNSUPPORTED, "ConvTranspose3d takes k = 3, stride 2, pad 1, output pad 0 or 1 "
                                         "(got k %d, stride %d, pad %d, output pad %d)", p->k, p->stride, p->pad, p->out_pad);
    if (p->C_out % 32 != 0) return fail(C1N_ERR_UNSUPPORTED, "C_out = %d: a multiple of 32 is taken", p->C_out);
    if ((long long)p->D * 4 * (p->C_out / 32) > 65535 || p->N > 65535)
        return fail(C1N_ERR_UNSUPPORTED, "grid too large (D * 4 * C_out / 32 and N must stay <= 65535)");
    const int Wo = 2 * p->W - 1 + p->out_pad;
    const bool tc_ok = p->C_in == 32 && p->C_out == 64 && Wo % 4 == 0;
    if (p->math == 2 && !tc_ok)
        return fail(C1N_ERR_UNSUPPORTED, "the tensor-core plan takes C_in = 32, C_out = 64 and Wo a multiple of 4");
    *tc = p->math == 2 || (p->math == 0 && tc_ok);
    return C1N_OK;
}
// The fused model kernel takes the page's shape only.
c1n_status convt3d_fused_check(const c1n_convt3d_params* p) {
    if (!p) return fail(C1N_ERR_INVALID_ARG, "params must be non-NULL");
    if (p->N < 1 || p->C_in < 1 || p->C_out < 1 || p->D < 1 || p->H < 1 || p->W < 1)
        return fail(C1N_ERR_INVALID_ARG, "N, C_in, C_out, D, H, W must be >= 1");
    if (p->C_in != 32 || p->C_out != 64 || p->W != 32 || p->k != 3 || p->stride != 2 || p->pad != 1 || p->out_pad != 1)
        return fail(C1N_ERR_UNSUPPORTED, "the fused model takes C_in 32, C_out 64, W 32, k 3, stride 2, pad 1, "
                                         "output pad 1 (got C_in %d, C_out %d, W %d, k %d, stride %d, pad %d, output pad %d)",
                    p->C_in, p->C_out, p->W, p->k, p->stride, p->pad, p->out_pad);
    if ((long long)p->N * p->D * ((p->H + 3) / 4) > 0x7fffffffLL) return fail(C1N_ERR_UNSUPPORTED, "too many tiles");
    return C1N_OK;
}
}  // namespace

extern "C" {

c1n_status conv1d_norm_desc_create(const c1n_params* params, c1n_desc** out) {
    g_last_error.clear();
    if (!out) return fail(C1N_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    c1n_status st = validate(params);
    if (st != C1N_OK) return st;
    Plan pl;
    st = make_plan(*params, pl);
    if (st != C1N_OK) return st;
    if (params->mainloop == C1N_MAINLOOP_PAIR && !pl.pair)
        return fail(C1N_ERR_UNSUPPORTED, "the chosen plan (path %d, MMA N %d) cannot run on CTA pairs", pl.path, pl.BN);
    c1n_desc* d = new (std::nothrow) c1n_desc();
    if (!d) return fail(C1N_ERR_INVALID_ARG, "out of host memory");
    d->p = *params;
    d->plan = pl;
    *out = d;
    return C1N_OK;
}

c1n_status conv1d_norm_workspace_size(const c1n_desc* desc, size_t* bytes) {
    if (!desc || !bytes) return fail(C1N_ERR_INVALID_ARG, "NULL argument");
    *bytes = desc->plan.ws_total;
    return C1N_OK;
}

c1n_status conv1d_norm_set_workspace(c1n_desc* desc, void* workspace, size_t bytes) {
    if (!desc) return fail(C1N_ERR_INVALID_ARG, "desc is NULL");
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(C1N_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    if (workspace && bytes < desc->plan.ws_total)
        return fail(C1N_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", desc->plan.ws_total, bytes);
    desc->ws = workspace;
    desc->ws_bytes = workspace ? bytes : 0;
    return C1N_OK;
}

c1n_status conv1d_norm_plan_info(const c1n_desc* desc, c1n_plan_info* info) {
    if (!desc || !info) return fail(C1N_ERR_INVALID_ARG, "NULL argument");
    const Plan& pl = desc->plan;
    std::memset(info, 0, sizeof(*info));
    info->path = pl.path;
    info->T_out = (int32_t)pl.T_out;
    info->tile_t = pl.path == C1N_PATH_SIMT ? 64 : (pl.pair ? 256 : 128);
    info->tile_co = pl.path == C1N_PATH_SIMT ? 64 : pl.BN;
    info->mma_n = pl.path == C1N_PATH_SIMT ? 0 : pl.BN;
    info->cluster = pl.cluster;
    info->n_tiles = pl.path == C1N_PATH_SIMT ? pl.n_units : pl.n_units;
    info->grid = pl.grid;
    info->kernels = pl.kernels;
    info->cta_pair = pl.pair;
    info->workspace_bytes = (int64_t)pl.ws_total;
    return C1N_OK;
}

c1n_status conv1d_norm_run(c1n_desc* desc, const void* x, const void* w, const float* b, const float* gamma,
                           const float* beta, void* y, c1n_stream_t stream) {
    g_last_error.clear();
    if (!desc) return fail(C1N_ERR_INVALID_ARG, "desc is NULL");
    if (desc->p.post == C1N_POST_ROWMIN_BIAS)
        return fail(C1N_ERR_INVALID_ARG, "row-min post-op needs conv1d_norm_run_ex (bias2)");
    c1n_args a;
    std::memset(&a, 0, sizeof(a));
    a.x = x; a.w = w; a.b = b; a.gamma = gamma; a.beta = beta; a.y = y;
    return run_impl(desc, &a, reinterpret_cast<cudaStream_t>(stream));
}

c1n_status conv1d_norm_run_ex(c1n_desc* desc, const c1n_args* args, c1n_stream_t stream) {
    g_last_error.clear();
    if (!desc || !args) return fail(C1N_ERR_INVALID_ARG, "NULL argument");
    return run_impl(desc, args, reinterpret_cast<cudaStream_t>(stream));
}

c1n_status conv1d_norm_pack_weights(c1n_desc* desc, const void* w, void* workspace, size_t workspace_bytes,
                                    c1n_stream_t stream) {
    g_last_error.clear();
    if (!desc || !w) return fail(C1N_ERR_INVALID_ARG, "desc and w must be non-NULL");
    const Plan& pl = desc->plan;
    if (pl.path == C1N_PATH_SIMT || pl.path == C1N_PATH_TC_LINEAR) return C1N_OK;
    void* ws = workspace ? workspace : desc->ws;
    size_t ws_bytes = workspace ? workspace_bytes : desc->ws_bytes;
    if (!ws || ws_bytes < pl.ws_total)
        return fail(C1N_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", pl.ws_total, ws ? ws_bytes : 0);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(C1N_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    unsigned* zero = pl.gx_words ? reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + pl.ws_gx) : nullptr;
    cudaError_t e = launch_pack_weights(desc->p, pl, w, static_cast<uint8_t*>(ws) + pl.ws_wp,
                                        reinterpret_cast<cudaStream_t>(stream), zero, pl.gx_words);
    if (e != cudaSuccess) return cuda_fail(e, "weight pack launch");
    return C1N_OK;
}

c1n_status conv1d_norm_check(const c1n_desc* desc, void* workspace, c1n_stream_t stream) {
    g_last_error.clear();
    if (!desc) return fail(C1N_ERR_INVALID_ARG, "desc is NULL");
    void* ws = workspace ? workspace : desc->ws;
    if (!ws) return fail(C1N_ERR_WORKSPACE, "no workspace");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int word[16] = {0};
    cudaError_t e = cudaMemcpyAsync(word, ws, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (word[0] != 0) {
        e = cudaMemsetAsync(ws, 0, sizeof(word), s);
        // A run that gave up may have left the fused GroupNorm exchange words with mixed epochs:
        // zero them (the state the weight pack leaves) so the next run agrees on its epoch.
        const Plan& pl = desc->plan;
        if (e == cudaSuccess && pl.gx_words > 0)
            e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + pl.ws_gx, 0, (size_t)pl.gx_words * 4, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "status reset");
        if (word[0] == C1N_ERR_TIMEOUT)
            return fail(C1N_ERR_TIMEOUT,
                        "device wait timed out (site %d, CTA %d; progress b_loads=%d a_consumed=%d mma_units=%d "
                        "a_written=%d epi_units=%d a_loads=%d; waiting: mma=%d epi=%d xp=%d tma=%d; mma_unit=%d "
                        "rings=0x%08x)",
                        word[1], word[2], word[3], word[4], word[5], word[6], word[7], word[8], word[9], word[10],
                        word[11], word[12], word[13], (unsigned)word[14]);
        return fail(C1N_ERR_DEVICE, "device status %d (detail %d)", word[0], word[1]);
    }
    return C1N_OK;
}

c1n_status conv1d_norm_set_profiling(c1n_desc* desc, int32_t enable) {
    if (!desc) return fail(C1N_ERR_INVALID_ARG, "desc is NULL");
    desc->profiling = enable ? 1 : 0;
    desc->n_marks = 0;
    return C1N_OK;
}

c1n_status conv1d_norm_kernel_times(c1n_desc* desc, c1n_kernel_time* out, int32_t capacity, int32_t* count) {
    if (!desc || !count || (capacity > 0 && !out)) return fail(C1N_ERR_INVALID_ARG, "NULL argument");
    *count = 0;
    const int n = desc->n_marks;
    if (n < 2) return C1N_OK;
    cudaError_t e = cudaEventSynchronize(desc->ev[n - 1]);
    if (e != cudaSuccess) {
        cudaGetLastError();  // not sticky: keep it from surfacing at the next launch
        return cuda_fail(e, "cudaEventSynchronize (profiling)");
    }
    int k = 0;
    for (int i = 0; i + 1 < n && k < capacity; ++i, ++k) {
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, desc->ev[i], desc->ev[i + 1]);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return cuda_fail(e, "cudaEventElapsedTime (profiling)");
        }
        std::memset(out[k].name, 0, sizeof(out[k].name));
        std::snprintf(out[k].name, sizeof(out[k].name), "%s", desc->ev_name[i]);
        out[k].ms = ms;
    }
    *count = n - 1;
    return C1N_OK;
}

void conv1d_norm_destroy(c1n_desc* desc) {
    if (desc && desc->events_ready)
        for (int i = 0; i < c1n_desc::kMaxMarks; ++i) cudaEventDestroy(desc->ev[i]);
    delete desc;
}

const char* conv1d_norm_status_string(c1n_status s) {
    switch (s) {
        case C1N_OK: return "ok";
        case C1N_ERR_INVALID_ARG: return "invalid argument";
        case C1N_ERR_UNSUPPORTED: return "unsupported on the requested path";
        case C1N_ERR_ALIGNMENT: return "misaligned pointer";
        case C1N_ERR_WORKSPACE: return "workspace missing or too small";
        case C1N_ERR_CUDA: return "CUDA runtime error";
        case C1N_ERR_TIMEOUT: return "device-side wait timed out";
        case C1N_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

const char* conv1d_norm_last_error(void) { return g_last_error.c_str(); }

c1n_status ln_avgpool3d_gelu_run(const c1n_lnpool_params* p, const float* z, float sum_weight, const float* gamma,
                                 const float* beta, float* out, c1n_stream_t stream) {
    g_last_error.clear();
    if (!p || !z || !out) return fail(C1N_ERR_INVALID_ARG, "params, z and out must be non-NULL");
    if (p->N < 1 || p->C < 1 || p->D < 1 || p->H < 1 || p->W < 1)
        return fail(C1N_ERR_INVALID_ARG, "N, C, D, H, W must be >= 1 (got %d, %d, %d, %d, %d)", p->N, p->C, p->D,
                    p->H, p->W);
    if (!(p->eps > 0.0f)) return fail(C1N_ERR_INVALID_ARG, "eps must be > 0");
    if (p->W != 64 && p->W != 128 && p->W != 256 && p->W != 512)
        return fail(C1N_ERR_UNSUPPORTED, "W = %d: the pass takes W = 64, 128, 256 or 512", p->W);
    if (!aligned16(z) || !aligned16(out)) return fail(C1N_ERR_ALIGNMENT, "z and out must be 16-byte aligned");
    if (p->D < 2 || p->H < 2) return C1N_OK;  // no pooling window: empty output
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    e = launch_ln_avgpool3d_gelu(*p, z, sum_weight, gamma, beta, out, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "LayerNorm + AvgPool3d + GELU launch");
    return C1N_OK;
}


c1n_status conv_transpose3d_workspace_size(const c1n_convt3d_params* p, size_t* bytes) {
    g_last_error.clear();
    if (!bytes) return fail(C1N_ERR_INVALID_ARG, "bytes must be non-NULL");
    bool tc = false;
    c1n_status st = convt3d_plan(p, &tc);
    if (st != C1N_OK) return st;
    *bytes = tc ? convt3d_tc_workspace_bytes(*p) : 0;
    return C1N_OK;
}

c1n_status conv_transpose3d_run(const c1n_convt3d_params* p, const float* x, const float* w, const float* b, float* y,
                                void* workspace, size_t workspace_bytes, c1n_stream_t stream) {
    g_last_error.clear();
    bool tc = false;
    c1n_status st = convt3d_plan(p, &tc);
    if (st != C1N_OK) return st;
    if (!x || !w || !y) return fail(C1N_ERR_INVALID_ARG, "x, w and y must be non-NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tc) {
        const size_t need = convt3d_tc_workspace_bytes(*p);
        if (!workspace || workspace_bytes < need)
            return fail(C1N_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? workspace_bytes : 0);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(C1N_ERR_ALIGNMENT, "workspace not 256-byte aligned");
        if (!aligned16(x) || !aligned16(y)) return fail(C1N_ERR_ALIGNMENT, "x and y must be 16-byte aligned");
        int dev = 0, sms = 0, major = 0, minor = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "device query");
        if (!(major == 10 && minor == 3))
            return fail(C1N_ERR_UNSUPPORTED, "the tensor-core plan is built for sm_103a; device is sm_%d%d", major, minor);
        e = launch_conv_transpose3d_tc(*p, x, w, b, y, workspace, sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "ConvTranspose3d (tensor cores) launch");
        return C1N_OK;
    }
    e = launch_conv_transpose3d(*p, x, w, b, y, s);
    if (e != cudaSuccess) return cuda_fail(e, "ConvTranspose3d launch");
    return C1N_OK;
}

c1n_status conv_transpose3d_ln_avgpool3d_gelu_workspace_size(const c1n_convt3d_params* p, size_t* bytes) {
    g_last_error.clear();
    if (!bytes) return fail(C1N_ERR_INVALID_ARG, "bytes is NULL");
    c1n_status st = convt3d_fused_check(p);
    if (st != C1N_OK) return st;
    *bytes = convt3d_lnpool_fused_workspace_bytes(*p);
    return C1N_OK;
}

c1n_status conv_transpose3d_ln_avgpool3d_gelu_run(const c1n_convt3d_params* p, float eps, float sum_weight,
                                                  const float* x, const float* w, const float* b,
                                                  const float* gamma, const float* beta, float* out,
                                                  void* workspace, size_t workspace_bytes, c1n_stream_t stream) {
    g_last_error.clear();
    c1n_status st = convt3d_fused_check(p);
    if (st != C1N_OK) return st;
    if (!(eps > 0.f)) return fail(C1N_ERR_INVALID_ARG, "eps must be > 0");
    if (!x || !w || !out) return fail(C1N_ERR_INVALID_ARG, "x, w and out must be non-NULL");
    const size_t need = convt3d_lnpool_fused_workspace_bytes(*p);
    if (!workspace || workspace_bytes < need)
        return fail(C1N_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? workspace_bytes : 0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(C1N_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    if (!aligned16(x) || !aligned16(out)) return fail(C1N_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
    int dev = 0, sms = 0, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    if (!(major == 10 && minor == 3))
        return fail(C1N_ERR_UNSUPPORTED, "the fused model kernel is built for sm_103a; device is sm_%d%d", major, minor);
    e = launch_convt3d_lnpool_fused(*p, eps, sum_weight, x, w, b, gamma, beta, out, workspace, sms,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fused ConvTranspose3d + LayerNorm / AvgPool3d / GELU launch");
    return C1N_OK;
}

int32_t conv1d_norm_version(void) { return 114; }

}  // extern "C"

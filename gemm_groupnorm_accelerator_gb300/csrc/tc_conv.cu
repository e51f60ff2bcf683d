// Tensor-core implicit-GEMM Conv1d (+ fused epilogues) for sm_103a.
//
// The convolution of the Kimi-K2.6 l1_p5 page (GEMM view: M = N*T_out, N = C_out, K = C_in*k) is
// computed tile by tile: one tile = 128 output time steps (MMA M, TMEM lanes) x BN <= 256 output
// channels (MMA N, TMEM columns) of one sample n, accumulated in fp32 TMEM.
//
//   D[t][co] = sum_kk sum_ci  x[n][ci][t + kk*dilation - pad_left] * wp[kk][co][ci]
//
//   * A operand (x, K-major): x[n][ci][t] arrives by TMA in time-contiguous boxes (a staging ring
//     several chunks deep), and eight "transposer" warps rewrite each box in shared memory as rows
//     of time steps, 128 bytes of input channels per row, in the 128-byte swizzled layout the
//     tensor core reads.
//     One tile holds 128 + (k-1)*dilation rows (the halo); tap kk uses the same tile with the
//     matrix-descriptor start moved down by kk*dilation rows, so the taps cost no extra copies.
//     Padding (causal or symmetric) and the ragged ends are zeros written by the transposer.
//   * B operand (weights, K-major): TMA boxes of the packed weights wp[kk][co][ci], one per
//     (input-channel chunk, channel block, tap).
//   * Accumulators sit at 256-column boundaries of TMEM; two of them on the persistent paths so
//     that the epilogue of one tile overlaps the mainloop of the next.
//
// Warp roles (480 threads): warp 0 issues the weight TMA loads, warp 1 owns TMEM and issues
// tcgen05.mma from one thread, warps 2-5 run the epilogue (each owns the 32 TMEM lanes of its
// quarter), warp 14 TMA-loads x boxes into a staging ring and warps 6-13 transpose them into the A
// ring (conv mode only).
//
// Linear mode (T = 1, k = 1; Kimi-K2.6 l2_p75 page): x is X[rows][in] and already K-major, so TMA
// loads the A operand as well; D[row][co].
//
// Epilogues: direct (bias, optional exact GELU, store), fused GroupNorm (Kimi-K2.6 l2_p35 page) and
// fused channel LayerNorm. Fused GroupNorm: the CTAs of one sample (a cooperative grid, or a
// thread-block cluster) together cover all its T_out steps, one tile each; the accumulator starts
// as the bias, so TMEM holds y; each CTA reduces per-group partial statistics over its tile (column
// sums across the 128 lanes by butterfly reduce-scatters), the partials are exchanged through
// global memory (epoch-tagged words) or distributed shared memory and merged with Chan's pairwise
// formula, and every CTA normalizes its tile straight from TMEM and stores it once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>

#include "c1n_internal.h"
#include "c1n_math.cuh"
#include "sm100_ptx.cuh"

namespace c1n {
namespace {

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpEpi0 = 2, kWarpXld = 14;
constexpr int kThreads = 32 * (kWarpXld + 1);  // 15 warps
// x transposer warps: fp32 data, warps 6-13 (16-byte column chunk per warp); bf16 data, warps 10-13
// (8x8 block transposes with ldmatrix / stmatrix); warps 6-9 then have no role.
template <bool BF16> __host__ __device__ constexpr int xp_first() { return BF16 ? 10 : 6; }
template <bool BF16> __host__ __device__ constexpr int xp_warps() { return BF16 ? 4 : 8; }

// Where a bounded wait gave up (status word detail).
enum WaitSite {
    kWaitAEmpty = 1, kWaitBEmpty, kWaitAFull, kWaitBFull, kWaitAccEmpty, kWaitAccFull, kWaitDrain, kWaitSEmpty,
    kWaitSFull, kWaitGridPeers, kWaitExchange, kWaitAccInit
};


__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Time-bounded wait that ignores the abort flag (used to drain copies and MMAs before exit).
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            if (status != nullptr && atomicCAS(status, 0, 6) == 0) atomicExch(status + 1, kWaitDrain);
            return;
        }
    }
}

// N consecutive floats from 16-byte aligned shared memory as N/4 vector loads (the epilogues read
// per-channel parameters for a whole chunk of columns at once, not one broadcast load per element).
template <int N>
__device__ __forceinline__ void lds_vec(const float* p, float (&out)[N]) {
    static_assert(N % 4 == 0, "whole float4s");
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const float4 t = reinterpret_cast<const float4*>(p)[k];
        out[4 * k] = t.x;
        out[4 * k + 1] = t.y;
        out[4 * k + 2] = t.z;
        out[4 * k + 3] = t.w;
    }
}

__device__ __forceinline__ void chan_merge(float& n_a, float& mu_a, float& m2_a, float n_b, float mu_b, float m2_b) {
    if (n_b <= 0.f) return;
    const float n = n_a + n_b;
    const float d = mu_b - mu_a;
    const float f = n_b / n;
    mu_a += d * f;
    m2_a += m2_b + d * d * n_a * f;
    n_a = n;
}

// Reduce-scatter over the warp of N <= 32 per-lane slots (N a power of two): lane l ends with the
// total over all 32 lanes of slot (l mod N) in v[0]. Lane distances 16 .. N add whole slot sets
// (both lanes keep the sum); the distances below N halve the slots each lane keeps.
template <int N>
__device__ __forceinline__ void warp_sum_scatter(float* v, int lane) {
#pragma unroll
    for (int d = 16; d >= N && d >= 1; d >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], d);
    }
#pragma unroll
    for (int d = N / 2; d >= 1; d >>= 1) {
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < d; ++i) {
            const float send = upper ? v[i] : v[i + d];
            const float keep = upper ? v[i + d] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
    }
}

// Moments of this warp's rows over columns [c_lo, c_hi) of its TMEM lane quarter (c_lo a multiple
// of 32), for every run of SUB consecutive channels (SUB = 4, 8, 16 divides the group size; SUB = 1
// is one run per channel), window by window (up to 32 runs): first the sum of acc over the run
// (red_s[q*256 + run]), then, with the run's mean m known to every lane, the sum over the run of
// (acc + bc[col] - m)^2 (red_m[q*256 + run]), where bc is the bias minus its mean over the run, so
// that this is the run's sum of squared deviations of y = acc + bias from its mean. Rows past T_out
// (row_ok false) count zero; n_rows is the number of valid rows of the warp.
template <int SUB>
__device__ __forceinline__ void gn_run_moments(uint32_t tb, int c_lo, int c_hi, bool row_ok, int n_rows,
                                               const float* bc, float* red_s, float* red_m, int q, int lane) {
    const float inv_n = n_rows > 0 ? 1.f / float(n_rows * SUB) : 0.f;
    if constexpr (SUB == 1) {
        for (int j0 = c_lo; j0 < c_hi; j0 += 32) {
            float v[32];
            tmem_load32(tb + uint32_t(j0), v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = row_ok ? v[i] : 0.f;
            warp_sum_scatter<32>(v, lane);
            if (j0 + lane < c_hi) red_s[q * 256 + j0 + lane] = v[0];
            const float m_lane = v[0] * inv_n;  // mean of column j0 + lane
            tmem_load32(tb + uint32_t(j0), v);
#pragma unroll
            for (int h = 0; h < 32; h += 8) {
                float b8[8];
                lds_vec(bc + j0 + h, b8);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float d = v[h + i] + b8[i] - __shfl_sync(0xffffffffu, m_lane, h + i);
                    v[h + i] = row_ok ? d * d : 0.f;
                }
            }
            warp_sum_scatter<32>(v, lane);
            if (j0 + lane < c_hi) red_m[q * 256 + j0 + lane] = v[0];
        }
    } else {
        constexpr int kRunsPerChunk = 32 / SUB;            // runs per 32-column TMEM load
        constexpr int kWin = 32 * SUB < 128 ? 32 * SUB : 128;
        constexpr int kRuns = kWin / SUB;                  // runs per window (one scatter)
        for (int w0 = c_lo; w0 < c_hi; w0 += kWin) {      // uniform over the warp
            float acc[kRuns];
#pragma unroll
            for (int i = 0; i < kRuns; ++i) acc[i] = 0.f;
#pragma unroll
            for (int c = 0; c < kWin / 32; ++c) {
                const int j0 = w0 + c * 32;
                if (j0 >= c_hi) break;  // uniform
                float v[32];
                tmem_load32(tb + uint32_t(j0), v);
#pragma unroll
                for (int r = 0; r < kRunsPerChunk; ++r) {
                    uint64_t p[SUB / 2];
#pragma unroll
                    for (int i = 0; i < SUB / 2; ++i) p[i] = f2_pack(v[r * SUB + 2 * i], v[r * SUB + 2 * i + 1]);
#pragma unroll
                    for (int w = SUB / 2; w > 1; w >>= 1) {
#pragma unroll
                        for (int i = 0; i < w / 2; ++i) p[i] = f2_add(p[i], p[i + w / 2]);
                    }
                    acc[c * kRunsPerChunk + r] = row_ok ? f2_hsum(p[0]) : 0.f;
                }
            }
            warp_sum_scatter<kRuns>(acc, lane);
            const bool mine = lane < kRuns && w0 + lane * SUB < c_hi;  // lane's run lies in this range
            if (mine) red_s[q * 256 + w0 / SUB + lane] = acc[0];
            const float m_lane = acc[0] * inv_n;  // mean of acc over run (lane mod kRuns)
#pragma unroll
            for (int i = 0; i < kRuns; ++i) acc[i] = 0.f;
#pragma unroll
            for (int c = 0; c < kWin / 32; ++c) {
                const int j0 = w0 + c * 32;
                if (j0 >= c_hi) break;  // uniform
                float v[32];
                tmem_load32(tb + uint32_t(j0), v);
#pragma unroll
                for (int r = 0; r < kRunsPerChunk; ++r) {
                    const int slot = c * kRunsPerChunk + r;
                    const float m = __shfl_sync(0xffffffffu, m_lane, slot);
                    const uint64_t mm = f2_pack(m, m);
                    float b[SUB];
                    lds_vec(bc + j0 + r * SUB, b);
                    uint64_t sq = 0ull;
#pragma unroll
                    for (int i = 0; i < SUB; i += 2) {
                        const uint64_t d = f2_sub(f2_add(f2_pack(v[r * SUB + i], v[r * SUB + i + 1]), f2_pack(b[i], b[i + 1])), mm);
                        sq = f2_fma(d, d, sq);
                    }
                    acc[slot] = row_ok ? f2_hsum(sq) : 0.f;
                }
            }
            warp_sum_scatter<kRuns>(acc, lane);
            if (mine) red_m[q * 256 + w0 / SUB + lane] = acc[0];
        }
    }
}

// Statistics of y over every run of SUB consecutive channels of this warp's columns [c_lo, c_hi)
// (c_lo a multiple of 32) and its valid rows (the accumulator holds y, bias included), from ONE sweep of TMEM (one wait per
// window of 32 or 64 columns): each run's values are summed as d = y - K with K a value of that run
// (row 0 of the warp, the run's first channel, the same for every lane), so the run's
// M2 = sum d^2 - (sum d)^2 / n does not cancel however far the data sit from zero. The sums go
// across the warp by reduce-scatters; lane l < runs-per-window then writes its run's mean and M2 to
// red_mean / red_m2[q * 256 + run]. Rows past T_out (row_ok false) count zero; n_rows is the number
// of valid rows of the warp (0: nothing is counted).
template <int SUB>
__device__ __forceinline__ void gn_run_stats(uint32_t tb, int c_lo, int c_hi, bool row_ok, int n_rows,
                                             float* red_mean, float* red_m2, int q, int lane) {
    constexpr int kWin = SUB == 1 ? 32 : (8 * SUB < 128 ? 8 * SUB : 128);
    constexpr int kRuns = kWin / SUB;         // runs per window: a power of two <= 32
    constexpr int kRunsPerChunk = 32 / SUB;   // runs per 32-column TMEM load
    const float inv_n = n_rows > 0 ? __fdividef(1.f, float(n_rows * SUB)) : 0.f;
#pragma unroll 1
    for (int w0 = c_lo; w0 < c_hi; w0 += kWin) {  // uniform over the warp
        float s1[kRuns], s2[kRuns];
        float k_mine = 0.f;  // K of run (lane mod kRuns) of this window
#pragma unroll
        for (int c = 0; c < kWin / 32; ++c) {
            const int j0 = w0 + c * 32;
            if (j0 >= c_hi) {  // uniform: runs past the range stay empty
#pragma unroll
                for (int r = 0; r < kRunsPerChunk; ++r) s1[c * kRunsPerChunk + r] = s2[c * kRunsPerChunk + r] = 0.f;
                continue;
            }
            float v[32];
            tmem_load32(tb + uint32_t(j0), v);
            // every run's shift K first (independent shuffles), then the runs' sums in two
            // interleaved chains each, so the runs overlap instead of waiting on one another
            if constexpr (SUB == 1) {
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const int slot = c * kRunsPerChunk + r;
                    const float K = __shfl_sync(0xffffffffu, v[r], 0);
                    if (lane == slot) k_mine = K;
                    const float d = row_ok ? v[r] - K : 0.f;
                    s1[slot] = d;
                    s2[slot] = d * d;
                }
            } else {
                float K[kRunsPerChunk];
#pragma unroll
                for (int r = 0; r < kRunsPerChunk; ++r) K[r] = __shfl_sync(0xffffffffu, v[r * SUB], 0);
#pragma unroll
                for (int r = 0; r < kRunsPerChunk; ++r) {
                    const int slot = c * kRunsPerChunk + r;
                    if ((lane & (kRuns - 1)) == slot) k_mine = K[r];
                    const uint64_t kk = f2_pack(K[r], K[r]);
                    uint64_t p1a = 0ull, p1b = 0ull, p2a = 0ull, p2b = 0ull;
#pragma unroll
                    for (int i = 0; i < SUB; i += 4) {
                        const uint64_t da = f2_sub(f2_pack(v[r * SUB + i], v[r * SUB + i + 1]), kk);
                        const uint64_t db = f2_sub(f2_pack(v[r * SUB + i + 2], v[r * SUB + i + 3]), kk);
                        p1a = f2_add(p1a, da);
                        p1b = f2_add(p1b, db);
                        p2a = f2_fma(da, da, p2a);
                        p2b = f2_fma(db, db, p2b);
                    }
                    s1[slot] = row_ok ? f2_hsum(f2_add(p1a, p1b)) : 0.f;
                    s2[slot] = row_ok ? f2_hsum(f2_add(p2a, p2b)) : 0.f;
                }
            }
        }
        float t1, t2;
        if constexpr (kRuns <= 16) {
            // one reduce-scatter over both sums: lane l ends with slot l mod 2kRuns, the sum of d for
            // lanes below kRuns, of d^2 for the next kRuns lanes
            float sv[2 * kRuns];
#pragma unroll
            for (int i = 0; i < kRuns; ++i) {
                sv[i] = s1[i];
                sv[kRuns + i] = s2[i];
            }
            warp_sum_scatter<2 * kRuns>(sv, lane);
            t1 = sv[0];
            t2 = __shfl_sync(0xffffffffu, sv[0], (lane + kRuns) & 31);
        } else {
            warp_sum_scatter<kRuns>(s1, lane);
            warp_sum_scatter<kRuns>(s2, lane);
            t1 = s1[0];
            t2 = s2[0];
        }
        if (lane < kRuns && w0 + lane * SUB < c_hi) {
            const float m = t1 * inv_n;
            red_mean[q * 256 + w0 / SUB + lane] = k_mine + m;
            red_m2[q * 256 + w0 / SUB + lane] = fmaxf(t2 - t1 * m, 0.f);
        }
    }
}

// Chan's pairwise merge of two (count, mean, M2) summaries, a first then b: the order is part of the
// result (floating point), so callers that must agree bit for bit merge in one fixed order.
__device__ __forceinline__ void stats_merge(float& n, float& mu, float& m2, float nb, float mub, float m2b) {
    const float nt = n + nb;
    if (nt <= 0.f) return;
    const float f = __fdividef(nb, nt);  // (counts are exact integers; 2-ulp quotient is plenty)
    const float d = mub - mu;
    mu = fmaf(d, f, mu);
    m2 = m2 + m2b + d * d * (n * f);
    n = nt;
}

// Merge with the summary held by lane (lane ^ d) of the warp, the lower lane's summary first, so
// both lanes of the pair end with the same bits.
__device__ __forceinline__ void stats_merge_xor(float& n, float& mu, float& m2, int d, int lane) {
    const float n_o = __shfl_xor_sync(0xffffffffu, n, d);
    const float mu_o = __shfl_xor_sync(0xffffffffu, mu, d);
    const float m2_o = __shfl_xor_sync(0xffffffffu, m2, d);
    const bool upper = (lane & d) != 0;  // the partner is the lower lane: its summary goes first
    float na = upper ? n_o : n, ma = upper ? mu_o : mu, Ma = upper ? m2_o : m2;
    stats_merge(na, ma, Ma, upper ? n : n_o, upper ? mu : mu_o, upper ? m2 : m2_o);
    n = na;
    mu = ma;
    m2 = Ma;
}

__device__ __forceinline__ void gn_run_stats_any(int sub, uint32_t tb, int c_lo, int c_hi, bool row_ok, int n_rows,
                                                 float* red_mean, float* red_m2, int q, int lane) {
    if (sub == 4) gn_run_stats<4>(tb, c_lo, c_hi, row_ok, n_rows, red_mean, red_m2, q, lane);
    else if (sub == 8) gn_run_stats<8>(tb, c_lo, c_hi, row_ok, n_rows, red_mean, red_m2, q, lane);
    else if (sub == 16) gn_run_stats<16>(tb, c_lo, c_hi, row_ok, n_rows, red_mean, red_m2, q, lane);
    else gn_run_stats<1>(tb, c_lo, c_hi, row_ok, n_rows, red_mean, red_m2, q, lane);
}

__device__ __forceinline__ void gn_run_moments_any(int sub, uint32_t tb, int c_lo, int c_hi, bool row_ok, int n_rows,
                                                   const float* bc, float* red_s, float* red_m, int q, int lane) {
    if (sub == 4) gn_run_moments<4>(tb, c_lo, c_hi, row_ok, n_rows, bc, red_s, red_m, q, lane);
    else if (sub == 8) gn_run_moments<8>(tb, c_lo, c_hi, row_ok, n_rows, bc, red_s, red_m, q, lane);
    else if (sub == 16) gn_run_moments<16>(tb, c_lo, c_hi, row_ok, n_rows, bc, red_s, red_m, q, lane);
    else gn_run_moments<1>(tb, c_lo, c_hi, row_ok, n_rows, bc, red_s, red_m, q, lane);
}

// GroupNorm of the runs of CPG consecutive channels held by one thread (CPG divides 32): two passes
// over the registers, population variance, then affine with the per-channel gamma / beta.
template <int CPG>
__device__ __forceinline__ void row_group_norm(float (&v)[32], const float* gamma_s, const float* beta_s, float eps) {
    float gamma[32], beta[32];
    lds_vec(gamma_s, gamma);
    lds_vec(beta_s, beta);
#pragma unroll
    for (int g = 0; g < 32 / CPG; ++g) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < CPG; ++i) s += v[g * CPG + i];
        const float mean = s * (1.f / CPG);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < CPG; ++i) {
            const float d = v[g * CPG + i] - mean;
            ss = fmaf(d, d, ss);
        }
        const float rstd = rsqrtf(ss * (1.f / CPG) + eps);
#pragma unroll
        for (int i = 0; i < CPG; ++i) {
            const int c = g * CPG + i;
            v[c] = fmaf((v[c] - mean) * rstd, gamma[c], beta[c]);
        }
    }
}

// 64-bit accesses are single-copy atomic: a word read with its epoch holds the value written with it.
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// At most one of this thread's bulk stores may still be reading its shared-memory source.
__device__ __forceinline__ void tma_store_wait_read_le1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Every bulk store issued by this thread has completed (its writes are done).
__device__ __forceinline__ void tma_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// LayerNorm of one 32-column chunk of a row from its mean and 1/sqrt(var + eps): per column
// ((v + bias) - mean) * rstd * gamma + beta, then GELU when asked, in paired fp32 arithmetic (each
// pair rounded as the scalar form ((v + (bias - mean)) * rstd) * gamma + beta).
__device__ __forceinline__ void ln_affine_gelu(float (&v)[32], const float* bias, const float* gamma, const float* beta,
                                               float mean, float rstd, bool gelu) {
    const uint64_t mp = f2_pack(mean, mean), rp = f2_pack(rstd, rstd);
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
        float bb[16], gg[16], be[16];
        lds_vec(bias + h, bb);
        lds_vec(gamma + h, gg);
        lds_vec(beta + h, be);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const uint64_t t = f2_add(f2_pack(v[h + i], v[h + i + 1]), f2_sub(f2_pack(bb[i], bb[i + 1]), mp));
            const uint64_t o = f2_fma(f2_mul(t, rp), f2_pack(gg[i], gg[i + 1]), f2_pack(be[i], be[i + 1]));
            f2_unpack(o, v[h + i], v[h + i + 1]);
        }
    }
    if (gelu) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) f2_unpack(gelu_erf2(f2_pack(v[i], v[i + 1])), v[i], v[i + 1]);
    }
}

// Fused GroupNorm output: out = acc * colscale + colshift (then GELU when asked) for this warp's
// columns [c_lo, c_hi), stored straight from registers. The 32 lanes of a warp hold 32 consecutive
// time steps of one channel, so each store writes 128 contiguous bytes (64 for bf16). The code runs
// once per launch: the chunk loop stays rolled so its instructions are fetched once and reused.
template <bool GELU, typename OutT>
__device__ __forceinline__ void gn_normalize_store(uint32_t tb, int c_lo, int c_hi, const float* colscale,
                                                   const float* colshift, OutT* ybase, int T_out, bool row_ok) {
    OutT* dst = ybase + (long long)c_lo * T_out;
    const long long step = T_out;
#pragma unroll 1
    for (int j0 = c_lo; j0 < c_hi; j0 += 32) {
        float v[32];
        tmem_load32(tb + uint32_t(j0), v);
        const int nv = row_ok ? min(32, c_hi - j0) : 0;  // columns of this chunk to store
#pragma unroll
        for (int h = 0; h < 32; h += 8) {
            float sc[8], sh[8];
            lds_vec(colscale + j0 + h, sc);
            lds_vec(colshift + j0 + h, sh);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float o = fmaf(v[h + i], sc[i], sh[i]);
                if constexpr (GELU) o = gelu_erf(o);
                if (h + i < nv) store_out(dst, o);
                dst += step;
            }
        }
    }
}

struct Unit {
    int n;     // sample (conv) / 0 (Linear)
    int row0;  // first output time step (conv) / first row (Linear)
    int cbu;   // index of the channel-block group
};

// A unit covers 128 rows (one CTA) or 256 rows (a CTA pair; `rank` selects the CTA's half).
// Linear mode walks the row tiles fastest, so the CTAs running at the same time share weight
// blocks in L2; conv mode walks the channel blocks fastest, so they share the x tile.
template <bool LINEAR, bool PAIR>
__device__ __forceinline__ Unit decode_unit(const TcArgs& a, int u, uint32_t rank) {
    Unit r;
    constexpr int kRows = PAIR ? 256 : 128;
    if (LINEAR) {
        r.n = 0;
        r.row0 = (u % a.n_t_tiles) * kRows + 128 * int(rank);
        r.cbu = u / a.n_t_tiles;
    } else {
        const int n_cbu = a.n_cb / a.cb_per_unit;
        r.cbu = u % n_cbu;
        const int rest = u / n_cbu;
        r.row0 = (rest % a.n_t_tiles) * kRows + 128 * int(rank);
        r.n = rest / a.n_t_tiles;
    }
    return r;
}

template <bool LINEAR, bool BF16, typename OutT, int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    tc_conv_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_y) {
    constexpr bool kFusedGN = EPI == kEpiClusterGN || EPI == kEpiGridGN;
    // kEpiLNX: the two CTAs of a cluster hold the two channel halves of the same 128 rows and
    // exchange per-row LayerNorm partial sums through distributed shared memory.
    constexpr bool kClusterX = EPI == kEpiLNX;
    static_assert(!(PAIR && (kFusedGN || kClusterX)), "the exchanging epilogues run one CTA per tile");
    // Epilogue warps: 4 (one per TMEM lane quarter), 8 (two per quarter, each taking a column range)
    // for the bf16 LayerNorm epilogues, whose transposer leaves warps 6-9 free, or 12 (warps 2-13,
    // three per quarter) for the fused GroupNorm: a fused-GroupNorm CTA has one tile, so its x
    // transposer warps first stage x and then, the mainloop's operands all staged, join the epilogue.
    constexpr int kEpiW = kFusedGN ? 12 : ((BF16 && (EPI == kEpiLN || EPI == kEpiLNX)) ? 8 : 4);
    constexpr int kEpiT = 32 * kEpiW;
    constexpr bool kShareXp = kFusedGN;
    static_assert(kShareXp || kWarpEpi0 + kEpiW <= xp_first<BF16>(), "epilogue and transposer warps overlap");
    using InT = typename std::conditional<BF16, __nv_bfloat16, float>::type;
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    const int SA = a.stages_a, SB = a.stages_b, SS = LINEAR ? 0 : a.stages_s;
    const uint32_t sA = smem_u32(base);
    const uint32_t sB = sA + uint32_t(SA * a.a_slot_bytes);
    const size_t s_off = size_t(SA) * a.a_slot_bytes + size_t(SB) * a.b_slot_bytes;  // x staging ring
    const uint32_t sS = sA + uint32_t(s_off);
    uint8_t* misc = base + s_off + size_t(SS) * a.s_slot_bytes + size_t(a.o_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    const int i_afull = 0, i_aempty = SA, i_bfull = 2 * SA, i_bempty = 2 * SA + SB, i_accfull = 2 * SA + 2 * SB,
              i_accempty = i_accfull + 2, i_drain = i_accempty + 2, i_sfull = i_drain + 1, i_sempty = i_sfull + SS,
              i_ex = i_sempty + SS, i_accinit = i_ex + 2, n_bars = i_ex + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + n_bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // progress counters: [0] B loads issued, [1] A chunks consumed by the MMA, [2] units issued by
    // the MMA, [3] A chunks written by transposer warp 0, [4] units finished by the epilogue,
    // [5] A loads issued (Linear); wait sites being waited on now: [6] MMA, [7] epilogue warp 0,
    // [8] transposer warp 0, [9] TMA; [10] MMA unit, [11] MMA ring indices (ai, aph, bi, bph).
    volatile int* prog = reinterpret_cast<volatile int*>(tmem_slot + 2);
    float* epi = reinterpret_cast<float*>(misc + 1024);  // epilogue scratch (kTcMiscBytes - 1024 bytes)
    const uint32_t bars_u32 = smem_u32(bars);
    auto bar = [&](int i) { return bars_u32 + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int taps = LINEAR ? 1 : a.k;
    // CTA pair (cta_group::2): rank 0 issues the MMAs over both CTAs' operands and owns the
    // full / accumulator-empty barriers; rank 1 signals those through the cluster.
    const uint32_t crank = (PAIR || kClusterX) ? (cluster_ctarank() & 1u) : 0u;
    const uint32_t rank = PAIR ? crank : 0u;
    const bool leader = rank == 0;
    // Bounded wait with an inline first test (the common case in a full pipeline costs no call).
    auto wait_bar = [&](int i, uint32_t parity, int site) -> bool {
        if constexpr (PAIR) {
            if (mbar_try_wait_cluster(bar(i), parity)) return true;
            return mbar_wait_cluster(bar(i), parity, abort_flag, a.status, site, prog);
        } else {
            if (mbar_try_wait(bar(i), parity)) return true;
            return mbar_wait(bar(i), parity, abort_flag, a.status, site, prog);
        }
    };
    auto leader_bar = [&](int i) -> uint32_t {
        if constexpr (PAIR) return map_shared_rank(bar(i), 0);
        else return bar(i);
    };
    // Unit u of this CTA; with kEpiLNX a unit is one (sample, 128-row tile) and the cluster rank
    // picks the channel half.
    auto decode = [&](int u) -> Unit {
        if constexpr (kClusterX) {
            Unit r;
            r.n = u / a.n_t_tiles;
            r.row0 = (u - r.n * a.n_t_tiles) * 128;
            r.cbu = int(crank);
            return r;
        } else {
            return decode_unit<LINEAR, PAIR>(a, u, rank);
        }
    };
    auto arrive_leader = [&](int i) {
        if (PAIR && !leader) mbar_arrive_cluster(leader_bar(i));
        else mbar_arrive(bar(i));
    };

    // This CTA's first unit, and how many of its x boxes are staged at entry: when the preceding
    // launch is this library's weight pack (which does not write x) and it released this kernel
    // only after its own wait for all earlier work, thread 0 arms the first x staging barriers
    // itself and issues those boxes before the CTA's setup; otherwise the unit's boxes head for L2. (A prefetch only fills L2, which every write reaches too, so it may run
    // ahead of the kernels this one depends on.)
    const int u0 = kFusedGN ? (blockIdx.z * a.n_t_tiles + blockIdx.x) * (a.n_cb / a.cb_per_unit) + blockIdx.y
                            : ((PAIR || kClusterX) ? int(blockIdx.x >> 1) : int(blockIdx.x));
    const int x_early = (!LINEAR && a.early_inputs && u0 < a.n_units) ? min(SS, a.n_ci_chunks) : 0;
    if (!LINEAR && threadIdx.x == 0 && u0 < a.n_units) {
        const Unit un0 = decode(u0);
        const int t0 = un0.row0 - a.pad_left - a.t_shift;
        const uint32_t box_bytes = uint32_t(a.RS * a.BK * (BF16 ? 2 : 4));
        for (int c = 0; c < x_early; ++c) mbar_init(bar(i_sfull + c), 1);
        if (x_early > 0) fence_mbar_init();
        for (int c = 0; c < x_early; ++c) {
            mbar_arrive_expect_tx(bar(i_sfull + c), box_bytes);
            tma_load_3d(sS + c * a.s_slot_bytes, &tm_a, bar(i_sfull + c), t0, c * a.BK, un0.n);
        }
        // With the first boxes in flight, prefetching the others would only delay them (every CTA's
        // loads share HBM at entry; the loader fetches the rest as slots free up). Without them,
        // the prefetch warms L2 for the loader.
        if (x_early == 0)
            for (int c = 0; c < a.n_ci_chunks; ++c) tma_prefetch_3d(&tm_a, t0, c * a.BK, un0.n);
    }
    if (warp == kWarpTma) {
        // barriers initialised by the 32 lanes together; arrival counts: A full: the TMA (Linear) or
        // one per transposer warp (of both CTAs of a pair); accumulator empty: one per epilogue warp
        // (of the pair); x staging empty: one per transposer warp; exchange: one per step, from the
        // peer's first 4 epilogue warps; accumulator initialised: one per warp 2-5; all others: one.
        for (int i = lane; i < n_bars; i += 32) {
            if (i >= i_sfull && i < i_sfull + x_early) continue;  // armed by thread 0 at entry
            uint32_t cnt = 1;
            if (i < i_aempty) cnt = LINEAR ? 1u : (PAIR ? 2u : 1u) * uint32_t(xp_warps<BF16>());
            else if (i >= i_accempty && i < i_drain) cnt = (PAIR ? 2u : 1u) * uint32_t(kEpiW);
            else if (i >= i_sempty && i < i_ex) cnt = uint32_t(xp_warps<BF16>());
            else if (i >= i_ex) cnt = 128;
            if (i == i_accinit) cnt = 4;
            mbar_init(bar(i), cnt);
        }
        if (lane == 0) *abort_flag = 0;
        if (lane < kProgSlots) prog[lane] = 0;
        fence_mbar_init();
        if (lane == 0) {
            prefetch_tensormap(&tm_a);
            prefetch_tensormap(&tm_b);
        }
    }
    if (warp == kWarpMma) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), uint32_t(a.tmem_cols));
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), uint32_t(a.tmem_cols));
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if (PAIR || kClusterX) cluster_sync_all();  // the peer's barriers exist before any remote arrival
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above (barriers, TMEM, tensor-map prefetch) may overlap the previous kernel of the
    // stream; no global memory it may write (x, weights, parameters, workspace) is touched before
    // this point. Two roles go on without waiting: the x transposer touches no global memory, and
    // the x loader reads only x, which the weight pack launched just before this kernel does not
    // write (the pack itself starts only after all earlier work of the stream has finished).
    {
        const bool xp_role = !LINEAR && warp >= xp_first<BF16>() && warp < xp_first<BF16>() + xp_warps<BF16>();
        if (!(xp_role || warp == kWarpTma || (warp == kWarpXld && a.early_inputs))) griddep_wait();
    }

    int first_unit, unit_step;
    if (kFusedGN) {
        first_unit = (blockIdx.z * a.n_t_tiles + blockIdx.x) * (a.n_cb / a.cb_per_unit) + blockIdx.y;
        unit_step = a.n_units;  // exactly one unit
    } else if (PAIR || kClusterX) {
        first_unit = blockIdx.x >> 1;  // one unit per cluster of two
        unit_step = gridDim.x >> 1;
    } else {
        first_unit = blockIdx.x;
        unit_step = gridDim.x;
    }

    // The producer and MMA warps run their loops with all 32 lanes (so loop state, addresses and
    // descriptors stay warp-uniform) and issue each copy / MMA / commit from one elected lane.
    // Every wait is taken by all lanes and agreed on with a vote.
    auto wait_warp = [&](int i, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, wait_bar(i, parity, site));
    };
    auto aborting = [&]() -> bool { return __any_sync(0xffffffffu, *abort_flag != 0); };
    if (warp == kWarpTma) {
        // ---------------------------------------------------------------- TMA producer
        // Linear mode: one ring of stages, each holding the A and the B chunk of one K step under
        // one full / empty barrier pair. Conv mode: the B (weight) ring only; A comes from the
        // transposer warps. A pair's full barriers (in the leader) expect both CTAs' bytes; each
        // CTA loads its own 128 rows of A and its half (BN/2 channels) of the B tile.
        int bi = 0;
        uint32_t bph = 0;
        long long b_cnt = 0;
        const uint32_t tx_mult = PAIR ? 2u : 1u;
        const uint32_t tx_stage = tx_mult * uint32_t(a.b_slot_bytes + (LINEAR ? a.a_slot_bytes : 0));
        const int co_half = PAIR ? int(rank) * (a.BN / 2) : 0;
        const int nparts = (!LINEAR && !BF16 && a.x3) ? 2 : 1;
        __syncwarp();
        griddep_wait();
        for (int u = first_unit; u < a.n_units && !aborting(); u += unit_step) {
            const Unit un = decode(u);
            for (int c = 0; c < a.n_ci_chunks; ++c) {
                for (int cbi = 0; cbi < a.cb_per_unit; ++cbi) {
                    const int co0 = (un.cbu * a.cb_per_unit + cbi) * a.BN + co_half;
                    for (int kkp = 0; kkp < taps * nparts; ++kkp) {
                        // 3xTF32: the head tile (part 0) then the tail tile (part 1) of each tap
                        const int kk = kkp / nparts, part = kkp - kk * nparts;
                        if (!wait_warp(i_bempty + bi, bph ^ 1, kWaitBEmpty)) goto tma_done;
                        const uint32_t full = leader_bar(i_bfull + bi);
                        const uint32_t dst_b = sB + uint32_t(bi * a.b_slot_bytes);
                        const uint32_t dst_a = sA + uint32_t(bi * a.a_slot_bytes);
                        if (elect_one()) {
                            if (leader) mbar_arrive_expect_tx(bar(i_bfull + bi), tx_stage);
                            if (LINEAR) {
                                if constexpr (PAIR) {
                                    tma_load_2d_pair(dst_a, &tm_a, full, c * a.BK, un.row0);
                                    tma_load_2d_pair(dst_b, &tm_b, full, c * a.BK, co0);
                                } else {
                                    tma_load_2d(dst_a, &tm_a, full, c * a.BK, un.row0);
                                    tma_load_2d(dst_b, &tm_b, full, c * a.BK, co0);
                                }
                            } else {
                                if constexpr (PAIR) tma_load_3d_pair(dst_b, &tm_b, full, c * a.BK, co0, kk + part * a.k);
                                else tma_load_3d(dst_b, &tm_b, full, c * a.BK, co0, kk + part * a.k);
                            }
                        }
                        __syncwarp();
                        ++b_cnt;
                        if (++bi == SB) { bi = 0; bph ^= 1; }
                    }
                }
            }
            if (lane == 0) prog[0] = int(b_cnt);
        }
    tma_done:
        if (aborting() && lane == 0) {
            // Let copies already in flight land before the CTA's shared memory goes away.
            if (leader) {
                for (int s = 0; s < SB; ++s)
                    if (b_cnt > s) mbar_drain(bar(i_bfull + s), s < bi ? bph : (bph ^ 1), a.status);
            } else {
                // the second CTA of a pair signals the leader's barriers and cannot watch its
                // own copies: give them a fixed 200 us to land
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------------- MMA issuer
        // Descriptors are built once: every operand slot is 128-byte swizzled, K-major, with
        // 8-row groups 1024 bytes apart, so only the start-address field (low word, in 16-byte
        // units) changes between MMAs: +2 per 32-byte K step, +8*dilation per tap (A tile
        // shifted down by dilation rows), + slot size per ring slot.
        if (leader) {
            int ai = 0, bi = 0;
            uint32_t aph = 0, bph = 0;
            int lt = 0;
            bool ok = true;
            const uint32_t a_lo0 = desc_lo_sw128(sA), b_lo0 = desc_lo_sw128(sB);
            const uint32_t a_step = uint32_t(a.a_slot_bytes) >> 4, b_step = uint32_t(a.b_slot_bytes) >> 4;
            const uint32_t tap_step = uint32_t(8 * a.dil);
            const uint32_t idesc = a.idesc;
            const bool x3 = !LINEAR && !BF16 && a.x3;  // 3xTF32: hi*hi + hi*lo + lo*hi per step
            const uint32_t a_tail = uint32_t(a.R * 8);  // the A tail tile follows the head tile (16-byte units)
            // Completion of the MMAs so far arrives on barrier i (in both CTAs of a pair).
            auto commit = [&](int i) {
                if constexpr (PAIR) mma_commit_pair(bar(i), 3);
                else mma_commit(bar(i));
            };
            for (int u = first_unit; u < a.n_units && ok && !aborting(); u += unit_step, ++lt) {
                const int ab = a.n_acc == 2 ? (lt & 1) : 0;
                const uint32_t acc_par = a.n_acc == 2 ? uint32_t((lt >> 1) & 1) : uint32_t(lt & 1);
                if (lane == 0) {
                    prog[10] = lt;
                    prog[11] = ai | (int(aph) << 8) | (bi << 16) | (int(bph) << 24);
                }
                if (!wait_warp(i_accempty + ab, acc_par ^ 1, kWaitAccEmpty)) break;
                // fused GroupNorm: the accumulator starts as the bias, written by warps 2-5
                if (kFusedGN && lt == 0 && !wait_warp(i_accinit, 0, kWaitAccInit)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + uint32_t(256 * ab * a.cb_per_unit);
                for (int c = 0; c < a.n_ci_chunks && ok; ++c) {
                    const uint32_t a_lo = a_lo0 + uint32_t(ai) * a_step;
                    if (!LINEAR) {
                        if (!wait_warp(i_afull + ai, aph, kWaitAFull)) { ok = false; break; }
                    }
                    for (int cbi = 0; cbi < a.cb_per_unit && ok; ++cbi) {
                        const uint32_t d = d0 + uint32_t(256 * cbi);
                        for (int kk = 0; kk < taps; ++kk) {
                            if (!wait_warp(i_bfull + bi, bph, kWaitBFull)) { ok = false; break; }
                            // 3xTF32: the tail tile of B is the next stage of the ring
                            const int bi2 = bi + 1 == SB ? 0 : bi + 1;
                            const uint32_t bph2 = bi + 1 == SB ? (bph ^ 1u) : bph;
                            if (x3 && !wait_warp(i_bfull + bi2, bph2, kWaitBFull)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t al = LINEAR ? a_lo0 + uint32_t(bi) * a_step : a_lo + uint32_t(kk) * tap_step;
                            const uint32_t bl = b_lo0 + uint32_t(bi) * b_step;
                            const uint32_t bl2 = b_lo0 + uint32_t(bi2) * b_step;
                            const uint32_t acc0 = (kFusedGN || (c | kk) != 0) ? 1u : 0u;
                            if (elect_one()) {
                                mma_issue<BF16, PAIR>(d, al, bl, idesc, acc0);
                                mma_issue<BF16, PAIR>(d, al + 2u, bl + 2u, idesc, 1u);
                                mma_issue<BF16, PAIR>(d, al + 4u, bl + 4u, idesc, 1u);
                                mma_issue<BF16, PAIR>(d, al + 6u, bl + 6u, idesc, 1u);
                                if (x3) {
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        mma_issue<BF16, PAIR>(d, al + 2u * j, bl2 + 2u * j, idesc, 1u);           // A head x B tail
                                        mma_issue<BF16, PAIR>(d, al + a_tail + 2u * j, bl + 2u * j, idesc, 1u);   // A tail x B head
                                    }
                                }
                                commit(i_bempty + bi);
                                if (x3) commit(i_bempty + bi2);
                            }
                            __syncwarp();
                            if (++bi == SB) { bi = 0; bph ^= 1; }
                            if (x3 && ++bi == SB) { bi = 0; bph ^= 1; }
                        }
                    }
                    if (!ok) break;
                    if (!LINEAR) {
                        if (elect_one()) commit(i_aempty + ai);
                        __syncwarp();
                        if (++ai == SA) { ai = 0; aph ^= 1; }
                    }
                }
                if (!ok) break;
                if (elect_one()) commit(i_accfull + ab);
                __syncwarp();
                if (lane == 0) prog[2] = lt + 1;
            }
            // Every MMA issued above has finished before TMEM is released (the commit comes from
            // the lane that issued them: elect.sync picks the lowest active lane each time).
            if (elect_one()) {
                if constexpr (PAIR) mma_commit_pair(bar(i_drain), 1);
                else mma_commit(bar(i_drain));
            }
            __syncwarp();
            if (lane == 0) mbar_drain(bar(i_drain), 0, a.status);
            // The MMAs are done: let the stream's next kernel launch now, so its launch overlaps this
            // kernel's epilogue (it waits for this kernel's completion before it reads or writes
            // anything this kernel touches: the library's weight pack does so first thing).
            griddep_launch_dependents();
        }
    } else if (warp == kWarpXld) {
        // ---------------------------------------------------------------- x staging loader (conv mode)
        // One TMA box per (tile, input-channel chunk): RS time steps (from a 16-byte aligned time
        // coordinate) x BK channels of one sample, time-contiguous. Boxes that reach past either
        // end of the sequence or past C_in are zero-filled by the TMA unit, which is exactly the
        // convolution's zero padding.
        if (!LINEAR && lane == 0) {
            const uint32_t box_bytes = uint32_t(a.RS * a.BK * (BF16 ? 2 : 4));
            // the first x_early boxes of the first unit were issued by thread 0 at entry
            int si = x_early == SS ? 0 : x_early;
            uint32_t sph = x_early == SS ? 1u : 0u;
            long long s_cnt = x_early;
            for (int u = first_unit; u < a.n_units && !*abort_flag; u += unit_step) {
                const Unit un = decode(u);
                const int t0 = un.row0 - a.pad_left - a.t_shift;  // multiple of 16 bytes of elements
                for (int c = u == first_unit ? x_early : 0; c < a.n_ci_chunks; ++c) {
                    if (!mbar_try_wait(bar(i_sempty + si), sph ^ 1) &&
                        !mbar_wait(bar(i_sempty + si), sph ^ 1, abort_flag, a.status, kWaitSEmpty, prog))
                        goto xld_done;
                    mbar_arrive_expect_tx(bar(i_sfull + si), box_bytes);
                    tma_load_3d(sS + si * a.s_slot_bytes, &tm_a, bar(i_sfull + si), t0, c * a.BK, un.n);
                    ++s_cnt;
                    if (++si == SS) { si = 0; sph ^= 1; }
                }
            }
        xld_done:
            if (*abort_flag)
                for (int s2 = 0; s2 < SS; ++s2)
                    if (s_cnt > s2) mbar_drain(bar(i_sfull + s2), s2 < si ? sph : (sph ^ 1), a.status);
        }
    } else {
        // x transposer and epilogue (with fp32 data the fused GroupNorm's warps 6-9 are both, in turn)
        if (warp >= xp_first<BF16>() && warp < xp_first<BF16>() + xp_warps<BF16>()) {
            // ---------------------------------------------------------------- x transposer (conv mode)
            // Staged x (rows = channels, time-contiguous) -> A tile (rows = time steps, 128 bytes of
            // channels per row, 128-byte swizzle).
            if (!LINEAR) {
                constexpr int kXp0 = xp_first<BF16>(), kXpW = xp_warps<BF16>();
                const int xw = warp - kXp0;
                const int R = a.R, RS = a.RS;
                int ai = 0, si = 0;
                uint32_t aph = 0, sph = 0;
                for (int u = first_unit; u < a.n_units; u += unit_step) {
                    for (int c = 0; c < a.n_ci_chunks; ++c) {
                        // One lane waits; the shuffle hands its answer to the warp and reconverges it.
                        int ok = 0;
                        if (lane == 0)
                            ok = mbar_wait(bar(i_sfull + si), sph, abort_flag, a.status, kWaitSFull, prog) &&
                                 wait_bar(i_aempty + ai, aph ^ 1, kWaitAEmpty);
                        if (!__shfl_sync(0xffffffffu, ok, 0)) goto xp_done;
                        uint8_t* slot = base + size_t(ai) * a.a_slot_bytes;
                        if constexpr (BF16) {
                            // 8x8 blocks (8 channels x 8 staged steps) through ldmatrix.trans + stmatrix,
                            // four blocks (channel groups 4*quad .. 4*quad+3) per instruction pair. Lane l
                            // gives row l%8 of block l/8: the source row is channel 8*cg + l%8 at staged
                            // steps 8*tg.., the destination row is A row 8*tg + l%8 - t_shift (rows
                            // outside the tile go to a scratch row). The staging row pitch RS is an odd
                            // multiple of 16 bytes, so the 8 rows of a block hit 8 different bank groups.
                            const uint32_t stg = sS + uint32_t(si * a.s_slot_bytes);
                            const uint32_t dslot = smem_u32(slot);
                            const uint32_t dummy = smem_u32(misc + 512) + uint32_t(lane * 16);
                            const int n_tg = (a.t_shift + R + 7) / 8;
                            const int mi = lane >> 3, ii = lane & 7;
                            for (int opi = xw; opi < 2 * n_tg; opi += kXpW) {
                                const int tg = opi >> 1, cg = (opi & 1) * 4 + mi;
                                uint32_t r[4];
                                ldmatrix_x4_trans(stg + uint32_t(((8 * cg + ii) * RS + 8 * tg) * 2), r);
                                const int rr = 8 * tg + ii - a.t_shift;
                                const uint32_t dst = (rr >= 0 && rr < R)
                                                         ? dslot + uint32_t(rr * 128 + ((cg ^ (rr & 7)) << 4))
                                                         : dummy;
                                stmatrix_x4(dst, r);
                            }
                        } else {
                            // Warp w owns the 16-byte column chunk w of every A row; its lanes take
                            // consecutive rows, so the staged reads are consecutive elements (one
                            // wavefront) and each group of 8 lanes writes 8 distinct swizzled chunks.
                            const int cg = xw;
                            const InT* col = reinterpret_cast<const InT*>(base + s_off + size_t(si) * a.s_slot_bytes) +
                                             (cg * 4) * RS + a.t_shift;
                            if (a.x3) {
                                // 3xTF32: the TF32 head (rounded) in the first tile, the tail x - head in
                                // the second (R rows further)
#pragma unroll 2
                                for (int r = lane; r < R; r += 32) {
                                    const InT* src = col + r;
                                    float v[4] = {float(src[0]), float(src[RS]), float(src[2 * RS]), float(src[3 * RS])};
                                    float h[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) h[e] = round_tf32(v[e]);
                                    const int off = r * 128 + ((cg ^ (r & 7)) << 4);
                                    *reinterpret_cast<uint4*>(slot + off) = make_uint4(
                                        __float_as_uint(h[0]), __float_as_uint(h[1]), __float_as_uint(h[2]), __float_as_uint(h[3]));
                                    *reinterpret_cast<uint4*>(slot + R * 128 + off) =
                                        make_uint4(__float_as_uint(v[0] - h[0]), __float_as_uint(v[1] - h[1]),
                                                   __float_as_uint(v[2] - h[2]), __float_as_uint(v[3] - h[3]));
                                }
                            } else {
#pragma unroll 2
                                for (int r = lane; r < R; r += 32) {
                                    const InT* src = col + r;
                                    const uint4 pk = make_uint4(__float_as_uint(src[0]), __float_as_uint(src[RS]),
                                                                __float_as_uint(src[2 * RS]), __float_as_uint(src[3 * RS]));
                                    // 16-byte chunk cg of row r sits at chunk position cg ^ (r & 7)
                                    *reinterpret_cast<uint4*>(slot + r * 128 + ((cg ^ (r & 7)) << 4)) = pk;
                                }
                            }
                        }
                        // Make the generic-proxy stores visible to the tensor core, then signal.
                        fence_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            arrive_leader(i_afull + ai);
                            mbar_arrive(bar(i_sempty + si));
                        }
                        if (threadIdx.x == kXp0 * 32) prog[3] = prog[3] + 1;
                        if (++ai == SA) { ai = 0; aph ^= 1; }
                        if (++si == SS) { si = 0; sph ^= 1; }
                    }
                }
            xp_done:;
            }
        }
        if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEpiW) {
            // ---------------------------------------------------------------- epilogue warps 2..(2+kEpiW-1)
            const int q = warp & 3;       // TMEM lane quarter this warp may access
            const int m = q * 32 + lane;  // tile row: time step (conv) or sample row (Linear)
            const int er = threadIdx.x - kWarpEpi0 * 32;  // index among the epilogue threads
            const int eg = (warp - kWarpEpi0) >> 2;       // column range (kEpiW / 4 warps per quarter)
            bool mid_sync_done = false;
            // Per-channel parameters of the current channel block, staged once in shared memory so the
            // element loops below read them with conflict-free broadcast loads instead of global loads.
            float* s_bias = epi + 3072;  // [256]
            int staged_co = -1;
            int obuf = 0;  // LayerNorm output staging: which of this warp's two tiles is next
            // Grid exchange of the fused GroupNorm: this launch's epoch is one past the one in this
            // CTA's own first word (all words of a (sample, channel block) carry the same epoch after
            // every launch), read here, while the mainloop runs, rather than on the epilogue's path.
            unsigned gx_target = 0;
            if (kFusedGN && first_unit < a.n_units) {
                // One unit per CTA: stage bias, gamma and beta of its channel block while the
                // mainloop runs (gamma and beta go where the column scale / shift end up). (Warps that
                // were x transposers have not waited for the preceding kernel yet.)
                griddep_wait();
                if (er < 128) {  // warps 2-5, which have no role in the mainloop
                    const int co_base = decode(first_unit).cbu * a.BN;
                    const int ncols = min(a.BN, a.C_out - co_base);
                    for (int col = er; col < 256; col += 128) {
                        const bool ok = col < ncols;
                        s_bias[col] = (ok && a.bias) ? __ldg(a.bias + co_base + col) : 0.f;
                        epi[2304 + col] = ok ? (a.gamma ? __ldg(a.gamma + co_base + col) : 1.f) : 0.f;
                        epi[2560 + col] = (ok && a.beta) ? __ldg(a.beta + co_base + col) : 0.f;
                    }
                    // (the epilogue's first barrier, at the accumulator wait, orders these for the
                    // other epilogue warps)
                    // The accumulator starts as the bias (every row of column j holds bias[j]) and the
                    // MMAs add the convolution to it, so the epilogue reads y itself from TMEM. Each of
                    // the four warps writes its lane quarter, then signals the MMA warp.
                    named_bar_sync(2, 128);
                    const uint32_t tq = tmem_base + (uint32_t(q * 32) << 16);
#pragma unroll 1
                    for (int j0 = 0; j0 < ncols; j0 += 32) {
                        float bv[32];
                        lds_vec(s_bias + j0, bv);
                        tmem_store32(tq + uint32_t(j0), bv);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(i_accinit));
                }
                // (after the accumulator's first operand, which the MMAs wait for)
                if (EPI == kEpiGridGN) {
                    const Unit un0 = decode(first_unit);
                    const size_t w0i = (size_t(un0.n * a.n_cb + un0.cbu) * a.n_t_tiles + un0.row0 / 128) * size_t(a.gstride) * 2;
                    gx_target = unsigned(ld_relaxed_gpu_u64(a.gx + w0i) >> 32) + 1u;
                }
            }
            int lt = 0;
            for (int u = first_unit; u < a.n_units; u += unit_step, ++lt) {
                const int ab = a.n_acc == 2 ? (lt & 1) : 0;
                const uint32_t acc_par = a.n_acc == 2 ? uint32_t((lt >> 1) & 1) : uint32_t(lt & 1);
                // One lane per warp waits; the shuffle reconverges the warp (the TMEM loads below are
                // warp-collective), and the barrier ORs what every epilogue thread saw, so all the
                // epilogue warps leave (or stay) together. False: give up.
                auto acc_wait = [&]() -> bool {
                    if (er == 0) prog[7] = kWaitAccFull;
                    int got = 0;
                    if (lane == 0) got = wait_bar(i_accfull + ab, acc_par, kWaitAccFull);
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (named_bar_any(1, kEpiT, !got || *abort_flag != 0)) return false;
                    __syncwarp();
                    if (er == 0) prog[7] = 0;
                    tc_fence_after();
                    return true;
                };
                // (the fused GroupNorm waits further down, once the index arithmetic of its tile,
                // which does not need the accumulator, is done)
                if constexpr (!kFusedGN) {
                    if (!acc_wait()) break;
                }
                const Unit un = decode(u);
                OutT* y = static_cast<OutT*>(a.y);
                const int row = un.row0 + m;
                const bool row_ok = LINEAR ? (row < a.N) : (row < a.T_out);

                if (EPI == kEpiDirect || EPI == kEpiDirectStats) {
                    for (int cbi = 0; cbi < a.cb_per_unit; ++cbi) {
                        const int cb = un.cbu * a.cb_per_unit + cbi;
                        const int co_base = cb * a.BN;
                        const int ncols = min(a.BN, a.C_out - co_base);
                        if (co_base != staged_co) {  // uniform over the epilogue threads
                            named_bar_sync(1, kEpiT);
                            for (int col = er; col < a.BN; col += kEpiT)
                                s_bias[col] = (a.bias && col < ncols) ? __ldg(a.bias + co_base + col) : 0.f;
                            named_bar_sync(1, kEpiT);
                            if (EPI == kEpiDirectStats && a.part_kind == 1) {
                                // the bias minus its mean over the column's run of `sub` channels
                                const int run = a.sub > 0 ? a.sub : 1;
                                for (int col = er; col < 256; col += kEpiT) {
                                    const int r0 = col - col % run;
                                    float mb = 0.f;
                                    for (int i = 0; i < run; ++i) mb += s_bias[r0 + i];
                                    epi[2816 + col] = s_bias[col] - mb * (1.f / float(run));
                                }
                                named_bar_sync(1, kEpiT);
                            }
                            staged_co = co_base;
                        }
                        const uint32_t tb =
                            tmem_base + (uint32_t(q * 32) << 16) + uint32_t(256 * (ab * a.cb_per_unit + cbi));
                        if (EPI == kEpiDirectStats && a.part_kind == 1) {
                            // GroupNorm partials of this 128-row tile: per-warp moments per run of
                            // `sub` channels, merged over the runs of each group and the four warps
                            // (Chan's formula) into the tile's (mean, M2) per group. Groups lie inside
                            // the channel block.
                            float* red_s = epi;         // [4][256] per-warp run sums
                            float* red_m = epi + 1024;  // [4][256] per-warp run sums of squared deviations
                            const int nvalid_t = min(128, a.T_out - un.row0);
                            const int nvalid_w = min(32, max(0, nvalid_t - q * 32));
                            gn_run_moments_any(a.sub, tb, 0, ncols, lane < nvalid_w, nvalid_w, epi + 2816, red_s, red_m,
                                               q, lane);
                            named_bar_sync(1, kEpiT);
                            const int run = a.sub > 0 ? a.sub : 1;
                            const int cpg = a.cpg;
                            const int ngroups = ncols / cpg;
                            for (int g = er; g < ngroups && nvalid_t > 0; g += kEpiT) {
                                float gn = 0.f, gmu = 0.f, gm2 = 0.f;
                                for (int j = g * cpg / run; j < (g + 1) * cpg / run; ++j) {
                                    float mb = 0.f;  // the bias mean of run j
                                    for (int i = 0; i < run; ++i) mb += s_bias[j * run + i];
                                    mb *= 1.f / float(run);
                                    for (int q2 = 0; q2 < 4; ++q2) {
                                        const int nr = min(32, max(0, nvalid_t - q2 * 32));
                                        if (nr == 0) continue;
                                        const float nq = float(nr * run);
                                        chan_merge(gn, gmu, gm2, nq, red_s[q2 * 256 + j] / nq + mb, red_m[q2 * 256 + j]);
                                    }
                                }
                                const size_t gi = size_t(un.n) * a.groups + co_base / cpg + g;
                                a.part[gi * a.part_tiles + un.row0 / 128] = make_float2(gmu, gm2);
                            }
                            // red_s / red_m are read above before the next tile's moments overwrite them
                            named_bar_sync(1, kEpiT);
                        } else if (EPI == kEpiDirectStats && a.part_kind == 2) {
                            // channel LayerNorm partials of this step over the block's channels: the
                            // mean, then the sum of squared deviations from it (two sweeps of TMEM)
                            float s1 = 0.f;
                            for (int j0 = 0; j0 < ncols; j0 += 16) {
                                float v[16], bb[16];
                                tmem_load16(tb + uint32_t(j0), v);
                                lds_vec(s_bias + j0, bb);
#pragma unroll
                                for (int i = 0; i < 16; ++i) s1 += (j0 + i < ncols) ? v[i] + bb[i] : 0.f;
                            }
                            const float mu = s1 / float(ncols);
                            float m2 = 0.f;
                            for (int j0 = 0; j0 < ncols; j0 += 16) {
                                float v[16], bb[16];
                                tmem_load16(tb + uint32_t(j0), v);
                                lds_vec(s_bias + j0, bb);
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const float d = v[i] + bb[i] - mu;
                                    m2 = (j0 + i < ncols) ? fmaf(d, d, m2) : m2;
                                }
                            }
                            if (row_ok) a.part[(size_t(un.n) * a.n_cb + cb) * a.T_out + row] = make_float2(mu, m2);
                        }
                        for (int j0 = 0; j0 < ncols; j0 += 16) {
                            float v[16];
                            tmem_load16(tb + uint32_t(j0), v);
                            {
                                float bb[16];
                                lds_vec(s_bias + j0, bb);
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] += bb[i];
                            }
                            if (a.gelu) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] = gelu_erf(v[i]);
                            }
                            if (!row_ok) continue;
                            if (LINEAR) {
                                OutT* dst = y + (long long)row * a.C_out + co_base + j0;
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (j0 + i < ncols) store_out(dst + i, v[i]);
                            } else {
                                OutT* dst = y + ((long long)un.n * a.C_out + co_base + j0) * a.T_out + row;
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (j0 + i < ncols) store_out(dst + (long long)i * a.T_out, v[i]);
                            }
                        }
                    }
                } else if (EPI == kEpiRowGN) {
                    // ------------------------------------------------ row epilogue (Linear mode)
                    // One thread owns one row (sample) and the channel block's columns: bias, optional
                    // GroupNorm over runs of row_cpg channels, affine, then either GELU + store or a
                    // running minimum (lowest channel on ties) for the row-min post-op.
                    const int co_base = un.cbu * a.BN;
                    const int ncols = min(a.BN, a.C_out - co_base);
                    float* s_gamma = epi + 2304;
                    float* s_beta = epi + 2560;
                    if (co_base != staged_co) {  // uniform over the epilogue threads
                        named_bar_sync(1, kEpiT);
                        for (int col = er; col < 256; col += kEpiT) {
                            const bool ok = col < ncols;
                            s_bias[col] = (ok && a.bias) ? __ldg(a.bias + co_base + col) : 0.f;
                            s_gamma[col] = ok ? (a.gamma ? __ldg(a.gamma + co_base + col) : 1.f) : 0.f;
                            s_beta[col] = (ok && a.beta) ? __ldg(a.beta + co_base + col) : 0.f;
                        }
                        named_bar_sync(1, kEpiT);
                        staged_co = co_base;
                    }
                    const uint32_t tb = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(256 * ab);
                    float best = __int_as_float(0x7f800000);
                    int best_i = 0x7fffffff;
                    OutT* dst = y + (long long)(row_ok ? row : 0) * a.C_out + co_base;
                    for (int j0 = 0; j0 < ncols; j0 += 32) {
                        float v[32];
                        tmem_load32(tb + uint32_t(j0), v);
                        {
                            float bb[32];
                            lds_vec(s_bias + j0, bb);
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] += bb[i];
                        }
                        if (a.row_cpg == 8) row_group_norm<8>(v, s_gamma + j0, s_beta + j0, a.eps);
                        else if (a.row_cpg == 16) row_group_norm<16>(v, s_gamma + j0, s_beta + j0, a.eps);
                        else if (a.row_cpg == 32) row_group_norm<32>(v, s_gamma + j0, s_beta + j0, a.eps);
                        if (a.rowmin) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (j0 + i < ncols && v[i] < best) { best = v[i]; best_i = co_base + j0 + i; }
                        } else {
                            if (a.gelu) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = gelu_erf(v[i]);
                            }
                            if (row_ok) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (j0 + i < ncols) store_out(dst + j0 + i, v[i]);
                            }
                        }
                    }
                    if (a.rowmin && row_ok)
                        a.rowpart[(size_t)row * a.n_cb + un.cbu] = make_float2(best, __int_as_float(best_i));
                } else if (EPI == kEpiLN || EPI == kEpiLNX) {
                    // ------------------------------------------------ channel LayerNorm (conv mode)
                    // One thread owns one time step. kEpiLN: this CTA holds every channel of the tile.
                    // kEpiLNX: it holds channels [crank*BN, crank*BN + BN) and its cluster peer the rest
                    // of the same 128 steps. With bf16 data two epilogue warps share each TMEM lane
                    // quarter and split the channels in two column ranges. Statistics: one pass of sums
                    // shifted by the range's first value gives each range's mean and M2; the ranges of
                    // a CTA are merged through shared memory, the CTA halves of kEpiLNX through
                    // distributed shared memory (remote stores + a remote arrival), all with Chan's
                    // formula in a fixed order, so every thread of both CTAs computes the same mean and
                    // variance. Then normalize + affine (+ GELU), staged per warp as [32 channels][32
                    // steps] tiles in shared memory and written by TMA bulk stores (or direct stores
                    // when y's layout does not allow TMA).
                    float* s_bias = epi;
                    float* s_gamma = epi + 256;
                    float* s_beta = epi + 512;
                    float* xbuf = epi + 768 + 256 * (lt & 1);  // [2 tiles][2][128]: the peer's mean and M2
                    float* hst = epi + 1280 + 512 * (lt & 1);  // [2 tiles][2 ranges][128][2]: range statistics
                    const int co_base = un.cbu * a.BN;
                    const int ncols = min(a.BN, a.C_out - co_base);
                    if (staged_co < 0) {
                        for (int c = er; c < 256; c += kEpiT) {
                            const bool ok = c < ncols;
                            s_bias[c] = (ok && a.bias) ? __ldg(a.bias + co_base + c) : 0.f;
                            s_gamma[c] = ok ? (a.gamma ? __ldg(a.gamma + co_base + c) : 1.f) : 0.f;
                            s_beta[c] = (ok && a.beta) ? __ldg(a.beta + co_base + c) : 0.f;
                        }
                        named_bar_sync(1, kEpiT);
                        staged_co = co_base;
                    }
                    // this warp's column range [c_lo, c_hi) (whole 32-column chunks but the last)
                    const int half = kEpiW == 8 ? ((ncols + 63) / 64) * 32 : ncols;
                    const int c_lo = eg == 0 ? 0 : min(half, ncols);
                    const int c_hi = eg == 0 ? min(half, ncols) : ncols;
                    const uint32_t tb = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(256 * ab);
                    float shift = 0.f, s1 = 0.f, s2 = 0.f;
                    for (int j0 = c_lo; j0 < c_hi; j0 += 32) {
                        float v[32];
                        tmem_load32(tb + uint32_t(j0), v);
                        float bb[32];
                        lds_vec(s_bias + j0, bb);
                        if (j0 == c_lo) shift = v[0] + bb[0];
                        if (j0 + 32 <= c_hi) {  // whole chunk (uniform): no per-column test, paired sums
                            const uint64_t sp = f2_pack(shift, shift);
                            uint64_t p1 = 0ull, p2 = 0ull;
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const uint64_t d = f2_sub(f2_add(f2_pack(v[i], v[i + 1]), f2_pack(bb[i], bb[i + 1])), sp);
                                p1 = f2_add(p1, d);
                                p2 = f2_fma(d, d, p2);
                            }
                            s1 += f2_hsum(p1);
                            s2 += f2_hsum(p2);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (j0 + i < c_hi) {
                                    const float d = v[i] + bb[i] - shift;
                                    s1 += d;
                                    s2 = fmaf(d, d, s2);
                                }
                        }
                    }
                    const float n_own = float(c_hi - c_lo);
                    float mean = n_own > 0.f ? shift + s1 / n_own : 0.f;
                    float m2 = n_own > 0.f ? fmaxf(s2 - s1 * (s1 / n_own), 0.f) : 0.f;
                    float n_cta = n_own;
                    if constexpr (kEpiW == 8) {
                        // the two column ranges of this CTA, merged in range order
                        hst[(eg * 128 + m) * 2] = mean;
                        hst[(eg * 128 + m) * 2 + 1] = m2;
                        named_bar_sync(1, kEpiT);
                        float n0 = float(min(half, ncols)), mu0 = hst[m * 2], m20 = hst[m * 2 + 1];
                        chan_merge(n0, mu0, m20, float(ncols) - float(min(half, ncols)), hst[(128 + m) * 2],
                                   hst[(128 + m) * 2 + 1]);
                        mean = mu0;
                        m2 = m20;
                        n_cta = n0;
                    }
                    if constexpr (kClusterX) {
                        const uint32_t peer = crank ^ 1u;
                        if (eg == 0) {
                            st_shared_cluster_f32(map_shared_rank(smem_u32(xbuf + m), peer), mean);
                            st_shared_cluster_f32(map_shared_rank(smem_u32(xbuf + 128 + m), peer), m2);
                            mbar_arrive_cluster(map_shared_rank(bar(i_ex), peer));
                        }
                        mbar_wait_cluster(bar(i_ex), uint32_t(lt & 1), abort_flag, a.status, kWaitExchange, prog);
                        const float n_peer = float(a.C_out - ncols);
                        const float p_mean = xbuf[m], p_m2 = xbuf[128 + m];
                        // Chan's merge of (rank 0 half, rank 1 half)
                        const float na = crank == 0 ? n_cta : n_peer, nb = crank == 0 ? n_peer : n_cta;
                        const float ma = crank == 0 ? mean : p_mean, mb = crank == 0 ? p_mean : mean;
                        const float Ma = crank == 0 ? m2 : p_m2, Mb = crank == 0 ? p_m2 : m2;
                        const float nt = na + nb, dlt = mb - ma;
                        mean = ma + dlt * (nb / nt);
                        m2 = Ma + Mb + dlt * dlt * (na * (nb / nt));
                    }
                    const float rstd = rsqrtf(m2 / float(a.C_out) + a.eps);
                    if (a.tma_store) {
                        OutT* ostage = reinterpret_cast<OutT*>(base + a.o_off) + (warp - kWarpEpi0) * (2 * 32 * 32);
                        for (int j0 = c_lo; j0 < c_hi; j0 += 32) {
                            float v[32];
                            tmem_load32(tb + uint32_t(j0), v);
                            ln_affine_gelu(v, s_bias + j0, s_gamma + j0, s_beta + j0, mean, rstd, a.gelu != 0);
                            // the store issued from this buffer two chunks ago has read it
                            if (lane == 0) tma_store_wait_read_le1();
                            __syncwarp();
                            OutT* ob = ostage + obuf * (32 * 32);
#pragma unroll
                            for (int i = 0; i < 32; ++i) store_out(ob + i * 32 + lane, v[i]);
                            fence_async_shared();
                            __syncwarp();
                            if (lane == 0)
                                tma_store_3d(&tm_y, smem_u32(ob), un.row0 + q * 32, co_base + j0, un.n);
                            obuf ^= 1;
                        }
                    } else {
                        OutT* dst = y + ((long long)un.n * a.C_out + co_base) * a.T_out + row;
                        for (int j0 = c_lo; j0 < c_hi; j0 += 32) {
                            float v[32];
                            tmem_load32(tb + uint32_t(j0), v);
                            ln_affine_gelu(v, s_bias + j0, s_gamma + j0, s_beta + j0, mean, rstd, a.gelu != 0);
                            if (row_ok) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (j0 + i < c_hi) store_out(dst + (long long)(j0 + i) * a.T_out, v[i]);
                            }
                        }
                    }
                } else {
                    // ------------------------------------------------ fused GroupNorm (conv mode)
                    // The CTAs of one (sample, channel block) together cover all T_out steps. Each
                    // takes the (mean, M2) of every group over its tile from one sweep of TMEM, the
                    // statistics are exchanged (global memory across a cooperative grid, or distributed
                    // shared memory inside a cluster) and merged, and each CTA normalizes its tile from
                    // TMEM and stores it once, straight from registers.
                    const int co_base = un.cbu * a.BN;
                    const int ncols = min(a.BN, a.C_out - co_base);
                    const int cpg = a.cpg;
                    const int ngroups = (ncols + cpg - 1) / cpg;
                    const int nvalid_t = min(128, a.T_out - un.row0);
                    const int tt = un.row0 / 128;
                    const int P = a.n_t_tiles;  // tiles (CTAs) whose statistics make up one group
                    // this warp's column range [c_lo, c_hi): the kEpiW / 4 warps of a lane quarter take
                    // one part each (whole 32-column chunks but the last)
                    constexpr int kParts = kEpiW / 4;
                    const int part = ((ncols + kParts - 1) / kParts + 31) / 32 * 32;
                    const int c_lo = min(eg * part, ncols);
                    const int c_hi = min(c_lo + part, ncols);
                    // grid exchange: per (sample, channel block, time tile, group) two 64-bit words,
                    // (mean | epoch) and (M2 | epoch), one epoch step per launch (the weight pack
                    // zeroes them); this launch's epoch was read before the accumulator wait
                    const size_t slot0 = size_t(un.n * a.n_cb + un.cbu) * a.n_t_tiles;
                    unsigned long long* gx_me = a.gx + (slot0 + tt) * size_t(a.gstride) * 2;
                    const unsigned target = gx_target;
                    float* red_mean = epi;         // [4][256] per lane quarter and run: mean of y over the run
                    float* red_m2 = epi + 1024;    // [4][256] ... and its M2
                    float* part_mu = epi + 2048;   // [256] this CTA's group means (cluster); peers' means (grid)
                    float* colscale = epi + 2304;  // [256]
                    float* colshift = epi + 2560;  // [256]
                    float* gmean = epi + 2816;     // [256] group mean over all CTAs
                    float* grstd = epi + 3328;     // [256] group 1/sqrt(var + eps)
                    float* part_m2 = epi + 3584;   // [256] this CTA's group M2 (cluster); peers' M2 (grid)
                    const uint32_t tb = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(256 * ab);
                    const int nvalid_w = min(32, max(0, nvalid_t - q * 32));
                    // Every loop over groups or columns below has one iteration at most per thread
                    // (ngroups <= 256 <= kEpiT), so its divisions are taken here, before the wait.
                    static_assert(!kFusedGN || kEpiT >= 256, "one group and one column per epilogue thread");
                    const int run = a.sub > 0 ? a.sub : 1;
                    float qn[4];  // count of one run's entry in lane quarter q2
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) qn[q2] = float(min(32, max(0, nvalid_t - q2 * 32)) * run);
                    const int g_me = er;  // this thread's group in the merge
                    const int j_lo = g_me * cpg / run, j_hi = (min(ncols, g_me * cpg + cpg) + run - 1) / run;
                    const int g_col = er < ncols ? er / cpg : 0;  // group of this thread's column
                    int x_g = er / P, x_p = er - (er / P) * P;     // (group, peer) of the exchange pair
                    if (!acc_wait()) break;
                    gn_run_stats_any(a.sub, tb, c_lo, c_hi, lane < nvalid_w, nvalid_w, red_mean, red_m2, q, lane);
                    named_bar_sync(1, kEpiT);
                    // This CTA's (mean, M2) per group from its (run, lane quarter) entries by the
                    // parallel-axis formula: the count-weighted mean, then the entries' M2 plus each
                    // entry's count times the squared distance of its mean from the group mean.
                    if (g_me < ngroups) {
                        const int g = g_me;
                        float n_tot = 0.f, s = 0.f;
                        for (int j = j_lo; j < j_hi; ++j) {
#pragma unroll
                            for (int q2 = 0; q2 < 4; ++q2) {
                                n_tot += qn[q2];
                                s = fmaf(qn[q2], red_mean[q2 * 256 + j], s);  // (qn = 0: the entry is finite)
                            }
                        }
                        const float gmu = n_tot > 0.f ? __fdividef(s, n_tot) : 0.f;
                        float gm2 = 0.f;
                        for (int j = j_lo; j < j_hi; ++j) {
#pragma unroll
                            for (int q2 = 0; q2 < 4; ++q2) {
                                const float d = red_mean[q2 * 256 + j] - gmu;
                                gm2 += fmaf(qn[q2] * d, d, red_m2[q2 * 256 + j]);
                            }
                        }
                        if (EPI == kEpiGridGN) {
                            // (testing aid: the first CTA withholds its words, so its sample's waits run out)
                            const bool withhold = a.test_stall && (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
                            const unsigned long long tag = (unsigned long long)target << 32;
                            if (!withhold) {
                                st_relaxed_gpu_u64(gx_me + 2 * g, tag | __float_as_uint(gmu));
                                st_relaxed_gpu_u64(gx_me + 2 * g + 1, tag | __float_as_uint(gm2));
                            }
                        } else {
                            part_mu[g] = gmu;
                            part_m2[g] = gm2;
                        }
                    }
                    if (EPI == kEpiClusterGN) {
                        // partials of every CTA in the cluster become visible
                        cluster_sync_all();
                        mid_sync_done = true;
                        for (int g = er; g < ngroups; g += kEpiT) {
                            const float cw = float(min(ncols, g * cpg + cpg) - g * cpg);
                            float gn = 0.f, gmu = 0.f, gm2 = 0.f;
                            const uint32_t pmu = smem_u32(part_mu + g), pm2 = smem_u32(part_m2 + g);
                            for (int rk = 0; rk < P; ++rk) {
                                const float cnt = cw * float(min(128, a.T_out - rk * 128));
                                chan_merge(gn, gmu, gm2, cnt, ld_shared_cluster_f32(map_shared_rank(pmu, uint32_t(rk))),
                                           ld_shared_cluster_f32(map_shared_rank(pm2, uint32_t(rk))));
                            }
                            gmean[g] = gmu;
                            grstd[g] = rsqrtf((gn > 0.f ? gm2 / gn : 0.f) + a.eps);
                        }
                    } else {
                        // Each (group, peer tile) pair has a thread that waits (bounded) for that peer's
                        // two words: a word carries its value and the epoch in one 64-bit access, so a
                        // word showing this launch's epoch holds this launch's value, with no fence on
                        // either side, and all peers' words are in flight at once. The P threads of a
                        // group then merge by shuffles (P a power of two, all pairs in one pass), or one
                        // thread per group merges them in peer order. Either way every CTA of the sample
                        // merges the same values in the same order and normalizes with identical bits.
                        const unsigned long long* gq = a.gx + slot0 * size_t(a.gstride) * 2;
                        const size_t tile_words = size_t(a.gstride) * 2;
                        const bool tree = (P & (P - 1)) == 0 && P <= 32 && ngroups * P <= kEpiT;
                        const bool in_smem = ngroups * P <= 256;  // peers' words kept for the serial merge
                        const uint64_t t0 = global_timer_ns();
                        for (int base = 0; base < ngroups * P; base += kEpiT) {  // uniform over the warp
                            const int idx = base + er;
                            if (base > 0) {
                                x_g = idx / P;
                                x_p = idx - x_g * P;
                            }
                            const int g = x_g, p = x_p;
                            unsigned long long wmu = 0ull, wm2 = 0ull;
                            if (g < ngroups) {
                                const unsigned long long* w = gq + size_t(p) * tile_words + 2 * g;
                                for (uint32_t it = 0;; ++it) {
                                    wmu = ld_relaxed_gpu_u64(w);
                                    wm2 = ld_relaxed_gpu_u64(w + 1);
                                    if ((unsigned(wmu >> 32) == target && unsigned(wm2 >> 32) == target) || *abort_flag)
                                        break;
                                    if ((it & 15u) == 15u && global_timer_ns() - t0 > kWaitLimitNs) {
                                        if (atomicCAS(a.status, 0, 6) == 0) {
                                            atomicExch(a.status + 1, kWaitGridPeers);
                                            atomicExch(a.status + 2, int(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)));
                                        }
                                        *abort_flag = 1;
                                        break;
                                    }
                                }
                            }
                            if (tree) {
                                float n = 0.f, mu = 0.f, m2 = 0.f;
                                if (g < ngroups) {
                                    n = float(min(ncols, g * cpg + cpg) - g * cpg) * float(min(128, a.T_out - p * 128));
                                    mu = __uint_as_float(unsigned(wmu));
                                    m2 = __uint_as_float(unsigned(wm2));
                                }
                                for (int d = 1; d < P; d <<= 1) stats_merge_xor(n, mu, m2, d, lane);
                                if (g < ngroups && p == 0) {
                                    gmean[g] = mu;
                                    grstd[g] = rsqrtf(__fdividef(m2, n) + a.eps);
                                }
                            } else if (in_smem && g < ngroups) {
                                part_mu[idx] = __uint_as_float(unsigned(wmu));
                                part_m2[idx] = __uint_as_float(unsigned(wm2));
                            }
                        }
                        if (!tree) {
                            named_bar_sync(1, kEpiT);
                            for (int g = er; g < ngroups; g += kEpiT) {
                                const float cw = float(min(ncols, g * cpg + cpg) - g * cpg);
                                float n = 0.f, mu = 0.f, m2 = 0.f;
                                for (int p = 0; p < P; ++p) {
                                    float pm, pv;
                                    if (in_smem) {
                                        pm = part_mu[g * P + p];
                                        pv = part_m2[g * P + p];
                                    } else {  // more pairs than fit: read the words again (they hold this
                                              // launch's values by now)
                                        const unsigned long long* w = gq + size_t(p) * tile_words + 2 * g;
                                        pm = __uint_as_float(unsigned(ld_relaxed_gpu_u64(w)));
                                        pv = __uint_as_float(unsigned(ld_relaxed_gpu_u64(w + 1)));
                                    }
                                    stats_merge(n, mu, m2, cw * float(min(128, a.T_out - p * 128)), pm, pv);
                                }
                                gmean[g] = mu;
                                grstd[g] = rsqrtf(m2 / n + a.eps);
                            }
                        }
                    }
                    named_bar_sync(1, kEpiT);
                    if (er < 256) {
                        const int col = er;
                        // colscale / colshift hold gamma / beta (staged before the mainloop)
                        float sc = 0.f, sh = 0.f;
                        if (col < ncols) {
                            const int g = g_col;
                            sc = grstd[g] * colscale[col];
                            sh = colshift[col] - gmean[g] * sc;  // (gmean: the mean of y = acc)
                        }
                        colscale[col] = sc;
                        colshift[col] = sh;
                    }
                    named_bar_sync(1, kEpiT);
                    // Normalize from TMEM and store straight from registers: the 32 lanes of a warp hold
                    // 32 consecutive time steps of a channel, so every store writes 128 contiguous bytes
                    // (64 for bf16). Two 32-column TMEM loads share one wait.
                    // (GELU or not is decided once, outside the unrolled loops, so the loop without it
                    // is compact straight-line code)
                    OutT* ybase = y + ((long long)un.n * a.C_out + co_base) * a.T_out + row;
                    if (a.gelu) gn_normalize_store<true>(tb, c_lo, c_hi, colscale, colshift, ybase, a.T_out, row_ok);
                    else gn_normalize_store<false>(tb, c_lo, c_hi, colscale, colshift, ybase, a.T_out, row_ok);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader(i_accempty + ab);
                if (threadIdx.x == kWarpEpi0 * 32) prog[4] = lt + 1;
            }
            if (EPI == kEpiClusterGN && !mid_sync_done) cluster_sync_all();
            if ((EPI == kEpiLN || EPI == kEpiLNX) && a.tma_store && lane == 0) tma_store_wait_all();
        }
    }

    if (EPI == kEpiClusterGN) {
        // Every thread of every CTA takes part in both cluster barriers, whatever happened above:
        // the epilogue's first one publishes the partial statistics (the other warps, or an
        // epilogue that gave up, arrive for it here), the second keeps each CTA's shared memory
        // alive until its peers have read it.
        if (warp < kWarpEpi0 || warp >= kWarpEpi0 + kEpiW) cluster_sync_all();
        cluster_sync_all();
    }
    __syncwarp();
    // A cluster leaves together: a pair leader's MMAs read the peer's shared memory and write its
    // TMEM, the peer's copies and arrivals target the leader's barriers, and exchanging epilogues
    // write into each other's shared memory.
    if (PAIR || kClusterX) cluster_sync_all();
    else __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, uint32_t(a.tmem_cols));
        else tmem_dealloc(tmem_base, uint32_t(a.tmem_cols));
    }
}

template <bool LINEAR, bool BF16, typename OutT, int EPI, bool PAIR>
cudaError_t launch_one(const Plan& pl, const TcArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                       const CUtensorMap& tm_y, int num_sms, cudaStream_t stream) {
    auto kern = tc_conv_kernel<LINEAR, BF16, OutT, EPI, PAIR>;
    // Host work per launch stays small: the shared-memory attribute and the resident-cluster count
    // are set / queried once per device and shared-memory size (per kernel instantiation).
    constexpr int kMaxDev = 64;
    static std::atomic<int> smem_set[kMaxDev];
    static std::atomic<long long> clusters_cached[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDev;
    if (!cacheable || smem_set[dev].load(std::memory_order_acquire) < pl.smem_bytes) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
        if (e != cudaSuccess) return e;
        if (cacheable) {
            int cur = smem_set[dev].load();
            while (cur < pl.smem_bytes && !smem_set[dev].compare_exchange_weak(cur, pl.smem_bytes)) {}
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = size_t(pl.smem_bytes);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (EPI == kEpiClusterGN) {
        cfg.gridDim = dim3(unsigned(a.n_t_tiles), unsigned(a.n_cb / a.cb_per_unit), unsigned(a.N));
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(a.n_t_tiles);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
    } else if (EPI == kEpiGridGN) {
        // every CTA of a sample waits for its peers: all CTAs must be resident at once
        cfg.gridDim = dim3(unsigned(a.n_t_tiles), unsigned(a.n_cb / a.cb_per_unit), unsigned(a.N));
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else if (PAIR || EPI == kEpiLNX) {
        // persistent clusters of two: as many as can be resident at once
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(unsigned(num_sms & ~1), 1, 1);
        int max_clusters = 0;
        const long long cached = cacheable ? clusters_cached[dev].load(std::memory_order_acquire) : 0;
        if (cached != 0 && int(cached >> 32) == pl.smem_bytes) {
            max_clusters = int(cached & 0xffffffff);
        } else {
            e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
            if (e != cudaSuccess) return e;
            if (cacheable) clusters_cached[dev].store((static_cast<long long>(pl.smem_bytes) << 32) | max_clusters);
        }
        if (max_clusters < 1) return cudaErrorInvalidConfiguration;
        const int pairs = a.n_units < max_clusters ? a.n_units : max_clusters;
        cfg.gridDim = dim3(unsigned(2 * pairs), 1, 1);
    } else {
        const int grid = a.n_units < num_sms ? a.n_units : num_sms;
        cfg.gridDim = dim3(unsigned(grid), 1, 1);
        cfg.numAttrs = 0;
    }
    // Programmatic dependent launch: the CTAs set up while the previous kernel (usually the weight
    // pack) finishes. If the driver refuses the combination, launch without it from then on.
    static std::atomic<int> pdl_refused{0};
    if (!pdl_refused.load(std::memory_order_relaxed)) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs += 1;
        e = cudaLaunchKernelEx(&cfg, kern, a, tm_a, tm_b, tm_y);
        if (e == cudaSuccess) return e;
        cudaGetLastError();
        pdl_refused.store(1);
        cfg.numAttrs -= 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a, tm_a, tm_b, tm_y);
}

}  // namespace

cudaError_t launch_tc(const Plan& pl, const TcArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                      const CUtensorMap& tm_y, bool linear, int epilogue, bool out_bf16, int num_sms,
                      cudaStream_t stream) {
#define C1N_LAUNCH(L, B, O, E, P) launch_one<L, B, O, E, P>(pl, a, tm_a, tm_b, tm_y, num_sms, stream)
#define C1N_LAUNCH2(L, B, O, E) (pl.pair ? C1N_LAUNCH(L, B, O, E, true) : C1N_LAUNCH(L, B, O, E, false))
    if (linear) {
        if (epilogue == kEpiRowGN) {
            if (pl.bf16) return C1N_LAUNCH2(true, true, __nv_bfloat16, kEpiRowGN);
            return C1N_LAUNCH2(true, false, float, kEpiRowGN);
        }
        if (pl.bf16 && out_bf16) return C1N_LAUNCH2(true, true, __nv_bfloat16, kEpiDirect);
        if (pl.bf16) return C1N_LAUNCH2(true, true, float, kEpiDirect);
        return C1N_LAUNCH2(true, false, float, kEpiDirect);
    }
    if (epilogue == kEpiLN) {
        if (pl.bf16) return C1N_LAUNCH2(false, true, __nv_bfloat16, kEpiLN);
        return C1N_LAUNCH2(false, false, float, kEpiLN);
    }
    if (epilogue == kEpiLNX) {
        if (pl.bf16) return C1N_LAUNCH(false, true, __nv_bfloat16, kEpiLNX, false);
        return C1N_LAUNCH(false, false, float, kEpiLNX, false);
    }
    if (epilogue == kEpiClusterGN) {
        if (pl.bf16) return C1N_LAUNCH(false, true, __nv_bfloat16, kEpiClusterGN, false);
        return C1N_LAUNCH(false, false, float, kEpiClusterGN, false);
    }
    if (epilogue == kEpiGridGN) {
        if (pl.bf16) return C1N_LAUNCH(false, true, __nv_bfloat16, kEpiGridGN, false);
        return C1N_LAUNCH(false, false, float, kEpiGridGN, false);
    }
    if (epilogue == kEpiDirectStats) {
        // raw fp32 tiles plus partial statistics (two-pass plans)
        if (pl.bf16) return C1N_LAUNCH2(false, true, float, kEpiDirectStats);
        return C1N_LAUNCH2(false, false, float, kEpiDirectStats);
    }
    if (pl.bf16) {
        if (out_bf16) return C1N_LAUNCH2(false, true, __nv_bfloat16, kEpiDirect);
        return C1N_LAUNCH2(false, true, float, kEpiDirect);
    }
    return C1N_LAUNCH2(false, false, float, kEpiDirect);
#undef C1N_LAUNCH2
#undef C1N_LAUNCH
}

}  // namespace c1n

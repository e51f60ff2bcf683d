// SIMT fp32 check path and the memory-bound passes shared by every path:
//   * simt_conv       — direct convolution from shared-memory tiles (fp32 FMA);
//   * gn_stats        — GroupNorm mean / rstd per (n, group), two passes over the group;
//   * ln_stats        — channel-LayerNorm mean / rstd per (n, t), two passes over channels;
//   * gn_merge, ln_merge — the same statistics from the partial (mean, M2) sets that the
//                       tensor-core epilogue of a two-pass plan writes (Chan's merge);
//   * normalize       — (raw - mean) * rstd * gamma + beta, then GELU, float4 when rows allow it;
//   * rowmin          — min (and lowest argmin) over channels of the normalized values per (n, t);
//   * broadcast       — y[n][c][t] = rowmin[n][t] + bias2[c];
//   * pack_weights    — w[co][ci][kk] -> wp[kk][co][ci_pad] (tf32-rounded for fp32 data).
// Operator definitions: Kimi-K2.6 l2_p35 page (Conv1d + GroupNorm), l2_p75 page (row-min + bias),
// l1_p5 page (causal padding), l2_p3 page (LayerNorm with affine, exact GELU).
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "c1n_internal.h"
#include "c1n_math.cuh"
#include "sm100_ptx.cuh"

namespace c1n {
namespace {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }



// ------------------------------------------------------------------------------ SIMT conv

constexpr int kSimtCo = 64, kSimtT = 64, kSimtCi = 8, kSimtThreads = 256;

struct SimtConvArgs {
    int N, C_in, C_out, T, T_out, k, stride, pad_left, dilation, span, gelu;
};

// One CTA computes a 64 (co) x 64 (t) output tile; each thread 4 x 4 outputs.
template <typename InT, typename OutT>
__global__ void __launch_bounds__(kSimtThreads) simt_conv_kernel(SimtConvArgs a, const InT* __restrict__ x,
                                                                 const InT* __restrict__ w,
                                                                 const float* __restrict__ b, OutT* __restrict__ out) {
    extern __shared__ float smem[];
    float* xs = smem;                          // [kSimtCi][span]
    float* ws = smem + kSimtCi * a.span;       // [kSimtCo][kSimtCi][k]
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int t0 = blockIdx.x * kSimtT, co0 = blockIdx.y * kSimtCo, n = blockIdx.z;
    const long long in_start = (long long)t0 * a.stride - a.pad_left;
    float acc[4][4] = {};
    for (int ci0 = 0; ci0 < a.C_in; ci0 += kSimtCi) {
        for (int idx = threadIdx.x; idx < kSimtCi * a.span; idx += kSimtThreads) {
            const int c = idx / a.span, p = idx % a.span;
            const int ci = ci0 + c;
            const long long pos = in_start + p;
            float v = 0.f;
            if (ci < a.C_in && pos >= 0 && pos < a.T) v = to_f32(x[((long long)n * a.C_in + ci) * a.T + pos]);
            xs[idx] = v;
        }
        const int wk = kSimtCi * a.k;
        for (int idx = threadIdx.x; idx < kSimtCo * wk; idx += kSimtThreads) {
            const int col = idx / wk, rem = idx % wk;
            const int c = rem / a.k, kk = rem % a.k;
            const int co = co0 + col, ci = ci0 + c;
            float v = 0.f;
            if (co < a.C_out && ci < a.C_in) v = to_f32(w[((long long)co * a.C_in + ci) * a.k + kk]);
            ws[idx] = v;
        }
        __syncthreads();
        for (int c = 0; c < kSimtCi; ++c) {
            for (int kk = 0; kk < a.k; ++kk) {
                float wv[4], xv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) wv[i] = ws[((ty + 16 * i) * kSimtCi + c) * a.k + kk];
#pragma unroll
                for (int j = 0; j < 4; ++j) xv[j] = xs[c * a.span + (tx + 16 * j) * a.stride + kk * a.dilation];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(wv[i], xv[j], acc[i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int co = co0 + ty + 16 * i;
        if (co >= a.C_out) continue;
        const float bias = b ? b[co] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = t0 + tx + 16 * j;
            if (t >= a.T_out) continue;
            float v = acc[i][j] + bias;
            if (a.gelu) v = gelu_erf(v);
            store_out(out + ((long long)n * a.C_out + co) * a.T_out + t, v);
        }
    }
}

// ------------------------------------------------------------------------------ block reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the CTA (blockDim.x multiple of 32, <= 1024); result broadcast to every thread.
__device__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < nw; ++i) s += red[i];
    return s;
}

// GroupNorm statistics: the channels of group g are contiguous rows, so the group is one
// contiguous span of cpg * T_out values, read once: sums of (v - shift) and of its square with the
// group's first value as the shift, then mean = shift + S1/n and variance = (S2 - S1^2/n) / n.
__global__ void __launch_bounds__(512) gn_stats_kernel(const float* __restrict__ raw, float2* __restrict__ stats,
                                                       int C, long long T_out, int G, float eps) {
    __shared__ float red[32];
    const int g = blockIdx.x, n = blockIdx.y;
    const long long cpg = C / G;
    const long long cnt = cpg * T_out;
    const float* src = raw + ((long long)n * C + g * cpg) * T_out;
    const float shift = __ldg(src);
    float s1 = 0.f, s2 = 0.f;
    if ((cnt & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const float4* s4 = reinterpret_cast<const float4*>(src);
        const long long n4 = cnt / 4;
#pragma unroll 4
        for (long long i = threadIdx.x; i < n4; i += blockDim.x) {
            const float4 v = __ldg(s4 + i);
            const float d0 = v.x - shift, d1 = v.y - shift, d2 = v.z - shift, d3 = v.w - shift;
            s1 += (d0 + d1) + (d2 + d3);
            s2 = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, s2))));
        }
    } else {
        for (long long i = threadIdx.x; i < cnt; i += blockDim.x) {
            const float d = src[i] - shift;
            s1 += d;
            s2 = fmaf(d, d, s2);
        }
    }
    s1 = block_sum(s1, red);
    s2 = block_sum(s2, red);
    const float inv = 1.f / (float)cnt;
    const float m1 = s1 * inv;
    const float var = fmaxf(s2 * inv - m1 * m1, 0.f);
    if (threadIdx.x == 0) stats[(long long)n * G + g] = make_float2(shift + m1, rsqrtf(var + eps));
}

// Chan's pairwise update of the moments (count n, mean mu, M2) with another set.
__device__ __forceinline__ void merge_moments(float& n, float& mu, float& m2, float nb, float mub, float m2b) {
    if (nb <= 0.f) return;
    const float nn = n + nb;
    const float d = mub - mu;
    const float f = nb / nn;
    mu += d * f;
    m2 += m2b + d * d * n * f;
    n = nn;
}

// GroupNorm statistics from the tensor-core epilogue's partials: one warp per (n, g); lane l
// merges the 128-step tiles l, l + 32, ... in order, then the 32 lane results are merged in a
// butterfly. Tile tt holds cpg * min(128, T_out - 128 tt) values.
__global__ void __launch_bounds__(256) gn_merge_kernel(const float2* __restrict__ part, float2* __restrict__ stats,
                                                       int NG, int n_tiles, int cpg, long long T_out, float eps) {
    const int lane = threadIdx.x & 31;
    const long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (i >= NG) return;
    float n = 0.f, mu = 0.f, m2 = 0.f;
    for (int tt = lane; tt < n_tiles; tt += 32) {
        const float2 v = __ldg(part + i * n_tiles + tt);
        const long long rows = T_out - 128LL * tt;
        merge_moments(n, mu, m2, float(cpg) * float(rows < 128 ? rows : 128), v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float nb = __shfl_xor_sync(0xffffffffu, n, o);
        const float mub = __shfl_xor_sync(0xffffffffu, mu, o);
        const float m2b = __shfl_xor_sync(0xffffffffu, m2, o);
        merge_moments(n, mu, m2, nb, mub, m2b);
    }
    if (lane == 0) stats[i] = make_float2(mu, rsqrtf((n > 0.f ? m2 / n : 0.f) + eps));
}

// Channel-LayerNorm statistics from the epilogue's partials: one thread per (n, t) merges the
// n_cb channel blocks (block cb holds min(BN, C - cb BN) channels); coalesced over t.
__global__ void __launch_bounds__(256) ln_merge_kernel(const float2* __restrict__ part, float2* __restrict__ stats,
                                                       int N, int C, int BN, int n_cb, long long T_out, float eps) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)N * T_out) return;
    const long long n = i / T_out, t = i - n * T_out;
    float cnt = 0.f, mu = 0.f, m2 = 0.f;
    for (int cb = 0; cb < n_cb; ++cb) {
        const float2 v = __ldg(part + (n * n_cb + cb) * T_out + t);
        const int c = C - cb * BN;
        merge_moments(cnt, mu, m2, float(c < BN ? c : BN), v.x, v.y);
    }
    stats[i] = make_float2(mu, rsqrtf(m2 / cnt + eps));
}

// Channel-LayerNorm statistics per (n, t), read once. A CTA covers 32 * VEC consecutive t of one
// sample; lane l of every warp owns t0 + VEC*l .. + VEC-1 (coalesced over t) and warp w the
// channels c = w, w + 8, ...; sums of (v - shift) and of its square with the channel-0 value as the
// shift, combined over the 8 warps in shared memory.
template <int VEC>
__global__ void __launch_bounds__(256) ln_stats_kernel(const float* __restrict__ raw, float2* __restrict__ stats,
                                                       int C, long long T_out, float eps) {
    __shared__ float part[2][8][32 * VEC];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int n = blockIdx.y;
    const long long t0 = (long long)blockIdx.x * (32 * VEC) + (long long)lane * VEC;
    const bool ok = t0 < T_out;  // with VEC = 4, T_out is a multiple of 4
    const float* src = raw + (long long)n * C * T_out + (ok ? t0 : 0);
    float sh[VEC], s1[VEC], s2[VEC];
    if (VEC == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src));
        sh[0] = v.x; sh[1] = v.y; sh[2] = v.z; sh[3] = v.w;
    } else {
        sh[0] = __ldg(src);
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) s1[j] = s2[j] = 0.f;
#pragma unroll 8
    for (int c = w; c < C; c += 8) {
        float v[VEC];
        if (VEC == 4) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(src + (long long)c * T_out));
            v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else {
            v[0] = __ldg(src + (long long)c * T_out);
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float d = v[j] - sh[j];
            s1[j] += d;
            s2[j] = fmaf(d, d, s2[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        part[0][w][lane * VEC + j] = s1[j];
        part[1][w][lane * VEC + j] = s2[j];
    }
    __syncthreads();
    for (int k = threadIdx.x; k < 32 * VEC; k += blockDim.x) {
        const long long t = (long long)blockIdx.x * (32 * VEC) + k;
        if (t >= T_out) continue;
        float a1 = 0.f, a2 = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) {
            a1 += part[0][ww][k];
            a2 += part[1][ww][k];
        }
        const float inv = 1.f / (float)C;
        const float m1 = a1 * inv;
        const float var = fmaxf(a2 * inv - m1 * m1, 0.f);
        const float shift = raw[(long long)n * C * T_out + t];
        stats[(long long)n * T_out + t] = make_float2(shift + m1, rsqrtf(var + eps));
    }
}

struct NormArgs {
    int N, C;
    long long T_out;
    int norm;   // 0 none, 1 group, 2 channel layer
    int cpg;    // channels per group (norm == 1)
    int G;
    int gelu;
};

__device__ __forceinline__ float2 stat_of(const NormArgs& a, const float2* stats, int n, int c, long long t) {
    if (a.norm == 1) return stats[(long long)n * a.G + c / a.cpg];
    if (a.norm == 2) return stats[(long long)n * a.T_out + t];
    return make_float2(0.f, 1.f);
}

// Normalize + affine + optional GELU. Grid: x over column chunks of a row, y over rows (n, c)
// in a grid-stride loop; rows of T_out contiguous values; float4 when T_out % 4 == 0.
template <typename OutT, bool VEC>
// `raw` and `y` may be the same buffer (in-place fp32 normalization): no __restrict__ on them.
__global__ void __launch_bounds__(256) normalize_kernel(NormArgs a, const float* raw,
                                                        const float2* __restrict__ stats,
                                                        const float* __restrict__ gamma,
                                                        const float* __restrict__ beta, OutT* y) {
    const long long rows = (long long)a.N * a.C;
    for (long long row = blockIdx.y; row < rows; row += gridDim.y) {
        const int n = (int)(row / a.C), c = (int)(row % a.C);
        const float ga = gamma ? gamma[c] : 1.f, be = beta ? beta[c] : 0.f;
        const float* src = raw + row * a.T_out;
        OutT* dst = y + row * a.T_out;
        if (VEC) {
            const long long n4 = a.T_out / 4;
            for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
                 i += (long long)gridDim.x * blockDim.x) {
                float4 v = reinterpret_cast<const float4*>(src)[i];
                float r[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 st = stat_of(a, stats, n, c, 4 * i + j);
                    float z = (r[j] - st.x) * st.y * ga + be;
                    if (a.gelu) z = gelu_erf(z);
                    r[j] = z;
                }
                if constexpr (sizeof(OutT) == 4) {
                    reinterpret_cast<float4*>(dst)[i] = make_float4(r[0], r[1], r[2], r[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) store_out(dst + 4 * i + j, r[j]);
                }
            }
        } else {
            for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < a.T_out;
                 t += (long long)gridDim.x * blockDim.x) {
                const float2 st = stat_of(a, stats, n, c, t);
                float z = (src[t] - st.x) * st.y * ga + be;
                if (a.gelu) z = gelu_erf(z);
                store_out(dst + t, z);
            }
        }
    }
}

// Normalize + affine + optional GELU, eight consecutive elements of a row per thread (two 16-byte
// loads; one 16- or two 16-byte stores), for rows whose length is a multiple of 8 and 16-byte
// aligned buffers. Grid: x over 2048-element segments of a row, y over rows (grid-stride).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}

template <typename OutT, int NORM, bool GELU>
__global__ void __launch_bounds__(256) normalize8_kernel(NormArgs a, const float* raw,
                                                         const float2* __restrict__ stats,
                                                         const float* __restrict__ gamma,
                                                         const float* __restrict__ beta, OutT* y) {
    const long long rows = (long long)a.N * a.C;
    const long long per_row = a.T_out / 8;
    for (long long row = blockIdx.y; row < rows; row += gridDim.y) {
        const int n = (int)(row / a.C), c = (int)(row % a.C);
        const float ga = gamma ? __ldg(gamma + c) : 1.f, be = beta ? __ldg(beta + c) : 0.f;
        float2 gs = make_float2(0.f, 1.f);
        if (NORM == 1) gs = __ldg(stats + (long long)n * a.G + c / a.cpg);
        const float4* src = reinterpret_cast<const float4*>(raw + row * a.T_out);
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < per_row;
             i += (long long)gridDim.x * blockDim.x) {
            const float4 v0 = src[2 * i], v1 = src[2 * i + 1];
            float r[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            if (NORM == 2) {
                const float4* st4 = reinterpret_cast<const float4*>(stats + (long long)n * a.T_out + 8 * i);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 q = __ldg(st4 + k);  // (mean, rstd) of two consecutive t
                    r[2 * k] = fmaf((r[2 * k] - q.x) * q.y, ga, be);
                    r[2 * k + 1] = fmaf((r[2 * k + 1] - q.z) * q.w, ga, be);
                }
            } else {
                const float sc = gs.y * ga, of = be - gs.x * gs.y * ga;
                const uint64_t sp = f2_pack(sc, sc), op = f2_pack(of, of);
#pragma unroll
                for (int j = 0; j < 8; j += 2) f2_unpack(f2_fma(f2_pack(r[j], r[j + 1]), sp, op), r[j], r[j + 1]);
            }
            if (GELU) {
#pragma unroll
                for (int j = 0; j < 8; j += 2) f2_unpack(gelu_erf2(f2_pack(r[j], r[j + 1])), r[j], r[j + 1]);
            }
            if constexpr (sizeof(OutT) == 4) {
                float4* dst = reinterpret_cast<float4*>(y + row * a.T_out);
                dst[2 * i] = make_float4(r[0], r[1], r[2], r[3]);
                dst[2 * i + 1] = make_float4(r[4], r[5], r[6], r[7]);
            } else {
                uint4* dst = reinterpret_cast<uint4*>(y + row * a.T_out);
                dst[i] = make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                                    pack_bf16x2(r[6], r[7]));
            }
        }
    }
}

// Channel-LayerNorm form of the above: statistics are per (n, t), so a thread keeps the (mean,
// rstd) of its eight consecutive t in registers and walks a block of 64 channels (rows) of one
// sample. Grid: x over 2048-step segments, y over 64-channel blocks, z over samples.
template <typename OutT, bool GELU>
__global__ void __launch_bounds__(256) normalize8_ln_kernel(NormArgs a, const float* raw,
                                                            const float2* __restrict__ stats,
                                                            const float* __restrict__ gamma,
                                                            const float* __restrict__ beta, OutT* y) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // 8-step chunk index
    if (i >= a.T_out / 8) return;
    const int n = blockIdx.z;
    float mu[8], rs[8];
    const float4* st4 = reinterpret_cast<const float4*>(stats + (long long)n * a.T_out + 8 * i);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 q = __ldg(st4 + k);
        mu[2 * k] = q.x;
        rs[2 * k] = q.y;
        mu[2 * k + 1] = q.z;
        rs[2 * k + 1] = q.w;
    }
    const int c_end = min(a.C, (int)(blockIdx.y + 1) * 64);
    // (four rows' loads in flight per thread; the raw tile is read once and y written once, so both
    // stream past L1 and are marked first to evict from L2)
#pragma unroll 4
    for (int c = blockIdx.y * 64; c < c_end; ++c) {
        const long long row = (long long)n * a.C + c;
        const float ga = gamma ? __ldg(gamma + c) : 1.f, be = beta ? __ldg(beta + c) : 0.f;
        const float4* src = reinterpret_cast<const float4*>(raw + row * a.T_out);
        const float4 v0 = __ldcs(src + 2 * i), v1 = __ldcs(src + 2 * i + 1);
        float r[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        const uint64_t gp = f2_pack(ga, ga), bp = f2_pack(be, be);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            uint64_t o = f2_fma(f2_mul(f2_sub(f2_pack(r[j], r[j + 1]), f2_pack(mu[j], mu[j + 1])),
                                       f2_pack(rs[j], rs[j + 1])), gp, bp);
            if (GELU) o = gelu_erf2(o);
            f2_unpack(o, r[j], r[j + 1]);
        }
        if constexpr (sizeof(OutT) == 4) {
            float4* dst = reinterpret_cast<float4*>(y + row * a.T_out);
            __stcs(dst + 2 * i, make_float4(r[0], r[1], r[2], r[3]));
            __stcs(dst + 2 * i + 1, make_float4(r[4], r[5], r[6], r[7]));
        } else {
            uint4* dst = reinterpret_cast<uint4*>(y + row * a.T_out);
            __stcs(dst + i, make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                                       pack_bf16x2(r[6], r[7])));
        }
    }
}

// Row-min over channels of the normalized values for one (n, t) per CTA; ties keep the lowest
// channel index.
__global__ void __launch_bounds__(256) rowmin_kernel(NormArgs a, const float* __restrict__ raw,
                                                     const float2* __restrict__ stats, const float* __restrict__ gamma,
                                                     const float* __restrict__ beta, float* __restrict__ rowmin,
                                                     int32_t* __restrict__ argmin) {
    __shared__ float sv[256];
    __shared__ int si[256];
    const long long t = blockIdx.x;
    const int n = blockIdx.y;
    float best = __int_as_float(0x7f800000);  // +inf
    int bi = 0x7fffffff;
    for (int c = threadIdx.x; c < a.C; c += blockDim.x) {
        const float2 st = stat_of(a, stats, n, c, t);
        const float ga = gamma ? gamma[c] : 1.f, be = beta ? beta[c] : 0.f;
        const float z = (raw[((long long)n * a.C + c) * a.T_out + t] - st.x) * st.y * ga + be;
        if (z < best) { best = z; bi = c; }
    }
    sv[threadIdx.x] = best;
    si[threadIdx.x] = bi;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) {
            const float ov = sv[threadIdx.x + s];
            const int oi = si[threadIdx.x + s];
            if (ov < sv[threadIdx.x] || (ov == sv[threadIdx.x] && oi < si[threadIdx.x])) {
                sv[threadIdx.x] = ov;
                si[threadIdx.x] = oi;
            }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        rowmin[(long long)n * a.T_out + t] = sv[0];
        if (argmin) argmin[(long long)n * a.T_out + t] = si[0];
    }
}

template <typename OutT>
__global__ void __launch_bounds__(256) broadcast_kernel(NormArgs a, const float* __restrict__ rowmin,
                                                        const float* __restrict__ bias2, OutT* __restrict__ y) {
    const long long total = (long long)a.N * a.C * a.T_out;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long t = e % a.T_out;
        const long long rc = e / a.T_out;
        const int c = (int)(rc % a.C), n = (int)(rc / a.C);
        store_out(y + e, rowmin[(long long)n * a.T_out + t] + bias2[c]);
    }
}

// T_out == 1 fast form: y[n][c] = rowmin[n] + bias2[c], float4 over c.
__global__ void __launch_bounds__(256) broadcast_rows_f32_kernel(int N, int C, const float* __restrict__ rowmin,
                                                                 const float* __restrict__ bias2, float* __restrict__ y) {
    const int c4 = C / 4;
    for (int n = blockIdx.y; n < N; n += gridDim.y) {
        const float m = rowmin[n];
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < c4; i += gridDim.x * blockDim.x) {
            const float4 bb = reinterpret_cast<const float4*>(bias2)[i];
            reinterpret_cast<float4*>(y + (long long)n * C)[i] = make_float4(m + bb.x, m + bb.y, m + bb.z, m + bb.w);
        }
    }
}

// Row-min finisher for the fused Linear epilogue: one CTA per row; the row's minimum (lowest channel
// on ties) over its per-block partials, then y[row][c] = min + bias2[c] (16-byte stores when the
// row length allows).
template <typename OutT>
__global__ void __launch_bounds__(256) rowmin_finish_kernel(int C, int n_cb, const float2* __restrict__ part,
                                                            const float* __restrict__ bias2, OutT* __restrict__ y,
                                                            int32_t* __restrict__ argmin) {
    __shared__ float sv[256];
    __shared__ int si[256];
    const int row = blockIdx.x;
    float best = __int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    for (int j = threadIdx.x; j < n_cb; j += blockDim.x) {
        const float2 pv = part[(size_t)row * n_cb + j];
        const int idx = __float_as_int(pv.y);
        if (pv.x < best || (pv.x == best && idx < bi)) { best = pv.x; bi = idx; }
    }
    sv[threadIdx.x] = best;
    si[threadIdx.x] = bi;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) {
            const float ov = sv[threadIdx.x + s];
            const int oi = si[threadIdx.x + s];
            if (ov < sv[threadIdx.x] || (ov == sv[threadIdx.x] && oi < si[threadIdx.x])) {
                sv[threadIdx.x] = ov;
                si[threadIdx.x] = oi;
            }
        }
        __syncthreads();
    }
    const float m = sv[0];
    if (threadIdx.x == 0 && argmin) argmin[row] = si[0];
    OutT* dst = y + (size_t)row * C;
    if (sizeof(OutT) == 4 && (C % 4) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(bias2) & 15) == 0) {
        for (int i = threadIdx.x; i < C / 4; i += blockDim.x) {
            const float4 b = reinterpret_cast<const float4*>(bias2)[i];
            reinterpret_cast<float4*>(dst)[i] = make_float4(m + b.x, m + b.y, m + b.z, m + b.w);
        }
    } else {
        for (int i = threadIdx.x; i < C; i += blockDim.x) store_out(dst + i, m + bias2[i]);
    }
}

// Weight pack: each thread walks (output channel co, input channel slot ci < ci_pad) slots, reads
// the k taps w[co][ci][0..k-1] and writes wp[kk][co][ci] for each tap, coalesced along ci (slots
// past C_in are zero). At most 2 CTAs of 128 threads per SM, no shared memory, at most 32
// registers: the conv kernel that follows (launched early through programmatic dependence; 480
// threads x 128 registers, ~224 KB of shared memory) fits on an SM beside them and stages x while
// the pack runs. fp32 weights are rounded to TF32; with tf32_mode 2 the TF32 tail w - tf32(w)
// goes to taps k..2k-1. Also zeroes `nzero` words at `zero`.
template <typename InT, typename PackT>
__global__ void __launch_bounds__(128, 16) pack_weights_kernel(int C_out, int C_in, int k, int ci_pad, int tf32_mode,
                                                           const InT* __restrict__ w, PackT* __restrict__ wp,
                                                           unsigned* __restrict__ zero, int nzero, int release_first) {
    // Launched with programmatic dependence, so its launch may overlap the end of the preceding
    // kernel: it waits for that kernel before it touches anything (that kernel may write w, or
    // still read the packed weights). The conv kernel that follows is released either after that
    // wait (it may then load x before waiting for this kernel: all earlier work is done) or, with
    // release_first, at once: its CTAs then take the SMs as the preceding kernel's leave, and it
    // waits for this kernel before it reads any global input.
    if (release_first) griddep_launch_dependents();
    griddep_wait();
    if (!release_first) griddep_launch_dependents();
    const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x, step = (long long)gridDim.x * blockDim.x;
    for (long long i = i0; i < nzero; i += step) zero[i] = 0u;
    const long long total = (long long)C_out * ci_pad;
    for (long long e = i0; e < total; e += step) {
        const int co = int(e / ci_pad), ci = int(e - (long long)co * ci_pad);
        const InT* src = w + ((long long)co * C_in + ci) * k;
        for (int kk = 0; kk < k; ++kk) {
            const float v = ci < C_in ? to_f32(src[kk]) : 0.f;
            PackT* dst = wp + ((long long)kk * C_out + co) * ci_pad + ci;
            if constexpr (sizeof(PackT) == 4) {
                const float hi = tf32_mode ? round_tf32(v) : v;
                *dst = hi;
                if (tf32_mode == 2) dst[(long long)k * C_out * ci_pad] = round_tf32(v - hi);
            } else {
                *dst = __float2bfloat16_rn(v);  // exact: v came from a bf16
            }
        }
    }
}

NormArgs norm_args(const c1n_params& p, const Plan& pl) {
    NormArgs a;
    a.N = p.N;
    a.C = p.C_out;
    a.T_out = pl.T_out;
    a.norm = p.norm;
    a.G = p.norm == C1N_NORM_GROUP ? p.groups : 1;
    a.cpg = p.C_out / a.G;
    a.gelu = p.post == C1N_POST_GELU_ERF;
    return a;
}

int grid_1d(long long work, int per_block = 256, int cap = 152 * 16) {
    long long g = (work + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

}  // namespace

cudaError_t launch_simt_conv(const c1n_params& p, const Plan& pl, const void* x, const void* w, const float* b,
                             void* out, bool out_is_raw_f32, cudaStream_t stream) {
    SimtConvArgs a;
    a.N = p.N; a.C_in = p.C_in; a.C_out = p.C_out; a.T = p.T; a.T_out = (int)pl.T_out; a.k = p.k;
    a.stride = p.stride; a.pad_left = p.pad_left; a.dilation = p.dilation;
    a.span = (kSimtT - 1) * p.stride + (p.k - 1) * p.dilation + 1;
    a.gelu = (!out_is_raw_f32 && p.norm == C1N_NORM_NONE && p.post == C1N_POST_GELU_ERF) ? 1 : 0;
    const size_t smem = sizeof(float) * ((size_t)kSimtCi * a.span + (size_t)kSimtCo * kSimtCi * p.k);
    dim3 grid((unsigned)((pl.T_out + kSimtT - 1) / kSimtT), (unsigned)((p.C_out + kSimtCo - 1) / kSimtCo),
              (unsigned)p.N);
    if (pl.bf16) {
        auto xi = static_cast<const __nv_bfloat16*>(x);
        auto wi = static_cast<const __nv_bfloat16*>(w);
        if (out_is_raw_f32) {
            auto k = simt_conv_kernel<__nv_bfloat16, float>;
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            k<<<grid, kSimtThreads, smem, stream>>>(a, xi, wi, b, static_cast<float*>(out));
        } else {
            auto k = simt_conv_kernel<__nv_bfloat16, __nv_bfloat16>;
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            k<<<grid, kSimtThreads, smem, stream>>>(a, xi, wi, b, static_cast<__nv_bfloat16*>(out));
        }
    } else {
        auto k = simt_conv_kernel<float, float>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k<<<grid, kSimtThreads, smem, stream>>>(a, static_cast<const float*>(x), static_cast<const float*>(w), b,
                                                static_cast<float*>(out));
    }
    return cudaGetLastError();
}

cudaError_t launch_gn_stats(const c1n_params& p, const Plan& pl, const float* raw, float2* stats,
                            cudaStream_t stream) {
    dim3 grid((unsigned)p.groups, (unsigned)p.N);
    gn_stats_kernel<<<grid, 512, 0, stream>>>(raw, stats, p.C_out, pl.T_out, p.groups, p.eps);
    return cudaGetLastError();
}

cudaError_t launch_gn_merge(const c1n_params& p, const Plan& pl, const float2* part, float2* stats,
                            cudaStream_t stream) {
    const int NG = p.N * p.groups;
    gn_merge_kernel<<<(NG + 7) / 8, 256, 0, stream>>>(part, stats, NG, pl.part_tiles, p.C_out / p.groups, pl.T_out,
                                                     p.eps);
    return cudaGetLastError();
}

cudaError_t launch_ln_merge(const c1n_params& p, const Plan& pl, const float2* part, float2* stats,
                            cudaStream_t stream) {
    const long long rows = (long long)p.N * pl.T_out;
    ln_merge_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, stream>>>(part, stats, p.N, p.C_out, pl.BN, pl.n_cb,
                                                                       pl.T_out, p.eps);
    return cudaGetLastError();
}

cudaError_t launch_ln_stats(const c1n_params& p, const Plan& pl, const float* raw, float2* stats,
                            cudaStream_t stream) {
    if (pl.T_out % 4 == 0) {
        dim3 grid((unsigned)((pl.T_out + 127) / 128), (unsigned)p.N);
        ln_stats_kernel<4><<<grid, 256, 0, stream>>>(raw, stats, p.C_out, pl.T_out, p.eps);
    } else {
        dim3 grid((unsigned)((pl.T_out + 31) / 32), (unsigned)p.N);
        ln_stats_kernel<1><<<grid, 256, 0, stream>>>(raw, stats, p.C_out, pl.T_out, p.eps);
    }
    return cudaGetLastError();
}

cudaError_t launch_normalize(const c1n_params& p, const Plan& pl, const float* raw, const float2* stats,
                             const float* gamma, const float* beta, void* y, cudaStream_t stream) {
    NormArgs a = norm_args(p, pl);
    const long long rows8 = (long long)p.N * p.C_out;
    if (pl.T_out % 8 == 0 && (reinterpret_cast<uintptr_t>(raw) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
        const long long per_row = pl.T_out / 8;
        int gx = (int)((per_row + 255) / 256);
        if (gx > 64) gx = 64;
        long long gy = (152LL * 16 + gx - 1) / gx;
        if (gy > rows8) gy = rows8;
        if (gy > 65535) gy = 65535;
        dim3 grid((unsigned)gx, (unsigned)gy);
#define C1N_NORM8(T, NORM)                                                                                  \
    (a.gelu ? (normalize8_kernel<T, NORM, true><<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, out), 0) \
            : (normalize8_kernel<T, NORM, false><<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, out), 0))
        if (a.norm == 2 && p.N <= 65535) {
            dim3 g3((unsigned)((per_row + 255) / 256), (unsigned)((p.C_out + 63) / 64), (unsigned)p.N);
            if (pl.bf16) {
                auto out = static_cast<__nv_bfloat16*>(y);
                if (a.gelu) normalize8_ln_kernel<__nv_bfloat16, true><<<g3, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
                else normalize8_ln_kernel<__nv_bfloat16, false><<<g3, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
            } else {
                auto out = static_cast<float*>(y);
                if (a.gelu) normalize8_ln_kernel<float, true><<<g3, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
                else normalize8_ln_kernel<float, false><<<g3, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
            }
            return cudaGetLastError();
        }
        if (pl.bf16) {
            auto out = static_cast<__nv_bfloat16*>(y);
            if (a.norm == 2) C1N_NORM8(__nv_bfloat16, 2);
            else if (a.norm == 1) C1N_NORM8(__nv_bfloat16, 1);
            else C1N_NORM8(__nv_bfloat16, 0);
        } else {
            auto out = static_cast<float*>(y);
            if (a.norm == 2) C1N_NORM8(float, 2);
            else if (a.norm == 1) C1N_NORM8(float, 1);
            else C1N_NORM8(float, 0);
        }
#undef C1N_NORM8
        return cudaGetLastError();
    }
    const bool vec = (pl.T_out % 4) == 0;
    const long long per_row = vec ? pl.T_out / 4 : pl.T_out;
    const long long rows = (long long)p.N * p.C_out;
    int gx = (int)((per_row + 255) / 256);
    if (gx > 64) gx = 64;
    long long gy = (152LL * 32 + gx - 1) / gx;
    if (gy > rows) gy = rows;
    if (gy > 65535) gy = 65535;
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (pl.bf16) {
        auto out = static_cast<__nv_bfloat16*>(y);
        if (vec) normalize_kernel<__nv_bfloat16, true><<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
        else normalize_kernel<__nv_bfloat16, false><<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
    } else {
        auto out = static_cast<float*>(y);
        if (vec) normalize_kernel<float, true><<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
        else normalize_kernel<float, false><<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, out);
    }
    return cudaGetLastError();
}

cudaError_t launch_rowmin(const c1n_params& p, const Plan& pl, const float* raw, const float2* stats,
                          const float* gamma, const float* beta, float* rowmin, int32_t* argmin,
                          cudaStream_t stream) {
    NormArgs a = norm_args(p, pl);
    dim3 grid((unsigned)pl.T_out, (unsigned)p.N);
    rowmin_kernel<<<grid, 256, 0, stream>>>(a, raw, stats, gamma, beta, rowmin, argmin);
    return cudaGetLastError();
}

cudaError_t launch_broadcast(const c1n_params& p, const Plan& pl, const float* rowmin, const float* bias2, void* y,
                             cudaStream_t stream) {
    NormArgs a = norm_args(p, pl);
    if (!pl.bf16 && pl.T_out == 1 && p.C_out % 4 == 0) {
        int gx = (p.C_out / 4 + 255) / 256;
        int gy = p.N < 4096 ? p.N : 4096;
        broadcast_rows_f32_kernel<<<dim3(gx, gy), 256, 0, stream>>>(p.N, p.C_out, rowmin, bias2,
                                                                    static_cast<float*>(y));
    } else {
        const long long total = (long long)p.N * p.C_out * pl.T_out;
        if (pl.bf16)
            broadcast_kernel<__nv_bfloat16><<<grid_1d(total), 256, 0, stream>>>(a, rowmin, bias2,
                                                                               static_cast<__nv_bfloat16*>(y));
        else
            broadcast_kernel<float><<<grid_1d(total), 256, 0, stream>>>(a, rowmin, bias2, static_cast<float*>(y));
    }
    return cudaGetLastError();
}

cudaError_t launch_rowmin_finish(const c1n_params& p, const Plan& pl, const float2* part, const float* bias2, void* y,
                                 int32_t* argmin, cudaStream_t stream) {
    if (pl.bf16)
        rowmin_finish_kernel<__nv_bfloat16><<<p.N, 256, 0, stream>>>(p.C_out, pl.n_cb, part, bias2,
                                                                      static_cast<__nv_bfloat16*>(y), argmin);
    else
        rowmin_finish_kernel<float><<<p.N, 256, 0, stream>>>(p.C_out, pl.n_cb, part, bias2, static_cast<float*>(y),
                                                             argmin);
    return cudaGetLastError();
}

// Set once the driver has refused programmatic dependence for the pack (then launched plainly).
static std::atomic<int> pdl_pack_refused{0};

cudaError_t launch_pack_weights(const c1n_params& p, const Plan& pl, const void* w, void* wp, cudaStream_t stream,
                                unsigned* zero, int nzero, bool release_first) {
    // One (co, ci) slot per thread where the grid allows, so the weight loads are in flight at once,
    // but at most 2 CTAs of 128 threads per SM (of 152): launched early, the CTAs wait beside the
    // preceding kernel's warps (8 per SM slowed the bf16 LayerNorm kernel's epilogue, 287 vs 269 us
    // per step), and the conv kernel launched behind them (1 CTA of 480 threads per SM) fits beside.
    const long long total = (long long)p.C_out * pl.ci_pad;
    const long long work = total > nzero ? total : nzero;
    const int grid = (int)std::min<long long>((work + 127) / 128, 152 * 2);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_pack_refused.load() ? 0 : 1;
    for (;;) {
        cudaError_t e;
        if (pl.bf16)
            e = cudaLaunchKernelEx(&cfg, pack_weights_kernel<__nv_bfloat16, __nv_bfloat16>, p.C_out, p.C_in, p.k,
                                   pl.ci_pad, 0, static_cast<const __nv_bfloat16*>(w),
                                   static_cast<__nv_bfloat16*>(wp), zero, nzero, release_first ? 1 : 0);
        else
            e = cudaLaunchKernelEx(&cfg, pack_weights_kernel<float, float>, p.C_out, p.C_in, p.k, pl.ci_pad,
                                   pl.x3 ? 2 : 1, static_cast<const float*>(w), static_cast<float*>(wp), zero,
                                   nzero, release_first ? 1 : 0);
        if (e == cudaSuccess || cfg.numAttrs == 0) return e;
        cudaGetLastError();  // the attribute refused: launch plainly from now on
        pdl_pack_refused.store(1);
        cfg.numAttrs = 0;
    }
}

}  // namespace c1n

// [p4]'s second operator (Kimi-K2.6 l2_p3 page, the model's steps after its ConvTranspose3d): a scalar
// added, LayerNorm over the last dimension W (affine per position w), AvgPool3d with kernel and
// stride 2, exact GELU. One memory-bound pass: z is read once, the pooled output written once.
//
// Work unit: one pooling group (n, c, d', h'), i.e. the four W-rows (2d'+a, 2h'+b), a, b in {0, 1},
// whose LayerNorm results feed the W/2 outputs (n, c, d', h', *). A group's rows reach shared
// memory by 16-byte asynchronous copies, several groups ahead of the arithmetic. A row is read by
// LPR lanes (16 or 32), V consecutive values per lane, so a lane's values contain whole pooling
// pairs along W. A warp holds 32/LPR rows at a time and makes 4 / (32/LPR) passes over a group;
// every pass reduces its rows' sums and squared deviations with shuffles inside the row's lanes
// (two-pass statistics on registers), normalizes, and adds the pairs into per-lane pool
// accumulators; half-warp rows are combined with one more shuffle.
#include <cuda_runtime.h>

#include <cstdint>

#include "c1n_internal.h"
#include "c1n_math.cuh"

namespace c1n {
namespace {

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// 16-byte asynchronous copy global -> shared (bypassing L1), grouped per stage.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Every warp walks its pooling groups (grid-stride) through a private ring of S shared-memory
// slots, one group per slot: the rows of the next S-1 groups are in flight (cp.async) while the
// oldest is reduced, so each SM keeps tens of kilobytes of z in flight.
template <int LPR, int V, int S>
__global__ void __launch_bounds__(256) ln_avgpool3d_gelu_kernel(int NC, int D, int H, float eps, float sum_weight,
                                                                const float* __restrict__ z,
                                                                const float* __restrict__ gamma,
                                                                const float* __restrict__ beta,
                                                                float* __restrict__ out) {
    constexpr int W = LPR * V;
    constexpr int RPP = 32 / LPR;    // rows a warp holds at once
    constexpr int PASSES = 4 / RPP;  // passes over the four rows of a group
    constexpr int SLOT = 4 * W;      // floats per slot: the group's four rows
    extern __shared__ float4 ring4[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* ring = reinterpret_cast<float*>(ring4) + warp * (S * SLOT);
    const int sub = lane / LPR;      // which of the warp's rows (RPP = 2: the h offset b)
    const int li = lane % LPR;       // lane within its row: columns li*V .. li*V+V-1
    const int D2 = D / 2, H2 = H / 2;
    float g[V], be[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        g[i] = gamma ? __ldg(gamma + li * V + i) : 1.f;
        be[i] = beta ? __ldg(beta + li * V + i) : 0.f;
    }
    // Work is handed out by plane pair: unit u = (n, c, d') covers the H/2 groups h' = 0 .. H/2-1,
    // walked in order, so a cursor moves from group to group by additions (one division per unit).
    const long long n_units = (long long)NC * D2;
    const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long plane = (long long)H * W;
    struct Cursor {
        long long unit, off;  // off: z offset of row (2d', 2h') of the current group
        int h2;
    };
    auto start = [&](Cursor& c, long long u) {
        c.unit = u;
        c.h2 = 0;
        c.off = u < n_units ? ((u / D2) * D + 2 * (u % D2)) * plane : 0;
    };
    auto advance = [&](Cursor& c) {
        if (++c.h2 == H2) start(c, c.unit + nwarps);
        else c.off += 2 * W;
    };
    // the group's four rows into slot `s`: W/4 16-byte pieces per row, spread over the lanes
    auto issue = [&](const Cursor& c, int s) {
        if (c.unit < n_units) {
            const uint32_t dst = smem_addr(ring + s * SLOT);
#pragma unroll
            for (int k = lane; k < W; k += 32) {  // k: 16-byte piece over the four rows (W / 4 per row)
                const int r = k / (W / 4), cc = k % (W / 4);
                cp_async16(dst + uint32_t((r * W + 4 * cc) * 4), z + c.off + (r >> 1) * plane + (r & 1) * W + 4 * cc);
            }
        }
        cp_async_commit();
    };
    Cursor cin, cur;
    start(cin, warp0);
    start(cur, warp0);
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        issue(cin, s);
        advance(cin);
    }
    int slot = 0;
    for (; cur.unit < n_units; advance(cur)) {
        issue(cin, (slot + S - 1) % S);
        advance(cin);
        cp_async_wait<S - 1>();  // this group's copies (the oldest group in flight) have landed
        __syncwarp();
        const float* sl = ring + slot * SLOT;
        float acc[V / 2];
#pragma unroll
        for (int j = 0; j < V / 2; ++j) acc[j] = 0.f;
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int r = RPP == 2 ? 2 * p + sub : p;  // rows (d offset, h offset) in slot order
            float v[V];
#pragma unroll
            for (int k = 0; k < V / 4; ++k) {
                const float4 f = reinterpret_cast<const float4*>(sl + r * W + li * V)[k];
                v[4 * k] = f.x;
                v[4 * k + 1] = f.y;
                v[4 * k + 2] = f.z;
                v[4 * k + 3] = f.w;
            }
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                v[i] += sum_weight;
                s += v[i];
            }
            const float mean = row_sum<LPR>(s) * (1.f / W);
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                v[i] -= mean;
                ss = fmaf(v[i], v[i], ss);
            }
            const float rstd = rsqrtf(row_sum<LPR>(ss) * (1.f / W) + eps);
#pragma unroll
            for (int j = 0; j < V / 2; ++j)
                acc[j] += fmaf(v[2 * j] * rstd, g[2 * j], be[2 * j]) + fmaf(v[2 * j + 1] * rstd, g[2 * j + 1], be[2 * j + 1]);
        }
        __syncwarp();  // every lane is done with the slot before it is refilled
        if (RPP == 2) {
#pragma unroll
            for (int j = 0; j < V / 2; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 16);
        }
        if (sub == 0) {
            float o[V / 2];
#pragma unroll
            for (int j = 0; j < V / 2; j += 2)
                f2_unpack(gelu_erf2(f2_pack(acc[j] * 0.125f, acc[j + 1] * 0.125f)), o[j], o[j + 1]);
            float* dst = out + (cur.unit * H2 + cur.h2) * (long long)(W / 2) + li * (V / 2);
            if constexpr (V / 2 == 2) {
                *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
            } else {
#pragma unroll
                for (int k = 0; k < V / 8; ++k)
                    reinterpret_cast<float4*>(dst)[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
            }
        }
        slot = slot + 1 == S ? 0 : slot + 1;
    }
    cp_async_wait<0>();  // no copy outlives the warp's shared memory
}

template <int LPR, int V, int S>
cudaError_t launch(const c1n_lnpool_params& p, const float* z, float sum_weight, const float* gamma,
                   const float* beta, float* out, int num_sms, cudaStream_t stream) {
    auto kern = ln_avgpool3d_gelu_kernel<LPR, V, S>;
    constexpr int kSmem = 8 * S * 4 * LPR * V * 4;  // 8 warps x S slots x 4 rows x W floats
    static_assert(kSmem <= 200 * 1024, "ring too large");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)p.N * p.C * (p.D / 2);  // plane pairs, one warp at a time each
    long long grid = (units + 7) / 8;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, kSmem);
    if (e != cudaSuccess) return e;
    const long long cap = (long long)num_sms * (per_sm > 0 ? per_sm : 1);  // one resident wave, then grid-stride
    if (grid > cap) grid = cap;
    kern<<<(unsigned)grid, 256, kSmem, stream>>>(p.N * p.C, p.D, p.H, p.eps, sum_weight, z, gamma, beta, out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ln_avgpool3d_gelu(const c1n_lnpool_params& p, const float* z, float sum_weight,
                                     const float* gamma, const float* beta, float* out, int num_sms,
                                     cudaStream_t stream) {
    switch (p.W) {
        case 64: return launch<16, 4, 6>(p, z, sum_weight, gamma, beta, out, num_sms, stream);
        case 128: return launch<32, 4, 4>(p, z, sum_weight, gamma, beta, out, num_sms, stream);
        case 256: return launch<32, 8, 3>(p, z, sum_weight, gamma, beta, out, num_sms, stream);
        case 512: return launch<32, 16, 2>(p, z, sum_weight, gamma, beta, out, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace c1n

// [p4]'s transposed 3-D convolution on the tensor cores (kernel 3, stride 2, padding 1, C_in = 32,
// C_out = 64; Kimi-K2.6 l2_p3 page).
//
// As a contraction: for every input voxel v = (n, i, j, l) and output parity p = (pd, ph, pw),
//   y[n][co][2i+pd][2j+ph][2l+pw] = b[co] + sum_{delta <= p} sum_ci x[n][ci][v + delta] * w[ci][co][k(p, delta)]
// with delta in {0, 1}^3 (componentwise at most p) and, per axis, k(0, 0) = 1, k(1, 0) = 2,
// k(1, 1) = 0 (inputs past the end count zero). For one (pd, ph) "class" the rows (pw, co) form
// M = 128, the voxels of a tile N = 128 (4 input rows j x 32 input columns l), and each shift delta
// one K = 32 step: D[(pw, co)][v] += A_delta[(pw, co)][ci] * X[v + delta][ci], where A_delta holds the
// weights of that tap (zero rows for pw = 0 when delta_w = 1). A class has 2, 4, 4 or 8 shifts.
//
// Operands: x is first rewritten channels-last (x_cl[n][d][h][w][ci]) so that a 32-voxel x 32-channel
// box of it is a K-major, 128-byte-swizzled MMA operand; the shift is just a TMA coordinate on the
// w / h / d dimensions (past the end -> zero fill). The class's A blocks (TF32-rounded, packed by a
// small kernel) stay in shared memory for the CTA's whole life. CTAs are split over the four
// classes in proportion to their shift counts; each walks its class's tiles.
//
// Roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2-5 epilogue
// (TMEM lane quarter q = rows 32q..32q+31: pw = q / 2, channels 32 (q % 2) ..). Two accumulators of
// 128 columns, so the epilogue of one tile overlaps the next tile's MMAs. The epilogue interleaves
// the two width parities through 128-byte-swizzled shared tiles [32 channels][32 ow] and sends them
// with TMA bulk stores. Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "c1n_internal.h"
#include "sm100_ptx.cuh"

namespace c1n {
namespace {

constexpr int kThreads = 192;
constexpr int kSB = 3;                    // B ring stages
constexpr int kTileBytes = 128 * 128;     // one 128-row x 128-byte operand tile (16 KB)
constexpr int kStageOut = 4 * 32 * 32 * 4;  // four 32 x 32 fp32 output tiles (16 KB), two buffers

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int c2,
                                            int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

__device__ __forceinline__ void tma_store_5d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2, int c3,
                                             int c4) {
    asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void store_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void store_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Time-bounded wait that ignores the abort flag: copies and MMAs in flight land before the CTA
// (and its shared memory / TMEM) goes away.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

struct ConvTArgs {
    int N, D, H, W, Do, Ho, Wo;
    int JT, LT;           // tiles along input rows (4 each) and input columns (32 each)
    int cta0[5];          // first CTA of each class (cta0[4] = grid)
    const float* bias;    // [64] or null
    int* status;          // [0] = 1 when a wait gave up (the output is then incomplete)
};

// Shift list of class c = (pd, ph): delta_d in [0, pd], delta_h in [0, ph], delta_w in {0, 1}; block
// index inside the packed weights: class base + position in this order.
__host__ __device__ constexpr int n_shifts(int c) { return 2 * ((c >> 1) + 1) * ((c & 1) + 1); }
__host__ __device__ constexpr int class_base(int c) {
    return c == 0 ? 0 : c == 1 ? n_shifts(0) : c == 2 ? n_shifts(0) + n_shifts(1) : n_shifts(0) + n_shifts(1) + n_shifts(2);
}

__global__ void __launch_bounds__(kThreads, 1)
    convt3d_tc_kernel(const __grid_constant__ ConvTArgs a, const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_y) {
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // class of this CTA and its place among the class's CTAs
    int cls = 0;
    while (cls < 3 && int(blockIdx.x) >= a.cta0[cls + 1]) ++cls;
    const int pd = cls >> 1, ph = cls & 1;
    const int ns = n_shifts(cls);
    const int cta_in = int(blockIdx.x) - a.cta0[cls], n_cta = a.cta0[cls + 1] - a.cta0[cls];
    const int tiles = a.N * a.D * a.JT * a.LT;
    // shared memory: A blocks (8 max) | B ring | output staging (2 buffers) | barriers
    const uint32_t sA = smem_u32(base);
    const uint32_t sB = sA + 8u * kTileBytes;
    uint8_t* so = base + 8 * kTileBytes + kSB * kTileBytes;  // 1024-byte aligned
    uint64_t* bars = reinterpret_cast<uint64_t*>(so + 2 * kStageOut);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };
    const int i_afull = 0, i_bfull = 1, i_bempty = 1 + kSB, i_accfull = 1 + 2 * kSB, i_accempty = i_accfull + 2,
              i_drain = i_accempty + 2, n_bars = i_drain + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + n_bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    if (warp == 0) {
        if (lane < n_bars) mbar_init(bar(lane), (lane >= i_accempty && lane < i_drain) ? 4u : 1u);
        if (lane == 0) *abort_flag = 0;
        fence_mbar_init();
        if (lane == 0) {
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_w);
            prefetch_tensormap(&tm_y);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 256u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    auto wait = [&](int i, uint32_t parity) -> bool {
        if (mbar_try_wait(bar(i), parity)) return true;
        return mbar_wait(bar(i), parity, abort_flag, a.status, 0, nullptr);
    };
    auto wait_warp = [&](int i, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(i, parity)); };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        long long b_cnt = 0;
        int bi = 0;
        uint32_t bph = 0;
        if (elect_one()) {
            mbar_arrive_expect_tx(bar(i_afull), uint32_t(ns * kTileBytes));
            for (int s = 0; s < ns; ++s) tma_load_2d(sA + s * kTileBytes, &tm_w, bar(i_afull), 0, (class_base(cls) + s) * 128);
        }
        __syncwarp();
        for (int t = cta_in; t < tiles && !__any_sync(0xffffffffu, *abort_flag != 0); t += n_cta) {
            const int lt = t % a.LT, jt = (t / a.LT) % a.JT, i = (t / (a.LT * a.JT)) % a.D, n = t / (a.LT * a.JT * a.D);
            for (int s = 0; s < ns; ++s) {
                const int dd = s / (2 * (ph + 1)), dh = (s / 2) % (ph + 1), dw = s & 1;
                if (!wait_warp(i_bempty + bi, bph ^ 1)) goto prod_done;
                if (elect_one()) {
                    mbar_arrive_expect_tx(bar(i_bfull + bi), kTileBytes);
                    tma_load_5d(sB + bi * kTileBytes, &tm_x, bar(i_bfull + bi), 0, lt * 32 + dw, jt * 4 + dh, i + dd, n);
                }
                __syncwarp();
                ++b_cnt;
                if (++bi == kSB) { bi = 0; bph ^= 1; }
            }
        }
    prod_done:
        if (*abort_flag && lane == 0) {
            // let the copies in flight land before the CTA leaves (bounded)
            drain_wait(bar(i_afull), 0);
            for (int s2 = 0; s2 < kSB; ++s2)
                if (b_cnt > s2) drain_wait(bar(i_bfull + s2), s2 < bi ? bph : (bph ^ 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = make_idesc(2u, 2u, 0u, 0u, 128u, 128u);
        int bi = 0, lt_ = 0;
        uint32_t bph = 0;
        bool ok = wait_warp(i_afull, 0);
        tc_fence_after();
        for (int t = cta_in; ok && t < tiles; t += n_cta, ++lt_) {
            const int ab = lt_ & 1;
            const uint32_t acc_par = uint32_t((lt_ >> 1) & 1);
            if (!wait_warp(i_accempty + ab, acc_par ^ 1)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + uint32_t(128 * ab);
            for (int s = 0; s < ns; ++s) {
                if (!wait_warp(i_bfull + bi, bph)) { ok = false; break; }
                tc_fence_after();
                const uint32_t al = desc_lo_sw128(sA + s * kTileBytes), bl = desc_lo_sw128(sB + bi * kTileBytes);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) mma_issue<false, false>(d, al + 2u * k, bl + 2u * k, idesc, (s | k) != 0 ? 1u : 0u);
                    mma_commit(bar(i_bempty + bi));
                }
                __syncwarp();
                if (++bi == kSB) { bi = 0; bph ^= 1; }
            }
            if (!ok) break;
            if (elect_one()) mma_commit(bar(i_accfull + ab));
            __syncwarp();
        }
        // every MMA issued has finished before TMEM is released
        if (elect_one()) mma_commit(bar(i_drain));
        __syncwarp();
        if (lane == 0) drain_wait(bar(i_drain), 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;            // TMEM lane quarter: rows 32q .. 32q+31
        const int pw = q >> 1, cb = q & 1;  // width parity, channel block (32 channels)
        const int co = cb * 32 + lane;
        const float bv = a.bias ? __ldg(a.bias + co) : 0.f;
        int lt_ = 0, ob = 0;
        for (int t = cta_in; t < tiles; t += n_cta, ++lt_) {
            const int ab = lt_ & 1;
            const uint32_t acc_par = uint32_t((lt_ >> 1) & 1);
            int got = 0;
            if (lane == 0) got = wait(i_accfull + ab, acc_par);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (named_bar_any(1, 128, !got || *abort_flag != 0)) break;
            tc_fence_after();
            const int lt = t % a.LT, jt = (t / a.LT) % a.JT, i = (t / (a.LT * a.JT)) % a.D, n = t / (a.LT * a.JT * a.D);
            const uint32_t tb = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(128 * ab);
            for (int jj = 0; jj < 4; ++jj) {
                float v[32];
                tmem_load32(tb + uint32_t(jj * 32), v);  // input columns l = 0..31 of row jj
                // buffer `ob` held the stores issued two rows ago: they must have read it
                if (lane == 0) store_wait_read_le1();
                named_bar_sync(1, 128);
                // tiles of buffer ob: [cb][half], each [32 channels][32 ow], 128-byte swizzle
                uint8_t* buf = so + ob * kStageOut;
#pragma unroll
                for (int l = 0; l < 32; ++l) {
                    const int h = l >> 4, c = 2 * (l & 15) + pw;  // ow = 2l + pw -> half h, column c
                    uint8_t* tile = buf + (cb * 2 + h) * 4096;
                    *reinterpret_cast<float*>(tile + lane * 128 + (((c >> 2) ^ (lane & 7)) << 4) + (c & 3) * 4) =
                        v[l] + bv;
                }
                fence_async_shared();
                named_bar_sync(1, 128);
                if (lane == 0) {
                    // warp q sends tile (channel block q & 1, half q >> 1)
                    const int tcb = q & 1, th = q >> 1;
                    tma_store_5d(&tm_y, smem_u32(buf + (tcb * 2 + th) * 4096), 64 * lt + 32 * th,
                                 2 * (jt * 4 + jj) + ph, 2 * i + pd, 32 * tcb, n);
                }
                __syncwarp();
                ob ^= 1;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(i_accempty + ab));
        }
        if (lane == 0) store_wait_read_all();
        __syncwarp();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 256u);
    }
}

// x [N][C][S] -> x_cl [N][S][C] (S = D*H*W), 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) to_channels_last_kernel(const float* __restrict__ x, float* __restrict__ xcl,
                                                               int C, long long S) {
    __shared__ float t[32][33];
    const int n = blockIdx.z;
    const long long s0 = (long long)blockIdx.x * 32;
    const int c0 = blockIdx.y * 32;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int c = c0 + r;
        const long long s = s0 + threadIdx.x;
        t[r][threadIdx.x] = (c < C && s < S) ? __ldg(x + ((long long)n * C + c) * S + s) : 0.f;
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const long long s = s0 + r;
        const int c = c0 + threadIdx.x;
        if (s < S && c < C) xcl[((long long)n * S + s) * C + c] = t[threadIdx.x][r];
    }
}

// Packed weights: 18 blocks [128 rows = (pw, co)][32 ci], TF32-rounded; block of class c and shift
// s (in the kernel's order) at row (class_base(c) + s) * 128. Rows whose tap does not exist are 0.
__global__ void __launch_bounds__(256) pack_convt_weights_kernel(const float* __restrict__ w, float* __restrict__ wp) {
    const int blk = blockIdx.x;  // 0 .. 17
    int cls = 0;
    while (cls < 3 && blk >= class_base(cls + 1)) ++cls;
    const int s = blk - class_base(cls);
    const int pd = cls >> 1, ph = cls & 1;
    const int dd = s / (2 * (ph + 1)), dh = (s / 2) % (ph + 1), dw = s & 1;
    auto tap = [](int p, int dl) { return p == 0 ? 1 : (dl == 0 ? 2 : 0); };
    const int kd = tap(pd, dd), kh = tap(ph, dh);
    for (int e = threadIdx.x; e < 128 * 32; e += blockDim.x) {
        const int row = e / 32, ci = e % 32, pw = row / 64, co = row % 64;
        float v = 0.f;
        if (!(pw == 0 && dw == 1)) {
            const int kw = tap(pw, dw);
            v = round_tf32(__ldg(w + (((ci * 64 + co) * 3 + kd) * 3 + kh) * 3 + kw));
        }
        wp[(size_t)blk * 128 * 32 + e] = v;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

bool encode_f32(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box) {
    auto fn = encoder();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t convt3d_tc_workspace_bytes(const c1n_convt3d_params& p) {
    const size_t xcl = (size_t)p.N * p.C_in * p.D * p.H * p.W * 4;
    return 256 + ((xcl + 1023) / 1024) * 1024 + 18 * (size_t)kTileBytes;
}

cudaError_t launch_conv_transpose3d_tc(const c1n_convt3d_params& p, const float* x, const float* w, const float* b,
                                       float* y, void* workspace, int num_sms, cudaStream_t stream) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    const size_t xcl_bytes = ((size_t)p.N * p.C_in * p.D * p.H * p.W * 4 + 1023) / 1024 * 1024;
    float* xcl = reinterpret_cast<float*>(ws + 256);
    float* wp = reinterpret_cast<float*>(ws + 256 + xcl_bytes);
    const int Do = 2 * p.D - 1 + p.out_pad, Ho = 2 * p.H - 1 + p.out_pad, Wo = 2 * p.W - 1 + p.out_pad;
    cudaError_t e = cudaMemsetAsync(status, 0, 256, stream);
    if (e != cudaSuccess) return e;
    const long long S = (long long)p.D * p.H * p.W;
    to_channels_last_kernel<<<dim3((unsigned)((S + 31) / 32), (unsigned)((p.C_in + 31) / 32), (unsigned)p.N),
                              dim3(32, 8), 0, stream>>>(x, xcl, p.C_in, S);
    pack_convt_weights_kernel<<<18, 256, 0, stream>>>(w, wp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tm_x, tm_w, tm_y;
    {
        const cuuint64_t dims[5] = {32, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)p.D, (cuuint64_t)p.N};
        const cuuint64_t str[4] = {32 * 4, (cuuint64_t)p.W * 32 * 4, (cuuint64_t)p.H * p.W * 32 * 4,
                                   (cuuint64_t)p.D * p.H * p.W * 32 * 4};
        const cuuint32_t box[5] = {32, 32, 4, 1, 1};
        if (!encode_f32(&tm_x, xcl, 5, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {32, 18 * 128};
        const cuuint64_t str[1] = {32 * 4};
        const cuuint32_t box[2] = {32, 128};
        if (!encode_f32(&tm_w, wp, 2, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[5] = {(cuuint64_t)Wo, (cuuint64_t)Ho, (cuuint64_t)Do, 64, (cuuint64_t)p.N};
        const cuuint64_t str[4] = {(cuuint64_t)Wo * 4, (cuuint64_t)Ho * Wo * 4, (cuuint64_t)Do * Ho * Wo * 4,
                                   (cuuint64_t)64 * Do * Ho * Wo * 4};
        const cuuint32_t box[5] = {32, 1, 1, 32, 1};
        if (!encode_f32(&tm_y, y, 5, dims, str, box)) return cudaErrorInvalidValue;
    }
    ConvTArgs a;
    a.N = p.N;
    a.D = p.D;
    a.H = p.H;
    a.W = p.W;
    a.Do = Do;
    a.Ho = Ho;
    a.Wo = Wo;
    a.JT = (p.H + 3) / 4;
    a.LT = (p.W + 31) / 32;
    a.bias = b;
    a.status = status;
    // CTAs per class in proportion to its shifts (2, 4, 4, 8 of 18), at least one each, no more than
    // the class has tiles
    const long long tiles = (long long)p.N * p.D * a.JT * a.LT;
    int grid = num_sms > 4 ? num_sms : 4;
    a.cta0[0] = 0;
    int left = grid;
    for (int c = 0; c < 4; ++c) {
        int k = c == 3 ? left : (grid * n_shifts(c) + 9) / 18;
        if (k < 1) k = 1;
        if (k > left - (3 - c)) k = left - (3 - c);
        if (k > tiles) k = (int)tiles;
        a.cta0[c + 1] = a.cta0[c] + k;
        left -= k;
    }
    grid = a.cta0[4];
    const int smem = 1024 + 8 * kTileBytes + kSB * kTileBytes + 2 * kStageOut + 256;
    e = cudaFuncSetAttribute(convt3d_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    convt3d_tc_kernel<<<grid, kThreads, smem, stream>>>(a, tm_x, tm_w, tm_y);
    return cudaGetLastError();
}

}  // namespace c1n

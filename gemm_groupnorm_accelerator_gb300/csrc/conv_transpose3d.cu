// [p4]'s transposed 3-D convolution (Kimi-K2.6 l2_p3 page: ConvTranspose3d, kernel 3, stride 2,
// padding 1, output padding 0 or 1, with bias), on the CUDA cores in fp32.
//
// Gather form split by output parity: along each axis an output o = 2i + p takes, for p = 0, only
// tap 1 from input i, and for p = 1, tap 2 from input i and tap 0 from input i + 1 (inputs past the
// end count zero). A CTA owns one sample n, one input depth i, one (depth, height) parity pair
// (pd, ph), 32 output channels and a tile of 8 input rows j by 32 input columns l; each thread
// computes both width parities of its (j, l) -- outputs ow = 2l and 2l + 1 -- for the 32 channels,
// so a warp stores 32 consecutive float2 per channel. Input channels are walked one at a time
// through shared memory: the (up to) 2 x 9 x 33 input values the tile's taps read (zero outside
// the input) and the 27 x 32 weights of that channel.
#include <cuda_runtime.h>

#include <cstdint>

#include "c1n_internal.h"

namespace c1n {
namespace {

constexpr int kTJ = 8, kTL = 32, kCo = 32;  // tile: input rows, input columns, output channels

__global__ void __launch_bounds__(256) conv_transpose3d_k3s2_kernel(int C_in, int C_out, int D, int H, int W,
                                                                    int Do, int Ho, int Wo,
                                                                    const float* __restrict__ x,
                                                                    const float* __restrict__ w,
                                                                    const float* __restrict__ b,
                                                                    float* __restrict__ y) {
    __shared__ float xs[2][kTJ + 1][kTL + 4];  // input planes i, i+1; rows j0..j0+8; columns l0..l0+32
    __shared__ float4 ws4[27][kCo / 4];        // weights of one input channel: tap (kd, kh, kw), 32 channels
    const int tid = threadIdx.x, jj = tid / kTL, ll = tid % kTL;
    // blockIdx.x: l tile, j tile; blockIdx.y: i, parity pair, channel block; blockIdx.z: sample
    const int n_lt = (W + kTL - 1) / kTL;
    const int l0 = (blockIdx.x % n_lt) * kTL, j0 = (blockIdx.x / n_lt) * kTJ;
    const int n_cb = C_out / kCo;
    const int cb = blockIdx.y % n_cb, pp = (blockIdx.y / n_cb) % 4, i = blockIdx.y / (n_cb * 4);
    const int pd = pp >> 1, ph = pp & 1;
    const int n = blockIdx.z;
    const int j = j0 + jj, l = l0 + ll;
    // taps along depth and height for this parity: (kernel index, input offset)
    const int nd = pd ? 2 : 1, nh = ph ? 2 : 1;
    const int kd_t[2] = {pd ? 2 : 1, 0}, dd_t[2] = {0, 1};
    const int kh_t[2] = {ph ? 2 : 1, 0}, dh_t[2] = {0, 1};
    float acc0[kCo], acc1[kCo];  // outputs ow = 2l (width parity 0) and 2l + 1 (parity 1)
#pragma unroll
    for (int c = 0; c < kCo; ++c) acc0[c] = acc1[c] = b ? __ldg(b + cb * kCo + c) : 0.f;
    const long long plane = (long long)H * W;
    for (int ci = 0; ci < C_in; ++ci) {
        __syncthreads();  // the previous channel's values are no longer read
        const float* xc = x + ((long long)n * C_in + ci) * D * plane;
        for (int e = tid; e < 2 * (kTJ + 1) * (kTL + 1); e += 256) {
            const int a = e / ((kTJ + 1) * (kTL + 1)), r = (e / (kTL + 1)) % (kTJ + 1), c = e % (kTL + 1);
            const int id = i + a, ih = j0 + r, iw = l0 + c;
            xs[a][r][c] = (id < D && ih < H && iw < W) ? __ldg(xc + id * plane + (long long)ih * W + iw) : 0.f;
        }
        const float* wc = w + ((long long)ci * C_out + cb * kCo) * 27;
        for (int e = tid; e < 27 * kCo; e += 256) {
            const int c = e / 27, t = e % 27;  // w[ci][co][t] is contiguous along t
            reinterpret_cast<float*>(ws4[t])[c] = __ldg(wc + e);
        }
        __syncthreads();
        for (int a = 0; a < nd; ++a) {
            for (int bh = 0; bh < nh; ++bh) {
                const float x0 = xs[dd_t[a]][jj + dh_t[bh]][ll];      // input column l
                const float x1 = xs[dd_t[a]][jj + dh_t[bh]][ll + 1];  // input column l + 1
                const int tb = (kd_t[a] * 3 + kh_t[bh]) * 3;         // tap index of (kd, kh, kw = 0)
#pragma unroll
                for (int q = 0; q < kCo / 4; ++q) {
                    const float4 w0 = ws4[tb][q], w1 = ws4[tb + 1][q], w2 = ws4[tb + 2][q];
                    acc0[4 * q] = fmaf(x0, w1.x, acc0[4 * q]);
                    acc0[4 * q + 1] = fmaf(x0, w1.y, acc0[4 * q + 1]);
                    acc0[4 * q + 2] = fmaf(x0, w1.z, acc0[4 * q + 2]);
                    acc0[4 * q + 3] = fmaf(x0, w1.w, acc0[4 * q + 3]);
                    acc1[4 * q] = fmaf(x1, w0.x, fmaf(x0, w2.x, acc1[4 * q]));
                    acc1[4 * q + 1] = fmaf(x1, w0.y, fmaf(x0, w2.y, acc1[4 * q + 1]));
                    acc1[4 * q + 2] = fmaf(x1, w0.z, fmaf(x0, w2.z, acc1[4 * q + 2]));
                    acc1[4 * q + 3] = fmaf(x1, w0.w, fmaf(x0, w2.w, acc1[4 * q + 3]));
                }
            }
        }
    }
    const int od = 2 * i + pd, oh = 2 * j + ph, ow = 2 * l;
    if (j >= H || l >= W || od >= Do || oh >= Ho) return;
    const bool pair = ow + 1 < Wo && (Wo & 1) == 0;  // even rows: 8-byte aligned pairs
    for (int c = 0; c < kCo; ++c) {
        float* dst = y + ((((long long)n * C_out + cb * kCo + c) * Do + od) * Ho + oh) * (long long)Wo + ow;
        if (pair) {
            *reinterpret_cast<float2*>(dst) = make_float2(acc0[c], acc1[c]);
        } else {
            dst[0] = acc0[c];
            if (ow + 1 < Wo) dst[1] = acc1[c];
        }
    }
}

}  // namespace

cudaError_t launch_conv_transpose3d(const c1n_convt3d_params& p, const float* x, const float* w, const float* b,
                                    float* y, cudaStream_t stream) {
    const int Do = 2 * p.D - 1 + p.out_pad, Ho = 2 * p.H - 1 + p.out_pad, Wo = 2 * p.W - 1 + p.out_pad;
    const unsigned gx = (unsigned)(((p.W + kTL - 1) / kTL) * ((p.H + kTJ - 1) / kTJ));
    const unsigned gy = (unsigned)(p.D * 4 * (p.C_out / kCo));
    conv_transpose3d_k3s2_kernel<<<dim3(gx, gy, (unsigned)p.N), 256, 0, stream>>>(p.C_in, p.C_out, p.D, p.H, p.W, Do, Ho,
                                                                                  Wo, x, w, b, y);
    return cudaGetLastError();
}

}  // namespace c1n

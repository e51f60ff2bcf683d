// Oracle for the fused Conv1d + normalization operator.
//
// TEST INFRASTRUCTURE ONLY. This file is a plain, slow, obviously correct CPU
// statement of what the operator computes. Only the test-suite, the smoke check
// and the benchmark's CPU-baseline leg may load it. It shares no code, header,
// table or helper with the CUDA library, and the CUDA library never calls it.
//
// Everything is direct loops in double precision; no BLAS, no SIMD intrinsics,
// no blocking or reordering beyond the definitions below. Inputs are float32
// values (bf16 workloads hand over the already-rounded values); outputs are double.
//
// Sources (web pages on the subject "gemm_groupnorm_accelerator"):
//   [p1] Kimi-K2.6 l2_p35 page: Conv1d(128->256, k=3, s=1, p=1) + GroupNorm(32).
//   [p2] Kimi-K2.6 l2_p75 page: Linear(8192->8192) + GroupNorm(512) + min(dim=1) + bias.
//   [p3] Kimi-K2.6 l1_p5 page: causal Conv1d, k=4, left pad (k-1)*dilation.
//   [p4] Kimi-K2.6 l2_p3 page: LayerNorm with affine and exact-erf GELU; its second operator
//        (scalar add, LayerNorm over the last dimension, AvgPool3d 2x2x2, GELU).
//
// Parity pins: every function below is pinned by tests that do not re-run this
// code's formulas (delta kernels, the worked causal example of [p3], GELU(1)
// from [p4], library routines in float64, and closed-form invariants).
// The whole-pipeline composition is pinned through those parts plus a float64
// library composition; no function here is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// Shape of one operator call, mirrored by a ctypes structure on the Python side.
struct OracleParams {
    int32_t N, C_in, C_out, T, k, stride, pad_left, pad_right, dilation;
    int32_t norm;    // 0 none, 1 GroupNorm, 2 channel LayerNorm
    int32_t groups;  // GroupNorm group count
    float eps;
    int32_t post;    // 0 none, 1 exact GELU, 2 row-min + broadcast bias
};

// Output length of a 1-D convolution with separate left/right padding
// ([p1] output-length paragraph; [p3] causal padding paragraph):
//   T_out = floor((T + pad_left + pad_right - dilation*(k-1) - 1) / stride) + 1.
long t_out_of(long T, long k, long s, long pl, long pr, long d) {
    long span = T + pl + pr - d * (k - 1) - 1;
    if (span < 0) return 0;
    return span / s + 1;
}

template <class F>
void parallel_for(long n, int nthreads, F f) {
    if (nthreads <= 1 || n <= 1) {
        for (long i = 0; i < n; ++i) f(i);
        return;
    }
    std::vector<std::thread> pool;
    long per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        long lo = t * per, hi = lo + per < n ? lo + per : n;
        if (lo >= hi) break;
        pool.emplace_back([=]() { for (long i = lo; i < hi; ++i) f(i); });
    }
    for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

long oracle_t_out(int T, int k, int stride, int pad_left, int pad_right, int dilation) {
    if (T < 1 || k < 1 || stride < 1 || dilation < 1 || pad_left < 0 || pad_right < 0) return -1;
    return t_out_of(T, k, stride, pad_left, pad_right, dilation);
}

// Direct convolution ([p1] convolution sum; [p3] causal form):
//   c[n][co][t] = b[co] + sum_{ci} sum_{kk} w[co][ci][kk] * X(n, ci, t*stride + kk*dilation - pad_left)
// with X = 0 outside [0, T). Tap kk = 0 is the oldest input of the window.
// Layouts: x [N][C_in][T], w [C_out][C_in][k], b [C_out] or null, out [N][C_out][T_out].
int oracle_conv1d(const OracleParams* p, const float* x, const float* w, const float* b, double* out,
                  int nthreads) {
    const long T_out = oracle_t_out(p->T, p->k, p->stride, p->pad_left, p->pad_right, p->dilation);
    if (T_out <= 0) return -1;
    const long N = p->N, Ci = p->C_in, Co = p->C_out, T = p->T, K = p->k;
    parallel_for(N * Co, nthreads, [&](long job) {
        const long n = job / Co, co = job % Co;
        for (long t = 0; t < T_out; ++t) {
            double acc = 0.0;
            for (long ci = 0; ci < Ci; ++ci) {
                for (long kk = 0; kk < K; ++kk) {
                    const long pos = t * p->stride + kk * p->dilation - p->pad_left;
                    if (pos < 0 || pos >= T) continue;
                    acc += (double)w[(co * Ci + ci) * K + kk] * (double)x[(n * Ci + ci) * T + pos];
                }
            }
            if (b) acc += (double)b[co];
            out[(n * Co + co) * T_out + t] = acc;
        }
    });
    return 0;
}

// GroupNorm ([p1] GroupNorm semantics; [p2] the 2-D [rows, channels] case):
// channels of group g are [g*C/G, (g+1)*C/G); statistics run over those
// channels and all L positions of one sample; variance is the population
// variance, computed in two passes; eps sits inside the square root; gamma and
// beta are per channel (null means 1 and 0).
int oracle_group_norm(int N, int C, long L, int G, float eps, const double* in, const float* gamma,
                      const float* beta, double* out) {
    if (G < 1 || C % G != 0 || !(eps > 0.0f)) return -1;
    const long cpg = C / G;
    for (long n = 0; n < N; ++n) {
        for (long g = 0; g < G; ++g) {
            const double* src = in + (n * C + g * cpg) * L;
            const long cnt = cpg * L;
            double sum = 0.0;
            for (long i = 0; i < cnt; ++i) sum += src[i];
            const double mean = sum / (double)cnt;
            double ss = 0.0;
            for (long i = 0; i < cnt; ++i) ss += (src[i] - mean) * (src[i] - mean);
            const double var = ss / (double)cnt;
            const double inv = 1.0 / std::sqrt(var + (double)eps);
            for (long c = 0; c < cpg; ++c) {
                const long ch = g * cpg + c;
                const double ga = gamma ? (double)gamma[ch] : 1.0;
                const double be = beta ? (double)beta[ch] : 0.0;
                for (long l = 0; l < L; ++l) {
                    const long idx = (n * C + ch) * L + l;
                    out[idx] = (in[idx] - mean) * inv * ga + be;
                }
            }
        }
    }
    return 0;
}

// Channel LayerNorm: for every (n, l) the statistics run over all C channels;
// population variance in two passes; eps inside the square root; per-channel
// gamma and beta ([p4] LayerNorm-with-affine paragraphs, applied along the
// channel axis as the operator's descriptor specifies).
int oracle_channel_layer_norm(int N, int C, long L, float eps, const double* in, const float* gamma,
                              const float* beta, double* out) {
    if (C < 1 || !(eps > 0.0f)) return -1;
    for (long n = 0; n < N; ++n) {
        for (long l = 0; l < L; ++l) {
            double sum = 0.0;
            for (long c = 0; c < C; ++c) sum += in[(n * C + c) * L + l];
            const double mean = sum / (double)C;
            double ss = 0.0;
            for (long c = 0; c < C; ++c) {
                const double d = in[(n * C + c) * L + l] - mean;
                ss += d * d;
            }
            const double inv = 1.0 / std::sqrt(ss / (double)C + (double)eps);
            for (long c = 0; c < C; ++c) {
                const long idx = (n * C + c) * L + l;
                const double ga = gamma ? (double)gamma[c] : 1.0;
                const double be = beta ? (double)beta[c] : 0.0;
                out[idx] = (in[idx] - mean) * inv * ga + be;
            }
        }
    }
    return 0;
}

// Exact GELU ([p4] GELU paragraphs): GELU(z) = 0.5 * z * (1 + erf(z / sqrt(2))).
void oracle_gelu_erf(long n, const double* in, double* out) {
    const double inv_sqrt2 = 1.0 / std::sqrt(2.0);
    for (long i = 0; i < n; ++i) out[i] = 0.5 * in[i] * (1.0 + std::erf(in[i] * inv_sqrt2));
}

// Row-min plus broadcast bias ([p2] min over dim=1 then + bias of shape
// (1, C, 1, 1)): for every (n, l), m = min over channels c of in[n][c][l],
// argmin = the lowest channel index attaining m, and out[n][c][l] = m + bias2[c].
int oracle_rowmin_bias(int N, int C, long L, const double* in, const float* bias2, double* out,
                       int32_t* argmin) {
    if (C < 1 || !bias2) return -1;
    for (long n = 0; n < N; ++n) {
        for (long l = 0; l < L; ++l) {
            double m = std::numeric_limits<double>::infinity();
            long am = 0;
            for (long c = 0; c < C; ++c) {
                const double v = in[(n * C + c) * L + l];
                if (v < m) { m = v; am = c; }
            }
            if (argmin) argmin[n * L + l] = (int32_t)am;
            for (long c = 0; c < C; ++c) out[(n * C + c) * L + l] = m + (double)bias2[c];
        }
    }
    return 0;
}

// The whole operator: conv (+ bias), then the normalization, then the post-op.
// y [N][C_out][T_out] (double); argmin [N][T_out] when post is row-min (nullable).
int oracle_conv1d_norm(const OracleParams* p, const float* x, const float* w, const float* b,
                       const float* gamma, const float* beta, const float* bias2, double* y,
                       int32_t* argmin, int nthreads) {
    const long T_out = oracle_t_out(p->T, p->k, p->stride, p->pad_left, p->pad_right, p->dilation);
    if (T_out <= 0) return -1;
    if (p->norm == 1 && (p->groups < 1 || p->C_out % p->groups != 0)) return -1;
    if (p->norm != 0 && !(p->eps > 0.0f)) return -1;
    if (p->post == 2 && !bias2) return -1;
    const long total = (long)p->N * p->C_out * T_out;
    if (oracle_conv1d(p, x, w, b, y, nthreads) != 0) return -1;
    std::vector<double> tmp;
    if (p->norm != 0) {
        tmp.assign(y, y + total);
        int rc = p->norm == 1
                     ? oracle_group_norm(p->N, p->C_out, T_out, p->groups, p->eps, tmp.data(), gamma, beta, y)
                     : oracle_channel_layer_norm(p->N, p->C_out, T_out, p->eps, tmp.data(), gamma, beta, y);
        if (rc != 0) return -1;
    }
    if (p->post == 1) {
        oracle_gelu_erf(total, y, y);
    } else if (p->post == 2) {
        tmp.assign(y, y + total);
        if (oracle_rowmin_bias(p->N, p->C_out, T_out, tmp.data(), bias2, y, argmin) != 0) return -1;
    }
    return 0;
}

// Sampled evaluation for large shapes: the full pipeline for the listed samples
// n (and for each of them every channel and time step) — used where the whole
// tensor is too large for the oracle but one sample's statistics are needed.
// y_n receives [count][C_out][T_out] for the samples in `ns`.
int oracle_conv1d_norm_samples(const OracleParams* p, const float* x, const float* w, const float* b,
                               const float* gamma, const float* beta, const float* bias2, const int32_t* ns,
                               int count, double* y_n, int32_t* argmin_n, int nthreads) {
    const long T_out = oracle_t_out(p->T, p->k, p->stride, p->pad_left, p->pad_right, p->dilation);
    if (T_out <= 0) return -1;
    OracleParams one = *p;
    one.N = 1;
    const long per_x = (long)p->C_in * p->T;
    const long per_y = (long)p->C_out * T_out;
    for (int i = 0; i < count; ++i) {
        if (ns[i] < 0 || ns[i] >= p->N) return -1;
        int rc = oracle_conv1d_norm(&one, x + (long)ns[i] * per_x, w, b, gamma, beta, bias2, y_n + i * per_y,
                                    argmin_n ? argmin_n + i * T_out : nullptr, nthreads);
        if (rc != 0) return rc;
    }
    return 0;
}

// [p4]'s transposed 3-D convolution (ConvTranspose3d, dilation 1), the plain gather form of its
// definition: output position o along each axis receives input i through tap k when
// o = i*stride - pad + k, so
//   y[n][co][od][oh][ow] = b[co] + sum_{ci, kd, kh, kw} x[n][ci][id][ih][iw] * w[ci][co][kd][kh][kw]
// over the taps for which id = (od + pad - kd) / stride (and likewise ih, iw) is a whole number
// inside the input. Output extent per axis: (in - 1)*stride - 2*pad + (k - 1) + output_pad + 1.
// Layouts: x [N][C_in][D][H][W], w [C_in][C_out][k][k][k] (cubic kernel), b [C_out] or null,
// y [N][C_out][Do][Ho][Wo] (double).
int oracle_conv_transpose3d(int N, int C_in, int C_out, int D, int H, int W, int k, int stride, int pad,
                            int out_pad, const float* x, const float* w, const float* b, double* y, int nthreads) {
    if (N < 1 || C_in < 1 || C_out < 1 || D < 1 || H < 1 || W < 1 || k < 1 || stride < 1 || pad < 0 ||
        out_pad < 0 || out_pad >= stride)
        return -1;
    const long Do = (long)(D - 1) * stride - 2 * pad + (k - 1) + out_pad + 1;
    const long Ho = (long)(H - 1) * stride - 2 * pad + (k - 1) + out_pad + 1;
    const long Wo = (long)(W - 1) * stride - 2 * pad + (k - 1) + out_pad + 1;
    if (Do < 1 || Ho < 1 || Wo < 1) return -1;
    // the input index of output o through tap kk, or -1 when there is none
    auto in_of = [&](long o, long kk, long extent) -> long {
        const long t = o + pad - kk;
        if (t < 0 || t % stride != 0) return -1;
        const long i = t / stride;
        return i < extent ? i : -1;
    };
    parallel_for((long)N * C_out, nthreads, [&](long job) {
        const long n = job / C_out, co = job % C_out;
        for (long od = 0; od < Do; ++od)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow) {
                    double acc = b ? (double)b[co] : 0.0;
                    for (long ci = 0; ci < C_in; ++ci)
                        for (long kd = 0; kd < k; ++kd) {
                            const long id = in_of(od, kd, D);
                            if (id < 0) continue;
                            for (long kh = 0; kh < k; ++kh) {
                                const long ih = in_of(oh, kh, H);
                                if (ih < 0) continue;
                                for (long kw = 0; kw < k; ++kw) {
                                    const long iw = in_of(ow, kw, W);
                                    if (iw < 0) continue;
                                    acc += (double)x[(((n * C_in + ci) * D + id) * H + ih) * W + iw] *
                                           (double)w[(((ci * C_out + co) * k + kd) * k + kh) * k + kw];
                                }
                            }
                        }
                    y[(((n * C_out + co) * Do + od) * Ho + oh) * Wo + ow] = acc;
                }
    });
    return 0;
}

// [p4]'s second operator, after its transposed convolution: add the scalar sum_weight, LayerNorm
// over the last (contiguous) dimension W with per-position gamma[W] / beta[W] (population variance
// in two passes, eps inside the square root), AvgPool3d with kernel 2 and stride 2 over (D, H, W)
// (floor: a trailing odd plane, row or column takes part in no window), then exact GELU.
// z [N][C][D][H][W]; out [N][C][D/2][H/2][W/2] (double). gamma / beta may be null (1 and 0).
// Only the (n, c) slices listed in `ncs` (count of them; null means all N*C in order) are
// evaluated, slice i of the output going to out + i * (D/2)*(H/2)*(W/2); z holds those slices
// in the same order (z + i * D*H*W).
int oracle_ln_avgpool3d_gelu(int D, int H, int W, float eps, float sum_weight, const float* z, const float* gamma,
                             const float* beta, int count, double* out, int nthreads) {
    if (D < 1 || H < 1 || W < 1 || count < 0 || !(eps > 0.0f)) return -1;
    const long D2 = D / 2, H2 = H / 2, W2 = W / 2;
    const double inv_sqrt2 = 1.0 / std::sqrt(2.0);
    parallel_for(count, nthreads, [&](long i) {
        const float* zs = z + i * (long)D * H * W;
        std::vector<double> ln((size_t)D * H * W);
        for (long d = 0; d < D; ++d) {
            for (long h = 0; h < H; ++h) {
                const float* row = zs + (d * H + h) * W;
                double* lr = ln.data() + (d * H + h) * W;
                double sum = 0.0;
                for (long w = 0; w < W; ++w) sum += (double)row[w] + (double)sum_weight;
                const double mean = sum / (double)W;
                double ss = 0.0;
                for (long w = 0; w < W; ++w) {
                    const double dv = (double)row[w] + (double)sum_weight - mean;
                    ss += dv * dv;
                }
                const double inv = 1.0 / std::sqrt(ss / (double)W + (double)eps);
                for (long w = 0; w < W; ++w) {
                    const double ga = gamma ? (double)gamma[w] : 1.0;
                    const double be = beta ? (double)beta[w] : 0.0;
                    lr[w] = ((double)row[w] + (double)sum_weight - mean) * inv * ga + be;
                }
            }
        }
        double* os = out + i * D2 * H2 * W2;
        for (long d2 = 0; d2 < D2; ++d2) {
            for (long h2 = 0; h2 < H2; ++h2) {
                for (long w2 = 0; w2 < W2; ++w2) {
                    double acc = 0.0;
                    for (long a = 0; a < 2; ++a)
                        for (long b = 0; b < 2; ++b)
                            for (long c = 0; c < 2; ++c)
                                acc += ln[((2 * d2 + a) * H + 2 * h2 + b) * W + 2 * w2 + c];
                    const double v = acc / 8.0;
                    os[(d2 * H2 + h2) * W2 + w2] = 0.5 * v * (1.0 + std::erf(v * inv_sqrt2));
                }
            }
        }
    });
    return 0;
}

}  // extern "C"

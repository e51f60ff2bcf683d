"""Seeded synthetic inputs for the fused Conv1d(implicit GEMM) + normalization operator.

This module is shared by the tests, the benchmark and the smoke check. It holds
only input generation (random numbers, value distributions and the five
workload shapes); none of the operator's arithmetic lives here.

Random numbers come from a counter-based generator: the SplitMix64 output
function (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) applied to ``stream_key + (i + 1) * 0x9E3779B97F4A7C15``
for element ``i``. Every tensor has its own stream key, derived from the seed and
a fixed tensor id, so tensors are independent of one another and of their
sizes, and the whole thing vectorises in numpy.

* uniform u in [0, 1): the top 53 bits of the 64-bit output times 2**-53;
* U(-a, a) = a * (2u - 1);
* N(mu, sigma): Box-Muller on two independent uniforms (element i uses the
  counter values 2i and 2i+1 of its stream), mu + sigma * sqrt(-2 ln(1-u1)) *
  cos(2 pi u2), computed in float64 and rounded once to float32.

bf16 inputs are float32 values rounded to the nearest bf16 (ties to even) by
``round_bf16``; both the oracle and the CUDA path consume exactly those values.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Dict, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Fixed stream ids, one per tensor role.
STREAM_X, STREAM_W, STREAM_B, STREAM_GAMMA, STREAM_BETA, STREAM_BIAS2 = 1, 2, 3, 4, 5, 6


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(stream) * _GOLDEN)
        return _mix64(np.array([k], dtype=np.uint64))[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """64-bit outputs for counters start .. start+count-1 of one stream."""
    key = _stream_key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GOLDEN)


def uniform01(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """float64 uniforms in [0, 1)."""
    return (raw_u64(seed, stream, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_CHUNK = 1 << 22
_pool = None


def _map_chunks(fn, count: int) -> None:
    """fn(s, n) for the chunks [s, s + n) of range(count), on a thread pool when there are several
    (numpy releases the interpreter lock in these array operations). Each chunk is a pure function
    of its counters, so the result does not depend on the thread count or order."""
    global _pool
    chunks = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]
    if len(chunks) <= 1:
        for s, n in chunks:
            fn(s, n)
        return
    if _pool is None:
        _pool = concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    list(_pool.map(lambda c: fn(*c), chunks))


def uniform_pm(seed: int, stream: int, count: int, a: float) -> np.ndarray:
    """float32 samples of U(-a, a)."""
    out = np.empty(count, dtype=np.float32)

    def fill(s, n):
        out[s:s + n] = (a * (2.0 * uniform01(seed, stream, n, start=s) - 1.0)).astype(np.float32)

    _map_chunks(fill, count)
    return out


def normal_slice(seed: int, stream: int, start: int, count: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """Elements start .. start+count-1 of the stream's N(mu, sigma) sequence (float32)."""
    out = np.empty(count, dtype=np.float32)

    def fill(s, n):
        u = uniform01(seed, stream, 2 * n, start=2 * (start + s))
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        out[s:s + n] = (mu + sigma * r * np.cos(2.0 * math.pi * u[1::2])).astype(np.float32)

    _map_chunks(fill, count)
    return out


def normal(seed: int, stream: int, count: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """float32 samples of N(mu, sigma) (sigma is the standard deviation)."""
    return normal_slice(seed, stream, 0, count, mu, sigma)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    r = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return (r & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-representable."""
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------------------------
# Workload shapes


NORM_NONE, NORM_GROUP, NORM_CHANNEL_LAYER = 0, 1, 2
POST_NONE, POST_GELU_ERF, POST_ROWMIN_BIAS = 0, 1, 2
DTYPE_F32, DTYPE_BF16 = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    """One operator configuration plus the distributions its inputs are drawn from."""

    name: str
    N: int
    C_in: int
    C_out: int
    T: int
    k: int
    stride: int = 1
    pad_left: int = 0
    pad_right: int = 0
    dilation: int = 1
    norm: int = NORM_NONE
    groups: int = 1
    eps: float = 1e-5
    post: int = POST_NONE
    dtype: int = DTYPE_F32
    has_bias: bool = True
    has_affine: bool = True
    w_bound: Optional[float] = None      # U(+-w_bound) for w and b; default 1/sqrt(C_in*k)
    description: str = ""

    @property
    def T_out(self) -> int:
        return (self.T + self.pad_left + self.pad_right - self.dilation * (self.k - 1) - 1) // self.stride + 1

    @property
    def gemm_mnk(self):
        return self.N * self.T_out, self.C_out, self.C_in * self.k

    @property
    def flops(self) -> float:
        m, n, k = self.gemm_mnk
        return 2.0 * m * n * k

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == DTYPE_BF16 else 4

    @property
    def algorithmic_bytes(self) -> int:
        """x + w read once, b/gamma/beta(/bias2) read once, y written once."""
        eb = self.elem_bytes
        b = self.N * self.C_in * self.T * eb + self.C_out * self.C_in * self.k * eb
        b += 4 * self.C_out * (int(self.has_bias) + 2 * int(self.has_affine and self.norm != NORM_NONE))
        if self.post == POST_ROWMIN_BIAS:
            b += 4 * self.C_out
        b += self.N * self.C_out * self.T_out * eb
        return b

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONV_GN_TINY = Workload(
    "conv1d_groupnorm_f32_n2_c16x32_t128", N=2, C_in=16, C_out=32, T=128, k=3, pad_left=1, pad_right=1,
    norm=NORM_GROUP, groups=4, description="Conv1d+GroupNorm fp32, N=2, C 16->32, T=128, k=3, pad 1/1, G=4")
CONV_GN = Workload(
    "conv1d_groupnorm_f32_n16_c128x256_t1024", N=16, C_in=128, C_out=256, T=1024, k=3, pad_left=1, pad_right=1,
    norm=NORM_GROUP, groups=32,
    description="Conv1d+GroupNorm fp32, N=16, C 128->256, T=1024, k=3, pad 1/1, G=32 (8 ch/group)")
CAUSAL_CONV = Workload(
    "causal_conv1d_f32_n32_c256x256_t8192_k4", N=32, C_in=256, C_out=256, T=8192, k=4, pad_left=3, pad_right=0,
    norm=NORM_NONE, w_bound=1.0 / 32.0,
    description="causal Conv1d fp32, no norm, N=32, C 256->256, T=8192, k=4, left pad 3")
LINEAR_GN_ROWMIN = Workload(
    "linear_groupnorm_rowmin_bias_f32_1024x8192x8192", N=1024, C_in=8192, C_out=8192, T=1, k=1,
    norm=NORM_GROUP, groups=512, post=POST_ROWMIN_BIAS,
    description="Linear 8192->8192 on 1024 rows + GroupNorm(512) + row-min + broadcast bias, fp32")
CONV_LN_GELU_BF16 = Workload(
    "conv1d_layernorm_gelu_bf16_n64_c256x512_t4096_k5_d2", N=64, C_in=256, C_out=512, T=4096, k=5, pad_left=4,
    pad_right=4, dilation=2, norm=NORM_CHANNEL_LAYER, post=POST_GELU_ERF, dtype=DTYPE_BF16,
    description="Conv1d+channel-LayerNorm+exact GELU bf16 (fp32 accumulate), N=64, C 256->512, T=4096, k=5, dil 2, pad 4/4")

WORKLOADS = [CONV_GN_TINY, CONV_GN, CAUSAL_CONV, LINEAR_GN_ROWMIN, CONV_LN_GELU_BF16]

# The largest fp32 output of the five with GroupNorm switched on (G = 32, 8 channels per group):
# the shape on which the memory-bound statistics / normalize passes of the two-pass plan are
# measured (268 MB of raw fp32 output read back and rewritten).
CAUSAL_CONV_GN32 = CAUSAL_CONV.replace(
    name="causal_conv1d_groupnorm32_f32_n32_c256x256_t8192_k4", norm=NORM_GROUP, groups=32,
    description="causal Conv1d fp32 + GroupNorm(32), N=32, C 256->256, T=8192, k=4, left pad 3")

BY_NAME: Dict[str, Workload] = {w.name: w for w in WORKLOADS + [CAUSAL_CONV_GN32]}


def make_inputs(wl: Workload, seed: int = 0, n_rows: Optional[int] = None, row_offset: int = 0) -> Dict[str, np.ndarray]:
    """Draw the inputs of ``wl`` (float32 arrays; bf16 workloads get bf16-rounded values).

    ``n_rows`` / ``row_offset`` draw only batch entries [row_offset, row_offset + n_rows) of x
    (the counter-based generator makes any such slice identical to the same rows of a larger
    draw); parameters are the same for every slice.
    """
    n = wl.N if n_rows is None else n_rows
    a = wl.w_bound if wl.w_bound is not None else 1.0 / math.sqrt(wl.C_in * wl.k)
    per_row = wl.C_in * wl.T
    x = normal_slice(seed, STREAM_X, row_offset * per_row, n * per_row).reshape(n, wl.C_in, wl.T)
    w = uniform_pm(seed, STREAM_W, wl.C_out * wl.C_in * wl.k, a).reshape(wl.C_out, wl.C_in, wl.k)
    out = {"x": x, "w": w}
    out["b"] = uniform_pm(seed, STREAM_B, wl.C_out, a) if wl.has_bias else None
    if wl.norm != NORM_NONE and wl.has_affine:
        out["gamma"] = normal(seed, STREAM_GAMMA, wl.C_out, 1.0, 0.1)
        out["beta"] = normal(seed, STREAM_BETA, wl.C_out, 0.0, 0.1)
    else:
        out["gamma"] = None
        out["beta"] = None
    out["bias2"] = normal(seed, STREAM_BIAS2, wl.C_out, 0.0, 1.0) if wl.post == POST_ROWMIN_BIAS else None
    if wl.dtype == DTYPE_BF16:
        out["x"] = round_bf16(out["x"])
        out["w"] = round_bf16(out["w"])
    return out


# ----------------------------------------------------------------------------------------------
# [p4]'s second operator: add a scalar, LayerNorm over the last dimension, AvgPool3d 2x2x2, GELU


@dataclasses.dataclass(frozen=True)
class LnPoolWorkload:
    """Shape of the LayerNorm(W) + AvgPool3d + GELU pass: z [N][C][D][H][W] fp32 (in [p4] the
    output of ConvTranspose3d(32 -> 64, k 3, stride 2, pad 1, output pad 1) on x [32, 32, 16, 32,
    32]); gamma / beta [W]; a scalar added before the LayerNorm."""

    name: str
    N: int
    C: int
    D: int
    H: int
    W: int
    eps: float = 1e-5
    sum_weight: float = 1.0
    has_affine: bool = True
    description: str = ""

    @property
    def out_shape(self):
        return (self.N, self.C, self.D // 2, self.H // 2, self.W // 2)

    @property
    def algorithmic_bytes(self) -> int:
        """z read once, gamma / beta read once, the pooled output written once (fp32)."""
        n_in = self.N * self.C * self.D * self.H * self.W
        n_out = self.N * self.C * (self.D // 2) * (self.H // 2) * (self.W // 2)
        return 4 * (n_in + n_out + (2 * self.W if self.has_affine else 0))

    def replace(self, **kw) -> "LnPoolWorkload":
        return dataclasses.replace(self, **kw)


LN_AVGPOOL3D_GELU = LnPoolWorkload(
    "layernorm_w_avgpool3d_gelu_f32_n32_c64_d32_h64_w64", N=32, C=64, D=32, H=64, W=64,
    description="+ scalar, LayerNorm over W=64, AvgPool3d 2x2x2, exact GELU, fp32, z [32,64,32,64,64]")


def make_lnpool_inputs(wl: LnPoolWorkload, seed: int = 0, n_slices: Optional[int] = None,
                       slice_offset: int = 0) -> Dict[str, np.ndarray]:
    """z ~ N(0, 1) (standing in for the transposed convolution's output), gamma ~ N(1, 0.1),
    beta ~ N(0, 0.1). ``n_slices`` / ``slice_offset`` draw only the (n, c) slices [slice_offset,
    slice_offset + n_slices) in n-major order, returned as [n_slices][D][H][W]."""
    per = wl.D * wl.H * wl.W
    total = wl.N * wl.C
    n = total if n_slices is None else n_slices
    z = normal_slice(seed, STREAM_X, slice_offset * per, n * per)
    z = z.reshape(wl.N, wl.C, wl.D, wl.H, wl.W) if n_slices is None else z.reshape(n, wl.D, wl.H, wl.W)
    out = {"z": z, "gamma": None, "beta": None}
    if wl.has_affine:
        out["gamma"] = normal(seed, STREAM_GAMMA, wl.W, 1.0, 0.1)
        out["beta"] = normal(seed, STREAM_BETA, wl.W, 0.0, 0.1)
    return out


@dataclasses.dataclass(frozen=True)
class ConvT3dWorkload:
    """[p4]'s ConvTranspose3d (cubic kernel, dilation 1, with bias) whose output feeds the
    LayerNorm(W) + AvgPool3d + GELU pass."""

    name: str
    N: int
    C_in: int
    C_out: int
    D: int
    H: int
    W: int
    k: int = 3
    stride: int = 2
    pad: int = 1
    out_pad: int = 1
    description: str = ""

    @property
    def out_dhw(self):
        f = lambda n: (n - 1) * self.stride - 2 * self.pad + (self.k - 1) + self.out_pad + 1
        return f(self.D), f(self.H), f(self.W)

    @property
    def macs(self) -> int:
        """Multiply-adds that meet an input voxel (taps that fall outside the input do not count)."""
        total = 0
        Do, Ho, Wo = self.out_dhw
        per_axis = []
        for n_in, n_out in ((self.D, Do), (self.H, Ho), (self.W, Wo)):
            cnt = 0
            for o in range(n_out):
                for kk in range(self.k):
                    t = o + self.pad - kk
                    if t >= 0 and t % self.stride == 0 and t // self.stride < n_in:
                        cnt += 1
            per_axis.append(cnt)
        total = per_axis[0] * per_axis[1] * per_axis[2]
        return self.N * self.C_out * self.C_in * total

    @property
    def flops(self) -> float:
        return 2.0 * self.macs

    @property
    def algorithmic_bytes(self) -> int:
        """fp32 x, w and b read once and y written once."""
        Do, Ho, Wo = self.out_dhw
        x = self.N * self.C_in * self.D * self.H * self.W
        w = self.C_in * self.C_out * self.k ** 3
        y = self.N * self.C_out * Do * Ho * Wo
        return 4 * (x + w + self.C_out + y)

    def replace(self, **kw) -> "ConvT3dWorkload":
        return dataclasses.replace(self, **kw)


CONV_TRANSPOSE3D = ConvT3dWorkload(
    "conv_transpose3d_f32_n32_c32x64_d16_h32_w32_k3_s2", N=32, C_in=32, C_out=64, D=16, H=32, W=32,
    description="ConvTranspose3d 32->64, k 3, stride 2, pad 1, output pad 1, fp32: x [32,32,16,32,32] -> [32,64,32,64,64]")


def make_convt3d_inputs(wl: ConvT3dWorkload, seed: int = 0, n_rows: Optional[int] = None,
                        row_offset: int = 0) -> Dict[str, np.ndarray]:
    """x ~ N(0, 1); w, b ~ U(+-1/sqrt(C_in*k^3)). ``n_rows`` / ``row_offset`` draw batch entries only."""
    n = wl.N if n_rows is None else n_rows
    per = wl.C_in * wl.D * wl.H * wl.W
    a = 1.0 / math.sqrt(wl.C_in * wl.k ** 3)
    x = normal_slice(seed, STREAM_X, row_offset * per, n * per).reshape(n, wl.C_in, wl.D, wl.H, wl.W)
    w = uniform_pm(seed, STREAM_W, wl.C_in * wl.C_out * wl.k ** 3, a).reshape(wl.C_in, wl.C_out, wl.k, wl.k, wl.k)
    return {"x": x, "w": w, "b": uniform_pm(seed, STREAM_B, wl.C_out, a)}

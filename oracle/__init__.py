"""CPU oracle for the fused Conv1d + normalization operator (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. It shares no code with the CUDA library and the CUDA
library never reaches it. The arithmetic lives in ``oracle.cpp`` (plain C++17,
double precision, direct loops); this module compiles it with g++ and marshals
numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("N", "C_in", "C_out", "T", "k", "stride", "pad_left", "pad_right", "dilation", "norm", "groups")]
    _fields_ += [("eps", ctypes.c_float), ("post", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile oracle.cpp into a shared library next to it (g++, -O2, portable flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            f32p, f64p, i32p = P(ctypes.c_float), P(ctypes.c_double), P(ctypes.c_int32)
            lib.oracle_t_out.restype = ctypes.c_long
            lib.oracle_t_out.argtypes = [ctypes.c_int] * 6
            lib.oracle_conv1d.argtypes = [P(OracleParams), f32p, f32p, f32p, f64p, ctypes.c_int]
            lib.oracle_group_norm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_float,
                                              f64p, f32p, f32p, f64p]
            lib.oracle_channel_layer_norm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_float,
                                                      f64p, f32p, f32p, f64p]
            lib.oracle_gelu_erf.argtypes = [ctypes.c_long, f64p, f64p]
            lib.oracle_gelu_erf.restype = None
            lib.oracle_rowmin_bias.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_long, f64p, f32p, f64p, i32p]
            lib.oracle_conv1d_norm.argtypes = [P(OracleParams), f32p, f32p, f32p, f32p, f32p, f32p, f64p, i32p,
                                               ctypes.c_int]
            lib.oracle_conv_transpose3d.argtypes = [ctypes.c_int] * 10 + [f32p, f32p, f32p, f64p, ctypes.c_int]
            lib.oracle_ln_avgpool3d_gelu.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                                     ctypes.c_float, f32p, f32p, f32p, ctypes.c_int, f64p, ctypes.c_int]
            lib.oracle_conv1d_norm_samples.argtypes = [P(OracleParams), f32p, f32p, f32p, f32p, f32p, f32p, i32p,
                                                       ctypes.c_int, f64p, i32p, ctypes.c_int]
            _lib = lib
    return _lib


def _f32(a: Optional[np.ndarray]):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f64(a: np.ndarray):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def params(N, C_in, C_out, T, k, stride=1, pad_left=0, pad_right=0, dilation=1, norm=0, groups=1, eps=1e-5,
           post=0) -> OracleParams:
    return OracleParams(N, C_in, C_out, T, k, stride, pad_left, pad_right, dilation, norm, groups, eps, post)


def params_of(wl) -> OracleParams:
    """OracleParams from a synth.Workload (shape fields only)."""
    return params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation, wl.norm,
                  wl.groups, wl.eps, wl.post)


def t_out(T, k, stride=1, pad_left=0, pad_right=0, dilation=1) -> int:
    return int(_load().oracle_t_out(T, k, stride, pad_left, pad_right, dilation))


def conv1d(p: OracleParams, x, w, b=None, nthreads: Optional[int] = None) -> np.ndarray:
    lib = _load()
    To = t_out(p.T, p.k, p.stride, p.pad_left, p.pad_right, p.dilation)
    x, xp = _f32(x)
    w, wp = _f32(w)
    b, bp = _f32(b)
    out = np.empty((p.N, p.C_out, To), dtype=np.float64)
    rc = lib.oracle_conv1d(ctypes.byref(p), xp, wp, bp, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                           nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_conv1d rejected its arguments")
    return out


def group_norm(inp: np.ndarray, G: int, eps: float, gamma=None, beta=None) -> np.ndarray:
    lib = _load()
    N, C, L = inp.shape
    inp, ip = _f64(inp)
    gamma, gp = _f32(gamma)
    beta, bp = _f32(beta)
    out = np.empty_like(inp)
    rc = lib.oracle_group_norm(N, C, L, G, eps, ip, gp, bp, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_group_norm rejected its arguments")
    return out


def channel_layer_norm(inp: np.ndarray, eps: float, gamma=None, beta=None) -> np.ndarray:
    lib = _load()
    N, C, L = inp.shape
    inp, ip = _f64(inp)
    gamma, gp = _f32(gamma)
    beta, bp = _f32(beta)
    out = np.empty_like(inp)
    rc = lib.oracle_channel_layer_norm(N, C, L, eps, ip, gp, bp, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_channel_layer_norm rejected its arguments")
    return out


def gelu_erf(inp: np.ndarray) -> np.ndarray:
    lib = _load()
    inp, ip = _f64(inp)
    out = np.empty_like(inp)
    lib.oracle_gelu_erf(inp.size, ip, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def rowmin_bias(inp: np.ndarray, bias2):
    lib = _load()
    N, C, L = inp.shape
    inp, ip = _f64(inp)
    bias2, bp = _f32(bias2)
    out = np.empty_like(inp)
    am = np.empty((N, L), dtype=np.int32)
    rc = lib.oracle_rowmin_bias(N, C, L, ip, bp, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                am.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    if rc != 0:
        raise ValueError("oracle_rowmin_bias rejected its arguments")
    return out, am


def conv1d_norm(p: OracleParams, x, w, b=None, gamma=None, beta=None, bias2=None, nthreads: Optional[int] = None):
    """The whole operator; returns (y float64 [N][C_out][T_out], argmin int32 [N][T_out] or None)."""
    lib = _load()
    To = t_out(p.T, p.k, p.stride, p.pad_left, p.pad_right, p.dilation)
    if To <= 0:
        raise ValueError("empty output length")
    arrs = [_f32(a) for a in (x, w, b, gamma, beta, bias2)]
    y = np.empty((p.N, p.C_out, To), dtype=np.float64)
    am = np.empty((p.N, To), dtype=np.int32) if p.post == 2 else None
    rc = lib.oracle_conv1d_norm(ctypes.byref(p), *[a[1] for a in arrs],
                                y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                None if am is None else am.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_conv1d_norm rejected its arguments")
    return y, am


def conv1d_norm_samples(p: OracleParams, ns, x, w, b=None, gamma=None, beta=None, bias2=None,
                        nthreads: Optional[int] = None):
    """The whole operator for the batch entries listed in ``ns`` only (x holds all N entries)."""
    lib = _load()
    To = t_out(p.T, p.k, p.stride, p.pad_left, p.pad_right, p.dilation)
    ns = np.ascontiguousarray(ns, dtype=np.int32)
    arrs = [_f32(a) for a in (x, w, b, gamma, beta, bias2)]
    y = np.empty((len(ns), p.C_out, To), dtype=np.float64)
    am = np.empty((len(ns), To), dtype=np.int32) if p.post == 2 else None
    rc = lib.oracle_conv1d_norm_samples(ctypes.byref(p), *[a[1] for a in arrs],
                                        ns.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(ns),
                                        y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                        None if am is None else am.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_conv1d_norm_samples rejected its arguments")
    return y, am


def ln_avgpool3d_gelu(z: np.ndarray, eps: float, sum_weight: float, gamma=None, beta=None,
                      nthreads: Optional[int] = None) -> np.ndarray:
    """[p4]'s add + LayerNorm(last dim) + AvgPool3d(2) + GELU on z [..., D, H, W] (float32), every
    leading index an independent slice; returns [..., D//2, H//2, W//2] in float64."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    *lead, D, H, W = z.shape
    count = int(np.prod(lead)) if lead else 1
    lib = _load()
    out = np.empty((count, D // 2, H // 2, W // 2), dtype=np.float64)
    gp, bp = _f32(gamma), _f32(beta)
    rc = lib.oracle_ln_avgpool3d_gelu(D, H, W, eps, sum_weight, z.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                      gp[1], bp[1], count, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                      nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_ln_avgpool3d_gelu rejected its arguments")
    return out.reshape(*lead, D // 2, H // 2, W // 2)


def conv_transpose3d_shape(D, H, W, k, stride, pad, out_pad):
    f = lambda n: (n - 1) * stride - 2 * pad + (k - 1) + out_pad + 1
    return f(D), f(H), f(W)


def conv_transpose3d(x: np.ndarray, w: np.ndarray, b=None, stride: int = 1, pad: int = 0, out_pad: int = 0,
                     nthreads: Optional[int] = None) -> np.ndarray:
    """[p4]'s ConvTranspose3d: x [N][C_in][D][H][W], w [C_in][C_out][k][k][k] float32 -> float64 output."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, C_in, D, H, W = x.shape
    _, C_out, k, _, _ = w.shape
    Do, Ho, Wo = conv_transpose3d_shape(D, H, W, k, stride, pad, out_pad)
    lib = _load()
    out = np.empty((N, C_out, Do, Ho, Wo), dtype=np.float64)
    bp = _f32(b)
    rc = lib.oracle_conv_transpose3d(N, C_in, C_out, D, H, W, k, stride, pad, out_pad,
                                     x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                     w.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), bp[1],
                                     out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_conv_transpose3d rejected its arguments")
    return out

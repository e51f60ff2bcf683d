"""Python binding of the conv1d_norm C ABI (``include/conv1d_norm.h``).

Argument marshalling only: every step of the operator runs in the CUDA library
(``libconv1dnorm.so``, built in-tree for sm_103a). The functions below carry the
C names; ``Conv1dNorm`` is a small convenience wrapper that allocates the workspace
and outputs with PyTorch and passes raw device pointers and the current stream.
There is no fallback: if the library is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build_lib

NORM_NONE, NORM_GROUP, NORM_CHANNEL_LAYER = 0, 1, 2
POST_NONE, POST_GELU_ERF, POST_ROWMIN_BIAS = 0, 1, 2
F32, BF16 = 0, 1
MATH_AUTO, MATH_SIMT, MATH_TENSOR, MATH_TENSOR_X3 = 0, 1, 2, 3
MAINLOOP_AUTO, MAINLOOP_SINGLE, MAINLOOP_PAIR = 0, 1, 2
PATH_AUTO, PATH_SIMT, PATH_TC_DIRECT, PATH_TC_FUSED_GN, PATH_TC_TWO_PASS, PATH_TC_LINEAR = -1, 0, 1, 2, 3, 4
PATH_TC_FUSED_GN_DSMEM, PATH_TC_FUSED_LN = 5, 6
PATH_NAMES = {0: "simt", 1: "tc_direct", 2: "tc_fused_gn", 3: "tc_two_pass", 4: "tc_linear", 5: "tc_fused_gn_dsmem",
              6: "tc_fused_ln"}

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(8)

EXPORTED_SYMBOLS = (
    "conv1d_norm_desc_create", "conv1d_norm_workspace_size", "conv1d_norm_set_workspace", "conv1d_norm_plan_info",
    "conv1d_norm_run", "conv1d_norm_run_ex", "conv1d_norm_pack_weights", "conv1d_norm_check", "conv1d_norm_destroy",
    "conv1d_norm_status_string", "conv1d_norm_last_error", "conv1d_norm_version", "conv1d_norm_run_static_scratch",
    "conv1d_norm_set_profiling", "conv1d_norm_kernel_times", "ln_avgpool3d_gelu_run",
    "conv_transpose3d_run", "conv_transpose3d_workspace_size",
    "conv_transpose3d_ln_avgpool3d_gelu_run", "conv_transpose3d_ln_avgpool3d_gelu_workspace_size",
)

STATIC_SCRATCH_BYTES = 4 << 20  # C1N_STATIC_SCRATCH_BYTES


class LnPoolParams(ctypes.Structure):
    """c1n_lnpool_params: z [N][C][D][H][W] fp32 and the LayerNorm eps."""
    _fields_ = [(n, ctypes.c_int32) for n in ("N", "C", "D", "H", "W")] + [("eps", ctypes.c_float)]


class ConvT3dParams(ctypes.Structure):
    """c1n_convt3d_params: x [N][C_in][D][H][W], cubic kernel k, stride, pad, output pad."""
    _fields_ = [(n, ctypes.c_int32) for n in ("N", "C_in", "C_out", "D", "H", "W", "k", "stride", "pad", "out_pad",
                                              "math")]


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("N", "C_in", "C_out", "T", "k", "stride", "pad_left", "pad_right", "dilation", "norm", "groups")]
    _fields_ += [("eps", ctypes.c_float)] + [(n, ctypes.c_int32) for n in ("post", "dtype", "math", "force_path",
                                                                          "mainloop")]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("path", "T_out", "tile_t", "tile_co", "mma_n", "cluster", "n_tiles", "grid", "kernels", "cta_pair")]
    _fields_ += [("workspace_bytes", ctypes.c_int64)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("ms", ctypes.c_float)]


class Args(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("w", ctypes.c_void_p), ("b", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("bias2", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("argmin", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("flags", ctypes.c_uint32)]


FLAG_WEIGHTS_PACKED = 1
FLAG_TEST_STALL_EXCHANGE = 2  # testing aid: see C1N_FLAG_TEST_STALL_EXCHANGE in the C header


class C1NError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"conv1d_norm status {status}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    return _build_lib.build(force=force)


def library_path() -> str:
    return _build_lib.LIB


def load(build_if_missing: bool = True):
    """Load libconv1dnorm.so (building it first if needed). Raises if it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build_lib.LIB
        if build_if_missing:
            path = _build_lib.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run build()")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER
        vp = ctypes.c_void_p
        lib.conv1d_norm_desc_create.argtypes = [P(Params), P(vp)]
        lib.conv1d_norm_workspace_size.argtypes = [vp, P(ctypes.c_size_t)]
        lib.conv1d_norm_set_workspace.argtypes = [vp, vp, ctypes.c_size_t]
        lib.conv1d_norm_plan_info.argtypes = [vp, P(PlanInfo)]
        lib.conv1d_norm_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        lib.conv1d_norm_run_ex.argtypes = [vp, P(Args), vp]
        lib.conv1d_norm_pack_weights.argtypes = [vp, vp, vp, ctypes.c_size_t, vp]
        lib.conv1d_norm_check.argtypes = [vp, vp, vp]
        lib.conv1d_norm_run_static_scratch.argtypes = [vp, P(Args), vp]
        lib.conv1d_norm_set_profiling.argtypes = [vp, ctypes.c_int32]
        lib.conv1d_norm_kernel_times.argtypes = [vp, P(KernelTime), ctypes.c_int32, P(ctypes.c_int32)]
        lib.conv1d_norm_destroy.argtypes = [vp]
        lib.conv1d_norm_destroy.restype = None
        lib.conv1d_norm_status_string.argtypes = [ctypes.c_int]
        lib.conv1d_norm_status_string.restype = ctypes.c_char_p
        lib.conv1d_norm_last_error.argtypes = []
        lib.conv1d_norm_last_error.restype = ctypes.c_char_p
        lib.conv1d_norm_version.restype = ctypes.c_int32
        lib.ln_avgpool3d_gelu_run.argtypes = [P(LnPoolParams), vp, ctypes.c_float, vp, vp, vp, vp]
        lib.ln_avgpool3d_gelu_run.restype = ctypes.c_int
        lib.conv_transpose3d_run.argtypes = [P(ConvT3dParams), vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.conv_transpose3d_run.restype = ctypes.c_int
        lib.conv_transpose3d_workspace_size.argtypes = [P(ConvT3dParams), P(ctypes.c_size_t)]
        lib.conv_transpose3d_workspace_size.restype = ctypes.c_int
        lib.conv_transpose3d_ln_avgpool3d_gelu_run.argtypes = [P(ConvT3dParams), ctypes.c_float, ctypes.c_float, vp, vp,
                                                               vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.conv_transpose3d_ln_avgpool3d_gelu_run.restype = ctypes.c_int
        lib.conv_transpose3d_ln_avgpool3d_gelu_workspace_size.argtypes = [P(ConvT3dParams), P(ctypes.c_size_t)]
        lib.conv_transpose3d_ln_avgpool3d_gelu_workspace_size.restype = ctypes.c_int
        for name in ("conv1d_norm_desc_create", "conv1d_norm_workspace_size", "conv1d_norm_set_workspace",
                     "conv1d_norm_plan_info", "conv1d_norm_run", "conv1d_norm_run_ex", "conv1d_norm_pack_weights",
                     "conv1d_norm_check", "conv1d_norm_run_static_scratch", "conv1d_norm_set_profiling",
                     "conv1d_norm_kernel_times"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int):
    if status != OK:
        lib = load()
        raise C1NError(status, (lib.conv1d_norm_last_error() or b"").decode() or
                       lib.conv1d_norm_status_string(status).decode())


# ------------------------------------------------------------------------------ C-named wrappers

def make_params(N, C_in, C_out, T, k, stride=1, pad_left=0, pad_right=0, dilation=1, norm=NORM_NONE, groups=1,
                eps=1e-5, post=POST_NONE, dtype=F32, math=MATH_AUTO, force_path=PATH_AUTO,
                mainloop=MAINLOOP_AUTO) -> Params:
    return Params(N, C_in, C_out, T, k, stride, pad_left, pad_right, dilation, norm, groups, eps, post, dtype, math,
                  force_path, mainloop)


def conv1d_norm_desc_create(params: Params) -> int:
    h = ctypes.c_void_p()
    _check(load().conv1d_norm_desc_create(ctypes.byref(params), ctypes.byref(h)))
    return h.value


def conv1d_norm_workspace_size(desc: int) -> int:
    n = ctypes.c_size_t()
    _check(load().conv1d_norm_workspace_size(desc, ctypes.byref(n)))
    return n.value


def conv1d_norm_set_workspace(desc: int, ptr: int, nbytes: int) -> None:
    _check(load().conv1d_norm_set_workspace(desc, ptr, nbytes))


def conv1d_norm_plan_info(desc: int) -> PlanInfo:
    info = PlanInfo()
    _check(load().conv1d_norm_plan_info(desc, ctypes.byref(info)))
    return info


def conv1d_norm_run(desc: int, x: int, w: int, b: Optional[int], gamma: Optional[int], beta: Optional[int], y: int,
                    stream: int) -> None:
    _check(load().conv1d_norm_run(desc, x, w, b, gamma, beta, y, stream))


def conv1d_norm_run_ex(desc: int, args: Args, stream: int) -> None:
    _check(load().conv1d_norm_run_ex(desc, ctypes.byref(args), stream))


def conv1d_norm_pack_weights(desc: int, w: int, workspace: Optional[int], workspace_bytes: int, stream: int) -> None:
    _check(load().conv1d_norm_pack_weights(desc, w, workspace, workspace_bytes, stream))


def conv1d_norm_run_static_scratch(desc: int, args: Args, stream: int) -> None:
    """Run without any allocation, using the library's fixed device scratch (see the C header)."""
    _check(load().conv1d_norm_run_static_scratch(desc, ctypes.byref(args), stream))


def ln_avgpool3d_gelu_run(params: LnPoolParams, z: int, sum_weight: float, gamma: Optional[int], beta: Optional[int],
                          out: int, stream: int) -> None:
    """[p4]'s scalar add + LayerNorm(last dim) + AvgPool3d(2) + GELU pass (see the C header)."""
    _check(load().ln_avgpool3d_gelu_run(ctypes.byref(params), z, sum_weight, gamma, beta, out, stream))


def ln_avgpool3d_gelu(z, sum_weight: float, gamma=None, beta=None, eps: float = 1e-5, out=None):
    """Torch convenience wrapper: z [N, C, D, H, W] float32 CUDA tensor (contiguous) -> a new (or the
    given) [N, C, D//2, H//2, W//2] float32 tensor, computed on the current stream."""
    import torch
    if z.dim() != 5:
        raise ValueError(f"z must be 5-D [N, C, D, H, W], got shape {tuple(z.shape)}")
    N, C, D, H, W = z.shape
    _check_tensor("z", z, (N, C, D, H, W), torch.float32)
    if not z.is_cuda:
        raise ValueError("z must be a CUDA tensor")
    for name, t in (("gamma", gamma), ("beta", beta)):
        _check_tensor(name, t, (W,), torch.float32, z.device, optional=True)
    _check_tensor("out", out, (N, C, D // 2, H // 2, W // 2), torch.float32, z.device, optional=True)
    if out is None:
        out = torch.empty((N, C, D // 2, H // 2, W // 2), dtype=torch.float32, device=z.device)
    p = LnPoolParams(N, C, D, H, W, eps)
    ln_avgpool3d_gelu_run(p, z.data_ptr(), float(sum_weight), _ptr(gamma), _ptr(beta), out.data_ptr(),
                          torch.cuda.current_stream(z.device).cuda_stream)
    return out


def _convt3d_shapes(x, w):
    """(N, C_in, D, H, W, C_out, k) of x [N, C_in, D, H, W] and w [C_in, C_out, k, k, k], both dense
    float32 CUDA tensors on one device; ValueError otherwise."""
    import torch
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError(f"x and w must be 5-D, got shapes {tuple(x.shape)} and {tuple(w.shape)}")
    N, C_in, D, H, W = x.shape
    C_out, k = w.shape[1], w.shape[2]
    _check_tensor("x", x, (N, C_in, D, H, W), torch.float32)
    _check_tensor("w", w, (C_in, C_out, k, k, k), torch.float32)
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    _check_tensor("w", w, (C_in, C_out, k, k, k), torch.float32, x.device)
    return N, C_in, D, H, W, C_out, k


def _check_workspace(ws, need: int, device) -> None:
    import torch
    if ws.dtype != torch.uint8 or ws.dim() != 1 or not ws.is_contiguous():
        raise ValueError("workspace must be a dense 1-D uint8 tensor")
    if ws.numel() < need:
        raise ValueError(f"workspace holds {ws.numel()} bytes, {need} needed")
    if not ws.is_cuda or ws.device != device:
        raise ValueError(f"workspace is on {ws.device}, expected {device}")


def conv_transpose3d_workspace_size(params: ConvT3dParams) -> int:
    """Workspace bytes of the chosen plan (0 for the CUDA-core plan)."""
    n = ctypes.c_size_t(0)
    _check(load().conv_transpose3d_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def conv_transpose3d_run(params: ConvT3dParams, x: int, w: int, b: Optional[int], y: int, workspace: Optional[int],
                         workspace_bytes: int, stream: int) -> None:
    """[p4]'s ConvTranspose3d (see the C header)."""
    _check(load().conv_transpose3d_run(ctypes.byref(params), x, w, b, y, workspace, workspace_bytes, stream))


def conv_transpose3d(x, w, b=None, stride: int = 2, pad: int = 1, out_pad: int = 1, out=None, math: int = 0,
                     workspace=None):
    """Torch convenience wrapper: x [N, C_in, D, H, W], w [C_in, C_out, k, k, k] float32 CUDA tensors
    (contiguous) -> a new (or the given) [N, C_out, Do, Ho, Wo] float32 tensor on the current stream.
    math: 0 auto, 1 CUDA cores, 2 tensor cores. The workspace (a uint8 CUDA tensor) is allocated here
    when the plan needs one and none is given."""
    import torch
    N, C_in, D, H, W, C_out, k = _convt3d_shapes(x, w)
    f = lambda n: (n - 1) * stride - 2 * pad + (k - 1) + out_pad + 1
    _check_tensor("b", b, (C_out,), torch.float32, x.device, optional=True)
    _check_tensor("out", out, (N, C_out, f(D), f(H), f(W)), torch.float32, x.device, optional=True)
    if out is None:
        out = torch.empty((N, C_out, f(D), f(H), f(W)), dtype=torch.float32, device=x.device)
    p = ConvT3dParams(N, C_in, C_out, D, H, W, k, stride, pad, out_pad, math)
    need = conv_transpose3d_workspace_size(p)
    if need and workspace is not None:
        _check_workspace(workspace, need, x.device)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    conv_transpose3d_run(p, x.data_ptr(), w.data_ptr(), _ptr(b), out.data_ptr(),
                         workspace.data_ptr() if need else None, need, torch.cuda.current_stream(x.device).cuda_stream)
    return out


def conv_transpose3d_ln_avgpool3d_gelu_workspace_size(params: ConvT3dParams) -> int:
    """Workspace bytes of the fused model kernel."""
    n = ctypes.c_size_t(0)
    _check(load().conv_transpose3d_ln_avgpool3d_gelu_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def conv_transpose3d_ln_avgpool3d_gelu_run(params: ConvT3dParams, eps: float, sum_weight: float, x: int, w: int,
                                           b: Optional[int], gamma: Optional[int], beta: Optional[int], out: int,
                                           workspace: int, workspace_bytes: int, stream: int) -> None:
    """[p4]'s whole model in one pass (see the C header)."""
    _check(load().conv_transpose3d_ln_avgpool3d_gelu_run(ctypes.byref(params), eps, sum_weight, x, w, b, gamma, beta,
                                                         out, workspace, workspace_bytes, stream))


def conv_transpose3d_ln_avgpool3d_gelu(x, w, b, sum_weight: float, gamma=None, beta=None, eps: float = 1e-5,
                                       stride: int = 2, pad: int = 1, out_pad: int = 1, out=None, workspace=None):
    """Torch convenience wrapper: x [N, 32, D, H, 32], w [32, 64, 3, 3, 3] float32 CUDA tensors
    (contiguous) -> a new (or the given) [N, 64, D, H, 32] float32 tensor on the current stream:
    GELU(AvgPool3d(2)(LayerNorm_W(ConvTranspose3d(x) + sum_weight))). The workspace (a uint8 CUDA
    tensor) is allocated here when none is given."""
    import torch
    N, C_in, D, H, W, C_out, k = _convt3d_shapes(x, w)
    w_out = (W - 1) * stride - 2 * pad + (k - 1) + out_pad + 1  # the LayerNorm width
    _check_tensor("b", b, (C_out,), torch.float32, x.device, optional=True)
    for name, t in (("gamma", gamma), ("beta", beta)):
        _check_tensor(name, t, (w_out,), torch.float32, x.device, optional=True)
    _check_tensor("out", out, (N, C_out, D, H, W), torch.float32, x.device, optional=True)
    if out is None:
        out = torch.empty((N, C_out, D, H, W), dtype=torch.float32, device=x.device)
    p = ConvT3dParams(N, C_in, C_out, D, H, W, k, stride, pad, out_pad, 2)
    need = conv_transpose3d_ln_avgpool3d_gelu_workspace_size(p)
    if workspace is not None:
        _check_workspace(workspace, need, x.device)
    else:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    conv_transpose3d_ln_avgpool3d_gelu_run(p, eps, sum_weight, x.data_ptr(), w.data_ptr(), _ptr(b), _ptr(gamma),
                                           _ptr(beta), out.data_ptr(), workspace.data_ptr(), need,
                                           torch.cuda.current_stream(x.device).cuda_stream)
    return out


def conv1d_norm_check(desc: int, workspace: Optional[int], stream: int) -> None:
    _check(load().conv1d_norm_check(desc, workspace, stream))


def conv1d_norm_set_profiling(desc: int, enable: bool) -> None:
    _check(load().conv1d_norm_set_profiling(desc, 1 if enable else 0))


def conv1d_norm_kernel_times(desc: int):
    """[(kernel name, ms)] of the last profiled run, in launch order (waits for it to finish)."""
    buf = (KernelTime * 8)()
    n = ctypes.c_int32()
    _check(load().conv1d_norm_kernel_times(desc, buf, 8, ctypes.byref(n)))
    return [(buf[i].name.decode(), float(buf[i].ms)) for i in range(min(n.value, 8))]


def conv1d_norm_destroy(desc: int) -> None:
    load().conv1d_norm_destroy(desc)


def conv1d_norm_status_string(status: int) -> str:
    return load().conv1d_norm_status_string(status).decode()


def conv1d_norm_version() -> int:
    return int(load().conv1d_norm_version())


# ------------------------------------------------------------------------------ convenience wrapper

def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_tensor(name: str, t, shape, dtype, device=None, optional: bool = False) -> None:
    """Raise ValueError unless `t` is a tensor of exactly `shape` and `dtype`, dense (contiguous) and,
    when `device` is given, a CUDA tensor on that device. Shape and dtype are checked first, so the
    checks also run on tensors of a machine without a GPU. The C library sees only raw pointers: a
    tensor of the wrong size would become out-of-bounds device accesses, not an error status."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and (not t.is_cuda or t.device != device):
        raise ValueError(f"{name} is on {t.device}, expected {device}")


class Conv1dNorm:
    """One descriptor plus its workspace; calls go through ``conv1d_norm_run_ex`` on the current stream."""

    def __init__(self, params: Params, device=None):
        import torch
        self.params = params
        self.desc = conv1d_norm_desc_create(params)
        self.info = conv1d_norm_plan_info(self.desc)
        self.T_out = self.info.T_out
        nbytes = conv1d_norm_workspace_size(self.desc)
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        conv1d_norm_set_workspace(self.desc, self.workspace.data_ptr(), self.workspace.numel())

    @property
    def path(self) -> str:
        return PATH_NAMES[self.info.path]

    def out_dtype(self):
        import torch
        return torch.bfloat16 if self.params.dtype == BF16 else torch.float32

    def _device(self):
        import torch
        return self.workspace.device if self.workspace.is_cuda else None

    def validate(self, x, w, b=None, gamma=None, beta=None, bias2=None, out=None, argmin=None) -> None:
        """Raise ValueError unless every tensor matches the descriptor: x [N, C_in, T] and w
        [C_out, C_in, k] in the descriptor's dtype; b, gamma, beta, bias2 [C_out] float32; out
        [N, C_out, T_out] in the output dtype; argmin [N, T_out] int32; all dense, on the workspace's
        device. bias2 is required with the row-min post-op."""
        import torch
        p = self.params
        dt = self.out_dtype()
        dev = self._device()
        _check_tensor("x", x, (p.N, p.C_in, p.T), dt, dev)
        _check_tensor("w", w, (p.C_out, p.C_in, p.k), dt, dev)
        for name, t in (("b", b), ("gamma", gamma), ("beta", beta)):
            _check_tensor(name, t, (p.C_out,), torch.float32, dev, optional=True)
        _check_tensor("bias2", bias2, (p.C_out,), torch.float32, dev, optional=p.post != POST_ROWMIN_BIAS)
        _check_tensor("out", out, (p.N, p.C_out, self.T_out), dt, dev, optional=True)
        _check_tensor("argmin", argmin, (p.N, self.T_out), torch.int32, dev, optional=True)

    def pack_weights(self, w, stream=None):
        import torch
        p = self.params
        _check_tensor("w", w, (p.C_out, p.C_in, p.k), self.out_dtype(), self._device())
        s = torch.cuda.current_stream(w.device).cuda_stream if stream is None else stream
        conv1d_norm_pack_weights(self.desc, w.data_ptr(), None, 0, s)

    def __call__(self, x, w, b=None, gamma=None, beta=None, bias2=None, out=None, argmin=None, stream=None,
                 weights_packed=False):
        import torch
        p = self.params
        self.validate(x, w, b, gamma, beta, bias2, out, argmin)
        if out is None:
            out = torch.empty((p.N, p.C_out, self.T_out), dtype=self.out_dtype(), device=x.device)
        args = Args(_ptr(x), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta), _ptr(bias2), _ptr(out), _ptr(argmin), None, 0,
                    FLAG_WEIGHTS_PACKED if weights_packed else 0)
        s = torch.cuda.current_stream(x.device).cuda_stream if stream is None else stream
        conv1d_norm_run_ex(self.desc, args, s)
        return out

    def check(self, stream=None):
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        conv1d_norm_check(self.desc, None, s)

    def set_profiling(self, enable: bool = True) -> None:
        conv1d_norm_set_profiling(self.desc, enable)

    def kernel_times(self):
        return conv1d_norm_kernel_times(self.desc)

    def close(self):
        if getattr(self, "desc", None):
            conv1d_norm_destroy(self.desc)
            self.desc = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

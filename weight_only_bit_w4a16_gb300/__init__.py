"""Python binding of libwq.so, the GB300 W4A16 dequantise-GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/wq.h.  There is no CPU path --
if the compiled library is missing, every call raises.

Low level (same names as the C ABI, integer pointers):
    wq_gemm, wq_gemm_ex, wq_dequant, wq_get_device_error, wq_selftest_timeout,
    wq_status_string, wq_version
Tensor level (torch CUDA tensors, raises WQError on a non-OK status):
    gemm(A, packed, scales, zeros, fmt, group=None, out_dtype="bf16", ...)
    dequant(packed, scales, zeros, fmt, group=None, out=None, ...)
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

# constants of include/wq.h
WQ_NVFP4, WQ_MXFP4, WQ_INT4 = 0, 1, 2
WQ_OUT_F32 = 0x100
WQ_PATH_AUTO, WQ_PATH_GEMV, WQ_PATH_TC = 0, 1, 2
WQ_LAUNCH_OVERLAP = 0x100
WQ_LAUNCH_INPUTS_READY = 0x200
WQ_OK = 0
WQ_ERR_INVALID_ARG = -1
WQ_ERR_UNSUPPORTED = -2
WQ_ERR_ALIGN = -3
WQ_ERR_CUDA = -4
WQ_ERR_DEVICE_TIMEOUT = -5

FORMATS = {"nvfp4": WQ_NVFP4, "mxfp4": WQ_MXFP4, "int4": WQ_INT4}
DEFAULT_GROUP = {"nvfp4": 16, "mxfp4": 32, "int4": 128}
PATHS = {"auto": WQ_PATH_AUTO, "gemv": WQ_PATH_GEMV, "tc": WQ_PATH_TC}

#: the C entry points include/wq.h declares: name -> (restype, argtypes)
_vp, _i = ctypes.c_void_p, ctypes.c_int
class wq_epilogue(ctypes.Structure):
    """The C struct of include/wq.h: bias, residual (device pointers or None), gated."""
    _fields_ = [("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p), ("gated", ctypes.c_int)]


SIGNATURES = {
    "wq_gemm": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i]),
    "wq_gemm_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i]),
    "wq_gemm_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _vp, _i]),
    "wq_gemm_workspace_size": (ctypes.c_size_t, [_i, _i, _i, _i, _i]),
    "wq_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i]),
    "wq_gemm_static": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i]),
    "wq_gemm_fused": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(wq_epilogue), _vp,
                           ctypes.c_size_t, _vp, _i]),
    "wq_prepack_bytes": (ctypes.c_size_t, [_i, _i, _i, _i]),
    "wq_prepack": (_i, [_vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i, _i, _vp]),
    "wq_gemm_prepacked": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(wq_epilogue), _vp,
                               ctypes.c_size_t, _vp, _i]),
    "wq_dequant": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "wq_get_device_error": (_i, []),
    "wq_selftest_timeout": (_i, [_vp]),
    "wq_status_string": (ctypes.c_char_p, [_i]),
    "wq_version": (_i, []),
}


class WQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libwq.so (built by __graft_entry__.build() / build.py); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
                    " (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


# -- the C ABI, same names ----------------------------------------------------
def wq_gemm(A, packed, scales, zeros, C, M, N, K, format, group) -> int:
    return lib().wq_gemm(A, packed, scales, zeros, C, M, N, K, format, group)


def wq_gemm_ex(A, packed, scales, zeros, C, M, N, K, format, group, stream, path) -> int:
    return lib().wq_gemm_ex(A, packed, scales, zeros, C, M, N, K, format, group, stream, path)


def wq_gemm_ws(A, packed, scales, zeros, C, M, N, K, format, group, workspace, workspace_bytes, stream,
               path) -> int:
    return lib().wq_gemm_ws(A, packed, scales, zeros, C, M, N, K, format, group, workspace, workspace_bytes,
                            stream, path)


def wq_gemm_static(A, packed, scales, zeros, C, M, N, K, format, group, stream, path) -> int:
    return lib().wq_gemm_static(A, packed, scales, zeros, C, M, N, K, format, group, stream, path)


def wq_gemm_fused(A, packed, scales, zeros, C, M, N, K, format, group, epilogue, workspace, workspace_bytes,
                  stream, path) -> int:
    return lib().wq_gemm_fused(A, packed, scales, zeros, C, M, N, K, format, group, epilogue, workspace,
                               workspace_bytes, stream, path)


def wq_gemm_workspace_size(M, N, K, format, group) -> int:
    return lib().wq_gemm_workspace_size(M, N, K, format, group)


def wq_workspace_bytes(M, N, K, format, group) -> int:
    return lib().wq_workspace_bytes(M, N, K, format, group)


def wq_prepack_bytes(N, K, format, group) -> int:
    return lib().wq_prepack_bytes(N, K, format, group)


def wq_prepack(packed, scales, zeros, prepacked, prepacked_bytes, N, K, format, group, stream) -> int:
    return lib().wq_prepack(packed, scales, zeros, prepacked, prepacked_bytes, N, K, format, group, stream)


def wq_gemm_prepacked(A, prepacked, C, M, N, K, format, group, epilogue, workspace, workspace_bytes, stream,
                      path) -> int:
    return lib().wq_gemm_prepacked(A, prepacked, C, M, N, K, format, group, epilogue, workspace, workspace_bytes,
                                   stream, path)


def wq_dequant(packed, scales, zeros, W, N, K, format, group, stream) -> int:
    return lib().wq_dequant(packed, scales, zeros, W, N, K, format, group, stream)


def wq_get_device_error() -> int:
    return lib().wq_get_device_error()


def wq_selftest_timeout(stream=None) -> int:
    return lib().wq_selftest_timeout(stream)


def wq_status_string(status: int) -> str:
    return lib().wq_status_string(int(status)).decode()


def wq_version() -> int:
    return lib().wq_version()


def status_string(status: int) -> str:
    try:
        return wq_status_string(status)
    except Exception:   # library not loadable: still give a message
        return f"wq status {status}"


# -- tensor-level helpers -------------------------------------------------------
def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _fmt_name(fmt) -> str:
    if isinstance(fmt, str):
        return fmt
    return {v: k for k, v in FORMATS.items()}[int(fmt)]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


_workspaces = {}


def workspace(M, N, K, fmt, group=None, device=None):
    """A zeroed device workspace for wq_gemm_ws on this shape (None if the
    shape needs none), cached per device and grown as needed.  Completed calls
    leave its flag words zero, so it is reused across calls on one stream."""
    import torch
    group = group or DEFAULT_GROUP[_fmt_name(fmt)]
    nbytes = wq_gemm_workspace_size(M, N, K, _fmt(fmt), int(group))
    if nbytes == 0:
        return None
    dev = torch.device(device if device is not None else "cuda")
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=torch.device("cuda", key))
        _workspaces[key] = ws
    return ws


def _launch_bits(overlap, inputs_ready):
    return (WQ_LAUNCH_OVERLAP if overlap else 0) | (WQ_LAUNCH_INPUTS_READY if inputs_ready else 0)


def gemm(A, packed, scales, zeros, fmt, group=None, out_dtype="bf16", out=None, path="auto", stream=None,
         overlap=False, workspace=None, bias=None, residual=None, gated=False, inputs_ready=False):
    """C = A . deq(packed, scales, zeros)^T on A's device and current stream.

    overlap=True sets WQ_LAUNCH_OVERLAP (programmatic dependent launch): the
    caller guarantees the preceding kernel on the stream does not write the
    weights.  inputs_ready=True sets WQ_LAUNCH_INPUTS_READY: A, too, is
    written by no kernel that may still be running (include/wq.h).  workspace: a zeroed uint8 CUDA tensor (see workspace()) that
    lets the tensor-core path split tiles over the SMs; "auto" takes the
    cached one.  bias (N,) bf16, residual (M, outputs) bf16 and gated select
    the fused epilogue of wq_gemm_fused (gated: C has N / 2 columns).

    A: (M, K) bf16; packed: (N, K/2) uint8; scales: (N, K/group) uint8
    (nvfp4 e4m3 / mxfp4 e8m0 bytes) or bf16 (int4); zeros: (N, K/group)
    uint8 for int4, None otherwise.  Returns C (M, N) bf16 or fp32.
    """
    import torch
    f = _fmt(fmt)
    group = group or DEFAULT_GROUP[_fmt_name(fmt)]
    M, K = A.shape
    N = packed.shape[0]
    if packed.shape[1] * 2 != K:
        raise ValueError(f"packed {tuple(packed.shape)} does not match K={K}")
    for t in (A, packed, scales, zeros, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if A.dtype != torch.bfloat16 or packed.dtype != torch.uint8:
        raise ValueError("A must be bf16 and packed uint8")
    odt = torch.float32 if out_dtype in ("fp32", torch.float32) else torch.bfloat16
    ncol = N // 2 if gated else N
    if out is None:
        out = torch.empty((M, ncol), dtype=odt, device=A.device)
    elif out.shape != (M, ncol) or out.dtype != odt:
        raise ValueError("out has the wrong shape or dtype")
    for t, shape in ((bias, (N,)), (residual, (M, ncol))):
        if t is not None and (t.dtype != torch.bfloat16 or tuple(t.shape) != shape or not t.is_cuda
                              or not t.is_contiguous()):
            raise ValueError(f"bias / residual must be contiguous bf16 CUDA tensors of shape {shape}")
    fmt_word = f | (WQ_OUT_F32 if odt == torch.float32 else 0)
    pcode = (PATHS[path] if isinstance(path, str) else int(path)) | _launch_bits(overlap, inputs_ready)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = globals()["workspace"](M, N, K, fmt, group, A.device)
    if bias is not None or residual is not None or gated:
        epi = wq_epilogue(None if bias is None else bias.data_ptr(),
                          None if residual is None else residual.data_ptr(), 1 if gated else 0)
        if workspace is not None and (not workspace.is_cuda or workspace.dtype != torch.uint8):
            raise ValueError("workspace must be a uint8 CUDA tensor")
        st = wq_gemm_fused(_ptr(A), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(out), M, N, K, fmt_word,
                           int(group), ctypes.byref(epi), _ptr(workspace),
                           0 if workspace is None else workspace.numel(), _stream_handle(stream, A.device), pcode)
    elif workspace is None:
        st = wq_gemm_ex(_ptr(A), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(out), M, N, K, fmt_word,
                        int(group), _stream_handle(stream, A.device), pcode)
    else:
        if not workspace.is_cuda or workspace.dtype != torch.uint8:
            raise ValueError("workspace must be a uint8 CUDA tensor")
        st = wq_gemm_ws(_ptr(A), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(out), M, N, K, fmt_word,
                        int(group), _ptr(workspace), workspace.numel(), _stream_handle(stream, A.device), pcode)
    if st != WQ_OK:
        raise WQError(st, "wq_gemm")
    return out


class Prepacked:
    """A weight in the prepacked layout (wq_prepack): the uint8 device buffer
    and the description it was made from."""

    def __init__(self, buf, N, K, fmt, group):
        self.buf, self.N, self.K, self.fmt, self.group = buf, N, K, _fmt_name(fmt), group


def prepack(packed, scales, zeros, fmt, group=None, stream=None, out=None) -> Prepacked:
    """Repack one weight (wq_prepack) into a new uint8 CUDA tensor, or into
    `out` (a uint8 CUDA tensor of at least wq_prepack_bytes() elements)."""
    import torch
    f = _fmt(fmt)
    group = group or DEFAULT_GROUP[_fmt_name(fmt)]
    N, Kh = packed.shape
    K = 2 * Kh
    for t in (packed, scales, zeros):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    nbytes = wq_prepack_bytes(N, K, f, int(group))
    if nbytes == 0:
        raise WQError(WQ_ERR_UNSUPPORTED, "wq_prepack_bytes")
    if out is None:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=packed.device)
    elif out.dtype != torch.uint8 or not out.is_cuda or not out.is_contiguous() or out.numel() < nbytes:
        raise ValueError(f"out must be a contiguous uint8 CUDA tensor of at least {nbytes} bytes")
    else:
        buf = out
    st = wq_prepack(_ptr(packed), _ptr(scales), _ptr(zeros), _ptr(buf), nbytes, N, K, f, int(group),
                    _stream_handle(stream, packed.device))
    if st != WQ_OK:
        raise WQError(st, "wq_prepack")
    return Prepacked(buf, N, K, fmt, int(group))


def gemm_prepacked(A, pre: Prepacked, out_dtype="bf16", out=None, stream=None, overlap=False, bias=None,
                   residual=None, gated=False, path="auto", workspace=None, inputs_ready=False):
    """C = A . deq(B)^T for a prepacked weight (wq_gemm_prepacked); the other
    arguments as for gemm()."""
    import torch
    M, K = A.shape
    N = pre.N
    if K != pre.K:
        raise ValueError(f"A has K={K}, the weight K={pre.K}")
    for t in (A, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if A.dtype != torch.bfloat16:
        raise ValueError("A must be bf16")
    odt = torch.float32 if out_dtype in ("fp32", torch.float32) else torch.bfloat16
    ncol = N // 2 if gated else N
    if out is None:
        out = torch.empty((M, ncol), dtype=odt, device=A.device)
    elif out.shape != (M, ncol) or out.dtype != odt:
        raise ValueError("out has the wrong shape or dtype")
    for t, shape in ((bias, (N,)), (residual, (M, ncol))):
        if t is not None and (t.dtype != torch.bfloat16 or tuple(t.shape) != shape or not t.is_cuda
                              or not t.is_contiguous()):
            raise ValueError(f"bias / residual must be contiguous bf16 CUDA tensors of shape {shape}")
    epi = None
    if bias is not None or residual is not None or gated:
        epi = ctypes.byref(wq_epilogue(None if bias is None else bias.data_ptr(),
                                       None if residual is None else residual.data_ptr(), 1 if gated else 0))
    fmt_word = _fmt(pre.fmt) | (WQ_OUT_F32 if odt == torch.float32 else 0)
    pcode = (PATHS[path] if isinstance(path, str) else int(path)) | _launch_bits(overlap, inputs_ready)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = globals()["workspace"](M, N, K, pre.fmt, pre.group, A.device)
    if workspace is not None and (not workspace.is_cuda or workspace.dtype != torch.uint8):
        raise ValueError("workspace must be a uint8 CUDA tensor")
    st = wq_gemm_prepacked(_ptr(A), _ptr(pre.buf), _ptr(out), M, N, K, fmt_word, pre.group, epi, _ptr(workspace),
                           0 if workspace is None else workspace.numel(), _stream_handle(stream, A.device), pcode)
    if st != WQ_OK:
        raise WQError(st, "wq_gemm_prepacked")
    return out


def dequant(packed, scales, zeros, fmt, group=None, out=None, stream=None):
    """W = deq(packed, scales, zeros) as an (N, K) bf16 tensor (bit-exact RNE)."""
    import torch
    f = _fmt(fmt)
    group = group or DEFAULT_GROUP[_fmt_name(fmt)]
    N, Kh = packed.shape
    K = 2 * Kh
    for t in (packed, scales, zeros, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=packed.device)
    st = wq_dequant(_ptr(packed), _ptr(scales), _ptr(zeros), _ptr(out), N, K, f, int(group),
                    _stream_handle(stream, packed.device))
    if st != WQ_OK:
        raise WQError(st, "wq_dequant")
    return out

"""Mamba-2 SSD chunked-scan forward on GB300: Python binding of libssd.so.

A thin ctypes layer over the C ABI declared in include/ssd.h. It only checks
and marshals arguments (shapes, dtypes, contiguity, device, stream handle);
every step of the forward runs in the library's CUDA kernels. There is no
fallback: if libssd.so is missing or fails to load, every call raises.

    from mamba_ssd_chunked_gb300 import ssd_fwd
    y, final_state = ssd_fwd(x, dt, dt_bias, A, B, C, D, init_state, chunk_len=256)

Tensors (torch, CUDA, contiguous):
    x [b, L, h, p] and B, C [b, L, g, n] in bf16 or fp32 (all three alike);
    dt [b, L, h], dt_bias [h], A [h], D [h] fp32; init_state [b, h, p, n] fp32.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

__all__ = [
    "SsdError", "library", "ssd_fwd", "ssd_fwd_host", "ssd_check_inputs", "ssd_device_status", "ssd_fwd_workspace_bytes",
    "ssd_select_path", "ssd_host_slices", "ssd_kernel_launches", "ssd_kernel_timing", "ssd_kernel_timing_read", "ssd_release", "ssd_step", "ssd_conv1d_silu", "ssd_conv1d_step",
    "ssd_gated_rmsnorm", "Dims", "ConvDims", "DtLimit", "PATHS", "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libssd.so")
LIBRARY_DEBUG = os.path.join(_HERE, "libssd_debug.so")  # the index-checked build (SSD_DEBUG)

STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_CUDA",
          4: "SSD_ERR_DEVICE_TIMEOUT", 5: "SSD_ERR_WORKSPACE", 6: "SSD_ERR_DEBUG_CHECK"}
PATHS = {"auto": 0, "simt": 1, "tc": 2, "chain": 3}
DTYPES = {"f32": 0, "bf16": 1}


class Dims(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int64) for k in ("batch", "seqlen", "nheads", "headdim", "ngroups", "dstate")]


class DtLimit(ctypes.Structure):
    _fields_ = [("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float)]


class ConvDims(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int64) for k in ("batch", "seqlen", "d_inner", "ngroups", "dstate", "kernel_size")]


class SsdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


_lib: Optional[ctypes.CDLL] = None


def use_library(path: str) -> str:
    """Make every later call go through the libssd build at `path` (for
    example LIBRARY_DEBUG); returns the path used until now."""
    global _lib, LIBRARY
    old = LIBRARY
    LIBRARY = path
    _lib = None
    return old


def library() -> ctypes.CDLL:
    """Load libssd.so (built by __graft_entry__.build() or mamba_ssd_chunked_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise RuntimeError(f"{LIBRARY} is missing: build it with `python -m mamba_ssd_chunked_gb300.build`")
    lib = ctypes.CDLL(LIBRARY)
    vp, fp, i, i64 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    pdims = ctypes.POINTER(Dims)
    lib.ssd_fwd.restype = i
    lib.ssd_fwd.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, i, i, vp, fp, vp]
    lib.ssd_fwd_ws.restype = i
    lib.ssd_fwd_ws.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, i, i, vp, fp, i, vp, ctypes.c_size_t, vp]
    lib.ssd_fwd_host.restype = i
    lib.ssd_fwd_host.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, i, i, vp, fp, vp]
    lib.ssd_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_fwd_workspace_bytes.argtypes = [pdims, i, i, i]
    lib.ssd_select_path.restype = i
    lib.ssd_select_path.argtypes = [pdims, i, i]
    lib.ssd_host_slices.restype = i
    lib.ssd_host_slices.argtypes = [pdims, i]
    lib.ssd_device_status.restype = i
    lib.ssd_check_inputs.restype = i
    lib.ssd_check_inputs.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, ctypes.POINTER(ctypes.c_int64), vp]
    lib.ssd_device_status.argtypes = [vp]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [i]
    lib.ssd_kernel_launches.restype = ctypes.c_uint64
    lib.ssd_kernel_launches.argtypes = []
    lib.ssd_kernel_timing.restype = None
    lib.ssd_kernel_timing.argtypes = [ctypes.c_int]
    lib.ssd_kernel_timing_read.restype = ctypes.c_int
    lib.ssd_kernel_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64)]
    lib.ssd_release.restype = None
    lib.ssd_release.argtypes = []
    lib.ssd_debug_build.restype = i
    lib.ssd_debug_build.argtypes = []
    lib.ssd_debug_failed_line.restype = ctypes.c_uint
    lib.ssd_debug_failed_line.argtypes = [vp]
    lib.ssd_step.restype = i
    lib.ssd_step.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, i, vp, vp]
    plim = ctypes.POINTER(DtLimit)
    lib.ssd_fwd_ex.restype = i
    lib.ssd_fwd_ex.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, i, i, vp, fp, plim, vp, i, vp, ctypes.c_size_t,
                               vp]
    lib.ssd_step_ex.restype = i
    lib.ssd_step_ex.argtypes = [pdims, i, vp, fp, fp, fp, vp, vp, fp, fp, i, vp, plim, vp]
    pconv = ctypes.POINTER(ConvDims)
    lib.ssd_conv1d_silu.restype = i
    lib.ssd_conv1d_silu.argtypes = [pconv, i, vp, i64, fp, fp, i, vp, vp, vp, vp, vp]
    lib.ssd_conv1d_step.restype = i
    lib.ssd_conv1d_step.argtypes = [pconv, i, vp, i64, fp, fp, i, vp, vp, vp, vp, vp]
    lib.ssd_gated_rmsnorm.restype = i
    lib.ssd_gated_rmsnorm.argtypes = [i, i64, i64, i64, vp, i64, vp, i64, fp, ctypes.c_float, vp, i64, vp]
    _lib = lib
    return lib


def _torch():
    import torch
    return torch


def _io_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DTYPES["bf16"]
    if t.dtype == torch.float32:
        return DTYPES["f32"]
    raise TypeError(f"x/B/C must be bf16 or fp32, got {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t, name, shape, dtype, device_type, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.type != device_type:
        raise ValueError(f"{name} must be on {device_type}, got {t.device}")


def _dims(x, B) -> Dims:
    b, L, h, p = x.shape
    g, n = B.shape[2], B.shape[3]
    return Dims(b, L, h, p, g, n)


def _check_all(x, dt, dt_bias, A, B, C, D, init_state, device_type):
    torch = _torch()
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [b, L, h, p] and B [b, L, g, n]")
    b, L, h, p = x.shape
    g, n = B.shape[2], B.shape[3]
    io = x.dtype
    _check(x, "x", (b, L, h, p), io, device_type)
    _check(B, "B", (b, L, g, n), io, device_type)
    _check(C, "C", (b, L, g, n), io, device_type)
    f32 = torch.float32
    _check(dt, "dt", (b, L, h), f32, device_type)
    _check(dt_bias, "dt_bias", (h,), f32, device_type)
    _check(A, "A", (h,), f32, device_type)
    _check(D, "D", (h,), f32, device_type, optional=True)
    _check(init_state, "init_state", (b, h, p, n), f32, device_type, optional=True)


INPUT_NAMES = ("x", "dt", "dt_bias", "A", "B", "C", "D", "init_state")


def ssd_check_inputs(x, dt, dt_bias, A, B, C, D=None, init_state=None, stream=None) -> dict:
    """Count the non-finite elements (NaN, +-Inf) of each forward input on the
    GPU through ssd_check_inputs; returns {name: count} over INPUT_NAMES (0 for
    an absent D / init_state). Synchronizes `stream` (default: torch's current
    stream)."""
    torch = _torch()
    _check_all(x, dt, dt_bias, A, B, C, D, init_state, "cuda")
    lib = library()
    dims = _dims(x, B)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    counts = (ctypes.c_int64 * len(INPUT_NAMES))()
    rc = lib.ssd_check_inputs(ctypes.byref(dims), _io_code(x), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B),
                              _ptr(C), _ptr(D), _ptr(init_state), counts, stream)
    if rc != 0:
        raise SsdError(rc, "ssd_check_inputs")
    return {name: int(c) for name, c in zip(INPUT_NAMES, counts)}


def ssd_fwd(x, dt, dt_bias, A, B, C, D=None, init_state=None, chunk_len: int = 256,
            ngroups: Optional[int] = None, y=None, final_state=None, return_final_state: bool = True,
            path: str = "auto", workspace=None, stream=None,
            dt_limit: Optional[Tuple[float, float]] = None, seq_idx=None,
            check_inputs: bool = False) -> Tuple[object, Optional[object]]:
    """Run the SSD forward on the GPU through ssd_fwd / ssd_fwd_ws (ssd_fwd_ex
    when a dt_limit = (lo, hi) clamp of softplus(dt + dt_bias) or packed
    sequences seq_idx [b, L] int32 are given: the state restarts from zero
    wherever seq_idx changes between consecutive tokens of a row).

    Returns (y, final_state); final_state is None when return_final_state is
    False. With path != "auto" or an explicit workspace (a uint8 CUDA tensor)
    the call goes through ssd_fwd_ws (a caller workspace must be zero-filled
    before its first use); otherwise through ssd_fwd with the library-owned
    workspace. Asynchronous on `stream` (default: torch's
    current stream). With check_inputs, the inputs first go through
    ssd_check_inputs (which synchronizes `stream`), and a non-finite element
    in any of them raises ValueError before the forward is launched.
    """
    torch = _torch()
    _check_all(x, dt, dt_bias, A, B, C, D, init_state, "cuda")
    lib = library()
    dims = _dims(x, B)
    if check_inputs:
        bad = {k: v for k, v in ssd_check_inputs(x, dt, dt_bias, A, B, C, D, init_state, stream=stream).items() if v}
        if bad:
            raise ValueError(f"ssd_fwd: non-finite input elements {bad}")
    if ngroups is None:
        ngroups = dims.ngroups
    if y is None:
        y = torch.empty_like(x)
    else:
        _check(y, "y", tuple(x.shape), x.dtype, "cuda")
    if final_state is None and return_final_state:
        final_state = torch.empty((dims.batch, dims.nheads, dims.headdim, dims.dstate), dtype=torch.float32,
                                  device=x.device)
    elif final_state is not None:
        _check(final_state, "final_state", (dims.batch, dims.nheads, dims.headdim, dims.dstate), torch.float32,
               "cuda")
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    io = _io_code(x)
    if seq_idx is not None:
        _check(seq_idx, "seq_idx", (dims.batch, dims.seqlen), torch.int32, "cuda")
    if dt_limit is not None or seq_idx is not None:
        lim = DtLimit(float(dt_limit[0]), float(dt_limit[1])) if dt_limit is not None else None
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_len = workspace.numel() if workspace is not None else 0
        rc = lib.ssd_fwd_ex(ctypes.byref(dims), io, _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
                            _ptr(D), _ptr(init_state), int(chunk_len), int(ngroups), _ptr(y), _ptr(final_state),
                            ctypes.byref(lim) if lim is not None else None, _ptr(seq_idx), PATHS[path], ws_ptr,
                            ws_len, stream)
    elif path == "auto" and workspace is None:
        rc = lib.ssd_fwd(ctypes.byref(dims), io, _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
                         _ptr(D), _ptr(init_state), int(chunk_len), int(ngroups), _ptr(y), _ptr(final_state),
                         stream)
    else:
        code = PATHS[path]
        need = lib.ssd_fwd_workspace_bytes(ctypes.byref(dims), io, int(chunk_len), code)
        if workspace is None:
            workspace = torch.zeros(max(int(need), 1), dtype=torch.uint8, device=x.device)
        rc = lib.ssd_fwd_ws(ctypes.byref(dims), io, _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
                            _ptr(D), _ptr(init_state), int(chunk_len), int(ngroups), _ptr(y), _ptr(final_state),
                            code, workspace.data_ptr(), workspace.numel(), stream)
    if rc != 0:
        raise SsdError(rc, "ssd_fwd")
    return y, final_state


def ssd_fwd_host(x, dt, dt_bias, A, B, C, D=None, init_state=None, chunk_len: int = 256,
                 ngroups: Optional[int] = None, y=None, final_state=None, return_final_state: bool = True,
                 stream=None):
    """End-to-end call on host (CPU, ideally pinned) torch tensors through ssd_fwd_host.

    Copies in, computes, copies out and synchronizes; returns CPU (y, final_state).
    """
    torch = _torch()
    _check_all(x, dt, dt_bias, A, B, C, D, init_state, "cpu")
    lib = library()
    dims = _dims(x, B)
    if ngroups is None:
        ngroups = dims.ngroups
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((dims.batch, dims.nheads, dims.headdim, dims.dstate), dtype=torch.float32)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    rc = lib.ssd_fwd_host(ctypes.byref(dims), _io_code(x), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B),
                          _ptr(C), _ptr(D), _ptr(init_state), int(chunk_len), int(ngroups), _ptr(y),
                          _ptr(final_state), stream)
    if rc != 0:
        raise SsdError(rc, "ssd_fwd_host")
    return y, final_state


def ssd_step(x, dt, dt_bias, A, B, C, D=None, state=None, ngroups: Optional[int] = None, y=None, stream=None,
             dt_limit: Optional[Tuple[float, float]] = None):
    """One decode step through ssd_step (ssd_step_ex with a dt_limit): x [b, h, p],
    dt [b, h], B/C [b, g, n] (CUDA tensors, x/B/C bf16 or fp32 alike), state
    [b, h, p, n] fp32 updated in place. Returns y [b, h, p] (x's dtype).
    Asynchronous on `stream`."""
    torch = _torch()
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [b, h, p] and B [b, g, n]")
    if state is None:
        raise ValueError("state is required (it is updated in place)")
    b, h, p = x.shape
    g, n = B.shape[1], B.shape[2]
    io = x.dtype
    _check(x, "x", (b, h, p), io, "cuda")
    _check(B, "B", (b, g, n), io, "cuda")
    _check(C, "C", (b, g, n), io, "cuda")
    f32 = torch.float32
    _check(dt, "dt", (b, h), f32, "cuda")
    _check(dt_bias, "dt_bias", (h,), f32, "cuda")
    _check(A, "A", (h,), f32, "cuda")
    _check(D, "D", (h,), f32, "cuda", optional=True)
    _check(state, "state", (b, h, p, n), f32, "cuda")
    if y is None:
        y = torch.empty_like(x)
    else:
        _check(y, "y", (b, h, p), io, "cuda")
    if ngroups is None:
        ngroups = g
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    dims = Dims(b, 1, h, p, g, n)
    if dt_limit is None:
        rc = library().ssd_step(ctypes.byref(dims), _io_code(x), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B),
                                _ptr(C), _ptr(D), _ptr(state), int(ngroups), _ptr(y), stream)
    else:
        lim = DtLimit(float(dt_limit[0]), float(dt_limit[1]))
        rc = library().ssd_step_ex(ctypes.byref(dims), _io_code(x), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A),
                                   _ptr(B), _ptr(C), _ptr(D), _ptr(state), int(ngroups), _ptr(y), ctypes.byref(lim),
                                   stream)
    if rc != 0:
        raise SsdError(rc, "ssd_step")
    return y


def _row_view(t, name, rows_shape, io):
    """Row stride (elements) of a CUDA tensor whose last dim is contiguous and
    whose leading dims are packed rows of that stride (e.g. a slice of the
    in_proj output along its last dimension)."""
    if t.dtype != io:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {io}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape[:-1]) != tuple(rows_shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, leading dims must be {tuple(rows_shape)}")
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must be contiguous in its last dimension")
    rs = t.stride(-2) if t.dim() >= 2 else t.shape[-1]
    expect = rs
    for k in range(t.dim() - 2, -1, -1):
        if t.shape[k] > 1 and t.stride(k) != expect:
            raise ValueError(f"{name}: leading dimensions must be packed rows of stride {rs}")
        expect *= t.shape[k]
    return rs


def ssd_conv1d_silu(xbc, weight, bias, d_inner: int, ngroups: int, dstate: int, activation: bool = True,
                    return_state: bool = False, stream=None):
    """Causal depthwise conv1d (+ SiLU) of xbc [b, L, >= conv_dim] (a CUDA
    tensor, bf16 or fp32, last dim contiguous, e.g. a slice of the in_proj
    output) with weight [conv_dim, K] fp32 and bias [conv_dim] fp32 or None.
    Returns x [b, L, d_inner], B [b, L, ngroups, dstate], C [b, L, ngroups, dstate]
    and, with return_state, the conv state [b, conv_dim, K] (else None)."""
    torch = _torch()
    b, L = xbc.shape[0], xbc.shape[1]
    io = xbc.dtype
    cd = d_inner + 2 * ngroups * dstate
    if xbc.shape[2] < cd:
        raise ValueError(f"xbc has {xbc.shape[2]} channels, need at least conv_dim = {cd}")
    rs = _row_view(xbc, "xbc", (b, L), io)
    K = weight.shape[1]
    _check(weight, "weight", (cd, K), torch.float32, "cuda")
    _check(bias, "bias", (cd,), torch.float32, "cuda", optional=True)
    x = torch.empty((b, L, d_inner), dtype=io, device=xbc.device)
    Bo = torch.empty((b, L, ngroups, dstate), dtype=io, device=xbc.device)
    Co = torch.empty_like(Bo)
    st = torch.empty((b, cd, K), dtype=io, device=xbc.device) if return_state else None
    if stream is None:
        stream = torch.cuda.current_stream(xbc.device).cuda_stream
    dims = ConvDims(b, L, d_inner, ngroups, dstate, K)
    rc = library().ssd_conv1d_silu(ctypes.byref(dims), _io_code(xbc), _ptr(xbc), int(rs), _ptr(weight), _ptr(bias),
                                   1 if activation else 0, _ptr(x), _ptr(Bo), _ptr(Co), _ptr(st), stream)
    if rc != 0:
        raise SsdError(rc, "ssd_conv1d_silu")
    return x, Bo, Co, st


def ssd_conv1d_step(xbc, conv_state, weight, bias, d_inner: int, ngroups: int, dstate: int,
                    activation: bool = True, stream=None):
    """One decode token through the conv: xbc [b, >= conv_dim] (last dim
    contiguous), conv_state [b, conv_dim, K] (xbc's dtype, contiguous) updated
    in place. Returns x [b, d_inner], B [b, ngroups, dstate], C [b, ngroups, dstate]."""
    torch = _torch()
    b = xbc.shape[0]
    io = xbc.dtype
    cd = d_inner + 2 * ngroups * dstate
    if xbc.shape[1] < cd:
        raise ValueError(f"xbc has {xbc.shape[1]} channels, need at least conv_dim = {cd}")
    rs = _row_view(xbc, "xbc", (b,), io)
    K = weight.shape[1]
    _check(weight, "weight", (cd, K), torch.float32, "cuda")
    _check(bias, "bias", (cd,), torch.float32, "cuda", optional=True)
    _check(conv_state, "conv_state", (b, cd, K), io, "cuda")
    x = torch.empty((b, d_inner), dtype=io, device=xbc.device)
    Bo = torch.empty((b, ngroups, dstate), dtype=io, device=xbc.device)
    Co = torch.empty_like(Bo)
    if stream is None:
        stream = torch.cuda.current_stream(xbc.device).cuda_stream
    dims = ConvDims(b, 1, d_inner, ngroups, dstate, K)
    rc = library().ssd_conv1d_step(ctypes.byref(dims), _io_code(xbc), _ptr(xbc), int(rs), _ptr(weight), _ptr(bias),
                                   1 if activation else 0, _ptr(conv_state), _ptr(x), _ptr(Bo), _ptr(Co), stream)
    if rc != 0:
        raise SsdError(rc, "ssd_conv1d_step")
    return x, Bo, Co


def ssd_gated_rmsnorm(y, z, weight, eps: float = 1e-5, group_size: Optional[int] = None, out=None, stream=None):
    """Gated RMSNorm (norm_before_gate=False) over the last dimension: y and z
    [..., dim] CUDA tensors of one dtype (last dim contiguous, leading dims
    packed rows; z may be None or a strided slice), weight [dim] fp32.
    Returns out [..., dim] (y's dtype, contiguous unless given)."""
    torch = _torch()
    dim = y.shape[-1]
    lead = tuple(y.shape[:-1])
    rows = 1
    for v in lead:
        rows *= v
    io = y.dtype
    ys = _row_view(y, "y", lead, io)
    zs = _row_view(z, "z", lead, io) if z is not None else 0
    _check(weight, "weight", (dim,), torch.float32, "cuda")
    if out is None:
        out = torch.empty(y.shape, dtype=io, device=y.device)
    os_ = _row_view(out, "out", lead, io)
    if stream is None:
        stream = torch.cuda.current_stream(y.device).cuda_stream
    rc = library().ssd_gated_rmsnorm(_io_code(y), int(rows), int(dim), int(group_size or 0), _ptr(y), int(ys), _ptr(z),
                                     int(zs), _ptr(weight), float(eps), _ptr(out), int(os_), stream)
    if rc != 0:
        raise SsdError(rc, "ssd_gated_rmsnorm")
    return out


def ssd_device_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device status code."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    return int(library().ssd_device_status(stream))


def ssd_fwd_workspace_bytes(batch, seqlen, nheads, headdim, ngroups, dstate, io="bf16", chunk_len=256,
                            path="auto") -> int:
    d = Dims(batch, seqlen, nheads, headdim, ngroups, dstate)
    return int(library().ssd_fwd_workspace_bytes(ctypes.byref(d), DTYPES[io], int(chunk_len), PATHS[path]))


def ssd_select_path(batch, seqlen, nheads, headdim, ngroups, dstate, io="bf16", chunk_len=256) -> str:
    d = Dims(batch, seqlen, nheads, headdim, ngroups, dstate)
    code = int(library().ssd_select_path(ctypes.byref(d), DTYPES[io], int(chunk_len)))
    return {v: k for k, v in PATHS.items()}[code]


def ssd_host_slices(batch, seqlen, nheads, headdim, ngroups, dstate, io="bf16") -> int:
    """Token slices ssd_fwd_host cuts a call of these dims into (0 for invalid dims)."""
    d = Dims(batch, seqlen, nheads, headdim, ngroups, dstate)
    return int(library().ssd_host_slices(ctypes.byref(d), DTYPES[io]))


def ssd_kernel_launches() -> int:
    return int(library().ssd_kernel_launches())


def ssd_kernel_timing(enable: bool) -> None:
    """Record CUDA events around each forward's main kernel (ssd_kernel_timing)."""
    library().ssd_kernel_timing(1 if enable else 0)


def ssd_kernel_timing_read() -> Tuple[float, int]:
    """(summed milliseconds, count) of the recorded main-kernel launches; clears them."""
    ms, n = ctypes.c_double(0.0), ctypes.c_uint64(0)
    rc = library().ssd_kernel_timing_read(ctypes.byref(ms), ctypes.byref(n))
    if rc != 0:
        raise SsdError(rc, "ssd_kernel_timing_read")
    return float(ms.value), int(n.value)


def ssd_release() -> None:
    library().ssd_release()

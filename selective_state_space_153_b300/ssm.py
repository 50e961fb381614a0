"""Thin Python binding of the C ABI in include/ssm_scan.h (libssm_scan.so), by ctypes.

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels. Tensors are torch tensors (device memory for the device entry points, host
memory for ``selective_scan_fwd_host``); their raw pointers are passed through unchanged.
There is no CPU fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssm_scan.so")

SSM_OK, SSM_ERR_NULL, SSM_ERR_SHAPE, SSM_ERR_DTYPE, SSM_ERR_ALIGN = 0, 1, 2, 3, 4
SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_WORKSPACE, SSM_ERR_CHECK = 5, 6, 7, 8, 9
SSM_F32, SSM_BF16 = 0, 1
SSM_DISC_EULER, SSM_DISC_ZOH = 0, 1
_DISC = {"euler": SSM_DISC_EULER, "zoh": SSM_DISC_ZOH}
MAX_DSTATE = 128
SCRATCH_MAX_BYTES = 48 * 1024 * 1024   # SSM_SCRATCH_MAX_BYTES: the no-alloc entry's fixed scratch

# every symbol include/ssm_scan.h declares
EXPORTS = ("ssm_selective_scan_fwd", "ssm_selective_scan_workspace_bytes",
           "ssm_selective_scan_fwd_ws", "ssm_state_update", "ssm_selective_scan_fwd_host",
           "ssm_stream_status", "ssm_status_string", "ssm_version",
           "ssm_selective_scan_fwd_noalloc", "ssm_selective_scan_fwd_disc", "ssm_state_update_disc",
           "ssm_conv_selective_scan_fwd", "ssm_conv_selective_scan_workspace_bytes",
           "ssm_selective_scan_bwd", "ssm_selective_scan_bwd_workspace_bytes",
           "ssm_set_structured_a", "ssm_set_workspace", "ssm_set_plan_override",
           "ssm_get_plan_override", "ssm_last_cuda_error", "ssm_cuda_error_string")

# ssm_kernel_t
SSM_KERNEL_AUTO, SSM_KERNEL_PAIR, SSM_KERNEL_SEQ, SSM_KERNEL_TC, SSM_KERNEL_TP = range(5)
_KERNELS = {"auto": SSM_KERNEL_AUTO, "pair": SSM_KERNEL_PAIR, "seq": SSM_KERNEL_SEQ, "tc": SSM_KERNEL_TC,
            "tp": SSM_KERNEL_TP}


class SsmDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("io_dtype", ctypes.c_int)]


class PlanOverride(ctypes.Structure):
    """ssm_plan_override_t: every field 0 = the planner's choice."""
    _fields_ = [("kernel", ctypes.c_int), ("pair_states_per_lane", ctypes.c_int), ("chunks", ctypes.c_int),
                ("seq_states_per_lane", ctypes.c_int), ("seq_lanes_per_channel", ctypes.c_int),
                ("decode_elementwise", ctypes.c_int), ("force_timeout", ctypes.c_int),
                ("check_probe", ctypes.c_int), ("bwd_states_per_lane", ctypes.c_int),
                ("bwd_chunks", ctypes.c_int)]


class SsmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {status_string(code)}"
        if code == SSM_ERR_CUDA and _lib is not None:
            e = _lib.ssm_last_cuda_error()
            msg += f" ({e}: {_lib.ssm_cuda_error_string(e).decode()})"
        super().__init__(msg)


_lib = None
_vp = ctypes.c_void_p


def load(path: str = LIB_PATH):
    """Load libssm_scan.so (raises if it is missing: build it with
    ``python -m selective_state_space_153_b300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = load_library(path)
    return _lib


@contextlib.contextmanager
def using(lib):
    """Route this module's calls to another loaded build of the library (for instance the
    checked build, -DSSM_CHECK) inside the block."""
    global _lib
    prev = load()
    _lib = lib
    try:
        yield lib
    finally:
        _lib = prev


def load_library(path: str):
    """Load a build of the library at ``path`` with its argument types set (not cached)."""
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path}")
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(SsmDims)
    scan_args = [dp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp]
    lib.ssm_selective_scan_fwd.argtypes = scan_args + [_vp]
    lib.ssm_selective_scan_fwd.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_ws.argtypes = scan_args + [_vp, ctypes.c_size_t, _vp]
    lib.ssm_selective_scan_fwd_ws.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_host.argtypes = scan_args + [_vp]
    lib.ssm_selective_scan_fwd_disc.argtypes = scan_args[:10] + [ctypes.c_int] + scan_args[10:] + [_vp, ctypes.c_size_t, _vp]
    lib.ssm_selective_scan_fwd_disc.restype = ctypes.c_int
    lib.ssm_state_update_disc.argtypes = [dp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp]
    lib.ssm_state_update_disc.restype = ctypes.c_int
    lib.ssm_conv_selective_scan_fwd.argtypes = [dp, _vp, _vp, _vp, ctypes.c_int] + scan_args[2:] + [_vp, ctypes.c_size_t, _vp]
    lib.ssm_conv_selective_scan_fwd.restype = ctypes.c_int
    lib.ssm_conv_selective_scan_workspace_bytes.argtypes = [dp]
    lib.ssm_conv_selective_scan_workspace_bytes.restype = ctypes.c_size_t
    lib.ssm_selective_scan_bwd.argtypes = scan_args[:10] + [_vp] * 10 + [_vp, ctypes.c_size_t, _vp]
    lib.ssm_selective_scan_bwd.restype = ctypes.c_int
    lib.ssm_selective_scan_bwd_workspace_bytes.argtypes = [dp]
    lib.ssm_selective_scan_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.ssm_selective_scan_fwd_noalloc.argtypes = scan_args + [_vp]
    lib.ssm_selective_scan_fwd_noalloc.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_host.restype = ctypes.c_int
    lib.ssm_selective_scan_workspace_bytes.argtypes = [dp]
    lib.ssm_selective_scan_workspace_bytes.restype = ctypes.c_size_t
    lib.ssm_state_update.argtypes = [dp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.ssm_state_update.restype = ctypes.c_int
    lib.ssm_stream_status.argtypes = [_vp]
    lib.ssm_stream_status.restype = ctypes.c_int
    lib.ssm_status_string.argtypes = [ctypes.c_int]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_version.argtypes = []
    lib.ssm_last_cuda_error.argtypes = []
    lib.ssm_last_cuda_error.restype = ctypes.c_int
    lib.ssm_cuda_error_string.argtypes = [ctypes.c_int]
    lib.ssm_cuda_error_string.restype = ctypes.c_char_p
    lib.ssm_version.restype = ctypes.c_int
    lib.ssm_set_structured_a.argtypes = [ctypes.c_int]
    lib.ssm_set_structured_a.restype = ctypes.c_int
    lib.ssm_set_workspace.argtypes = [_vp, ctypes.c_size_t]
    lib.ssm_set_workspace.restype = ctypes.c_int
    lib.ssm_set_plan_override.argtypes = [ctypes.POINTER(PlanOverride)]
    lib.ssm_set_plan_override.restype = ctypes.c_int
    lib.ssm_get_plan_override.argtypes = [ctypes.POINTER(PlanOverride)]
    lib.ssm_get_plan_override.restype = ctypes.c_int
    return lib


def status_string(code: int) -> str:
    return load().ssm_status_string(int(code)).decode()


def _io_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    if t.dtype == torch.float32:
        return SSM_F32
    raise TypeError(f"io dtype must be bfloat16 or float32, got {t.dtype}")


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return _vp(t.data_ptr())


def _stream_ptr(stream) -> Optional[ctypes.c_void_p]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream) if hasattr(stream, "cuda_stream") else _vp(int(stream))


def dims(batch, dim, seqlen, dstate, io) -> SsmDims:
    return SsmDims(int(batch), int(dim), int(seqlen), int(dstate), int(io))


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                       y=None, last_state=None, return_last_state=False, stream=None,
                       workspace=None, discretization="euler") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Device scan. u, delta, z [Bt, D, L]; B, C [Bt, N, L] (io dtype); A [D, N], D, bias [D]
    fp32. Returns (y, last_state or None). ``workspace``: optional uint8 device tensor for
    ssm_selective_scan_fwd_ws. ``discretization``: "euler" (B_bar = dt*B) or "zoh" (exact
    zero-order hold, through ssm_selective_scan_fwd_disc)."""
    lib = load()
    Bt, Dm, L = u.shape
    N = A.shape[1]
    io = _io_code(u)
    if y is None:
        y = torch.empty_like(u)
    if return_last_state and last_state is None:
        last_state = torch.empty((Bt, Dm, N), dtype=torch.float32, device=u.device)
    dm = dims(Bt, Dm, L, N, io)
    args = [ctypes.byref(dm), _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
            int(bool(delta_softplus)), _p(y), _p(last_state)]
    if discretization != "euler":
        ws_p = None if workspace is None else _p(workspace)
        ws_n = 0 if workspace is None else workspace.numel() * workspace.element_size()
        rc = lib.ssm_selective_scan_fwd_disc(*args[:10], _DISC[discretization], *args[10:], ws_p, ws_n,
                                             _stream_ptr(stream))
    elif workspace is None:
        rc = lib.ssm_selective_scan_fwd(*args, _stream_ptr(stream))
    else:
        rc = lib.ssm_selective_scan_fwd_ws(*args, _p(workspace), workspace.numel() * workspace.element_size(),
                                           _stream_ptr(stream))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_selective_scan_fwd")
    return y, last_state


def selective_scan_fwd_noalloc(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                               y=None, last_state=None, return_last_state=False, stream=None
                               ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Device scan through ssm_selective_scan_fwd_noalloc: no device allocation inside the
    library; its scratch is the library's fixed per-device array of SCRATCH_MAX_BYTES.
    Raises SsmError (SSM_ERR_WORKSPACE) for a shape whose scratch exceeds that size. Calls
    that overlap on the GPU share the scratch and race: keep them on one stream."""
    lib = load()
    Bt, Dm, L = u.shape
    N = A.shape[1]
    io = _io_code(u)
    if y is None:
        y = torch.empty_like(u)
    if return_last_state and last_state is None:
        last_state = torch.empty((Bt, Dm, N), dtype=torch.float32, device=u.device)
    dm = dims(Bt, Dm, L, N, io)
    rc = lib.ssm_selective_scan_fwd_noalloc(ctypes.byref(dm), _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D),
                                            _p(z), _p(delta_bias), int(bool(delta_softplus)), _p(y),
                                            _p(last_state), _stream_ptr(stream))
    if rc != SSM_OK:
        need = workspace_bytes(Bt, Dm, L, N, io)
        raise SsmError(rc, f"ssm_selective_scan_fwd_noalloc (scratch needed {need} B, "
                           f"fixed size {SCRATCH_MAX_BYTES} B)")
    return y, last_state


def conv_selective_scan_fwd(x, conv_w, conv_b, delta, A, B, C, D=None, z=None, delta_bias=None,
                            delta_softplus=True, y=None, last_state=None, return_last_state=False,
                            stream=None, workspace=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Causal depthwise conv (conv_w [D, K] fp32, K <= 4; conv_b [D] or None) + SiLU fused in
    front of the scan, through ssm_conv_selective_scan_fwd. x: [Bt, D, L] io dtype (the conv
    input); other tensors as selective_scan_fwd."""
    lib = load()
    Bt, Dm, L = x.shape
    N = A.shape[1]
    io = _io_code(x)
    if y is None:
        y = torch.empty_like(x)
    if return_last_state and last_state is None:
        last_state = torch.empty((Bt, Dm, N), dtype=torch.float32, device=x.device)
    dm = dims(Bt, Dm, L, N, io)
    ws_p = None if workspace is None else _p(workspace)
    ws_n = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.ssm_conv_selective_scan_fwd(ctypes.byref(dm), _p(x), _p(conv_w), _p(conv_b), int(conv_w.shape[1]),
                                         _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                         int(bool(delta_softplus)), _p(y), _p(last_state), ws_p, ws_n,
                                         _stream_ptr(stream))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_conv_selective_scan_fwd")
    return y, last_state


def selective_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=True,
                       dlast_state=None, stream=None, workspace=None):
    """Gradients of sum(y*dy) (+ sum(last_state*dlast_state)) through the device scan, via
    ssm_selective_scan_bwd. Returns a dict of fp32 device tensors: u, delta, A, B, C, and
    D / z / delta_bias when those inputs are given."""
    lib = load()
    Bt, Dm, L = u.shape
    N = A.shape[1]
    io = _io_code(u)
    f32 = dict(dtype=torch.float32, device=u.device)
    g = {"u": torch.empty((Bt, Dm, L), **f32), "delta": torch.empty((Bt, Dm, L), **f32),
         "A": torch.empty((Dm, N), **f32), "B": torch.empty((Bt, N, L), **f32), "C": torch.empty((Bt, N, L), **f32),
         "D": torch.empty((Dm,), **f32) if D is not None else None,
         "z": torch.empty((Bt, Dm, L), **f32) if z is not None else None,
         "delta_bias": torch.empty((Dm,), **f32) if delta_bias is not None else None}
    dm = dims(Bt, Dm, L, N, io)
    ws_p = None if workspace is None else _p(workspace)
    ws_n = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.ssm_selective_scan_bwd(ctypes.byref(dm), _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z),
                                    _p(delta_bias), int(bool(delta_softplus)), _p(dy), _p(dlast_state),
                                    _p(g["u"]), _p(g["delta"]), _p(g["A"]), _p(g["B"]), _p(g["C"]), _p(g["D"]),
                                    _p(g["z"]), _p(g["delta_bias"]), ws_p, ws_n, _stream_ptr(stream))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_selective_scan_bwd")
    return g


def workspace_bytes(Bt, Dm, L, N, io=SSM_BF16) -> int:
    return int(load().ssm_selective_scan_workspace_bytes(ctypes.byref(dims(Bt, Dm, L, N, io))))


def selective_scan_fwd_host(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                            y=None, last_state=None, return_last_state=False, stream=None):
    """Host-buffer scan: every tensor on the CPU (pinned for speed); copies in, scans on
    the GPU, copies out, returns when the results are in the host tensors."""
    lib = load()
    Bt, Dm, L = u.shape
    N = A.shape[1]
    io = _io_code(u)
    if y is None:
        y = torch.empty_like(u)
    if return_last_state and last_state is None:
        last_state = torch.empty((Bt, Dm, N), dtype=torch.float32)
    dm = dims(Bt, Dm, L, N, io)
    rc = lib.ssm_selective_scan_fwd_host(ctypes.byref(dm), _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D),
                                         _p(z), _p(delta_bias), int(bool(delta_softplus)), _p(y),
                                         _p(last_state), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_selective_scan_fwd_host")
    return y, last_state


def state_update(state, x, dt, A, B, C, D=None, z=None, y=None, stream=None,
                 discretization="euler") -> torch.Tensor:
    """In-place recurrent step on ``state`` [Bt, D, N] fp32; x, dt, z [Bt, D]; B, C [Bt, N]
    (io dtype); A [D, N]; D [D]. Returns y [Bt, D]. ``discretization``: "euler" or "zoh"."""
    lib = load()
    Bt, Dm, N = state.shape
    io = _io_code(x)
    if y is None:
        y = torch.empty_like(x)
    dm = dims(Bt, Dm, 1, N, io)
    if discretization != "euler":
        rc = lib.ssm_state_update_disc(ctypes.byref(dm), _p(state), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D),
                                       _p(z), _DISC[discretization], _p(y), _stream_ptr(stream))
    else:
        rc = lib.ssm_state_update(ctypes.byref(dm), _p(state), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D),
                                  _p(z), _p(y), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_state_update")
    return y


def stream_status(stream=None) -> int:
    return int(load().ssm_stream_status(_stream_ptr(stream)))


def set_structured_a(enable: bool) -> bool:
    """Switch the forward scans' run-time structured-A test (A[d, n] == (n + 1) * A[d, 0]
    for every state of a warp's channels; such warps form the decays from powers of
    exp(dt * A[d, 0])). Off by default; returns the previous setting. Process-wide."""
    return bool(load().ssm_set_structured_a(1 if enable else 0))


def set_workspace(workspace: Optional[torch.Tensor]) -> None:
    """Register ``workspace`` (a device tensor, any dtype, 16-byte aligned) as the current
    device's default scan workspace (ssm_set_workspace), or unregister it with None. While one
    is registered, scans without a workspace of their own use it and never allocate; keep the
    tensor alive until those calls have completed."""
    lib = load()
    if workspace is None:
        rc = lib.ssm_set_workspace(None, 0)
    else:
        rc = lib.ssm_set_workspace(_p(workspace), workspace.numel() * workspace.element_size())
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_set_workspace")


def get_plan_override() -> PlanOverride:
    ov = PlanOverride()
    rc = load().ssm_get_plan_override(ctypes.byref(ov))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_get_plan_override")
    return ov


def set_plan_override(ov: Optional[PlanOverride]) -> None:
    rc = load().ssm_set_plan_override(None if ov is None else ctypes.byref(ov))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_set_plan_override")


@contextlib.contextmanager
def plan_override(kernel: str = "auto", pair_states_per_lane: int = 0, chunks: int = 0,
                  seq_split: Optional[Tuple[int, int]] = None, decode_elementwise: bool = False,
                  force_timeout: bool = False, check_probe: bool = False, bwd_states_per_lane: int = 0,
                  bwd_chunks: int = 0):
    """Force a launch plan for the calls inside the block (ssm_set_plan_override; a test and
    tuning hook), then restore the override that was in force before."""
    prev = get_plan_override()
    ov = PlanOverride(_KERNELS[kernel], int(pair_states_per_lane), int(chunks),
                      int(seq_split[0]) if seq_split else 0, int(seq_split[1]) if seq_split else 0,
                      int(bool(decode_elementwise)), int(bool(force_timeout)), int(bool(check_probe)),
                      int(bwd_states_per_lane), int(bwd_chunks))
    set_plan_override(ov)
    try:
        yield ov
    finally:
        set_plan_override(prev)


def version() -> Tuple[int, int]:
    v = int(load().ssm_version())
    return v >> 16, v & 0xFFFF

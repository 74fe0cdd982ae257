"""Python binding of the GB300 fused RMSNorm library (librms_norm_gb300.so).

Argument marshalling only: every step of the forward and the backward runs
in the library's CUDA kernels.  PyTorch supplies device memory and the
current CUDA stream.  There is no CPU fallback: without the built library,
or with tensors that are not on a CUDA device, every call raises.

The functions carry the names of the C entry points declared in
``include/rms_norm.h``:

* ``rms_norm_fwd(x, gamma, eps, offset=0, cast_mode="round_once")``
  -> ``(y, rstd)``
* ``rms_norm_bwd(dy, x, gamma, rstd, offset=0)`` -> ``(dx, dw)``
* ``rms_norm_bwd_workspace_size(rows, hidden, dtype)``
* ``rms_norm_status_string(status)``
* ``rms_norm_bwd_noalloc(dy, x, gamma, rstd, offset=0)`` -> ``(dx, dw)``
* ``rms_norm_bwd_blocked(dy, x, gamma, rstd, block_rows, offset=0)`` ->
  ``(dx, chunk_sums)``; ``rms_norm_dw_sum(chunk_sums)`` -> ``dw``;
  ``rms_norm_dw_chunk_count(rows, block_rows)``;
  ``rms_norm_bwd_blocked_workspace_size(rows, hidden, block_rows)``;
  ``rms_norm_rank_rows(rows, block_rows, world, rank)`` -> ``(lo, hi)`` (the
  weight gradient in an order that any split of the rows reproduces)
* ``rms_norm_set_sm_budget(sms)``, ``rms_norm_sm_budget()
* ``rms_norm_fwd_fp8(x, gamma, scale, eps, offset=0)`` -> ``(y8, rstd)``
  (``y8`` a torch.float8_e4m3fn tensor, ``scale`` a one-element fp32
  device tensor)
* ``softmax_fwd(x)`` -> ``y``; ``softmax_bwd(dy, y)`` -> ``dx`` (last
  dimension)
* ``group_norm_fwd(x, gamma, beta, groups, eps)`` -> ``(y, mean, rstd)``;
  ``group_norm_bwd(dy, x, gamma, mean, rstd, groups)`` ->
  ``(dx, dgamma, dbeta)`` (x of shape [n, channels, *spatial])
* ``layer_norm_fwd(x, gamma, beta, eps)`` -> ``(y, mean, rstd)``
* ``layer_norm_bwd(dy, x, gamma, mean, rstd)`` -> ``(dx, dgamma, dbeta)``

For autograd: ``rms_norm(x, weight, eps, offset=0, cast_mode="round_once")``
(a ``torch.autograd.Function`` over rms_norm_fwd / rms_norm_bwd) and the
module ``RMSNorm(hidden, eps, offset=0, cast_mode="round_once")``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

LIB_NAME = "librms_norm_gb300.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

# Values of the C enums (include/rms_norm.h).
RMSN_F32, RMSN_BF16, RMSN_F16 = 0, 1, 2
RMSN_ROUND_ONCE, RMSN_ROUND_TWICE = 0, 1
RMSN_OK = 0
RMSN_MAX_HIDDEN = 65536
RMSN_MAX_PARTIALS = 1024
RMSN_DW_CHUNK_BLOCKS = 32

DTYPE_CODES = {torch.float32: RMSN_F32, torch.bfloat16: RMSN_BF16, torch.float16: RMSN_F16}
CAST_MODES = {"round_once": RMSN_ROUND_ONCE, "round_twice": RMSN_ROUND_TWICE}

EXPORTED = (
    "rms_norm_fwd",
    "rms_norm_bwd_workspace_size",
    "rms_norm_bwd",
    "rms_norm_status_string",
    "rms_norm_last_cuda_error",
    "rms_norm_last_launch_count",
    "rms_norm_last_kernels",
    "rms_norm_bwd_noalloc",
    "rms_norm_bwd_blocked_workspace_size",
    "rms_norm_dw_chunk_count",
    "rms_norm_bwd_blocked",
    "rms_norm_dw_sum",
    "rms_norm_rank_rows",
    "rms_norm_set_sm_budget",
    "rms_norm_sm_budget",
    "rms_norm_wait_timeouts",
    "rms_norm_selftest_wait_limit",
    "rms_norm_fwd_fp8",
    "layer_norm_fwd",
    "layer_norm_bwd_workspace_size",
    "layer_norm_bwd",
    "softmax_fwd",
    "softmax_bwd",
    "group_norm_fwd",
    "group_norm_bwd_workspace_size",
    "group_norm_bwd",
)


class RMSNormError(RuntimeError):
    """A C entry point returned an error status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({rms_norm_status_string(status)})")


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library and declare the C signatures (once)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -m bwd_rms_norm_gb300.build)")
    lib = ctypes.CDLL(path)
    P, I64, I, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.rms_norm_fwd.argtypes = [P, P, P, P, I64, I64, F, I, I, I, P]
    lib.rms_norm_fwd.restype = I
    lib.rms_norm_bwd_workspace_size.argtypes = [I64, I64, I]
    lib.rms_norm_bwd_workspace_size.restype = SZ
    lib.rms_norm_bwd.argtypes = [P, P, P, P, P, P, I64, I64, I, I, P, SZ, P]
    lib.rms_norm_bwd.restype = I
    lib.rms_norm_status_string.argtypes = [I]
    lib.rms_norm_status_string.restype = ctypes.c_char_p
    lib.rms_norm_last_cuda_error.argtypes = []
    lib.rms_norm_last_cuda_error.restype = I
    lib.rms_norm_last_kernels.argtypes = [ctypes.POINTER(ctypes.c_char_p), I]
    lib.rms_norm_last_kernels.restype = I
    lib.rms_norm_last_launch_count.argtypes = []
    lib.rms_norm_last_launch_count.restype = I
    lib.rms_norm_bwd_noalloc.argtypes = [P, P, P, P, P, P, I64, I64, I, I, P]
    lib.rms_norm_bwd_noalloc.restype = I
    lib.rms_norm_bwd_blocked_workspace_size.argtypes = [I64, I64, I64]
    lib.rms_norm_bwd_blocked_workspace_size.restype = SZ
    lib.rms_norm_dw_chunk_count.argtypes = [I64, I64]
    lib.rms_norm_dw_chunk_count.restype = I64
    lib.rms_norm_bwd_blocked.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P]
    lib.rms_norm_bwd_blocked.restype = I
    lib.rms_norm_dw_sum.argtypes = [P, I64, I64, P, P]
    lib.rms_norm_dw_sum.restype = I
    lib.rms_norm_rank_rows.argtypes = [I64, I64, I, I, ctypes.POINTER(I64), ctypes.POINTER(I64)]
    lib.rms_norm_rank_rows.restype = I
    lib.rms_norm_set_sm_budget.argtypes = [I]
    lib.rms_norm_set_sm_budget.restype = I
    lib.rms_norm_sm_budget.argtypes = []
    lib.rms_norm_sm_budget.restype = I
    lib.rms_norm_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.rms_norm_wait_timeouts.restype = I
    lib.rms_norm_selftest_wait_limit.argtypes = [ctypes.POINTER(ctypes.c_uint),
                                                 ctypes.POINTER(ctypes.c_double)]
    lib.rms_norm_selftest_wait_limit.restype = I
    lib.rms_norm_fwd_fp8.argtypes = [P, P, P, P, P, I64, I64, F, I, I, P]
    lib.rms_norm_fwd_fp8.restype = I
    lib.group_norm_fwd.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, F, I, P]
    lib.group_norm_fwd.restype = I
    lib.group_norm_bwd_workspace_size.argtypes = [I64, I64, I64, I64, I]
    lib.group_norm_bwd_workspace_size.restype = SZ
    lib.group_norm_bwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, I, P, SZ, P]
    lib.group_norm_bwd.restype = I
    lib.softmax_fwd.argtypes = [P, P, I64, I64, I, P]
    lib.softmax_fwd.restype = I
    lib.softmax_bwd.argtypes = [P, P, P, I64, I64, I, P]
    lib.softmax_bwd.restype = I
    lib.layer_norm_fwd.argtypes = [P, P, P, P, P, P, I64, I64, F, I, P]
    lib.layer_norm_fwd.restype = I
    lib.layer_norm_bwd_workspace_size.argtypes = [I64, I64, I]
    lib.layer_norm_bwd_workspace_size.restype = SZ
    lib.layer_norm_bwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I, P, SZ, P]
    lib.layer_norm_bwd.restype = I
    _lib = lib
    return lib


def rms_norm_status_string(status: int) -> str:
    return load_library().rms_norm_status_string(int(status)).decode()


def rms_norm_bwd_workspace_size(rows: int, hidden: int, dtype) -> int:
    """Bytes of workspace ``rms_norm_bwd`` needs (``dtype`` a torch dtype or
    a C code)."""
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().rms_norm_bwd_workspace_size(int(rows), int(hidden), code))


def last_launch_count() -> int:
    """Kernels enqueued by the last successful call on this thread."""
    return int(load_library().rms_norm_last_launch_count())


def last_kernels() -> list:
    """Symbol names of the kernels the last call on this thread launched."""
    buf = (ctypes.c_char_p * 4)()
    n = load_library().rms_norm_last_kernels(buf, 4)
    return [buf[i].decode() for i in range(max(n, 0))]


def wait_timeouts() -> int:
    """Bounded device waits that ran out since the library was loaded (0 in
    correct operation); synchronises with the device."""
    n = ctypes.c_uint(0)
    st = load_library().rms_norm_wait_timeouts(ctypes.byref(n))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_wait_timeouts", st)
    return int(n.value)


def selftest_wait_limit() -> Tuple[int, float]:
    """Run the bounded-wait self-test (a wait on a barrier nothing completes
    runs out after about a second): returns (waits that ran out, seconds)."""
    n, t = ctypes.c_uint(0), ctypes.c_double(0.0)
    st = load_library().rms_norm_selftest_wait_limit(ctypes.byref(n), ctypes.byref(t))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_selftest_wait_limit", st)
    return int(n.value), float(t.value)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None or t.numel() == 0 else t.data_ptr()


def _stream_handle(device: torch.device, stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _check_cuda(name: str, t: torch.Tensor, device: Optional[torch.device] = None) -> None:
    if not t.is_cuda:
        raise RuntimeError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if device is not None and t.device != device:
        raise RuntimeError(f"{name} is on {t.device}, the other tensors on {device}")
    if not t.is_contiguous():
        raise RuntimeError(f"{name} must be contiguous")


def _check_like(name: str, t: Optional[torch.Tensor], dtype: torch.dtype, numel: int,
                shape=None) -> None:
    """A tensor the kernels read or write a fixed extent of: its dtype and
    size are checked on the host before anything reaches the device (a short
    buffer would be read or written out of bounds)."""
    if t is None:
        return
    if t.dtype != dtype:
        raise RuntimeError(f"{name} must be {dtype}, not {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise RuntimeError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    if t.numel() != numel:
        raise RuntimeError(f"{name} must have {numel} elements, not {t.numel()}")


def _check_bwd_args(dy, x, gamma, rstd, dx, dw) -> Tuple[int, int]:
    """Host-side checks shared by the RMSNorm backward entry points: dtypes,
    shapes and element counts of every tensor, caller-supplied outputs
    included.  Returns (rows, hidden)."""
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    rows, hidden = _as_rows(x)
    _check_like("dy", dy, x.dtype, x.numel(), x.shape)
    _check_like("gamma", gamma, x.dtype, hidden)
    _check_like("rstd", rstd, torch.float32, rows)
    _check_like("dx", dx, x.dtype, x.numel(), x.shape)
    _check_like("dw", dw, torch.float32, hidden)
    return rows, hidden


def _as_rows(x: torch.Tensor) -> Tuple[int, int]:
    if x.dim() < 1:
        raise RuntimeError("x must have at least one dimension")
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden > 0 else 0
    return rows, hidden


def rms_norm_fwd(x: torch.Tensor, gamma: torch.Tensor, eps: float, offset: int = 0,
                 cast_mode: str = "round_once", y: Optional[torch.Tensor] = None,
                 rstd: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None):
    """Forward over the last dimension of ``x``; returns ``(y, rstd)`` with
    ``y`` shaped like ``x`` and ``rstd`` fp32 of shape ``x.shape[:-1]``."""
    lib = load_library()
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    if cast_mode not in CAST_MODES:
        raise RuntimeError(f"cast_mode must be one of {sorted(CAST_MODES)}")
    rows, hidden = _as_rows(x)
    _check_like("gamma", gamma, x.dtype, hidden)
    _check_like("y", y, x.dtype, x.numel(), x.shape)
    _check_like("rstd", rstd, torch.float32, rows)
    _check_cuda("x", x)
    _check_cuda("gamma", gamma, x.device)
    if y is None:
        y = torch.empty_like(x)
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _check_cuda("y", y, x.device)
    _check_cuda("rstd", rstd, x.device)
    with torch.cuda.device(x.device):
        st = lib.rms_norm_fwd(_ptr(x), _ptr(gamma), _ptr(y), _ptr(rstd), rows, hidden,
                              float(eps), int(offset), DTYPE_CODES[x.dtype],
                              CAST_MODES[cast_mode], _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_fwd", st)
    return y, rstd


FP8_DTYPE = torch.float8_e4m3fn


def rms_norm_fwd_fp8(x: torch.Tensor, gamma: torch.Tensor, scale: torch.Tensor, eps: float,
                     offset: int = 0, y: Optional[torch.Tensor] = None,
                     rstd: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None):
    """Forward with an FP8 E4M3 output: ``y = e4m3(x_hat * gain * scale)``
    (saturating).  ``scale`` is a one-element fp32 tensor on the device (read
    by the kernel); returns ``(y, rstd)`` with ``y`` of dtype
    torch.float8_e4m3fn shaped like ``x``."""
    lib = load_library()
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    rows, hidden = _as_rows(x)
    _check_like("gamma", gamma, x.dtype, hidden)
    _check_like("scale", scale, torch.float32, 1)
    _check_like("y", y, FP8_DTYPE, x.numel(), x.shape)
    _check_like("rstd", rstd, torch.float32, rows)
    _check_cuda("x", x)
    _check_cuda("gamma", gamma, x.device)
    _check_cuda("scale", scale, x.device)
    if y is None:
        y = torch.empty(x.shape, dtype=FP8_DTYPE, device=x.device)
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _check_cuda("y", y, x.device)
    _check_cuda("rstd", rstd, x.device)
    with torch.cuda.device(x.device):
        st = lib.rms_norm_fwd_fp8(_ptr(x), _ptr(gamma), _ptr(scale), _ptr(y), _ptr(rstd), rows,
                                  hidden, float(eps), int(offset), DTYPE_CODES[x.dtype],
                                  _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_fwd_fp8", st)
    return y, rstd


def rms_norm_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, rstd: torch.Tensor,
                 offset: int = 0, dx: Optional[torch.Tensor] = None,
                 dw: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None):
    """Backward; returns ``(dx, dw)`` with ``dw`` fp32 of shape ``[hidden]``.
    ``workspace`` (a byte or float tensor of at least
    ``rms_norm_bwd_workspace_size`` bytes) is allocated when not given."""
    lib = load_library()
    rows, hidden = _check_bwd_args(dy, x, gamma, rstd, dx, dw)
    for name, t in (("x", x), ("dy", dy), ("gamma", gamma), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    code = DTYPE_CODES[x.dtype]
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(hidden, dtype=torch.float32, device=x.device)
    need = int(lib.rms_norm_bwd_workspace_size(rows, hidden, code))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check_cuda("dx", dx, x.device)
    _check_cuda("dw", dw, x.device)
    _check_cuda("workspace", workspace, x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(x.device):
        st = lib.rms_norm_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx), _ptr(dw),
                              rows, hidden, int(offset), code, workspace.data_ptr(), ws_bytes,
                              _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_bwd", st)
    return dx, dw


def rms_norm_bwd_noalloc(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor,
                         rstd: torch.Tensor, offset: int = 0, dx: Optional[torch.Tensor] = None,
                         dw: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None):
    """Backward for callers that cannot allocate device scratch: the library
    keeps the weight-gradient partials in its own fixed 16 MiB device array
    (sizes needing more are refused).  Pass ``dx`` and ``dw`` to avoid any
    allocation on the Python side as well.  Calls that may overlap on the GPU
    share that array and must be ordered on one stream."""
    lib = load_library()
    rows, hidden = _check_bwd_args(dy, x, gamma, rstd, dx, dw)
    for name, t in (("x", x), ("dy", dy), ("gamma", gamma), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(hidden, dtype=torch.float32, device=x.device)
    _check_cuda("dx", dx, x.device)
    _check_cuda("dw", dw, x.device)
    with torch.cuda.device(x.device):
        st = lib.rms_norm_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx),
                                      _ptr(dw), rows, hidden, int(offset), DTYPE_CODES[x.dtype],
                                      _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_bwd_noalloc", st)
    return dx, dw


def rms_norm_dw_chunk_count(rows: int, block_rows: int) -> int:
    """Chunk sums ``rms_norm_bwd_blocked`` writes for ``rows`` rows."""
    n = int(load_library().rms_norm_dw_chunk_count(int(rows), int(block_rows)))
    if n < 0:
        raise RMSNormError("rms_norm_dw_chunk_count", -n)
    return n


def rms_norm_bwd_blocked_workspace_size(rows: int, hidden: int, block_rows: int) -> int:
    """Bytes of workspace ``rms_norm_bwd_blocked`` needs."""
    return int(load_library().rms_norm_bwd_blocked_workspace_size(int(rows), int(hidden),
                                                                  int(block_rows)))


def rms_norm_rank_rows(rows: int, block_rows: int, world: int, rank: int) -> Tuple[int, int]:
    """Rank ``rank``'s slab [lo, hi) of ``rows`` rows in whole chunks of
    ``RMSN_DW_CHUNK_BLOCKS * block_rows`` rows (no device needed)."""
    lo, hi = ctypes.c_int64(0), ctypes.c_int64(0)
    st = load_library().rms_norm_rank_rows(int(rows), int(block_rows), int(world), int(rank),
                                           ctypes.byref(lo), ctypes.byref(hi))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_rank_rows", st)
    return int(lo.value), int(hi.value)


def rms_norm_bwd_blocked(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor,
                         rstd: torch.Tensor, block_rows: int, offset: int = 0,
                         dx: Optional[torch.Tensor] = None,
                         chunk_sums: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None):
    """Backward with the weight gradient left as chunk sums over fixed blocks
    of ``block_rows`` rows; returns ``(dx, chunk_sums)``, ``chunk_sums`` fp32
    of shape [rms_norm_dw_chunk_count(rows, block_rows), hidden].  Adding
    them with ``rms_norm_dw_sum`` gives the same dw for any split of the rows
    into whole chunks (see ``rms_norm_rank_rows``)."""
    lib = load_library()
    rows, hidden = _check_bwd_args(dy, x, gamma, rstd, dx, None)
    if int(block_rows) < 1:
        raise RuntimeError("block_rows must be at least 1")
    nchunks = rms_norm_dw_chunk_count(rows, block_rows)
    _check_like("chunk_sums", chunk_sums, torch.float32, nchunks * hidden)
    for name, t in (("x", x), ("dy", dy), ("gamma", gamma), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    if dx is None:
        dx = torch.empty_like(x)
    if chunk_sums is None:
        chunk_sums = torch.empty(nchunks, hidden, dtype=torch.float32, device=x.device)
    need = rms_norm_bwd_blocked_workspace_size(rows, hidden, block_rows)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    for name, t in (("dx", dx), ("chunk_sums", chunk_sums), ("workspace", workspace)):
        _check_cuda(name, t, x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(x.device):
        st = lib.rms_norm_bwd_blocked(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx),
                                      _ptr(chunk_sums), rows, hidden, int(block_rows),
                                      int(offset), DTYPE_CODES[x.dtype], workspace.data_ptr(),
                                      ws_bytes, _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_bwd_blocked", st)
    return dx, chunk_sums


def rms_norm_dw_sum(chunk_sums: torch.Tensor, dw: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """dw [hidden] = the chunk sums [nchunks, hidden] added in chunk order."""
    lib = load_library()
    if chunk_sums.dim() != 2 or chunk_sums.dtype != torch.float32:
        raise RuntimeError("chunk_sums must be a float32 [nchunks, hidden] tensor")
    nchunks, hidden = chunk_sums.shape
    _check_like("dw", dw, torch.float32, hidden)
    _check_cuda("chunk_sums", chunk_sums)
    if dw is None:
        dw = torch.empty(hidden, dtype=torch.float32, device=chunk_sums.device)
    _check_cuda("dw", dw, chunk_sums.device)
    with torch.cuda.device(chunk_sums.device):
        st = lib.rms_norm_dw_sum(_ptr(chunk_sums), nchunks, hidden, _ptr(dw),
                                 _stream_handle(chunk_sums.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_dw_sum", st)
    return dw


def rms_norm_set_sm_budget(sms: int) -> None:
    """Let the persistent kernels use at most ``sms`` SMs' worth of
    resident CTAs (0: every SM); process-wide, read at each launch."""
    st = load_library().rms_norm_set_sm_budget(int(sms))
    if st != RMSN_OK:
        raise RMSNormError("rms_norm_set_sm_budget", st)


def rms_norm_sm_budget() -> int:
    return int(load_library().rms_norm_sm_budget())


def layer_norm_fwd(x: torch.Tensor, gamma: torch.Tensor, beta: Optional[torch.Tensor], eps: float,
                   y: Optional[torch.Tensor] = None, mean: Optional[torch.Tensor] = None,
                   rstd: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """LayerNorm forward over the last dimension; returns ``(y, mean, rstd)``
    (``beta`` may be None)."""
    lib = load_library()
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    rows, hidden = _as_rows(x)
    _check_like("gamma", gamma, x.dtype, hidden)
    _check_like("beta", beta, x.dtype, hidden)
    _check_like("y", y, x.dtype, x.numel(), x.shape)
    _check_like("mean", mean, torch.float32, rows)
    _check_like("rstd", rstd, torch.float32, rows)
    _check_cuda("x", x)
    _check_cuda("gamma", gamma, x.device)
    if beta is not None:
        _check_cuda("beta", beta, x.device)
    y = torch.empty_like(x) if y is None else y
    mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if mean is None else mean
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if rstd is None else rstd
    for name, t in (("y", y), ("mean", mean), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    with torch.cuda.device(x.device):
        st = lib.layer_norm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean), _ptr(rstd),
                                rows, hidden, float(eps), DTYPE_CODES[x.dtype],
                                _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("layer_norm_fwd", st)
    return y, mean, rstd


def layer_norm_bwd_workspace_size(rows: int, hidden: int, dtype) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().layer_norm_bwd_workspace_size(int(rows), int(hidden), code))


def layer_norm_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, mean: torch.Tensor,
                   rstd: torch.Tensor, dx: Optional[torch.Tensor] = None,
                   dgamma: Optional[torch.Tensor] = None, dbeta: Optional[torch.Tensor] = None,
                   with_dbeta: bool = True, workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """LayerNorm backward; returns ``(dx, dgamma, dbeta)`` (dbeta None when
    ``with_dbeta`` is False)."""
    lib = load_library()
    rows, hidden = _check_bwd_args(dy, x, gamma, rstd, dx, dgamma)
    _check_like("mean", mean, torch.float32, rows)
    _check_like("dbeta", dbeta if with_dbeta else None, torch.float32, hidden)
    for name, t in (("x", x), ("dy", dy), ("gamma", gamma), ("mean", mean), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    code = DTYPE_CODES[x.dtype]
    dx = torch.empty_like(x) if dx is None else dx
    dgamma = torch.empty(hidden, dtype=torch.float32, device=x.device) if dgamma is None else dgamma
    if with_dbeta and dbeta is None:
        dbeta = torch.empty(hidden, dtype=torch.float32, device=x.device)
    need = int(lib.layer_norm_bwd_workspace_size(rows, hidden, code))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    for name, t in (("dx", dx), ("dgamma", dgamma), ("workspace", workspace)):
        _check_cuda(name, t, x.device)
    if with_dbeta:
        _check_cuda("dbeta", dbeta, x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(x.device):
        st = lib.layer_norm_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dx),
                                _ptr(dgamma), _ptr(dbeta) if with_dbeta else None, rows, hidden,
                                code, workspace.data_ptr(), ws_bytes,
                                _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("layer_norm_bwd", st)
    return dx, dgamma, (dbeta if with_dbeta else None)


def softmax_fwd(x: torch.Tensor, y: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Softmax over the last dimension of ``x`` (fp32 arithmetic, one
    rounding to x's dtype at the store)."""
    lib = load_library()
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    rows, cols = _as_rows(x)
    _check_like("y", y, x.dtype, x.numel(), x.shape)
    _check_cuda("x", x)
    y = torch.empty_like(x) if y is None else y
    _check_cuda("y", y, x.device)
    with torch.cuda.device(x.device):
        st = lib.softmax_fwd(_ptr(x), _ptr(y), rows, cols, DTYPE_CODES[x.dtype],
                             _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("softmax_fwd", st)
    return y


def softmax_bwd(dy: torch.Tensor, y: torch.Tensor, dx: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Backward of softmax_fwd from its output: dx = y * (dy - sum(dy * y))
    per row, the sum in fp32."""
    lib = load_library()
    if y.dtype not in DTYPE_CODES:
        raise RuntimeError(f"y must be float32, bfloat16 or float16, not {y.dtype}")
    rows, cols = _as_rows(y)
    _check_like("dy", dy, y.dtype, y.numel(), y.shape)
    _check_like("dx", dx, y.dtype, y.numel(), y.shape)
    _check_cuda("y", y)
    _check_cuda("dy", dy, y.device)
    dx = torch.empty_like(y) if dx is None else dx
    _check_cuda("dx", dx, y.device)
    with torch.cuda.device(y.device):
        st = lib.softmax_bwd(_ptr(dy), _ptr(y), _ptr(dx), rows, cols, DTYPE_CODES[y.dtype],
                             _stream_handle(y.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("softmax_bwd", st)
    return dx


def _gn_shape(x: torch.Tensor, groups: int):
    if x.dim() < 2:
        raise RuntimeError("x must be [n, channels, *spatial]")
    n, c = x.shape[0], x.shape[1]
    spatial = 1
    for d in x.shape[2:]:
        spatial *= d
    if c % groups:
        raise RuntimeError("channels must be a multiple of groups")
    return n, c, spatial


def group_norm_fwd(x: torch.Tensor, gamma: torch.Tensor, beta: Optional[torch.Tensor],
                   groups: int, eps: float, y: Optional[torch.Tensor] = None,
                   mean: Optional[torch.Tensor] = None, rstd: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """GroupNorm forward over x [n, channels, *spatial]; returns ``(y, mean,
    rstd)`` with mean and rstd fp32 [n, groups] (``beta`` may be None)."""
    lib = load_library()
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    n, c, sp = _gn_shape(x, groups)
    _check_like("gamma", gamma, x.dtype, c)
    _check_like("beta", beta, x.dtype, c)
    _check_like("y", y, x.dtype, x.numel(), x.shape)
    _check_like("mean", mean, torch.float32, n * groups)
    _check_like("rstd", rstd, torch.float32, n * groups)
    _check_cuda("x", x)
    _check_cuda("gamma", gamma, x.device)
    if beta is not None:
        _check_cuda("beta", beta, x.device)
    y = torch.empty_like(x) if y is None else y
    mean = torch.empty(n, groups, dtype=torch.float32, device=x.device) if mean is None else mean
    rstd = torch.empty(n, groups, dtype=torch.float32, device=x.device) if rstd is None else rstd
    for name, t in (("y", y), ("mean", mean), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    with torch.cuda.device(x.device):
        st = lib.group_norm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean), _ptr(rstd),
                                n, c, sp, int(groups), float(eps), DTYPE_CODES[x.dtype],
                                _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("group_norm_fwd", st)
    return y, mean, rstd


def group_norm_bwd_workspace_size(n: int, channels: int, spatial: int, groups: int,
                                  dtype) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().group_norm_bwd_workspace_size(int(n), int(channels), int(spatial),
                                                            int(groups), code))


def group_norm_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, mean: torch.Tensor,
                   rstd: torch.Tensor, groups: int, dx: Optional[torch.Tensor] = None,
                   dgamma: Optional[torch.Tensor] = None, dbeta: Optional[torch.Tensor] = None,
                   with_dbeta: bool = True, workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """GroupNorm backward; returns ``(dx, dgamma, dbeta)`` (fp32 weight
    gradients; dbeta None when ``with_dbeta`` is False)."""
    lib = load_library()
    if x.dtype not in DTYPE_CODES:
        raise RuntimeError(f"x must be float32, bfloat16 or float16, not {x.dtype}")
    n, c, sp = _gn_shape(x, groups)
    _check_like("dy", dy, x.dtype, x.numel(), x.shape)
    _check_like("gamma", gamma, x.dtype, c)
    _check_like("mean", mean, torch.float32, n * groups)
    _check_like("rstd", rstd, torch.float32, n * groups)
    _check_like("dx", dx, x.dtype, x.numel(), x.shape)
    _check_like("dgamma", dgamma, torch.float32, c)
    _check_like("dbeta", dbeta if with_dbeta else None, torch.float32, c)
    for name, t in (("x", x), ("dy", dy), ("gamma", gamma), ("mean", mean), ("rstd", rstd)):
        _check_cuda(name, t, x.device)
    code = DTYPE_CODES[x.dtype]
    dx = torch.empty_like(x) if dx is None else dx
    dgamma = torch.empty(c, dtype=torch.float32, device=x.device) if dgamma is None else dgamma
    if with_dbeta and dbeta is None:
        dbeta = torch.empty(c, dtype=torch.float32, device=x.device)
    need = int(lib.group_norm_bwd_workspace_size(n, c, sp, int(groups), code))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    for name, t in (("dx", dx), ("dgamma", dgamma), ("workspace", workspace)):
        _check_cuda(name, t, x.device)
    if with_dbeta:
        _check_cuda("dbeta", dbeta, x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(x.device):
        st = lib.group_norm_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dx),
                                _ptr(dgamma), _ptr(dbeta) if with_dbeta else None, n, c, sp,
                                int(groups), code, workspace.data_ptr(), ws_bytes,
                                _stream_handle(x.device, stream))
    if st != RMSN_OK:
        raise RMSNormError("group_norm_bwd", st)
    return dx, dgamma, (dbeta if with_dbeta else None)


class RMSNormFunction(torch.autograd.Function):
    """RMSNorm over the last dimension with this library's forward and
    backward.  The backward's weight gradient, summed in fp32 by the library,
    is cast to the weight's dtype (autograd wants the parameter's dtype)."""

    @staticmethod
    def forward(ctx, x, weight, eps, offset, cast_mode):
        x = x.contiguous()
        weight = weight.contiguous()
        y, rstd = rms_norm_fwd(x, weight, eps, offset, cast_mode)
        ctx.save_for_backward(x, weight, rstd)
        ctx.offset = offset
        return y

    @staticmethod
    def backward(ctx, dy):
        x, weight, rstd = ctx.saved_tensors
        dx, dw = rms_norm_bwd(dy.contiguous(), x, weight, rstd, ctx.offset)
        return dx, dw.to(weight.dtype), None, None, None


def rms_norm(x: torch.Tensor, weight: torch.Tensor, eps: float, offset: int = 0,
             cast_mode: str = "round_once") -> torch.Tensor:
    """Differentiable RMSNorm of ``x`` over its last dimension (gain
    ``weight``, or ``1 + weight`` with ``offset=1``)."""
    return RMSNormFunction.apply(x, weight, eps, offset, cast_mode)


class RMSNorm(torch.nn.Module):
    """RMSNorm layer over the last dimension of its input.  The weight starts
    at 1 (gain ``weight``) or at 0 with ``offset=1`` (gain ``1 + weight``)."""

    def __init__(self, hidden: int, eps: float = 1e-6, offset: int = 0,
                 cast_mode: str = "round_once", device=None, dtype=None):
        super().__init__()
        if offset not in (0, 1):
            raise ValueError("offset must be 0 or 1")
        if cast_mode not in CAST_MODES:
            raise ValueError(f"cast_mode must be one of {sorted(CAST_MODES)}")
        self.weight = torch.nn.Parameter(
            torch.full((hidden,), 0.0 if offset else 1.0, device=device, dtype=dtype))
        self.eps, self.offset, self.cast_mode = eps, offset, cast_mode

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return rms_norm(x, self.weight, self.eps, self.offset, self.cast_mode)

    def extra_repr(self) -> str:
        return (f"{self.weight.numel()}, eps={self.eps}, offset={self.offset}, "
                f"cast_mode={self.cast_mode!r}")

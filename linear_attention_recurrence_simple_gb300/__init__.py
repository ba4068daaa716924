"""GB300 (sm_103a) Simple GLA mixer: a thin binding over the C ABI of ``libgla.so``.

The functions keep the C names (``include/gla.h``) and only marshal arguments: they check
torch tensors, allocate outputs with torch, and pass raw device pointers and the current CUDA
stream to the library.  Every step of the computation runs in the library's CUDA kernels; there
is no other code path, and a missing library raises instead of falling back.

Layouts (see ``include/gla.h``): q, k ``[B, T, H, 96]``; v ``[B, T, H, 192]``; packed inputs
``[T_total, H, d]`` (or ``[1, T_total, H, d]``) with ``cu_seqlens``; states ``[B, H, 96, 192]`` fp32.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

__all__ = [
    "GlaError", "load_library", "library_path", "gla_workspace_bytes", "gla_bwd_workspace_bytes",
    "gla_chunk_fwd",
    "gla_chunk_bwd", "gla_decode_step", "gla_chunk_fwd_noalloc", "gla_head_norm_gate", "gla_chunk_fwd_split",
    "gla_split_choose_seg_chunks", "gla_get_device_error",
    "gla_set_wait_limit_ns", "gla_debug_bounds", "debug_bounds_library", "gla_chunk_fwd_host",
    "gla_chunk_fwd_host_workspace_bytes",
    "gla_status_string", "DK", "DV", "CHUNK", "EXPORTS",
]

DK, DV, CHUNK = 96, 192, 128
GLA_BF16, GLA_F32 = 0, 1
EXPORTS = ("gla_workspace_bytes", "gla_bwd_workspace_bytes", "gla_chunk_fwd", "gla_chunk_bwd",
           "gla_decode_step", "gla_chunk_fwd_aug", "gla_decode_step_aug", "gla_head_norm_gate",
           "gla_decode_step_bf16_state", "gla_split_workspace_bytes", "gla_chunk_fwd_split",
           "gla_decode_step_norm_gate", "gla_decode_step_mxfp8_state", "gla_state_to_mxfp8",
           "gla_state_from_mxfp8",
           "gla_split_choose_seg_chunks", "gla_chunk_fwd_noalloc", "gla_get_device_error", "gla_set_wait_limit_ns",
           "gla_debug_bounds", "gla_chunk_fwd_host", "gla_chunk_fwd_host_workspace_bytes", "gla_status_string")
NOALLOC_MAX_SEQS = 16384

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgla.so")
_LIB_DEBUG_PATH = os.path.join(_PKG, "libgla_debug.so")  # the debug-bounds build
_lock = threading.Lock()
_libs = {}          # False: release build, True: debug-bounds build
_use_debug = False  # which one the calls go to (see debug_bounds_library)


class GlaError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {gla_status_string(status)} ({status})" if where else
                         f"{gla_status_string(status)} ({status})")


def library_path(debug: bool = False) -> str:
    return _LIB_DEBUG_PATH if debug else _LIB_PATH


def load_library(build: bool = True, debug: bool | None = None):
    """Loads libgla.so, or with ``debug`` (default: inside :func:`debug_bounds_library`) its
    debug-bounds build libgla_debug.so, building it first if missing and ``build``; raises if it
    cannot."""
    if debug is None:
        debug = _use_debug
    with _lock:
        if debug in _libs:
            return _libs[debug]
        path = library_path(debug)
        if build:
            from . import _build
            _build.build(debug=debug)
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} is missing ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P, I, F, Z, U = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                         ctypes.c_ulonglong)
        lib.gla_workspace_bytes.argtypes = [I, I]
        lib.gla_workspace_bytes.restype = Z
        lib.gla_bwd_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.gla_bwd_workspace_bytes.restype = Z
        lib.gla_chunk_fwd.argtypes = [P, P, P, P, P, F, P, P, P, I, I, I, I, I, I, P, Z, P]
        lib.gla_chunk_fwd.restype = I
        lib.gla_chunk_bwd.argtypes = [P, P, P, P, P, F, P, P, P, P, P, P, P, I, I, I, I, I, I, P, Z, P]
        lib.gla_chunk_bwd.restype = I
        lib.gla_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, F, P, P, P, I, I, I, I, I, I, P]
        lib.gla_chunk_fwd_noalloc.restype = I
        lib.gla_decode_step.argtypes = [P, P, P, P, F, P, P, I, P, I, I, I, I, I, P]
        lib.gla_decode_step.restype = I
        lib.gla_chunk_fwd_aug.argtypes = [P, P, P, P, P, F, P, P, P, P, I, I, I, I, I, I, P, Z, P]
        lib.gla_chunk_fwd_aug.restype = I
        lib.gla_decode_step_aug.argtypes = [P, P, P, P, F, P, P, P, I, P, I, I, I, I, I, P]
        lib.gla_decode_step_aug.restype = I
        lib.gla_head_norm_gate.argtypes = [P, P, P, P, I, F, P, ctypes.c_longlong, I, I, I, P]
        lib.gla_decode_step_bf16_state.argtypes = [P, P, P, P, F, P, P, P, I, P, I, I, I, I, I, P]
        lib.gla_decode_step_bf16_state.restype = I
        lib.gla_decode_step_norm_gate.argtypes = [P, P, P, P, F, P, P, P, I, P, P, P, I, F, P, I, I, I, I, I, P]
        lib.gla_decode_step_norm_gate.restype = I
        lib.gla_decode_step_mxfp8_state.argtypes = [P, P, P, P, F, P, P, P, P, I, P, I, I, I, I, I, P]
        lib.gla_decode_step_mxfp8_state.restype = I
        lib.gla_state_to_mxfp8.argtypes = [P, P, P, ctypes.c_longlong, P]
        lib.gla_state_to_mxfp8.restype = I
        lib.gla_state_from_mxfp8.argtypes = [P, P, P, ctypes.c_longlong, P]
        lib.gla_state_from_mxfp8.restype = I
        lib.gla_split_workspace_bytes.argtypes = [P, I, I, I]
        lib.gla_split_workspace_bytes.restype = Z
        lib.gla_chunk_fwd_split.argtypes = [P, P, P, P, P, F, P, P, P, P, I, I, I, I, I, I, I, P, Z, P]
        lib.gla_chunk_fwd_split.restype = I
        lib.gla_split_choose_seg_chunks.argtypes = [P, I, I]
        lib.gla_split_choose_seg_chunks.restype = I
        lib.gla_head_norm_gate.restype = I
        lib.gla_get_device_error.argtypes = [P]
        lib.gla_get_device_error.restype = I
        lib.gla_set_wait_limit_ns.argtypes = [U]
        lib.gla_set_wait_limit_ns.restype = I
        lib.gla_status_string.argtypes = [I]
        lib.gla_status_string.restype = ctypes.c_char_p
        lib.gla_debug_bounds.argtypes = []
        lib.gla_debug_bounds.restype = I
        lib.gla_chunk_fwd_host_workspace_bytes.argtypes = [I, I, I, I]
        lib.gla_chunk_fwd_host_workspace_bytes.restype = Z
        lib.gla_chunk_fwd_host.argtypes = [P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, P, Z, P]
        lib.gla_chunk_fwd_host.restype = I
        _libs[debug] = lib
        return lib


@contextlib.contextmanager
def debug_bounds_library():
    """Within the block every call goes to the debug-bounds build (libgla_debug.so: device index
    checks that record GLA_ERR_BOUNDS and skip the access).  Not for concurrent use from several
    threads.  Each build keeps its own device error word."""
    global _use_debug
    lib = load_library(debug=True)
    prev, _use_debug = _use_debug, True
    try:
        yield lib
    finally:
        _use_debug = prev


def gla_debug_bounds() -> int:
    """1 when calls go to the debug-bounds build, 0 for the release build."""
    return int(load_library().gla_debug_bounds())


def gla_status_string(status: int) -> str:
    return load_library().gla_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise GlaError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GLA_BF16
    if t.dtype == torch.float32:
        return GLA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _need(t: torch.Tensor, name: str, dtype=None, device=None, numel=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def _layout(q, k, v, cu_seqlens):
    """Returns (n_seq, T, H, packed_shape_prefix) for fixed-length or packed inputs."""
    if cu_seqlens is None:
        if q.dim() != 4:
            raise ValueError("without cu_seqlens, q must be [B, T, H, 96]")
        B, T, H, dk = q.shape
        n_seq = B
    else:
        if q.dim() == 4:
            if q.shape[0] != 1:
                raise ValueError("packed inputs must be [T_total, H, d] or [1, T_total, H, d]")
            T, H, dk = q.shape[1:]
        elif q.dim() == 3:
            T, H, dk = q.shape
        else:
            raise ValueError("packed q must be [T_total, H, 96]")
        n_seq = cu_seqlens.numel() - 1
    if dk != DK or k.shape != q.shape or v.shape[:-1] != q.shape[:-1] or v.shape[-1] != DV:
        raise ValueError("expected q, k [..., H, 96] and v [..., H, 192] with matching leading dims")
    return n_seq, T, H


def gla_workspace_bytes(n_seq: int, H: int) -> int:
    return int(load_library().gla_workspace_bytes(int(n_seq), int(H)))


def gla_bwd_workspace_bytes(n_seq: int, T: int, H: int, packed: bool, dtype_code: int) -> int:
    return int(load_library().gla_bwd_workspace_bytes(int(n_seq), int(T), int(H), int(bool(packed)),
                                                      int(dtype_code)))


def _workspace(cu_seqlens, n_seq, H, device, workspace):
    if cu_seqlens is None:
        return None, 0
    need = gla_workspace_bytes(n_seq, H)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def gla_chunk_fwd(q, k, v, log_lambda, scale=None, h0=None, cu_seqlens=None,
                  output_final_state: bool = True, o=None, hT=None, workspace=None, aug=None):
    """Chunked forward.  Returns ``(o, hT)`` (``hT`` is None if not requested).

    ``aug`` (aug_balance, fp32 ``[H, 96]``) adds the self-augmentation copy
    ``sigmoid(q_t . (aug[h] * k_t)) v_t`` to each output row (``gla_chunk_fwd_aug``)."""
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_seq, T, H = _layout(q, k, v, cu_seqlens)
    if log_lambda.numel() != H:
        raise ValueError("log_lambda must have H entries")
    if h0 is not None:
        _need(h0, "h0", torch.float32, dev)
        if h0.shape != (n_seq, H, DK, DV):
            raise ValueError("h0 must be [n_seq, H, 96, 192]")
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "o", v.dtype, dev, v.numel())
    if output_final_state and hT is None:
        hT = torch.empty((n_seq, H, DK, DV), dtype=torch.float32, device=dev)
    if hT is not None:
        _need(hT, "hT", torch.float32, dev, n_seq * H * DK * DV)
    ws, ws_bytes = _workspace(cu_seqlens, n_seq, H, dev, workspace)
    s = float(DK ** -0.5) if scale is None else float(scale)
    if aug is not None:
        _need(aug, "aug", torch.float32, dev)
        if aug.shape != (H, DK):
            raise ValueError("aug must be [H, 96]")
    with torch.cuda.device(dev):
        if aug is None:
            rc = lib.gla_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), s, _ptr(o),
                                   _ptr(hT), _ptr(cu_seqlens), n_seq, T, H, DK, DV, dt, _ptr(ws),
                                   ws_bytes, _stream(dev))
        else:
            rc = lib.gla_chunk_fwd_aug(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), s,
                                       _ptr(aug), _ptr(o), _ptr(hT), _ptr(cu_seqlens), n_seq, T, H, DK,
                                       DV, dt, _ptr(ws), ws_bytes, _stream(dev))
    _check(rc, "gla_chunk_fwd" if aug is None else "gla_chunk_fwd_aug")
    return o, hT


def gla_chunk_fwd_noalloc(q, k, v, log_lambda, scale=None, h0=None, cu_seqlens=None, o=None, hT=None):
    """The forward with no device allocation inside the library and no workspace argument.

    For callers that cannot allocate device memory per call (for instance a serving engine that
    hands all device memory to its own pool at start-up): pass preallocated ``o`` and ``hT`` and
    nothing is allocated here either.  The packed schedule lives in a 64 KB library-owned device
    array, so ``cu_seqlens`` may describe at most ``NOALLOC_MAX_SEQS`` sequences, and calls that
    overlap on the GPU (unordered streams) race on it.  Returns ``(o, hT)``."""
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_seq, T, H = _layout(q, k, v, cu_seqlens)
    if h0 is not None:
        _need(h0, "h0", torch.float32, dev, n_seq * H * DK * DV)
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "o", v.dtype, dev, v.numel())
    if hT is not None:
        _need(hT, "hT", torch.float32, dev, n_seq * H * DK * DV)
    s = float(DK ** -0.5) if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = lib.gla_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), s,
                                       _ptr(o), _ptr(hT), _ptr(cu_seqlens), n_seq, T, H, DK, DV, dt,
                                       _stream(dev))
    _check(rc, "gla_chunk_fwd_noalloc")
    return o, hT


def gla_chunk_fwd_host_workspace_bytes(n_seq: int, T: int, H: int, dtype_code: int) -> int:
    return int(load_library().gla_chunk_fwd_host_workspace_bytes(n_seq, T, H, dtype_code))


def gla_chunk_fwd_host(q, k, v, log_lambda, scale=None, h0=None, o=None, hT=None, pieces=16, workspace=None,
                       output_final_state: bool = True):
    """The forward on HOST tensors (``gla_chunk_fwd_host``): q, k ``[B, T, H, 96]``, v
    ``[B, T, H, 192]`` and h0 (fp32, optional) on the CPU (page-locked for overlapped copies);
    log_lambda on the device.  Returns host ``(o, hT)``, written once the current stream has run
    (synchronise it before reading).  The library copies ``pieces`` pieces in, runs them and
    copies them out, pipelined; ``workspace`` is a device buffer of at least
    :func:`gla_chunk_fwd_host_workspace_bytes` bytes (allocated when not given)."""
    lib = load_library()
    dev = log_lambda.device
    if dev.type != "cuda":
        raise ValueError("log_lambda must be on the device")
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.device.type != "cpu" or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor of q's dtype")
    if q.dim() != 4 or q.shape[3] != DK or k.shape != q.shape or v.shape != (*q.shape[:3], DV):
        raise ValueError("expected q, k [B, T, H, 96] and v [B, T, H, 192]")
    B, T, H = q.shape[:3]
    _need(log_lambda, "log_lambda", torch.float32, dev, H)
    if h0 is not None and (h0.device.type != "cpu" or h0.dtype != torch.float32 or not h0.is_contiguous()
                           or h0.shape != (B, H, DK, DV)):
        raise ValueError("h0 must be a contiguous CPU fp32 tensor [B, H, 96, 192]")
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype).pin_memory()
    if hT is None and output_final_state:
        hT = torch.empty((B, H, DK, DV), dtype=torch.float32).pin_memory()
    for name, t, shape, dtype in (("o", o, v.shape, v.dtype), ("hT", hT, (B, H, DK, DV), torch.float32)):
        if t is not None and (t.device.type != "cpu" or t.dtype != dtype or t.shape != shape or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor {tuple(shape)} of {dtype}")
    need = gla_chunk_fwd_host_workspace_bytes(B, T, H, dt)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if workspace.numel() < need:
        raise ValueError(f"workspace has {workspace.numel()} bytes, needs {need}")
    s = float(DK ** -0.5) if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = lib.gla_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), s, _ptr(o), _ptr(hT),
                                    B, T, H, DK, DV, dt, int(pieces), _ptr(workspace), workspace.numel(),
                                    _stream(dev))
    _check(rc, "gla_chunk_fwd_host")
    return o, hT


def gla_chunk_bwd(q, k, v, log_lambda, dO, scale=None, h0=None, dhT=None, cu_seqlens=None,
                  need_dh0: bool = True, workspace=None, dq=None, dk=None, dv=None, dh0=None):
    """Chunked backward.  Returns ``(dq, dk, dv, dh0)`` (``dh0`` None if not requested).
    ``dq``, ``dk``, ``dv``, ``dh0``: optional preallocated outputs (contiguous, sized like q, k, v
    and [n_seq, H, 96, 192] fp32)."""
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    n_seq, T, H = _layout(q, k, v, cu_seqlens)
    if dO.shape != v.shape:
        raise ValueError("dO must have the shape of v")
    for name, t in (("h0", h0), ("dhT", dhT)):
        if t is not None:
            _need(t, name, torch.float32, dev)
            if t.shape != (n_seq, H, DK, DV):
                raise ValueError(f"{name} must be [n_seq, H, 96, 192]")
    dq = torch.empty(q.shape, dtype=q.dtype, device=dev) if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype, device=dev) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, device=dev) if dv is None else dv
    if dh0 is None and need_dh0:
        dh0 = torch.empty((n_seq, H, DK, DV), dtype=torch.float32, device=dev)
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _need(t, name, q.dtype, dev, ref.numel())
    if dh0 is not None:
        _need(dh0, "dh0", torch.float32, dev, n_seq * H * DK * DV)
    need = gla_bwd_workspace_bytes(n_seq, T, H, cu_seqlens is not None, dt)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = float(DK ** -0.5) if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = lib.gla_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), s, _ptr(dO),
                               _ptr(dhT), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dh0), _ptr(cu_seqlens),
                               n_seq, T, H, DK, DV, dt, _ptr(workspace), ws_bytes, _stream(dev))
    _check(rc, "gla_chunk_bwd")
    return dq, dk, dv, dh0


def gla_decode_step(q, k, v, log_lambda, state, scale=None, slot=None, o=None, aug=None):
    """One decode step on the state pool ``state [P, H, 96, 192]`` (updated in place).

    q, k ``[N, H, 96]``; v ``[N, H, 192]``; ``slot`` ``[N]`` int32 pool rows or None (row n).
    ``aug`` (fp32 ``[H, 96]``) adds the self-augmentation copy of v (``gla_decode_step_aug``).
    A bf16 ``state`` pool runs ``gla_decode_step_bf16_state`` (the state is rounded to bf16 when
    it is written back).  Returns ``o [N, H, 192]``."""
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    if state.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("state must be float32 or bfloat16")
    _need(state, "state", state.dtype, dev)
    if q.dim() != 3 or q.shape[2] != DK or k.shape != q.shape or v.shape != (*q.shape[:2], DV):
        raise ValueError("expected q, k [N, H, 96] and v [N, H, 192]")
    N, H = q.shape[:2]
    if state.dim() != 4 or state.shape[1:] != (H, DK, DV):
        raise ValueError("state must be [P, H, 96, 192]")
    if slot is not None:
        _need(slot, "slot", torch.int32, dev)
        if slot.shape != (N,):
            raise ValueError("slot must be [N]")
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "o", v.dtype, dev, v.numel())
    s = float(DK ** -0.5) if scale is None else float(scale)
    if aug is not None:
        _need(aug, "aug", torch.float32, dev)
        if aug.shape != (H, DK):
            raise ValueError("aug must be [H, 96]")
    with torch.cuda.device(dev):
        if state.dtype == torch.bfloat16:
            rc = lib.gla_decode_step_bf16_state(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), s, _ptr(aug),
                                                _ptr(state), _ptr(slot), state.shape[0], _ptr(o), N, H, DK,
                                                DV, dt, _stream(dev))
            _check(rc, "gla_decode_step_bf16_state")
            return o
        if aug is None:
            rc = lib.gla_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), s, _ptr(state),
                                     _ptr(slot), state.shape[0], _ptr(o), N, H, DK, DV, dt, _stream(dev))
        else:
            rc = lib.gla_decode_step_aug(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), s, _ptr(aug),
                                         _ptr(state), _ptr(slot), state.shape[0], _ptr(o), N, H, DK, DV,
                                         dt, _stream(dev))
    _check(rc, "gla_decode_step" if aug is None else "gla_decode_step_aug")
    return o


def gla_decode_step_norm_gate(q, k, v, log_lambda, state, g, weight, tier, scale=None, slot=None,
                              eps=1e-6, y=None, aug=None):
    """One decode step (fp32 state pool, updated in place) whose readout goes straight through the
    per-tier Head RMSNorm and the SiLU(g) gate: returns ``y [N, H, 192]``,
    ``y = o / sqrt(mean(o^2) + eps) * weight[tier[h]] * SiLU(g)`` with o the step's readout (plus
    the self-augmentation copy when ``aug`` is given).  ``g`` ``[N, H, 192]`` (dtype of q),
    ``weight`` fp32 ``[n_tiers, 192]``, ``tier`` int32 ``[H]``."""
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    _need(state, "state", torch.float32, dev)
    if q.dim() != 3 or q.shape[2] != DK or k.shape != q.shape or v.shape != (*q.shape[:2], DV):
        raise ValueError("expected q, k [N, H, 96] and v [N, H, 192]")
    N, H = q.shape[:2]
    if state.dim() != 4 or state.shape[1:] != (H, DK, DV):
        raise ValueError("state must be [P, H, 96, 192]")
    _need(g, "g", q.dtype, dev, v.numel())
    _need(weight, "weight", torch.float32, dev)
    _need(tier, "tier", torch.int32, dev, H)
    if weight.dim() != 2 or weight.shape[1] != DV:
        raise ValueError("weight must be [n_tiers, 192]")
    if slot is not None:
        _need(slot, "slot", torch.int32, dev, N)
    if aug is not None:
        _need(aug, "aug", torch.float32, dev, H * DK)
    if y is None:
        y = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(y, "y", v.dtype, dev, v.numel())
    s = float(DK ** -0.5) if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = lib.gla_decode_step_norm_gate(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), s, _ptr(aug),
                                           _ptr(state), _ptr(slot), state.shape[0], _ptr(g), _ptr(weight),
                                           _ptr(tier), weight.shape[0], float(eps), _ptr(y), N, H, DK, DV,
                                           dt, _stream(dev))
    _check(rc, "gla_decode_step_norm_gate")
    return y


def gla_state_to_mxfp8(x, codes=None, scales=None):
    """fp32 state rows ``x [..., 192]`` to MXFP8: returns ``(codes uint8 [..., 192],
    scales uint8 [..., 6])`` (the format of :func:`gla_decode_step_mxfp8_state`)."""
    lib = load_library()
    dev = x.device
    _need(x, "x", torch.float32, dev)
    if x.shape[-1] != DV:
        raise ValueError("x must be [..., 192]")
    rows = x.numel() // DV
    codes = torch.empty(x.shape, dtype=torch.uint8, device=dev) if codes is None else codes
    scales = torch.empty(x.shape[:-1] + (DV // 32,), dtype=torch.uint8, device=dev) if scales is None else scales
    _need(codes, "codes", torch.uint8, dev, x.numel())
    _need(scales, "scales", torch.uint8, dev, rows * (DV // 32))
    with torch.cuda.device(dev):
        rc = lib.gla_state_to_mxfp8(_ptr(x), _ptr(codes), _ptr(scales), rows, _stream(dev))
    _check(rc, "gla_state_to_mxfp8")
    return codes, scales


def gla_state_from_mxfp8(codes, scales, x=None):
    """MXFP8 state rows back to fp32 (exact); returns ``x [..., 192]``."""
    lib = load_library()
    dev = codes.device
    _need(codes, "codes", torch.uint8, dev)
    if codes.shape[-1] != DV:
        raise ValueError("codes must be [..., 192]")
    rows = codes.numel() // DV
    _need(scales, "scales", torch.uint8, dev, rows * (DV // 32))
    x = torch.empty(codes.shape, dtype=torch.float32, device=dev) if x is None else x
    _need(x, "x", torch.float32, dev, codes.numel())
    with torch.cuda.device(dev):
        rc = lib.gla_state_from_mxfp8(_ptr(codes), _ptr(scales), _ptr(x), rows, _stream(dev))
    _check(rc, "gla_state_from_mxfp8")
    return x


def gla_decode_step_mxfp8_state(q, k, v, log_lambda, codes, scales, scale=None, slot=None, o=None, aug=None):
    """One decode step on an MXFP8 state pool (``codes`` uint8 ``[P, H, 96, 192]``, ``scales``
    uint8 ``[P, H, 96, 6]``, both updated in place).  Returns ``o [N, H, 192]``."""
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    if q.dim() != 3 or q.shape[2] != DK or k.shape != q.shape or v.shape != (*q.shape[:2], DV):
        raise ValueError("expected q, k [N, H, 96] and v [N, H, 192]")
    N, H = q.shape[:2]
    _need(codes, "codes", torch.uint8, dev)
    if codes.dim() != 4 or codes.shape[1:] != (H, DK, DV):
        raise ValueError("codes must be [P, H, 96, 192]")
    _need(scales, "scales", torch.uint8, dev, codes.shape[0] * H * DK * (DV // 32))
    if slot is not None:
        _need(slot, "slot", torch.int32, dev, N)
    if aug is not None:
        _need(aug, "aug", torch.float32, dev, H * DK)
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "o", v.dtype, dev, v.numel())
    s = float(DK ** -0.5) if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = lib.gla_decode_step_mxfp8_state(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), s, _ptr(aug),
                                             _ptr(codes), _ptr(scales), _ptr(slot), codes.shape[0], _ptr(o), N,
                                             H, DK, DV, dt, _stream(dev))
    _check(rc, "gla_decode_step_mxfp8_state")
    return o


def _host_offsets(lengths):
    import numpy as np
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return cu


def gla_split_choose_seg_chunks(lengths, H):
    """Chunks per segment that ``gla_chunk_fwd_split(..., seg_chunks=0)`` uses for these sequence
    lengths and H heads; 0 when every sequence stays one segment (the plain forward)."""
    cu = _host_offsets(lengths)
    rc = load_library().gla_split_choose_seg_chunks(cu.ctypes.data_as(ctypes.c_void_p), len(lengths), int(H))
    if rc < 0:
        _check(rc, "gla_split_choose_seg_chunks")
    return rc


def gla_chunk_fwd_split(q, k, v, log_lambda, lengths, seg_chunks=0, scale=None, h0=None, aug=None,
                        output_final_state: bool = True, o=None, hT=None, workspace=None):
    """Sequence-split forward (``gla_chunk_fwd_split``) for long sequences.

    ``lengths``: the sequences' token counts (host ints); q, k ``[T_total, H, 96]``, v
    ``[T_total, H, 192]`` packed in that order (a fixed-length batch may pass ``[B, T, H, d]``
    tensors with ``lengths = [T] * B``).  Segments hold at most ``seg_chunks`` chunks of 128
    tokens; 0 lets the library choose (:func:`gla_split_choose_seg_chunks`), which may keep every
    sequence whole.  Returns ``(o, hT)`` like :func:`gla_chunk_fwd`."""
    import numpy as np
    lib = load_library()
    dev = q.device
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, q.dtype, dev)
    _need(log_lambda, "log_lambda", torch.float32, dev)
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, np.int64))
    n_seq, H = len(lengths), q.shape[-2]
    T = int(cu[-1])
    if q.numel() != T * H * DK or k.shape != q.shape or v.numel() != T * H * DV or q.shape[-1] != DK:
        raise ValueError("q, k, v must hold sum(lengths) tokens of H heads")
    if log_lambda.numel() != H:
        raise ValueError("log_lambda must have H entries")
    if h0 is not None:
        _need(h0, "h0", torch.float32, dev, n_seq * H * DK * DV)
        if h0.shape != (n_seq, H, DK, DV):
            raise ValueError("h0 must be [n_seq, H, 96, 192]")
    if aug is not None:
        _need(aug, "aug", torch.float32, dev)
        if aug.shape != (H, DK):
            raise ValueError("aug must be [H, 96]")
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "o", v.dtype, dev, v.numel())
    if output_final_state and hT is None:
        hT = torch.empty((n_seq, H, DK, DV), dtype=torch.float32, device=dev)
    if hT is not None:
        _need(hT, "hT", torch.float32, dev, n_seq * H * DK * DV)
    cu_p = cu.ctypes.data_as(ctypes.c_void_p)
    need = lib.gla_split_workspace_bytes(cu_p, n_seq, H, int(seg_chunks))
    if need == 0 and n_seq > 0:
        raise ValueError("bad lengths or seg_chunks")
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    s = float(DK ** -0.5) if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = lib.gla_chunk_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), s, _ptr(aug),
                                     _ptr(o), _ptr(hT), cu_p, n_seq, T, H, DK, DV, dt, int(seg_chunks),
                                     _ptr(workspace), workspace.numel(), _stream(dev))
    _check(rc, "gla_chunk_fwd_split")
    return o, hT


def gla_head_norm_gate(o, g, weight, tier, eps=1e-6, y=None):
    """Per-tier Head RMSNorm of each head's output row and the SiLU(g) gate.

    o, g ``[..., H, 192]`` (same dtype, bf16 or fp32); weight fp32 ``[n_tiers, 192]``; tier int32
    ``[H]``.  Returns ``y`` like ``o``."""
    lib = load_library()
    dev = o.device
    dt = _dtype_code(o)
    _need(o, "o", o.dtype, dev)
    _need(g, "g", o.dtype, dev)
    _need(weight, "weight", torch.float32, dev)
    _need(tier, "tier", torch.int32, dev)
    if o.dim() < 2 or o.shape[-1] != DV or g.shape != o.shape:
        raise ValueError("expected o, g [..., H, 192] of one shape")
    H = o.shape[-2]
    rows = o.numel() // (H * DV)
    if weight.dim() != 2 or weight.shape[1] != DV or tier.shape != (H,):
        raise ValueError("weight must be [n_tiers, 192] and tier [H]")
    if y is None:
        y = torch.empty_like(o)
    _need(y, "y", o.dtype, dev)
    with torch.cuda.device(dev):
        rc = lib.gla_head_norm_gate(_ptr(o), _ptr(g), _ptr(weight), _ptr(tier), weight.shape[0], float(eps),
                                    _ptr(y), rows, H, DV, dt, _stream(dev))
    _check(rc, "gla_head_norm_gate")
    return y


def gla_get_device_error(device=None) -> int:
    """Synchronises the current stream; returns and clears the device's sticky error status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(load_library().gla_get_device_error(_stream(dev)))


def gla_set_wait_limit_ns(ns: int) -> None:
    _check(load_library().gla_set_wait_limit_ns(int(ns)), "gla_set_wait_limit_ns")

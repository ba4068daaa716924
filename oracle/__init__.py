"""fp64 CPU oracle of the Simple GLA mixer.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use this
package.  The GPU library never imports, links or calls it, and it never calls the GPU library.
The arithmetic lives in ``gla_oracle.cpp`` (plain per-token loops in double precision); this
module compiles it with g++ and marshals numpy arrays through ctypes.

Every entry returns fp64 arrays.  Inputs are converted to fp32 first: bf16 workloads pass their
bf16-rounded values, which fp32 holds exactly.  Layouts: q, k ``[T, H, dk]``; v, dO ``[T, H, dv]``
(token-major, packed over sequences by ``cu_seqlens``); states ``[n_seq, H, dk, dv]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (g++, -O2, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_fwd.argtypes = [P, P, P, P, P, D, P, I, I, I, I, P, P, I]
    lib.oracle_fwd_chunked.argtypes = [P, P, P, P, P, D, P, I, I, I, I, I, P, P, I]
    lib.oracle_decode_step.argtypes = [P, P, P, P, D, P, P, I, I, I, I, I]
    lib.oracle_bwd.argtypes = [P, P, P, P, P, D, P, P, P, I, I, I, I, P, P, P, P, I]
    lib.oracle_self_aug.argtypes = [P, P, P, P, ctypes.c_longlong, I, I, I, P]
    lib.oracle_head_norm_gate.argtypes = [P, P, P, P, I, D, ctypes.c_longlong, I, I, P]
    lib.oracle_decode_step_bf16_state.argtypes = [P, P, P, P, D, P, P, I, I, I, I]
    lib.oracle_round_to_bf16.argtypes = [P, P, ctypes.c_longlong]
    lib.oracle_mxfp8_quantize.argtypes = [P, ctypes.c_longlong, I, P, P]
    lib.oracle_mxfp8_dequantize.argtypes = [P, P, ctypes.c_longlong, I, P]
    lib.oracle_decode_step_mxfp8_state.argtypes = [P, P, P, P, D, P, P, P, I, I, I, I, P]
    lib.oracle_hardware_threads.argtypes = []
    for f in (lib.oracle_fwd, lib.oracle_fwd_chunked, lib.oracle_decode_step, lib.oracle_bwd,
              lib.oracle_self_aug, lib.oracle_head_norm_gate, lib.oracle_decode_step_bf16_state,
              lib.oracle_round_to_bf16, lib.oracle_mxfp8_quantize, lib.oracle_mxfp8_dequantize,
              lib.oracle_decode_step_mxfp8_state, lib.oracle_hardware_threads):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def _f32(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cu(cu_seqlens, T_total):
    if cu_seqlens is None:
        cu = np.array([0, T_total], np.int32)
    else:
        cu = np.ascontiguousarray(cu_seqlens, np.int32)
    if cu[-1] != T_total:
        raise ValueError("cu_seqlens[-1] must equal the packed token count")
    return cu


def _shapes(q, k, v):
    if q.ndim != 3 or k.shape != q.shape or v.ndim != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [T, H, dk] and v [T, H, dv]")
    return q.shape[0], q.shape[1], q.shape[2], v.shape[2]


def fwd(q, k, v, log_lambda, scale, h0=None, cu_seqlens=None, nthreads=0, _lib_override=None):
    """Per-token recurrence.  Returns ``(o [T, H, dv], hT [n_seq, H, dk, dv])`` in fp64."""
    q, k, v, ll, h0 = _f32(q), _f32(k), _f32(v), _f32(log_lambda), _f32(h0)
    T, H, dk, dv = _shapes(q, k, v)
    cu = _cu(cu_seqlens, T)
    n = len(cu) - 1
    if h0 is not None and h0.shape != (n, H, dk, dv):
        raise ValueError("h0 must be [n_seq, H, dk, dv]")
    o = np.zeros((T, H, dv), np.float64)
    hT = np.zeros((n, H, dk, dv), np.float64)
    rc = (_lib_override or _load()).oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), _ptr(h0), float(scale), _ptr(cu),
                            n, H, dk, dv, _ptr(o), _ptr(hT), int(nthreads))
    if rc:
        raise ValueError(f"oracle_fwd rejected its arguments ({rc})")
    return o, hT


def fwd_chunked(q, k, v, log_lambda, scale, C, h0=None, cu_seqlens=None, nthreads=0,
                _lib_override=None):
    """The chunked decomposition in fp64 (chunk size ``C``); for invariance checks only."""
    q, k, v, ll, h0 = _f32(q), _f32(k), _f32(v), _f32(log_lambda), _f32(h0)
    T, H, dk, dv = _shapes(q, k, v)
    cu = _cu(cu_seqlens, T)
    n = len(cu) - 1
    o = np.zeros((T, H, dv), np.float64)
    hT = np.zeros((n, H, dk, dv), np.float64)
    rc = (_lib_override or _load()).oracle_fwd_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), _ptr(h0), float(scale),
                                    _ptr(cu), n, H, dk, dv, int(C), _ptr(o), _ptr(hT), int(nthreads))
    if rc:
        raise ValueError(f"oracle_fwd_chunked rejected its arguments ({rc})")
    return o, hT


def decode_step(q, k, v, log_lambda, scale, state, nthreads=0, _lib_override=None):
    """One decode step.  ``state`` is an fp64 ``[N, H, dk, dv]`` array updated in place.

    q, k ``[N, H, dk]``; v ``[N, H, dv]``.  Returns ``o [N, H, dv]`` (fp64)."""
    q, k, v, ll = _f32(q), _f32(k), _f32(v), _f32(log_lambda)
    N, H, dk = q.shape
    dv = v.shape[2]
    if state.dtype != np.float64 or not state.flags.c_contiguous or state.shape != (N, H, dk, dv):
        raise ValueError("state must be a C-contiguous fp64 [N, H, dk, dv] array")
    o = np.zeros((N, H, dv), np.float64)
    rc = (_lib_override or _load()).oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), float(scale), _ptr(state),
                                    _ptr(o), N, H, dk, dv, int(nthreads))
    if rc:
        raise ValueError(f"oracle_decode_step rejected its arguments ({rc})")
    return o


def self_aug(q, k, v, aug, _lib_override=None):
    """The self-augmentation term ``sigmoid(q_t . (a_h * k_t)) v_t`` for every row (token or
    sequence) and head, fp64 ``[rows, H, dv]``; add it to :func:`fwd`'s or :func:`decode_step`'s
    output.  q, k ``[rows, H, dk]``; v ``[rows, H, dv]``; aug ``[H, dk]``."""
    q, k, v, a = _f32(q), _f32(k), _f32(v), _f32(aug)
    rows, H, dk, dv = _shapes(q, k, v)
    if a.shape != (H, dk):
        raise ValueError("aug must be [H, dk]")
    out = np.zeros((rows, H, dv), np.float64)
    rc = (_lib_override or _load()).oracle_self_aug(_ptr(q), _ptr(k), _ptr(v), _ptr(a), rows, H, dk, dv,
                                                    _ptr(out))
    if rc:
        raise ValueError(f"oracle_self_aug rejected its arguments ({rc})")
    return out


def head_norm_gate(o, g, weight, tier, eps, _lib_override=None):
    """Per-tier Head RMSNorm of each head's output row and the SiLU(g) gate, fp64
    ``[rows, H, dv]``.  o, g ``[rows, H, dv]``; weight ``[n_tiers, dv]``; tier ``[H]`` int."""
    o, g, w = _f32(o), _f32(g), _f32(weight)
    tr = np.ascontiguousarray(tier, np.int32)
    if o.ndim != 3 or g.shape != o.shape or w.ndim != 2 or w.shape[1] != o.shape[2] or tr.shape != (o.shape[1],):
        raise ValueError("expected o, g [rows, H, dv], weight [n_tiers, dv], tier [H]")
    rows, H, dv = o.shape
    y = np.zeros((rows, H, dv), np.float64)
    rc = (_lib_override or _load()).oracle_head_norm_gate(_ptr(o), _ptr(g), _ptr(w), _ptr(tr), w.shape[0],
                                                          float(eps), rows, H, dv, _ptr(y))
    if rc:
        raise ValueError(f"oracle_head_norm_gate rejected its arguments ({rc})")
    return y


def round_to_bf16(x, _lib_override=None):
    """fp64 values rounded to the nearest bf16 (ties to even), as fp64."""
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty_like(x)
    (_lib_override or _load()).oracle_round_to_bf16(_ptr(x), _ptr(y), x.size)
    return y


def decode_step_bf16_state(q, k, v, log_lambda, scale, state, _lib_override=None):
    """One decode step with a bf16-stored state: ``state`` (fp64 ``[N, H, dk, dv]`` holding bf16
    values) is updated in place to the update rounded to bf16; returns ``o`` read out from the
    update before that rounding."""
    q, k, v, ll = _f32(q), _f32(k), _f32(v), _f32(log_lambda)
    N, H, dk = q.shape
    dv = v.shape[2]
    if state.dtype != np.float64 or not state.flags.c_contiguous or state.shape != (N, H, dk, dv):
        raise ValueError("state must be a C-contiguous fp64 [N, H, dk, dv] array")
    o = np.zeros((N, H, dv), np.float64)
    rc = (_lib_override or _load()).oracle_decode_step_bf16_state(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), float(scale),
                                                                  _ptr(state), _ptr(o), N, H, dk, dv)
    if rc:
        raise ValueError(f"oracle_decode_step_bf16_state rejected its arguments ({rc})")
    return o


def mxfp8_quantize(x, _lib_override=None):
    """MXFP8 (E4M3 elements, one E8M0 scale per 32 along the last axis) of fp32 values
    ``x [..., 32 m]``: returns ``(codes uint8 [..., 32 m], scales uint8 [..., m])``."""
    x = _f32(x)
    cols = x.shape[-1]
    rows = x.size // cols if cols else 0
    codes = np.zeros(x.shape, np.uint8)
    scales = np.zeros(x.shape[:-1] + (cols // 32,), np.uint8)
    rc = (_lib_override or _load()).oracle_mxfp8_quantize(_ptr(x), rows, cols, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError(f"oracle_mxfp8_quantize rejected its arguments ({rc})")
    return codes, scales


def mxfp8_dequantize(codes, scales, _lib_override=None):
    """The fp64 values of MXFP8 ``codes [..., 32 m]`` with ``scales [..., m]``."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    cols = codes.shape[-1]
    if scales.shape != codes.shape[:-1] + (cols // 32,):
        raise ValueError("scales must be [..., cols / 32]")
    x = np.zeros(codes.shape, np.float64)
    rc = (_lib_override or _load()).oracle_mxfp8_dequantize(_ptr(codes), _ptr(scales), codes.size // cols, cols,
                                                            _ptr(x))
    if rc:
        raise ValueError(f"oracle_mxfp8_dequantize rejected its arguments ({rc})")
    return x


def decode_step_mxfp8_state(q, k, v, log_lambda, scale, codes, scales, return_pre=False, _lib_override=None):
    """One decode step with an MXFP8-stored state (``codes`` uint8 ``[N, H, dk, dv]``, ``scales``
    uint8 ``[N, H, dk, dv / 32]``, both updated in place); returns ``o`` (fp64, read out from the
    update before it is stored), and with ``return_pre`` also the fp32 update that was quantised."""
    q, k, v, ll = _f32(q), _f32(k), _f32(v), _f32(log_lambda)
    N, H, dk = q.shape
    dv = v.shape[2]
    for a, shape in ((codes, (N, H, dk, dv)), (scales, (N, H, dk, dv // 32))):
        if a.dtype != np.uint8 or not a.flags.c_contiguous or a.shape != shape:
            raise ValueError("codes / scales must be C-contiguous uint8 [N, H, dk, dv] / [N, H, dk, dv/32]")
    o = np.zeros((N, H, dv), np.float64)
    pre = np.zeros((N, H, dk, dv), np.float32) if return_pre else None
    rc = (_lib_override or _load()).oracle_decode_step_mxfp8_state(
        _ptr(q), _ptr(k), _ptr(v), _ptr(ll), float(scale), _ptr(codes), _ptr(scales), _ptr(o), N, H, dk, dv,
        _ptr(pre))
    if rc:
        raise ValueError(f"oracle_decode_step_mxfp8_state rejected its arguments ({rc})")
    return (o, pre) if return_pre else o


def bwd(q, k, v, log_lambda, scale, dO, h0=None, dhT=None, cu_seqlens=None, nthreads=0,
        _lib_override=None):
    """Adjoint of :func:`fwd`.  Returns ``(dq, dk, dv, dh0)`` in fp64."""
    q, k, v, ll, h0, dO, dhT = (_f32(q), _f32(k), _f32(v), _f32(log_lambda), _f32(h0), _f32(dO),
                                _f32(dhT))
    T, H, dk, dv = _shapes(q, k, v)
    cu = _cu(cu_seqlens, T)
    n = len(cu) - 1
    dq = np.zeros((T, H, dk), np.float64)
    dkk = np.zeros((T, H, dk), np.float64)
    dvv = np.zeros((T, H, dv), np.float64)
    dh0 = np.zeros((n, H, dk, dv), np.float64)
    rc = (_lib_override or _load()).oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), _ptr(h0), float(scale), _ptr(dO),
                            _ptr(dhT), _ptr(cu), n, H, dk, dv, _ptr(dq), _ptr(dkk), _ptr(dvv),
                            _ptr(dh0), int(nthreads))
    if rc:
        raise ValueError(f"oracle_bwd rejected its arguments ({rc})")
    return dq, dkk, dvv, dh0


class Variant:
    """The same entry points bound to another build of the oracle source (a compiled copy).

    Used by the tests that plant a mistake in a copy of ``gla_oracle.cpp`` and check that the
    pins catch it; the oracle itself is never modified."""

    def __init__(self, so_path):
        self._lib = _bind(so_path)

    def fwd(self, *a, **kw):
        return fwd(*a, _lib_override=self._lib, **kw)

    def fwd_chunked(self, *a, **kw):
        return fwd_chunked(*a, _lib_override=self._lib, **kw)

    def decode_step(self, *a, **kw):
        return decode_step(*a, _lib_override=self._lib, **kw)

    def bwd(self, *a, **kw):
        return bwd(*a, _lib_override=self._lib, **kw)

    def self_aug(self, *a, **kw):
        return self_aug(*a, _lib_override=self._lib, **kw)

    def head_norm_gate(self, *a, **kw):
        return head_norm_gate(*a, _lib_override=self._lib, **kw)

    def round_to_bf16(self, *a, **kw):
        return round_to_bf16(*a, _lib_override=self._lib, **kw)

    def decode_step_bf16_state(self, *a, **kw):
        return decode_step_bf16_state(*a, _lib_override=self._lib, **kw)

    def mxfp8_quantize(self, *a, **kw):
        return mxfp8_quantize(*a, _lib_override=self._lib, **kw)

    def mxfp8_dequantize(self, *a, **kw):
        return mxfp8_dequantize(*a, _lib_override=self._lib, **kw)

    def decode_step_mxfp8_state(self, *a, **kw):
        return decode_step_mxfp8_state(*a, _lib_override=self._lib, **kw)


def source_path() -> str:
    return _SRC

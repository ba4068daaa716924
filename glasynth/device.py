"""Device-side filling of torch CUDA tensors with the seeded inputs of :mod:`glasynth`.

Same generator, same bits as the numpy implementation; used where an input is too large to
generate on the host (the 36 GB decode state pool) or to copy every time."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import torch

from . import stream_key

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.cu")
_LIB = os.path.join(_HERE, "libglasynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.glasynth_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong,
                                                 ctypes.c_ulonglong, ctypes.c_ulonglong,
                                                 ctypes.c_double, ctypes.c_void_p]
            lib.glasynth_fill_normal.restype = ctypes.c_int
            _lib = lib
    return _lib


def fill_normal_(t: torch.Tensor, seed: int, tid: int, sigma: float = 1.0, start: int = 0) -> torch.Tensor:
    """Fills contiguous CUDA tensor ``t`` (fp32 or bf16) with elements ``start ..`` of the stream."""
    if not t.is_cuda or not t.is_contiguous() or t.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("fill_normal_ needs a contiguous fp32/bf16 CUDA tensor")
    with torch.cuda.device(t.device):
        rc = _load().glasynth_fill_normal(
            ctypes.c_void_p(t.data_ptr()), int(t.dtype == torch.bfloat16), t.numel(), int(start),
            stream_key(seed, tid), float(sigma),
            ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream))
    if rc:
        raise RuntimeError("glasynth_fill_normal launch failed")
    return t


def normal(shape, seed: int, tid: int, sigma: float = 1.0, dtype=torch.bfloat16, device="cuda",
           start: int = 0) -> torch.Tensor:
    return fill_normal_(torch.empty(shape, dtype=dtype, device=device), seed, tid, sigma, start)

"""Seeded synthetic inputs for the GLA mixer: one counter-based generator, two implementations.

This module holds no part of the GLA arithmetic.  It only turns (seed, tensor id, element
index) into numbers, identically on the host (numpy, here) and on the device (the CUDA kernel
in ``synth_gen.cu``, loaded through :mod:`glasynth.device`).  The oracle's inputs come from
the host side, the GPU path's from either side; both give the same bits.

Generator (the "published definition" both sides implement):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014; the finaliser constants are those of Vigna's public-domain C version).
  Output ``i`` (0-based) of the stream seeded with ``key`` is ``mix64(key + (i + 1) * GAMMA)``.
* Stream key of tensor ``tid`` under run seed ``seed``: ``mix64((seed * 2**16 + tid + 1) * GAMMA)``.
* Normal variate (approximate): the four 16-bit fields of one 64-bit output are summed
  (Irwin-Hall with n = 4 discrete uniforms), centred and scaled in fp32:
  ``x = (float(sum) - 131070.0f) * c``, ``c = fp32(sigma / sqrt(4 * (65536**2 - 1) / 12))``.
  Every step is exact or a single IEEE fp32 rounding, so host and device agree bit for bit.
  The distribution has mean 0, standard deviation sigma, and tails cut at 3.46 sigma.
* bf16 inputs are the fp32 variates rounded to nearest-even.
* Uniform integers in [lo, hi]: ``lo + u64 % (hi - lo + 1)``.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1
IH4_SD = float(np.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0))
IH4_MEAN = 131070.0

# Tensor ids of the streams.  A config's run seed picks the stream family.
TID = {
    "q": 1, "k": 2, "v": 3, "h0": 4, "dO": 5, "dhT": 6, "state": 7, "lengths": 8,
}


def tid_decode(step: int, name: str) -> int:
    """Tensor id of the decode-step input ``name`` (q, k or v) at step ``step``."""
    return 64 + 3 * step + {"q": 0, "k": 1, "v": 2}[name]


def _mix64_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int) -> int:
    return _mix64_int(((seed * 65536 + tid + 1) * GAMMA) & _MASK)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def u64_at(seed: int, tid: int, idx: np.ndarray) -> np.ndarray:
    """Outputs number ``idx`` (any array of non-negative ints) of the stream of (seed, tid)."""
    key = np.uint64(stream_key(seed, tid))
    i = np.asarray(idx, dtype=np.uint64) + np.uint64(1)
    with np.errstate(over="ignore"):
        return _mix64(key + i * np.uint64(GAMMA))


def u64(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream of (seed, tid)."""
    return u64_at(seed, tid, np.arange(start, start + count, dtype=np.uint64))


def ih4_scale(sigma: float) -> np.float32:
    """The fp32 constant ``c`` that both sides multiply by."""
    return np.float32(sigma / IH4_SD)


def _ih4(x: np.ndarray, sigma: float) -> np.ndarray:
    m = np.uint64(0xFFFF)
    s = ((x & m) + ((x >> np.uint64(16)) & m) + ((x >> np.uint64(32)) & m)
         + ((x >> np.uint64(48)) & m))
    return ((s.astype(np.float32) - np.float32(IH4_MEAN)) * ih4_scale(sigma)).astype(np.float32)


def normal(seed: int, tid: int, shape, sigma: float = 1.0, start: int = 0) -> np.ndarray:
    """fp32 approximate-normal variates, elements ``start ..`` of the stream, in C order."""
    count = int(np.prod(shape, dtype=np.int64))
    return _ih4(u64(seed, tid, count, start), sigma).reshape(shape)


def normal_rows(seed: int, tid: int, row_shape, rows, sigma: float = 1.0) -> np.ndarray:
    """Rows ``rows`` (flat indices of the leading axis) of a C-order tensor ``[*, *row_shape]``.

    Lets a test regenerate a sampled slice of a device-generated tensor without the rest."""
    row_len = int(np.prod(row_shape, dtype=np.int64))
    rows = np.asarray(rows, dtype=np.uint64)
    idx = rows[:, None] * np.uint64(row_len) + np.arange(row_len, dtype=np.uint64)[None, :]
    return _ih4(u64_at(seed, tid, idx), sigma).reshape((len(rows),) + tuple(row_shape))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the 16-bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 values rounded to the nearest bf16 (ties to even), returned as fp32."""
    return (bf16_bits(x).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform_int(seed: int, tid: int, count: int, lo: int, hi: int) -> np.ndarray:
    x = u64(seed, tid, count)
    return (np.uint64(lo) + x % np.uint64(hi - lo + 1)).astype(np.int64)


# ----------------------------------------------------------------------------------------------
# Workloads: shapes, seeds and distributions of the five measured configurations.
# ----------------------------------------------------------------------------------------------
H = 16
DK = 96
DV = 192
SCALE = np.float32(1.0 / np.sqrt(96.0))


def laplace_log_lambda(H: int = 16) -> np.ndarray:
    """log of the per-head decay 1 - 2^-(5 + 7h/15), rounded to fp32 (the workloads' schedule)."""
    h = np.arange(H, dtype=np.float64)
    return np.log1p(-np.exp2(-(5.0 + 7.0 * h / 15.0))).astype(np.float32)


def halflife_log_lambda(H: int = 16, t_min: float = 1.0, t_max: float = 2048.0) -> np.ndarray:
    """log-decay of a geometric half-life schedule from t_min to t_max tokens (lambda_0 = 0.5)."""
    h = np.arange(H, dtype=np.float64)
    t_half = t_min * (t_max / t_min) ** (h / max(H - 1, 1))
    return (-np.log(2.0) / t_half).astype(np.float32)


def varlen_lengths(seed: int = 3, n_seq: int = 32, lo: int = 128, hi: int = 16384) -> np.ndarray:
    return uniform_int(seed, TID["lengths"], n_seq, lo, hi)


def cu_seqlens_of(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return cu

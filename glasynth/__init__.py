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
* Normal variate (Box-Muller; Box and Muller, "A note on the generation of random normal
  deviates", Ann. Math. Statist. 1958): from one 64-bit output x, a = x >> 32 and b = x mod 2^32,
  u1 = (a + 1/2) / 2^32 in (0, 1), u2 = b / 2^32 in [0, 1), and
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, ``value = fp32(z * sigma)``.  Only the cosine half of the
  pair is used, so element i of a tensor is a function of output i alone.  Tails reach
  sqrt(-2 ln(2^-33)) = 6.77 sigma.  The logarithm and cosine are not library calls but the
  series below, evaluated in fp64 with IEEE-rounded +, -, x, / and sqrt only, in one fixed
  order, so that numpy here and the CUDA kernel give the same bits:
    ln u1 = (e - 32) ln 2 + ln m, with a + 1/2 = 2^e m, m in [1/sqrt 2, sqrt 2], and
    ln m = 2 t (1 + t^2/3 + t^4/5 + ... + t^20/21), t = (m - 1)/(m + 1), |t| <= 0.1716
    (the atanh series; truncation below 1e-17 relative);
    2 pi u2 = n pi/2 + phi with 4 u2 = n + f, n = floor(4 u2 + 1/2), |f| <= 1/2, phi = f pi/2, and
    cos phi, sin phi by their Taylor series through phi^20/20!, phi^21/21! (|phi| <= pi/4;
    truncation below 1e-20); cos(2 pi u2) is cos phi, -sin phi, -cos phi, sin phi for n mod 4 =
    0, 1, 2, 3.  The series coefficients 1/(2j+1) and +-1/k! are correctly rounded doubles (k! is
    exact in fp64 for k <= 22).  The result agrees with the exact Box-Muller value to about 1e-15
    relative before the final fp32 rounding.
* bf16 inputs are the fp32 variates rounded to nearest-even.
* Uniform integers in [lo, hi]: ``lo + u64 % (hi - lo + 1)``.
"""
from __future__ import annotations

import numpy as np

import math

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# fp64 constants of the Box-Muller evaluation (the CUDA kernel uses the same values)
LN2 = 0.6931471805599453      # ln 2, rounded to double
PIO2 = 1.5707963267948966     # pi / 2, rounded to double
SQRT2 = 1.4142135623730951    # sqrt 2, rounded to double
LOG_C = tuple(1.0 / (2 * j + 1) for j in range(11))                            # atanh series
COS_C = tuple((-1) ** j / float(math.factorial(2 * j)) for j in range(11))      # cos Taylor
SIN_C = tuple((-1) ** j / float(math.factorial(2 * j + 1)) for j in range(11))  # sin Taylor

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


def _horner(coef, s):
    p = np.full_like(s, coef[-1])
    for c in coef[-2::-1]:
        p = p * s + c
    return p


def ln_u1(a: np.ndarray) -> np.ndarray:
    """ln((a + 1/2) / 2^32) for 32-bit integers a, by the atanh series (see the module text)."""
    y = a.astype(np.float64) + 0.5
    mant, ex = np.frexp(y)                       # y = mant 2^ex, mant in [1/2, 1): exact
    m = mant * 2.0
    e = ex.astype(np.int64) - 1
    big = m > SQRT2
    m = np.where(big, m * 0.5, m)
    e = np.where(big, e + 1, e)
    t = (m - 1.0) / (m + 1.0)
    lnm = (2.0 * t) * _horner(LOG_C, t * t)
    return (e - 32).astype(np.float64) * LN2 + lnm


def cos_2pi(b: np.ndarray) -> np.ndarray:
    """cos(2 pi b / 2^32) for 32-bit integers b, by quadrant reduction and Taylor series."""
    w = b.astype(np.float64) * (2.0 ** -30)      # 4 u2, exact
    n = np.floor(w + 0.5)
    phi = (w - n) * PIO2
    s = phi * phi
    c = _horner(COS_C, s)
    sn = phi * _horner(SIN_C, s)
    q = n.astype(np.int64) & 3
    return np.where(q == 0, c, np.where(q == 1, -sn, np.where(q == 2, -c, sn)))


def _box_muller(x: np.ndarray, sigma: float) -> np.ndarray:
    a = x >> np.uint64(32)
    b = x & np.uint64(0xFFFFFFFF)
    z = np.sqrt(-2.0 * ln_u1(a)) * cos_2pi(b)
    return (z * float(sigma)).astype(np.float32)


def normal(seed: int, tid: int, shape, sigma: float = 1.0, start: int = 0) -> np.ndarray:
    """fp32 N(0, sigma^2) variates (Box-Muller), elements ``start ..`` of the stream, in C order."""
    count = int(np.prod(shape, dtype=np.int64))
    out = np.empty(count, np.float32)
    step = 1 << 22                               # bounded temporaries for large tensors
    for i in range(0, count, step):
        out[i:i + step] = _box_muller(u64(seed, tid, min(step, count - i), start + i), sigma)
    return out.reshape(shape)


def normal_rows(seed: int, tid: int, row_shape, rows, sigma: float = 1.0) -> np.ndarray:
    """Rows ``rows`` (flat indices of the leading axis) of a C-order tensor ``[*, *row_shape]``.

    Lets a test regenerate a sampled slice of a device-generated tensor without the rest."""
    row_len = int(np.prod(row_shape, dtype=np.int64))
    rows = np.asarray(rows, dtype=np.uint64)
    idx = rows[:, None] * np.uint64(row_len) + np.arange(row_len, dtype=np.uint64)[None, :]
    return _box_muller(u64_at(seed, tid, idx), sigma).reshape((len(rows),) + tuple(row_shape))


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

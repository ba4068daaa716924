"""Shared pieces of the GPU parity tests: inputs built on the host (so the oracle sees exactly
the same values), the error metric, and per-sequence comparison."""
import numpy as np

import glasynth as gs

BF16_TOL = 2e-2   # max |gpu - oracle| / rms(oracle), bf16 operands, fp32 state and accumulation
F32_TOL = 1e-4    # same metric, all-fp32 mode


def half_ulp_bf16(ref):
    """Half a unit in the last place of bf16 at |ref|: the error of rounding ref itself to bf16."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


class RelErr(float):
    """The bounded figure (a float, compared against the bar) that also carries the raw
    max |x - ref| / rms(ref) without the half-ulp allowance; formatting shows both, so a
    failure message tells how far the plain error sits from the bar."""

    def __new__(cls, value, raw):
        obj = super().__new__(cls, value)
        obj.raw = raw
        return obj

    def __format__(self, spec):
        return f"{float(self):{spec or '.3e'}} (raw {self.raw:{spec or '.3e'}})"

    def __repr__(self):
        return format(self, ".3e")


def rel_err(x, ref, bf16_out=False):
    """max |x - ref| / rms(ref).  For outputs stored in bf16 (``bf16_out``), each element's error
    is first reduced by half a bf16 ulp of ref: the rounding that even the exact answer takes
    when stored in the output's format, which the bound is not meant to measure.  The result
    (a float) also carries the raw figure, shown when formatted."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return RelErr(0.0, 0.0)
    rms = max(float(np.sqrt(np.mean(ref ** 2))), 1e-30)
    d = np.abs(x - ref)
    raw = float(np.max(d) / rms)
    if bf16_out:
        d = np.maximum(d - half_ulp_bf16(ref), 0.0)
    return RelErr(float(np.max(d) / rms), raw)


def within_one_bf16_rounding(x, y):
    """True when two bf16 results of the same fp32 sum, added up in different orders, differ
    element by element by at most one bf16 ulp of the larger (2^-7 of its magnitude: adjacent
    bf16 values), plus 1e-5 of the RMS for values near zero, where a reordered fp32 sum can
    change sign."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    rms = float(np.sqrt(np.mean(y ** 2))) if y.size else 0.0
    return bool(np.all(np.abs(x - y) <= np.exp2(-7) * np.maximum(np.abs(x), np.abs(y)) + 1e-5 * rms))


def host_chunk_inputs(seed, lengths, H, bf16, with_h0, packed, log_lambda=None, grad=False,
                      qk_sigma=1 / np.sqrt(96), v_sigma=1.0):
    """Numpy inputs in oracle layout ([T_total, H, d], cu_seqlens) plus the GPU layout shape."""
    cu = gs.cu_seqlens_of(lengths)
    Tt = int(cu[-1])
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    d = {
        "q": rnd(gs.normal(seed, 1, (Tt, H, 96), qk_sigma)),
        "k": rnd(gs.normal(seed, 2, (Tt, H, 96), qk_sigma)),
        "v": rnd(gs.normal(seed, 3, (Tt, H, 192), v_sigma)),
        "h0": gs.normal(seed, 4, (len(lengths), H, 96, 192), 0.1) if with_h0 else None,
        "log_lambda": gs.laplace_log_lambda(H) if log_lambda is None else
        np.asarray(log_lambda, np.float32),
        "cu": cu,
    }
    if grad:
        d["dO"] = rnd(gs.normal(seed, 5, (Tt, H, 192)))
        d["dhT"] = gs.normal(seed, 6, (len(lengths), H, 96, 192), 0.01)
    if not packed:
        assert len(set(lengths)) == 1
    d["gpu_prefix"] = (Tt,) if packed else (len(lengths), lengths[0])
    return d


def to_device(d, bf16, packed):
    import torch
    dt = torch.bfloat16 if bf16 else torch.float32
    out = {}
    for name in ("q", "k", "v", "dO"):
        if name in d:
            x = torch.from_numpy(np.ascontiguousarray(d[name]))
            x = x.reshape(d["gpu_prefix"] + tuple(d[name].shape[1:]))
            out[name] = x.to("cuda").to(dt).contiguous()
    for name in ("h0", "dhT"):
        out[name] = None if d.get(name) is None else torch.from_numpy(d[name]).cuda()
    out["log_lambda"] = torch.from_numpy(d["log_lambda"]).cuda()
    out["cu_seqlens"] = torch.from_numpy(d["cu"]).cuda() if packed else None
    return out


def flat(t, packed):
    """GPU tensor -> numpy [T_total, H, d] (fp64)."""
    x = t.float().cpu().numpy().astype(np.float64)
    return x if packed else x.reshape((-1,) + x.shape[2:])

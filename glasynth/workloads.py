"""The five measured workloads: shapes, seeds and distributions, generated on the device, with
any sampled slice regenerable bit-for-bit on the host for the oracle.

  tiny      B=1, T=256, H=2; fp32 q, k, v ~ N(0,1); lambda = {0.97, 0.999}; h0 = 0; seed 0
  layer     B=8, T=2048, H=16; bf16 q, k ~ N(0,1)/sqrt(96), v ~ N(0,1); lambda_h = 1 - 2^-(5+7h/15);
            h0 = 0; seed 1
  decode    1,280 sequences x 24 layers (= 30,720 pool rows) x H=16 fp32 states ~ N(0, 0.1);
            per step bf16 q, k, v as in `layer`; lambda as in `layer`; 64 steps; seed 2
  varlen    32 sequences, lengths uniform in [128, 16384] (seed 3), packed; h0 ~ N(0, 0.1);
            bf16 q, k, v as in `layer`; seed 3
  bwd       `layer` shapes; dO ~ N(0,1) bf16, dhT ~ N(0, 0.01) fp32; seed 4

"N(0, s)" is read with s the standard deviation; the variates are Box-Muller normals (tails
to 6.77 sigma), documented in :mod:`glasynth`.  No part of the GLA arithmetic is here.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import (DK, DV, SCALE, TID, bf16_round, cu_seqlens_of, laplace_log_lambda, normal_rows,
               tid_decode, varlen_lengths)

QK_SIGMA = float(1.0 / np.sqrt(96.0))


@dataclass
class ChunkWorkload:
    name: str
    seed: int
    lengths: list               # per-sequence lengths
    H: int
    bf16: bool
    packed: bool                # True: [T_total, H, d] with cu_seqlens; False: [B, T, H, d]
    log_lambda: np.ndarray
    h0_sigma: float = 0.0       # 0: h0 absent (zeros)
    qk_sigma: float = QK_SIGMA
    v_sigma: float = 1.0
    with_grad: bool = False     # backward inputs dO, dhT
    dO_sigma: float = 1.0
    dhT_sigma: float = 0.01
    scale: float = float(SCALE)
    cu: np.ndarray = field(init=False)

    def __post_init__(self):
        self.cu = cu_seqlens_of(self.lengths)

    @property
    def n_seq(self):
        return len(self.lengths)

    @property
    def tokens(self):
        return int(self.cu[-1])

    def shape(self, d):
        if self.packed:
            return (self.tokens, self.H, d)
        return (self.n_seq, self.lengths[0], self.H, d)

    # ---- device tensors -------------------------------------------------------------------
    def device_inputs(self, device="cuda"):
        import torch

        from .device import normal
        dt = torch.bfloat16 if self.bf16 else torch.float32
        out = {
            "q": normal(self.shape(DK), self.seed, TID["q"], self.qk_sigma, dt, device),
            "k": normal(self.shape(DK), self.seed, TID["k"], self.qk_sigma, dt, device),
            "v": normal(self.shape(DV), self.seed, TID["v"], self.v_sigma, dt, device),
            "log_lambda": torch.from_numpy(self.log_lambda).to(device),
            "h0": None, "cu_seqlens": None,
        }
        if self.h0_sigma:
            out["h0"] = normal((self.n_seq, self.H, DK, DV), self.seed, TID["h0"], self.h0_sigma,
                               torch.float32, device)
        if self.packed:
            out["cu_seqlens"] = torch.from_numpy(self.cu).to(device)
        if self.with_grad:
            out["dO"] = normal(self.shape(DV), self.seed, TID["dO"], self.dO_sigma, dt, device)
            out["dhT"] = normal((self.n_seq, self.H, DK, DV), self.seed, TID["dhT"],
                                self.dhT_sigma, torch.float32, device)
        return out

    # ---- host regeneration of one (sequence, head) --------------------------------------------
    def _token_rows(self, n, h):
        t0, t1 = int(self.cu[n]), int(self.cu[n + 1])
        return [(t * self.H + h) for t in range(t0, t1)]

    def host_unit(self, n, h):
        """fp32 arrays of sequence n, head h in oracle layout (H = 1): q, k [T,1,96], v [T,1,192],
        h0 [1,1,96,192] or None, dO, dhT when the workload has them."""
        rows = self._token_rows(n, h)
        rnd = bf16_round if self.bf16 else (lambda x: x)
        out = {
            "q": rnd(normal_rows(self.seed, TID["q"], (DK,), rows, self.qk_sigma))[:, None],
            "k": rnd(normal_rows(self.seed, TID["k"], (DK,), rows, self.qk_sigma))[:, None],
            "v": rnd(normal_rows(self.seed, TID["v"], (DV,), rows, self.v_sigma))[:, None],
            "h0": None,
            "log_lambda": self.log_lambda[h:h + 1],
        }
        if self.h0_sigma:
            out["h0"] = normal_rows(self.seed, TID["h0"], (DK, DV), [n * self.H + h],
                                    self.h0_sigma)[:, None]
        if self.with_grad:
            out["dO"] = rnd(normal_rows(self.seed, TID["dO"], (DV,), rows, self.dO_sigma))[:, None]
            out["dhT"] = normal_rows(self.seed, TID["dhT"], (DK, DV), [n * self.H + h],
                                     self.dhT_sigma)[:, None]
        return out


def tiny():
    return ChunkWorkload("tiny GLA fwd B=1 T=256 H=2 fp32", 0, [256], 2, bf16=False, packed=False,
                         log_lambda=np.log(np.array([0.97, 0.999], np.float32)),
                         qk_sigma=1.0, v_sigma=1.0)


def layer(with_grad=False, B=8, T=2048, H=16):
    name = (f"Laplace-layer chunked {'bwd' if with_grad else 'fwd'} B={B} T={T} H={H} dk=96 dv=192 bf16")
    return ChunkWorkload(name, 4 if with_grad else 1, [T] * B, H, bf16=True, packed=False,
                         log_lambda=laplace_log_lambda(H), with_grad=with_grad)


def varlen(n_seq=32, lo=128, hi=16384, H=16):
    lens = [int(x) for x in varlen_lengths(3, n_seq, lo, hi)]
    return ChunkWorkload(f"packed varlen fwd {n_seq} seqs len U[{lo},{hi}] H={H} bf16 h0", 3, lens,
                         H, bf16=True, packed=True, log_lambda=laplace_log_lambda(H), h0_sigma=0.1)


@dataclass
class DecodeWorkload:
    name: str = "decode 1280 seqs x 24 layers H=16 fp32 state bf16 io"
    seed: int = 2
    seqs: int = 1280
    layers: int = 24
    H: int = 16
    steps: int = 64
    state_sigma: float = 0.1
    qk_sigma: float = QK_SIGMA
    v_sigma: float = 1.0
    scale: float = float(SCALE)

    @property
    def N(self):  # pool rows: one per (sequence, layer)
        return self.seqs * self.layers

    @property
    def log_lambda(self):
        return laplace_log_lambda(self.H)

    def device_state(self, device="cuda"):
        import torch

        from .device import normal
        return normal((self.N, self.H, DK, DV), self.seed, TID["state"], self.state_sigma,
                      torch.float32, device)

    def device_step(self, step, device="cuda", out=None):
        import torch

        from .device import fill_normal_, normal
        shapes = {"q": (self.N, self.H, DK), "k": (self.N, self.H, DK), "v": (self.N, self.H, DV)}
        sig = {"q": self.qk_sigma, "k": self.qk_sigma, "v": self.v_sigma}
        if out is None:
            return {nm: normal(shapes[nm], self.seed, tid_decode(step, nm), sig[nm], torch.bfloat16,
                               device) for nm in ("q", "k", "v")}
        for nm in ("q", "k", "v"):
            fill_normal_(out[nm], self.seed, tid_decode(step, nm), sig[nm])
        return out

    def host_state(self, rows_nh):
        """fp32 initial states of the (row, head) pairs, as [len, 96, 192]."""
        return normal_rows(self.seed, TID["state"], (DK, DV), [r * self.H + h for r, h in rows_nh],
                           self.state_sigma)

    def host_step(self, step, rows_nh):
        idx = [r * self.H + h for r, h in rows_nh]
        q = bf16_round(normal_rows(self.seed, tid_decode(step, "q"), (DK,), idx, self.qk_sigma))
        k = bf16_round(normal_rows(self.seed, tid_decode(step, "k"), (DK,), idx, self.qk_sigma))
        v = bf16_round(normal_rows(self.seed, tid_decode(step, "v"), (DV,), idx, self.v_sigma))
        return q, k, v

"""GPU parity of gla_head_norm_gate (per-tier Head RMSNorm and SiLU(g) gate, "Beyond the KV
cache", section "i14 and the Laplace 3B architecture") against the fp64 oracle.  Bar as for the
mixer: max |gpu - oracle| / rms(oracle) <= 2e-2 for bf16 data (half a bf16 ulp of allowance on
the stored output), <= 1e-4 in fp32."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from tests.gpu_helpers import BF16_TOL, F32_TOL, flat, host_chunk_inputs, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


def _inputs(seed, rows, H, n_tiers, bf16):
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    o = rnd(gs.normal(seed, 1, (rows, H, 192)))
    g = rnd(gs.normal(seed, 2, (rows, H, 192), 2.0))
    w = (1.0 + gs.normal(seed, 3, (n_tiers, 192), 0.3)).astype(np.float32)
    tier = (np.arange(H) * n_tiers // H).astype(np.int32)
    return o, g, w, tier


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("rows,H,n_tiers", [(1, 1, 1), (37, 16, 4), (300, 5, 3), (7, 2, 2), (11, 3, 3),
                                             (9, 40, 33)])
def test_head_norm_gate_matches_oracle(bf16, rows, H, n_tiers):
    o, g, w, tier = _inputs(900 + rows + H, rows, H, n_tiers, bf16)
    dt = torch.bfloat16 if bf16 else torch.float32
    y = gla.gla_head_norm_gate(torch.from_numpy(o).cuda().to(dt), torch.from_numpy(g).cuda().to(dt),
                               torch.from_numpy(w).cuda(), torch.from_numpy(tier).cuda(), eps=1e-6)
    ref = oracle.head_norm_gate(o, g, w, tier, 1e-6)
    assert rel_err(y.float().cpu().numpy(), ref, bf16_out=bf16) <= (BF16_TOL if bf16 else F32_TOL)


def test_head_norm_gate_zero_rows_and_large_eps():
    """A row of zeros gives zeros; a huge eps gives o * w * SiLU(g) / sqrt(eps)."""
    o, g, w, tier = _inputs(950, 8, 4, 2, False)
    o[3] = 0.0
    y = gla.gla_head_norm_gate(torch.from_numpy(o).cuda(), torch.from_numpy(g).cuda(),
                               torch.from_numpy(w).cuda(), torch.from_numpy(tier).cuda(), eps=1e-6)
    assert torch.count_nonzero(y[3]) == 0
    y = gla.gla_head_norm_gate(torch.from_numpy(o).cuda(), torch.from_numpy(g).cuda(),
                               torch.from_numpy(w).cuda(), torch.from_numpy(tier).cuda(), eps=1e8)
    assert rel_err(y.cpu().numpy(), oracle.head_norm_gate(o, g, w, tier, 1e8)) <= F32_TOL


def test_head_norm_gate_bad_tier_is_reported_and_skipped():
    o, g, w, tier = _inputs(960, 6, 3, 2, False)
    tier[1] = 7
    y = torch.full(o.shape, 5.0, device="cuda")
    gla.gla_head_norm_gate(torch.from_numpy(o).cuda(), torch.from_numpy(g).cuda(), torch.from_numpy(w).cuda(),
                           torch.from_numpy(tier).cuda(), y=y)
    assert gla.gla_get_device_error() == -2  # GLA_ERR_SHAPE, cleared by the read
    assert torch.all(y[:, 1] == 5.0)
    ok = [0, 2]
    assert rel_err(y[:, ok].cpu().numpy(), oracle.head_norm_gate(o, g, w, tier.clip(0, 1), 1e-6)[:, ok]) <= F32_TOL


def test_forward_then_norm_gate_end_to_end():
    """The mixer's bf16 output [B, T, H, 192] through the norm and gate, against the oracle's norm
    of that same output (each stage meets its own bar: the forward's error, up to 2e-2 of o's
    RMS, is scaled by SiLU(g) here and is not a property of this stage)."""
    B, H, T = 2, 16, 300
    d = host_chunk_inputs(970, [T] * B, H, True, with_h0=True, packed=False)
    d["scale"] = float(gs.SCALE)
    gd = to_device(d, True, packed=False)
    o, _ = gla.gla_chunk_fwd(gd["q"], gd["k"], gd["v"], gd["log_lambda"], d["scale"], h0=gd["h0"])
    _, g, w, tier = _inputs(971, B * T, H, 4, True)
    y = gla.gla_head_norm_gate(o, torch.from_numpy(g).cuda().to(torch.bfloat16).view(B, T, H, 192),
                               torch.from_numpy(w).cuda(), torch.from_numpy(tier).cuda())
    ref = oracle.head_norm_gate(flat(o, False), g, w, tier, 1e-6)
    assert rel_err(flat(y, False), ref, bf16_out=True) <= BF16_TOL


def test_head_norm_gate_benchmark_size_in_full():
    """16,384 rows x 16 heads x 192 bf16, four tiers (the benchmark row's shape and inputs),
    compared in full (the oracle is a single pass)."""
    rows, H = 16384, 16
    o = gs.bf16_round(gs.normal(13, 1, (rows, H, 192)))
    g = gs.bf16_round(gs.normal(13, 2, (rows, H, 192), 2.0))
    w = (1.0 + gs.normal(13, 3, (4, 192), 0.3)).astype(np.float32)
    tier = (np.arange(H) // 4).astype(np.int32)
    y = gla.gla_head_norm_gate(torch.from_numpy(o).cuda().to(torch.bfloat16),
                               torch.from_numpy(g).cuda().to(torch.bfloat16), torch.from_numpy(w).cuda(),
                               torch.from_numpy(tier).cuda())
    ref = oracle.head_norm_gate(o, g, w, tier, 1e-6)
    assert rel_err(y.float().cpu().numpy(), ref, bf16_out=True) <= BF16_TOL

"""GPU parity of gla_decode_step_norm_gate: the decode step with the per-tier Head RMSNorm and the
SiLU(g) gate fused into its epilogue ("Beyond the KV cache", section "i14 and the Laplace 3B
architecture": Head RMSNorm per tier, then the SiLU gate; "Decay schedule's reach": tiers of
heads share a norm).  Reference: the oracle's decode step followed by the oracle's Head RMSNorm +
gate, in fp64.  Bar: max |gpu - oracle| / rms(oracle) <= 2e-2 with bf16 data (half a bf16 ulp of
allowance on the stored y), <= 1e-4 in fp32; the state pool itself as for gla_decode_step."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from glasynth import workloads as wl
from tests.gpu_helpers import BF16_TOL, F32_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


def _norm_inputs(seed, H, n_tiers):
    w = (1.0 + gs.normal(seed, 3, (n_tiers, 192), 0.3)).astype(np.float32)
    tier = (np.arange(H) * n_tiers // H).astype(np.int32)
    return w, tier


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("with_aug", [False, True])
def test_decode_norm_gate_matches_oracle(bf16, with_aug):
    N, H, P, steps, n_tiers = 5, 16, 7, 6, 4
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    dt = torch.bfloat16 if bf16 else torch.float32
    ll = gs.laplace_log_lambda(H)
    w, tier = _norm_inputs(71, H, n_tiers)
    aug = gs.normal(71, 9, (H, 96), 10.0) if with_aug else None
    slot_h = np.array([6, 0, 3, 5, 1], np.int32)
    s0 = gs.normal(71, 7, (P, H, 96, 192), 0.1)
    state = torch.from_numpy(s0).cuda()
    ref_state = s0.astype(np.float64)[slot_h].copy()
    args = dict(weight=torch.from_numpy(w).cuda(), tier=torch.from_numpy(tier).cuda(),
                slot=torch.from_numpy(slot_h).cuda(), eps=1e-6,
                aug=None if aug is None else torch.from_numpy(aug).cuda())
    tol = BF16_TOL if bf16 else F32_TOL
    for t in range(steps):
        q = rnd(gs.normal(71, 100 + 4 * t, (N, H, 96), 1 / np.sqrt(96)))
        k = rnd(gs.normal(71, 101 + 4 * t, (N, H, 96), 1 / np.sqrt(96)))
        v = rnd(gs.normal(71, 102 + 4 * t, (N, H, 192)))
        g = rnd(gs.normal(71, 103 + 4 * t, (N, H, 192), 2.0))
        dev = [torch.from_numpy(x).cuda().to(dt) for x in (q, k, v, g)]
        y = gla.gla_decode_step_norm_gate(dev[0], dev[1], dev[2], torch.from_numpy(ll).cuda(), state,
                                          dev[3], scale=float(gs.SCALE), **args)
        o_ref = oracle.decode_step(q, k, v, ll, float(gs.SCALE), ref_state)
        if aug is not None:
            o_ref = o_ref + oracle.self_aug(q, k, v, aug)
        y_ref = oracle.head_norm_gate(o_ref, g, w, tier, 1e-6)
        e = rel_err(y.float().cpu().numpy(), y_ref, bf16)
        assert e <= tol, f"step {t}: {e:.3e}"
    assert rel_err(state[slot_h].cpu().numpy(), ref_state) <= 1e-4
    untouched = [r for r in range(P) if r not in slot_h]
    assert np.array_equal(state[untouched].cpu().numpy(), s0[untouched])


def test_decode_norm_gate_matches_unfused_path():
    """The fused step against the unfused calls (gla_decode_step, then gla_head_norm_gate on its
    output), in fp32 (with bf16 data the unfused path rounds o to bf16 before the norm, an error
    of its own that the fused step does not make); the state update is the same kernel code."""
    N, H = 9, 16
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    w, tier = _norm_inputs(72, H, 4)
    w, tier = torch.from_numpy(w).cuda(), torch.from_numpy(tier).cuda()
    s0 = torch.from_numpy(gs.normal(72, 7, (N, H, 96, 192), 0.1)).cuda()
    q, k = (torch.from_numpy(gs.normal(72, i, (N, H, 96), 0.1)).cuda() for i in (1, 2))
    v, g = (torch.from_numpy(gs.normal(72, i, (N, H, 192))).cuda() for i in (3, 4))
    sa, sb = s0.clone(), s0.clone()
    y = gla.gla_decode_step_norm_gate(q, k, v, ll, sa, g, w, tier, scale=float(gs.SCALE))
    o = gla.gla_decode_step(q, k, v, ll, sb, float(gs.SCALE))
    y2 = gla.gla_head_norm_gate(o, g, w, tier, eps=1e-6)
    assert torch.equal(sa, sb)
    assert rel_err(y.cpu().numpy(), y2.cpu().numpy()) <= F32_TOL


def test_decode_norm_gate_bad_tier_is_reported_and_skipped():
    N, H = 3, 4
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    w = torch.ones((2, 192), device="cuda")
    tier = torch.tensor([0, 1, 5, 0], dtype=torch.int32, device="cuda")
    state = torch.zeros((N, H, 96, 192), device="cuda")
    q = k = torch.full((N, H, 96), 0.1, device="cuda")
    v = g = torch.ones((N, H, 192), device="cuda")
    y = torch.full((N, H, 192), 7.0, device="cuda")
    gla.gla_decode_step_norm_gate(q, k, v, ll, state, g, w, tier, y=y)
    assert gla.gla_get_device_error() == -2
    assert torch.all(y[:, 2] == 7.0)                    # head 2's rows untouched
    assert not torch.any(y[:, 0] == 7.0)
    assert torch.all(state[:, 2] != 0.0)                # its state still advanced


def test_decode_norm_gate_workload_sampled_64_steps():
    """The benchmark's pool (1,280 sequences x 24 layers x 16 heads, fp32 states), 64 steps with a
    gate stream g ~ N(0, 2^2) per step and four tiers of four heads; 12 sampled (pool row, head)
    states followed by the oracle's step and norm + gate."""
    w_ = wl.DecodeWorkload()
    state = w_.device_state()
    ll = torch.from_numpy(w_.log_lambda).cuda()
    wt, tier = _norm_inputs(73, w_.H, 4)
    wt_d, tier_d = torch.from_numpy(wt).cuda(), torch.from_numpy(tier).cuda()
    rng = np.random.default_rng(5)
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, w_.N, 10), rng.integers(0, w_.H, 10))]
    rows += [(0, 0), (w_.N - 1, w_.H - 1)]
    ref = w_.host_state(rows).astype(np.float64)[:, None]
    ri = torch.tensor([r for r, _ in rows], device="cuda")
    hi = torch.tensor([h for _, h in rows], device="cuda")
    bufs = w_.device_step(0)
    g = torch.empty((w_.N, w_.H, 192), dtype=torch.bfloat16, device="cuda")
    from glasynth.device import fill_normal_
    worst = 0.0
    for step in range(w_.steps):
        w_.device_step(step, out=bufs)
        fill_normal_(g, 73, 300 + step, 2.0)
        y = gla.gla_decode_step_norm_gate(bufs["q"], bufs["k"], bufs["v"], ll, state, g, wt_d, tier_d,
                                          scale=w_.scale)
        yg = y[ri, hi].float().cpu().numpy()
        q, k, v = w_.host_step(step, rows)
        gh = gs.bf16_round(gs.normal_rows(73, 300 + step, (192,), [r * w_.H + h for r, h in rows], 2.0))
        for i, (r, h) in enumerate(rows):
            o_ref = oracle.decode_step(q[i:i + 1, None], k[i:i + 1, None], v[i:i + 1, None],
                                       w_.log_lambda[h:h + 1], w_.scale, ref[i:i + 1])
            y_ref = oracle.head_norm_gate(o_ref, gh[i:i + 1, None], wt, tier[h:h + 1], 1e-6)[0, 0]
            worst = max(worst, rel_err(yg[i], y_ref, bf16_out=True))
    assert worst <= BF16_TOL, worst
    assert rel_err(state[ri, hi].cpu().numpy(), ref[:, 0]) <= 1e-4

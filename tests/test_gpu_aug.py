"""GPU parity of the self-augmentation entry points (gla_chunk_fwd_aug, gla_decode_step_aug)
against the fp64 oracle: the mixer's output plus sigmoid(q_t . (a_h * k_t)) v_t ("Beyond the KV
cache", section "i14 and the Laplace 3B architecture", the paragraph after the state readout).
Bar as for the plain forward: max |gpu - oracle| / rms(oracle) <= 2e-2 in bf16 mode, <= 1e-4 in
fp32 mode.  The final states do not involve the augmentation and must equal the plain forward's
bit for bit."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from tests.gpu_helpers import BF16_TOL, F32_TOL, flat, host_chunk_inputs, rel_err, to_device

pytestmark = pytest.mark.gpu

# q, k ~ N(0, 1/96): q . (a * k) has a standard deviation of about sigma_a / sqrt(96), so
# sigma_a = 10 spreads the gate over most of the sigmoid.
AUG_SIGMA = 10.0


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


def _aug(seed, H):
    return gs.normal(seed, 9, (H, 96), AUG_SIGMA)


def _run(d, aug, bf16, packed):
    g = to_device(d, bf16, packed)
    a = torch.from_numpy(aug).cuda()
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"],
                              cu_seqlens=g["cu_seqlens"], aug=a)
    o_plain, hT_plain = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"],
                                          h0=g["h0"], cu_seqlens=g["cu_seqlens"])
    return o, hT, o_plain, hT_plain


def _check(d, aug, o, hT, hT_plain, packed, tol):
    bf = o.dtype == torch.bfloat16
    o_ref, hT_ref = oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], d["scale"], h0=d["h0"],
                               cu_seqlens=d["cu"])
    o_ref = o_ref + oracle.self_aug(d["q"], d["k"], d["v"], aug)
    x = flat(o, packed)
    assert np.all(np.isfinite(x))
    cu = d["cu"]
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b > a:
            e = rel_err(x[a:b], o_ref[a:b], bf)
            assert e <= tol, f"o of sequence {n} (len {b - a}): {e:.3e}"
        e = rel_err(hT[n].cpu().numpy(), hT_ref[n])
        assert e <= tol, f"hT of sequence {n}: {e:.3e}"
    assert torch.equal(hT, hT_plain)


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T", [1, 129, 300])
def test_fwd_aug_fixed_length(bf16, T):
    B, H = 2, 3
    d = host_chunk_inputs(700 + T, [T] * B, H, bf16, with_h0=(T % 2 == 1), packed=False)
    d["scale"] = float(gs.SCALE)
    aug = _aug(700 + T, H)
    o, hT, _, hT_plain = _run(d, aug, bf16, packed=False)
    _check(d, aug, o, hT, hT_plain, False, BF16_TOL if bf16 else F32_TOL)


@pytest.mark.parametrize("B,H,T", [(5, 10, 1000), (2, 40, 640)])
def test_fwd_aug_balanced_ranges(B, H, T):
    """Balanced chunk ranges with hand-over pieces (as test_fwd_balanced_ranges), augmented."""
    d = host_chunk_inputs(760 + B * H, [T] * B, H, True, with_h0=False, packed=False)
    d["scale"] = float(gs.SCALE)
    aug = _aug(761, H)
    o, hT, _, hT_plain = _run(d, aug, True, packed=False)
    _check(d, aug, o, hT, hT_plain, False, BF16_TOL)


@pytest.mark.parametrize("bf16", [True, False])
def test_fwd_aug_varlen(bf16):
    lens = [5, 0, 200, 1, 128, 129, 300]
    H = 4
    d = host_chunk_inputs(780, lens, H, bf16, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    aug = _aug(781, H)
    o, hT, _, hT_plain = _run(d, aug, bf16, packed=True)
    _check(d, aug, o, hT, hT_plain, True, BF16_TOL if bf16 else F32_TOL)


def test_fwd_aug_zero_balance_adds_half_the_value():
    """a = 0: the page's half-strength copy, o_aug - o = v / 2 (up to the bf16 output rounding)."""
    B, H, T = 2, 4, 300
    d = host_chunk_inputs(790, [T] * B, H, True, with_h0=True, packed=False)
    d["scale"] = float(gs.SCALE)
    o, _, o_plain, _ = _run(d, np.zeros((H, 96), np.float32), True, packed=False)
    diff = flat(o, False) - flat(o_plain, False)
    assert rel_err(diff, 0.5 * np.asarray(d["v"], np.float64)) <= 2 * BF16_TOL


@pytest.mark.parametrize("bf16", [True, False])
def test_decode_aug_steps_match_oracle(bf16):
    N, H, steps = 5, 3, 6
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    dt = torch.bfloat16 if bf16 else torch.float32
    ll = gs.laplace_log_lambda(H)
    aug = _aug(800, H)
    a = torch.from_numpy(aug).cuda()
    s0 = gs.normal(800, 7, (N, H, 96, 192), 0.1)
    state = torch.from_numpy(s0).cuda()
    ref_state = s0.astype(np.float64).copy()
    for t in range(steps):
        q = rnd(gs.normal(800, 100 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        k = rnd(gs.normal(800, 101 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        v = rnd(gs.normal(800, 102 + 3 * t, (N, H, 192)))
        o = gla.gla_decode_step(torch.from_numpy(q).cuda().to(dt), torch.from_numpy(k).cuda().to(dt),
                                torch.from_numpy(v).cuda().to(dt), torch.from_numpy(ll).cuda(), state,
                                float(gs.SCALE), aug=a)
        o_ref = oracle.decode_step(q, k, v, ll, float(gs.SCALE), ref_state) + oracle.self_aug(q, k, v, aug)
        tol = BF16_TOL if bf16 else F32_TOL
        assert rel_err(o.float().cpu().numpy(), o_ref, bf16_out=bf16) <= tol, t
    assert rel_err(state.cpu().numpy(), ref_state) <= 1e-5


def test_fwd_aug_layer_workload_sampled():
    """B=8, T=2048, H=16 bf16 with aug_balance (the benchmark's augmented forward), 5 sampled
    (sequence, head) units against the oracle's forward plus its self-augmentation term."""
    from glasynth import workloads as wl
    w = wl.layer()
    g = w.device_inputs()
    aug = gs.normal(11, 9, (16, 96), 10.0)   # as the benchmark row
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale,
                              aug=torch.from_numpy(aug).cuda())
    torch.cuda.synchronize()
    for n, h in [(0, 0), (7, 15), (3, 5), (5, 14), (2, 9)]:
        u = w.host_unit(n, h)
        o_ref, hT_ref = oracle.fwd(u["q"], u["k"], u["v"], u["log_lambda"], w.scale, h0=u["h0"])
        o_ref = o_ref + oracle.self_aug(u["q"], u["k"], u["v"], aug[h:h + 1])
        og = o[n, :, h].float().cpu().numpy()
        assert rel_err(og, o_ref[:, 0], bf16_out=True) <= BF16_TOL, (n, h)
        assert rel_err(hT[n, h].cpu().numpy(), hT_ref[0, 0]) <= BF16_TOL, (n, h)

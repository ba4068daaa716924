"""GPU parity of gla_decode_step against the fp64 oracle over consecutive steps."""
import numpy as np
import pytest

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from glasynth import workloads as wl
from tests.gpu_helpers import BF16_TOL, F32_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


@pytest.mark.parametrize("bf16", [True, False])
def test_decode_steps_match_oracle(bf16):
    import torch
    N, H, steps = 5, 3, 10
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    dt = torch.bfloat16 if bf16 else torch.float32
    ll = gs.laplace_log_lambda(H)
    s0 = gs.normal(40, 7, (N, H, 96, 192), 0.1)
    state = torch.from_numpy(s0).cuda()
    ref_state = s0.astype(np.float64).copy()
    for t in range(steps):
        q = rnd(gs.normal(40, 100 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        k = rnd(gs.normal(40, 101 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        v = rnd(gs.normal(40, 102 + 3 * t, (N, H, 192)))
        o = gla.gla_decode_step(torch.from_numpy(q).cuda().to(dt), torch.from_numpy(k).cuda().to(dt),
                                torch.from_numpy(v).cuda().to(dt), torch.from_numpy(ll).cuda(), state,
                                float(gs.SCALE))
        o_ref = oracle.decode_step(q, k, v, ll, float(gs.SCALE), ref_state)
        tol = BF16_TOL if bf16 else F32_TOL
        assert rel_err(o.float().cpu().numpy(), o_ref, bf16_out=bf16) <= tol, t
    assert rel_err(state.cpu().numpy(), ref_state) <= 1e-5  # fp32 state, exact inputs


def test_decode_slots_touch_only_their_rows():
    import torch
    P, N, H = 9, 4, 2
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    pool = torch.from_numpy(gs.normal(41, 7, (P, H, 96, 192), 0.1)).cuda()
    before = pool.clone()
    slot = torch.tensor([7, 0, 3, 5], dtype=torch.int32, device="cuda")
    q = torch.from_numpy(gs.normal(41, 1, (N, H, 96), 0.1)).cuda()
    k = torch.from_numpy(gs.normal(41, 2, (N, H, 96), 0.1)).cuda()
    v = torch.from_numpy(gs.normal(41, 3, (N, H, 192))).cuda()
    o = gla.gla_decode_step(q, k, v, ll, pool, 0.5, slot=slot)
    ref_state = before.cpu().numpy()[[7, 0, 3, 5]].astype(np.float64).copy()
    o_ref = oracle.decode_step(q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy(), ll.cpu().numpy(),
                               0.5, ref_state)
    assert rel_err(o.cpu().numpy(), o_ref) <= F32_TOL
    for r in range(P):
        if r in (7, 0, 3, 5):
            assert not torch.equal(pool[r], before[r])
        else:
            assert torch.equal(pool[r], before[r])
    assert rel_err(pool[[7, 0, 3, 5]].cpu().numpy(), ref_state) <= 1e-5


def test_decode_bad_slot_is_reported_and_skipped():
    import torch
    P, N, H = 3, 2, 1
    pool = torch.zeros(P, H, 96, 192, device="cuda")
    q = torch.ones(N, H, 96, device="cuda")
    v = torch.ones(N, H, 192, device="cuda")
    slot = torch.tensor([1, 3], dtype=torch.int32, device="cuda")   # 3 is outside the pool
    gla.gla_decode_step(q, q, v, torch.zeros(H, device="cuda"), pool, 1.0, slot=slot)
    assert gla.gla_get_device_error() == -2
    assert gla.gla_get_device_error() == 0          # the word is cleared once read
    assert torch.count_nonzero(pool[0]) == 0 and torch.count_nonzero(pool[2]) == 0
    assert torch.all(pool[1] == 1.0)


def test_decode_workload_sampled_64_steps():
    """1,280 sequences x 24 layers x 16 heads (36 GB of fp32 state), 64 steps, as benchmarked;
    12 sampled (pool row, head) states are followed by the oracle through all 64 steps."""
    import torch
    w = wl.DecodeWorkload()
    state = w.device_state()
    ll = torch.from_numpy(w.log_lambda).cuda()
    rng = np.random.default_rng(2)
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, w.N, 12), rng.integers(0, w.H, 12))]
    rows += [(0, 0), (w.N - 1, w.H - 1)]
    ref = w.host_state(rows).astype(np.float64)[:, None]      # [n, 1, 96, 192]
    bufs = w.device_step(0)
    ri = torch.tensor([r for r, _ in rows], device="cuda")
    hi = torch.tensor([h for _, h in rows], device="cuda")
    worst = 0.0
    for step in range(w.steps):
        w.device_step(step, out=bufs)
        o = gla.gla_decode_step(bufs["q"], bufs["k"], bufs["v"], ll, state, w.scale)
        og = o[ri, hi].float().cpu().numpy()
        q, k, v = w.host_step(step, rows)
        lls = np.array([w.log_lambda[h] for _, h in rows], np.float32)
        o_ref = np.stack([oracle.decode_step(q[i:i + 1, None], k[i:i + 1, None], v[i:i + 1, None],
                                             lls[i:i + 1], w.scale, ref[i:i + 1])[0, 0]
                          for i in range(len(rows))])
        worst = max(worst, rel_err(og, o_ref, bf16_out=True))
    assert worst <= BF16_TOL
    sg = state[ri, hi].cpu().numpy()
    assert rel_err(sg, ref[:, 0]) <= 1e-4


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("with_aug", [False, True])
def test_decode_bf16_state_matches_oracle(bf16, with_aug):
    """bf16-stored state pool: each step against the oracle's step with the state rounded to bf16
    on write-back (the readout from the update before rounding); the pool itself against the
    oracle's rounded state (bf16 values: half a bf16 ulp of allowance).  The bar is the bf16 one
    for either i/o dtype: the kernel rounds its fp32 update and the oracle its fp64 update, so a
    value within an fp32 rounding of a bf16 tie may round the other way (one bf16 ulp, 2^-8
    relative, in that state element), which the next readouts carry; 1e-4 is the all-fp32 bar."""
    import torch
    N, H, steps = 5, 3, 10
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    dt = torch.bfloat16 if bf16 else torch.float32
    ll = gs.laplace_log_lambda(H)
    aug = gs.normal(41, 9, (H, 96), 10.0) if with_aug else None
    s0 = gs.bf16_round(gs.normal(41, 7, (N, H, 96, 192), 0.1))
    state = torch.from_numpy(s0).cuda().to(torch.bfloat16)
    ref_state = s0.astype(np.float64).copy()
    tol = BF16_TOL
    for t in range(steps):
        q = rnd(gs.normal(41, 100 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        k = rnd(gs.normal(41, 101 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        v = rnd(gs.normal(41, 102 + 3 * t, (N, H, 192)))
        o = gla.gla_decode_step(torch.from_numpy(q).cuda().to(dt), torch.from_numpy(k).cuda().to(dt),
                                torch.from_numpy(v).cuda().to(dt), torch.from_numpy(ll).cuda(), state,
                                float(gs.SCALE), aug=None if aug is None else torch.from_numpy(aug).cuda())
        o_ref = oracle.decode_step_bf16_state(q, k, v, ll, float(gs.SCALE), ref_state)
        if aug is not None:
            o_ref = o_ref + oracle.self_aug(q, k, v, aug)
        assert rel_err(o.float().cpu().numpy(), o_ref, bf16_out=bf16) <= tol, t
        assert rel_err(state.float().cpu().numpy(), ref_state, bf16_out=True) <= BF16_TOL, t


def test_decode_bf16_state_workload_sampled():
    """The benchmark's pool (1,280 sequences x 24 layers x 16 heads) stored in bf16, 16 steps as
    benchmarked; 8 sampled (pool row, head) states followed by the oracle's rounded step."""
    import torch
    w = wl.DecodeWorkload()
    state = w.device_state().to(torch.bfloat16)
    ll = torch.from_numpy(w.log_lambda).cuda()
    rng = np.random.default_rng(3)
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, w.N, 6), rng.integers(0, w.H, 6))]
    rows += [(0, 0), (w.N - 1, w.H - 1)]
    ref = oracle.round_to_bf16(w.host_state(rows).astype(np.float64))[:, None]
    bufs = w.device_step(0)
    ri = torch.tensor([r for r, _ in rows], device="cuda")
    hi = torch.tensor([h for _, h in rows], device="cuda")
    worst = 0.0
    for step in range(16):
        w.device_step(step, out=bufs)
        o = gla.gla_decode_step(bufs["q"], bufs["k"], bufs["v"], ll, state, w.scale)
        og = o[ri, hi].float().cpu().numpy()
        q, k, v = w.host_step(step, rows)
        lls = np.array([w.log_lambda[h] for _, h in rows], np.float32)
        o_ref = np.stack([oracle.decode_step_bf16_state(q[i:i + 1, None], k[i:i + 1, None], v[i:i + 1, None],
                                                        lls[i:i + 1], w.scale, ref[i:i + 1])[0, 0]
                          for i in range(len(rows))])
        worst = max(worst, rel_err(og, o_ref, bf16_out=True))
    assert worst <= BF16_TOL
    sg = state[ri, hi].float().cpu().numpy()
    assert rel_err(sg, ref[:, 0], bf16_out=True) <= BF16_TOL
    del state

"""A sweep of shapes and decays against the fp64 oracle, beyond the cases of the per-row test files.

Heads 1, 5, 17 and 64; lengths on both sides of every chunk boundary up to three chunks; many
short packed sequences (the longest-first schedule with hundreds of entries); lambda = 1 (causal
linear attention) and lambda = 0 (only the current token) exactly; a balanced persistent forward
whose chunk ranges cut pairs at odd places; the backward at the same head counts; decode steps
with a permuted pool.  Bar as everywhere: max |gpu - oracle| / rms(oracle) <= 2e-2 (bf16, half a
bf16 ulp allowed on bf16-stored outputs), <= 1e-4 (fp32)."""
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


def _fwd_check(d, bf16, packed, tol):
    g = to_device(d, bf16, packed=packed)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"],
                              cu_seqlens=g["cu_seqlens"])
    o_ref, hT_ref = oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE), h0=d["h0"],
                               cu_seqlens=d["cu"])
    on, cu = flat(o, packed), d["cu"]
    assert np.all(np.isfinite(on))
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b > a:
            e = rel_err(on[a:b], o_ref[a:b], bf16)
            assert e <= tol, f"o of sequence {n} (len {b - a}): {e:.3e}"
        e = rel_err(hT[n].cpu().numpy(), hT_ref[n])
        assert e <= tol, f"hT of sequence {n}: {e:.3e}"


@pytest.mark.parametrize("H", [1, 5, 17])
@pytest.mark.parametrize("T", [1, 2, 3, 127, 128, 129, 255, 256, 257, 383, 384, 385])
def test_fwd_heads_and_chunk_boundaries(H, T):
    d = host_chunk_inputs(1000 + 7 * H + T, [T] * 2, H, True, with_h0=True, packed=False)
    _fwd_check(d, True, False, BF16_TOL)


def test_fwd_many_heads():
    d = host_chunk_inputs(1101, [300, 129], 64, True, with_h0=True, packed=True)
    _fwd_check(d, True, True, BF16_TOL)


@pytest.mark.parametrize("bf16", [True, False])
def test_fwd_hundreds_of_short_packed_sequences(bf16):
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(0, 41, 300)]
    d = host_chunk_inputs(1102, lens, 2, bf16, with_h0=True, packed=True)
    _fwd_check(d, bf16, True, BF16_TOL if bf16 else F32_TOL)


@pytest.mark.parametrize("bf16", [True, False])
def test_fwd_lambda_one_and_zero(bf16):
    """log lambda = 0 (lambda = 1: causal linear attention, nothing decays) and -inf (lambda = 0:
    each output sees only its own token; h0 vanishes after the first token)."""
    ll = np.array([0.0, -np.inf], np.float32)
    d = host_chunk_inputs(1103, [300, 1, 129], 2, bf16, with_h0=True, packed=True, log_lambda=ll)
    _fwd_check(d, bf16, True, BF16_TOL if bf16 else F32_TOL)


def test_fwd_balanced_launch_ragged_batch():
    """17 sequences of 257 tokens, 16 heads: 272 (sequence, head) pairs of 3 chunks (the last one
    token long) cut into equal chunk ranges over the persistent CTA groups, so pairs straddle
    ranges at odd places and hand their states over through hT."""
    d = host_chunk_inputs(1104, [257] * 17, 16, True, with_h0=True, packed=False)
    _fwd_check(d, True, False, BF16_TOL)


@pytest.mark.parametrize("H", [1, 5, 17])
@pytest.mark.parametrize("bf16", [True, False])
def test_bwd_heads(H, bf16):
    lens = [385, 1, 128, 0, 130]
    d = host_chunk_inputs(1200 + H, lens, H, bf16, with_h0=True, packed=True, grad=True)
    g = to_device(d, bf16, packed=True)
    res = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], float(gs.SCALE),
                            h0=g["h0"], dhT=g["dhT"], cu_seqlens=g["cu_seqlens"])
    ref = oracle.bwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE), d["dO"], h0=d["h0"],
                     dhT=d["dhT"], cu_seqlens=d["cu"])
    tol = BF16_TOL if bf16 else F32_TOL
    cu = d["cu"]
    for name, x, r in zip(("dq", "dk", "dv"), res[:3], ref[:3]):
        xs = flat(x, True)
        for n in range(len(lens)):
            a, b = cu[n], cu[n + 1]
            if b > a:
                e = rel_err(xs[a:b], r[a:b], bf16)
                assert e <= tol, f"{name} of sequence {n}: {e:.3e}"
    assert rel_err(res[3].cpu().numpy(), ref[3]) <= tol


@pytest.mark.parametrize("bf16", [True, False])
def test_decode_permuted_pool(bf16):
    N, H, P = 257, 3, 300
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    dt = torch.bfloat16 if bf16 else torch.float32
    rng = np.random.default_rng(13)
    slot = rng.permutation(P)[:N].astype(np.int32)
    s0 = gs.normal(1300, 7, (P, H, 96, 192), 0.1)
    pool = torch.from_numpy(s0).cuda()
    ref = s0.astype(np.float64)[slot].copy()
    ll = gs.laplace_log_lambda(H)
    for t in range(3):
        q = rnd(gs.normal(1300, 10 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        k = rnd(gs.normal(1300, 11 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        v = rnd(gs.normal(1300, 12 + 3 * t, (N, H, 192)))
        o = gla.gla_decode_step(*(torch.from_numpy(x).cuda().to(dt) for x in (q, k, v)),
                                torch.from_numpy(ll).cuda(), pool, float(gs.SCALE),
                                slot=torch.from_numpy(slot).cuda())
        o_ref = oracle.decode_step(q, k, v, ll, float(gs.SCALE), ref)
        assert rel_err(o.float().cpu().numpy(), o_ref, bf16) <= (BF16_TOL if bf16 else F32_TOL), t
    assert rel_err(pool[slot].cpu().numpy(), ref) <= 1e-4
    untouched = np.setdiff1d(np.arange(P), slot)
    assert np.array_equal(pool[untouched].cpu().numpy(), s0[untouched])

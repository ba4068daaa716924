"""Pins of the fp64 oracle against facts fixed by the mathematics, not by the oracle's own code.

The oracle computes the per-token recurrence S_t = lambda S_{t-1} + k_t v_t^T, o_t = S_t^T(s q_t)
("Beyond the KV cache" blog post on Laplace 3B, section "i14 and the Laplace 3B architecture",
GLA mixer update and readout equations).  Each test below checks it against an independent
formulation: the closed-form sum, the O(T^2) decay-masked attention form, exact rational
arithmetic, the lambda = 1 and lambda = 0 reductions, chunk-size invariance, resume and varlen
invariance, linearity, and for the backward, finite differences of the forward.
"""
from fractions import Fraction

import numpy as np
import pytest

import glasynth as gs


def _rand(seed, tid, shape, sigma=1.0):
    return gs.normal(seed, tid, shape, sigma)


def _case(seed, T, H=2, dk=5, dv=7, with_h0=True):
    q = _rand(seed, 1, (T, H, dk))
    k = _rand(seed, 2, (T, H, dk))
    v = _rand(seed, 3, (T, H, dv))
    h0 = _rand(seed, 4, (1, H, dk, dv), 0.5) if with_h0 else None
    ll = np.log(np.array([0.9, 0.6, 0.99, 0.3][:H], np.float32)).astype(np.float32)
    return q, k, v, h0, ll


def _f64(x):
    return None if x is None else np.asarray(x, np.float64)


def _closed_form(q, k, v, ll, s, h0):
    """o_t = s sum_{j<=t} lam^(t-j) (q_t.k_j) v_j + s lam^(t+1) h0^T q_t (0-based t);
    hT = lam^T h0 + sum_j lam^(T-1-j) k_j v_j^T.  Written as sums, not as a recurrence."""
    q, k, v, h0 = _f64(q), _f64(k), _f64(v), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    lam = np.exp(ll.astype(np.float64))
    t = np.arange(T)
    o = np.zeros((T, H, dv))
    hT = np.zeros((1, H, dk, dv))
    for h in range(H):
        diff = t[:, None] - t[None, :]
        D = np.where(diff >= 0, lam[h] ** np.maximum(diff, 0), 0.0)
        A = (q[:, h] @ k[:, h].T) * D
        o[:, h] = s * A @ v[:, h]
        w = lam[h] ** (T - 1 - t)
        hT[0, h] = np.einsum("j,ja,jb->ab", w, k[:, h], v[:, h])
        if h0 is not None:
            o[:, h] += s * (lam[h] ** (t + 1))[:, None] * (q[:, h] @ h0[0, h])
            hT[0, h] += lam[h] ** T * h0[0, h]
    return o, hT


def _relerr(x, ref):
    ref = np.asarray(ref)
    return np.max(np.abs(np.asarray(x) - ref)) / max(np.sqrt(np.mean(ref ** 2)), 1e-300)


@pytest.mark.parametrize("T", [1, 2, 17, 64])
@pytest.mark.parametrize("with_h0", [False, True])
def test_fwd_matches_quadratic_and_closed_form(oracle_mod, T, with_h0):
    q, k, v, h0, ll = _case(10 + T, T, with_h0=with_h0)
    s = 0.37
    o, hT = oracle_mod.fwd(q, k, v, ll, s, h0=h0)
    o_ref, hT_ref = _closed_form(q, k, v, ll, s, h0)
    assert _relerr(o, o_ref) < 1e-12
    assert _relerr(hT, hT_ref) < 1e-12


def test_exact_rational_worked_example(oracle_mod):
    """T=3, H=1, dk=dv=2, lambda=1/2, s=1/2: every value is a dyadic rational, so the exact
    answer of the closed form (Fraction arithmetic) must be met to the last bit."""
    q = np.array([[1, 2], [0, 1], [3, -1]], np.float32)[:, None, :]
    k = np.array([[1, 0], [2, 1], [-1, 1]], np.float32)[:, None, :]
    v = np.array([[1, 1], [0, 2], [4, -3]], np.float32)[:, None, :]
    h0 = np.array([[1, 0], [0, 2]], np.float32)[None, None]
    lam, s = Fraction(1, 2), Fraction(1, 2)
    T = 3
    o_exact = [[Fraction(0)] * 2 for _ in range(T)]
    for t in range(T):
        for b in range(2):
            acc = Fraction(0)
            for j in range(t + 1):
                qk = sum(Fraction(int(q[t, 0, a])) * Fraction(int(k[j, 0, a])) for a in range(2))
                acc += s * lam ** (t - j) * qk * Fraction(int(v[j, 0, b]))
            acc += s * lam ** (t + 1) * sum(Fraction(int(h0[0, 0, a, b])) * Fraction(int(q[t, 0, a]))
                                            for a in range(2))
            o_exact[t][b] = acc
    hT_exact = [[lam ** T * Fraction(int(h0[0, 0, a, b])) +
                 sum(lam ** (T - 1 - j) * Fraction(int(k[j, 0, a])) * Fraction(int(v[j, 0, b]))
                     for j in range(T)) for b in range(2)] for a in range(2)]
    ll = np.array([np.log(0.5)], np.float32)
    assert np.exp(np.float64(ll[0])) == 0.5 or abs(np.exp(np.float64(ll[0])) - 0.5) < 1e-7
    o, hT = oracle_mod.fwd(q, k, v, ll, 0.5, h0=h0)
    # lambda is exp(fp32(log 0.5)) in double: not exactly 1/2, so allow its 1e-7 relative offset.
    lam64 = np.exp(np.float64(ll[0]))
    tol = 1e-6 if lam64 != 0.5 else 0.0
    for t in range(T):
        for b in range(2):
            assert abs(o[t, 0, b] - float(o_exact[t][b])) <= tol * max(1.0, abs(float(o_exact[t][b])))
    for a in range(2):
        for b in range(2):
            assert abs(hT[0, 0, a, b] - float(hT_exact[a][b])) <= tol * max(1.0, abs(float(hT_exact[a][b])))
    # A value worked by hand: lam*h0 = [[.5, 0], [0, 1]], k_1 v_1^T = [[1, 1], [0, 0]], so
    # S_1 = [[1.5, 1], [0, 1]] and o_1 = s * S_1^T q_1 = 0.5 * [1.5*1 + 0*2, 1*1 + 1*2] = [0.75, 1.5].
    assert abs(o[0, 0, 0] - 0.75) <= 1e-6 and abs(o[0, 0, 1] - 1.5) <= 1e-6


def test_lambda_one_is_causal_linear_attention(oracle_mod):
    T, H, dk, dv = 40, 1, 6, 5
    q, k, v = _rand(1, 1, (T, H, dk)), _rand(1, 2, (T, H, dk)), _rand(1, 3, (T, H, dv))
    s = 0.25
    o, hT = oracle_mod.fwd(q, k, v, np.zeros(1, np.float32), s)
    kv = np.einsum("ta,tb->tab", _f64(k[:, 0]), _f64(v[:, 0]))
    S = np.cumsum(kv, axis=0)
    o_ref = s * np.einsum("tab,ta->tb", S, _f64(q[:, 0]))
    assert _relerr(o[:, 0], o_ref) < 1e-12
    assert _relerr(hT[0, 0], S[-1]) < 1e-12


def test_lambda_zero_keeps_only_current_token(oracle_mod):
    T, H, dk, dv = 9, 1, 4, 3
    q, k, v = _rand(2, 1, (T, H, dk)), _rand(2, 2, (T, H, dk)), _rand(2, 3, (T, H, dv))
    h0 = _rand(2, 4, (1, H, dk, dv))
    s = 1.5
    o, hT = oracle_mod.fwd(q, k, v, np.array([-np.inf], np.float32), s, h0=h0)
    qk = np.sum(_f64(q[:, 0]) * _f64(k[:, 0]), axis=1)
    assert _relerr(o[:, 0], s * qk[:, None] * _f64(v[:, 0])) < 1e-14
    assert _relerr(hT[0, 0], np.outer(_f64(k[-1, 0]), _f64(v[-1, 0]))) < 1e-14


def test_single_token(oracle_mod):
    q, k, v, h0, ll = _case(3, 1, H=2)
    s = 0.8
    o, hT = oracle_mod.fwd(q, k, v, ll, s, h0=h0)
    lam = np.exp(ll.astype(np.float64))
    for h in range(2):
        S1 = lam[h] * _f64(h0[0, h]) + np.outer(_f64(k[0, h]), _f64(v[0, h]))
        assert _relerr(hT[0, h], S1) < 1e-15
        assert _relerr(o[0, h], s * S1.T @ _f64(q[0, h])) < 1e-14


def test_linear_in_v_and_h0(oracle_mod):
    q, k, v1, h1, ll = _case(4, 23)
    _, _, v2, h2, _ = _case(5, 23)
    s = 0.3
    a, b = 2.0, -0.5
    o1, s1 = oracle_mod.fwd(q, k, v1, ll, s, h0=h1)
    o2, s2 = oracle_mod.fwd(q, k, v2, ll, s, h0=h2)
    # The combined inputs are rounded to fp32 on the way in, hence the 1e-6 bound.
    o3, s3 = oracle_mod.fwd(q, k, a * v1 + b * v2, ll, s, h0=a * h1 + b * h2)
    assert _relerr(o3, a * o1 + b * o2) < 1e-6
    assert _relerr(s3, a * s1 + b * s2) < 1e-6


def test_resume_from_final_state(oracle_mod):
    q, k, v, h0, ll = _case(6, 50)
    s = 0.5
    o, hT = oracle_mod.fwd(q, k, v, ll, s, h0=h0)
    oa, ha = oracle_mod.fwd(q[:19], k[:19], v[:19], ll, s, h0=h0)
    ob, hb = oracle_mod.fwd(q[19:], k[19:], v[19:], ll, s, h0=ha)
    # ha is fp64; the second call takes fp32 h0, so compare with that rounding in mind.
    assert _relerr(np.concatenate([oa, ob]), o) < 1e-6
    assert _relerr(hb, hT) < 1e-6
    assert _relerr(oa, o[:19]) < 1e-15


@pytest.mark.parametrize("cuts", [[19], [1, 2, 30], [10, 20, 30, 40]])
def test_segment_states_chain_to_the_final_state(oracle_mod, cuts):
    """The sequence-split forward's algebra: each segment's final state from a ZERO state, U_i,
    chained as S_in[0] = h0, S_in[i+1] = lam^(L_i) S_in[i] + U_i, gives every segment's starting
    state (the last link is hT), and the segments run from those states give the unsplit
    outputs.  Checked against the closed form for hT and the unsplit oracle for the outputs."""
    q, k, v, h0, ll = _case(16, 50)
    s = 0.5
    o, hT = oracle_mod.fwd(q, k, v, ll, s, h0=h0)
    _, hT_closed = _closed_form(q, k, v, ll, s, h0)
    lam = np.exp(ll.astype(np.float64))
    bounds = [0] + list(cuts) + [50]
    S = np.asarray(h0, np.float64)
    outs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        oi, _ = oracle_mod.fwd(q[a:b], k[a:b], v[a:b], ll, s, h0=S.astype(np.float32))
        outs.append(oi)
        _, U = oracle_mod.fwd(q[a:b], k[a:b], v[a:b], ll, s)
        S = (lam ** (b - a))[None, :, None, None] * S + U
    assert _relerr(S, hT_closed) < 1e-12
    assert _relerr(np.concatenate(outs), o) < 1e-6   # (segment starts rounded to fp32 h0)


@pytest.mark.parametrize("C", [1, 7, 64, 128, 200])
def test_chunk_size_invariance(oracle_mod, C):
    q, k, v, h0, ll = _case(7, 200, dk=6, dv=4)
    s = 0.41
    o, hT = oracle_mod.fwd(q, k, v, ll, s, h0=h0)
    oc, hc = oracle_mod.fwd_chunked(q, k, v, ll, s, C, h0=h0)
    assert _relerr(oc, o) < 1e-12
    assert _relerr(hc, hT) < 1e-12


def test_chunked_form_small_decay_does_not_overflow(oracle_mod):
    """lambda = 0.5 (the pages' head 0): lambda^127 is tiny but the chunked form never divides."""
    T = 300
    q, k, v = _rand(8, 1, (T, 1, 4)), _rand(8, 2, (T, 1, 4)), _rand(8, 3, (T, 1, 3))
    ll = np.array([np.log(0.5)], np.float32)
    o, hT = oracle_mod.fwd(q, k, v, ll, 1.0)
    oc, hc = oracle_mod.fwd_chunked(q, k, v, ll, 1.0, 128)
    assert np.all(np.isfinite(oc)) and _relerr(oc, o) < 1e-12 and _relerr(hc, hT) < 1e-12


def test_varlen_equals_separate_sequences(oracle_mod):
    lens = [5, 0, 33, 1, 128, 129]
    cu = gs.cu_seqlens_of(lens)
    T = int(cu[-1])
    H, dk, dv = 2, 4, 6
    q, k, v = _rand(9, 1, (T, H, dk)), _rand(9, 2, (T, H, dk)), _rand(9, 3, (T, H, dv))
    h0 = _rand(9, 4, (len(lens), H, dk, dv), 0.1)
    ll = np.log(np.array([0.97, 0.5], np.float32))
    o, hT = oracle_mod.fwd(q, k, v, ll, 0.3, h0=h0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, hn = oracle_mod.fwd(q[a:b], k[a:b], v[a:b], ll, 0.3, h0=h0[n:n + 1])
        assert np.array_equal(o[a:b], on)
        assert np.array_equal(hT[n], hn[0])
    # An empty sequence hands its initial state through unchanged.
    assert np.array_equal(hT[1], h0[1].astype(np.float64))


def test_decode_steps_equal_prefill(oracle_mod):
    T, N, H, dk, dv = 12, 3, 2, 5, 4
    q, k, v = _rand(11, 1, (T, N, H, dk)), _rand(11, 2, (T, N, H, dk)), _rand(11, 3, (T, N, H, dv))
    h0 = _rand(11, 4, (N, H, dk, dv), 0.1)
    ll = np.log(np.array([0.9, 0.8], np.float32))
    state = h0.astype(np.float64).copy()
    outs = [oracle_mod.decode_step(q[t], k[t], v[t], ll, 0.7, state) for t in range(T)]
    for n in range(N):
        o, hT = oracle_mod.fwd(q[:, n], k[:, n], v[:, n], ll, 0.7, h0=h0[n:n + 1])
        assert _relerr(np.stack([x[n] for x in outs]), o) < 1e-13
        assert _relerr(state[n], hT[0]) < 1e-13


def test_pages_decay_schedule_endpoints():
    """Half-life schedule from 1 to 2,048 tokens: head 0 decays by one half per token and head 15
    keeps about 0.9997 (section "Decay schedule's reach")."""
    lam = np.exp(gs.halflife_log_lambda().astype(np.float64))
    assert abs(lam[0] - 0.5) < 1e-7
    assert abs(lam[15] - 0.9997) < 1e-4
    lam_w = np.exp(gs.laplace_log_lambda().astype(np.float64))
    assert abs(lam_w[0] - 0.96875) < 1e-7 and abs(lam_w[15] - (1 - 2.0 ** -12)) < 1e-7


# ---------------------------------------------------------------------------------------------
# Backward: the adjoint of the recurrence, pinned by finite differences of the forward.
# Each scalar input enters the forward linearly, so a central difference in one coordinate is
# exact up to rounding.
# ---------------------------------------------------------------------------------------------
def _loss(oracle_mod, q, k, v, ll, s, h0, dO, dhT, cu=None):
    o, hT = oracle_mod.fwd(q, k, v, ll, s, h0=h0, cu_seqlens=cu)
    return float(np.sum(o * dO) + np.sum(hT * dhT))


@pytest.mark.parametrize("lens", [[6], [3, 0, 5]])
def test_backward_matches_finite_differences(oracle_mod, lens):
    cu = gs.cu_seqlens_of(lens)
    T, H, dk, dv = int(cu[-1]), 2, 3, 4
    n = len(lens)
    rng = np.random.default_rng(0)
    # Dyadic inputs (multiples of 1/8) make the forward nearly exact in fp64.
    q = (rng.integers(-8, 9, (T, H, dk)) / 8).astype(np.float32)
    k = (rng.integers(-8, 9, (T, H, dk)) / 8).astype(np.float32)
    v = (rng.integers(-8, 9, (T, H, dv)) / 8).astype(np.float32)
    h0 = (rng.integers(-8, 9, (n, H, dk, dv)) / 8).astype(np.float32)
    dO = (rng.integers(-8, 9, (T, H, dv)) / 8).astype(np.float32)
    dhT = (rng.integers(-8, 9, (n, H, dk, dv)) / 8).astype(np.float32)
    ll = np.log(np.array([0.75, 0.5], np.float32))
    s = 0.5
    dq, dk_, dv_, dh0 = oracle_mod.bwd(q, k, v, ll, s, dO, h0=h0, dhT=dhT, cu_seqlens=cu)
    eps = 0.125
    for name, x, g in (("q", q, dq), ("k", k, dk_), ("v", v, dv_), ("h0", h0, dh0)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = dict(q=q, k=k, v=v, h0=h0)
            args[name] = xp
            lp = _loss(oracle_mod, args["q"], args["k"], args["v"], ll, s, args["h0"], dO, dhT, cu)
            args[name] = xm
            lm = _loss(oracle_mod, args["q"], args["k"], args["v"], ll, s, args["h0"], dO, dhT, cu)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-9 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


@pytest.mark.parametrize("lens", [[40], [17, 0, 33, 1]])
def test_backward_adjoint_identity_random_directions(oracle_mod, lens):
    """The forward is linear in each of q, k, v, h0 alone (the others fixed), so for a random
    direction d of one of them the loss L = <dO, o> + <dhT, hT> changes by exactly
    L(x + d) - L(x) = <dx, d>: the backward is the adjoint of the forward.  Full-size random
    directions (every element at once), real-valued inputs, longer sequences than the
    finite-difference pin."""
    cu = gs.cu_seqlens_of(lens)
    T, H, dk, dv = int(cu[-1]), 3, 5, 7
    n = len(lens)
    x = {"q": _rand(30, 1, (T, H, dk)), "k": _rand(30, 2, (T, H, dk)), "v": _rand(30, 3, (T, H, dv)),
         "h0": _rand(30, 4, (n, H, dk, dv), 0.5)}
    dO = _rand(30, 5, (T, H, dv))
    dhT = _rand(30, 6, (n, H, dk, dv), 0.3)
    ll = np.log(np.array([0.9, 0.6, 0.99], np.float32))
    s = 0.37
    grads = dict(zip(("q", "k", "v", "h0"),
                     oracle_mod.bwd(x["q"], x["k"], x["v"], ll, s, dO, h0=x["h0"], dhT=dhT, cu_seqlens=cu)))
    base = _loss(oracle_mod, x["q"], x["k"], x["v"], ll, s, x["h0"], dO, dhT, cu)
    for i, name in enumerate(("q", "k", "v", "h0")):
        d = _rand(31, 10 + i, x[name].shape)
        args = dict(x)
        shifted = (np.asarray(x[name], np.float64) + np.asarray(d, np.float64)).astype(np.float32)
        d_eff = shifted.astype(np.float64) - np.asarray(x[name], np.float64)  # the step actually taken
        args[name] = shifted
        change = _loss(oracle_mod, args["q"], args["k"], args["v"], ll, s, args["h0"], dO, dhT, cu) - base
        pred = float(np.sum(np.asarray(grads[name], np.float64) * d_eff))
        assert abs(change - pred) <= 1e-9 * max(1.0, abs(pred)), (name, change, pred)


def test_backward_lambda_one_closed_form(oracle_mod):
    """lambda = 1: G_t = dhT + s sum_{u>=t} q_u dO_u^T, so dk_t = G_t v_t and dv_t = G_t^T k_t;
    dq_t = s (h0 + sum_{j<=t} k_j v_j^T) dO_t."""
    T, H, dk, dv = 15, 1, 4, 6
    q, k, v = _rand(12, 1, (T, H, dk)), _rand(12, 2, (T, H, dk)), _rand(12, 3, (T, H, dv))
    dO, dhT = _rand(12, 5, (T, H, dv)), _rand(12, 6, (1, H, dk, dv))
    h0 = _rand(12, 4, (1, H, dk, dv))
    s = 0.6
    dq, dk_, dv_, dh0 = oracle_mod.bwd(q, k, v, np.zeros(1, np.float32), s, dO, h0=h0, dhT=dhT)
    q64, k64, v64, g64 = _f64(q[:, 0]), _f64(k[:, 0]), _f64(v[:, 0]), _f64(dO[:, 0])
    qg = s * np.einsum("ta,tb->tab", q64, g64)
    G = _f64(dhT[0, 0])[None] + np.cumsum(qg[::-1], axis=0)[::-1]
    assert _relerr(dk_[:, 0], np.einsum("tab,tb->ta", G, v64)) < 1e-12
    assert _relerr(dv_[:, 0], np.einsum("tab,ta->tb", G, k64)) < 1e-12
    assert _relerr(dh0[0, 0], G[0]) < 1e-12
    S = _f64(h0[0, 0])[None] + np.cumsum(np.einsum("ta,tb->tab", k64, v64), axis=0)
    assert _relerr(dq[:, 0], s * np.einsum("tab,tb->ta", S, g64)) < 1e-12


def test_backward_empty_sequence_passes_dhT(oracle_mod):
    cu = gs.cu_seqlens_of([0, 4])
    H, dk, dv = 1, 2, 3
    q, k, v = _rand(13, 1, (4, H, dk)), _rand(13, 2, (4, H, dk)), _rand(13, 3, (4, H, dv))
    dO, dhT = _rand(13, 5, (4, H, dv)), _rand(13, 6, (2, H, dk, dv))
    _, _, _, dh0 = oracle_mod.bwd(q, k, v, np.log(np.array([0.9], np.float32)), 1.0, dO, dhT=dhT,
                                  cu_seqlens=cu)
    assert np.array_equal(dh0[0], dhT[0].astype(np.float64))


# --- self-augmentation term -------------------------------------------------------------------
# The page (section "i14 and the Laplace 3B architecture", the paragraph after the readout) adds a
# gated copy of the value, sigmoid(q_t . (a (*) k_t)) v_t, and states that a = 0 gives a
# half-strength copy of the value.  The pins below use facts of the sigmoid and of the gate's
# arguments that do not depend on how the oracle evaluates it.

def _aug_case(seed, rows=9, H=2, dk=5, dv=7):
    q = _rand(seed, 11, (rows, H, dk))
    k = _rand(seed, 12, (rows, H, dk))
    v = _rand(seed, 13, (rows, H, dv))
    a = _rand(seed, 14, (H, dk), 0.7)
    return q, k, v, a


def test_self_aug_zero_balance_is_half_the_value(oracle_mod):
    q, k, v, _ = _aug_case(21)
    add = oracle_mod.self_aug(q, k, v, np.zeros((q.shape[1], q.shape[2]), np.float32))
    assert np.array_equal(add, 0.5 * np.asarray(v, np.float64))


def test_self_aug_opposite_balances_sum_to_the_value(oracle_mod):
    # sigmoid(x) + sigmoid(-x) = 1 for every gate argument x = q . (a * k)
    q, k, v, a = _aug_case(22)
    s = oracle_mod.self_aug(q, k, v, a) + oracle_mod.self_aug(q, k, v, -a)
    assert np.allclose(s, np.asarray(v, np.float64), rtol=0, atol=1e-14)


def test_self_aug_single_channel_saturates_by_sign_of_q_times_k(oracle_mod):
    # a = M e_c on one channel c: the gate argument is M q_c k_c, so for large M the copy is the
    # whole value where q_c k_c > 0 and nothing where q_c k_c < 0 (per row and head).
    q, k, v, _ = _aug_case(23, rows=16, H=2, dk=6, dv=3)
    for c in (0, 4):
        a = np.zeros((2, 6), np.float32)
        a[0, c] = 1e4
        a[1, (c + 1) % 6] = -1e4
        add = oracle_mod.self_aug(q, k, v, a)
        for h, ch, sign in ((0, c, 1.0), (1, (c + 1) % 6, -1.0)):
            prod = sign * np.asarray(q[:, h, ch], np.float64) * np.asarray(k[:, h, ch], np.float64)
            want = np.where(prod[:, None] > 0, np.asarray(v[:, h], np.float64), 0.0)
            keep = np.abs(prod) > 1e-2  # stay clear of the gate's middle
            assert np.allclose(add[keep, h], want[keep], rtol=0, atol=1e-12)


def test_self_aug_gate_against_exact_value(oracle_mod):
    # One row, one head, dk = 2: q . (a * k) = 0.5*2*1 + (-1)*0.25*4 = 1 - 1 = 0 -> gate 1/2;
    # and with a = (1, 0): 0.5*1*2 = 1 -> gate 1 / (1 + e^-1).
    q = np.array([[[0.5, -1.0]]], np.float32)
    k = np.array([[[2.0, 4.0]]], np.float32)
    v = np.array([[[1.0, -3.0, 8.0]]], np.float32)
    add = oracle_mod.self_aug(q, k, v, np.array([[1.0, 0.25]], np.float32))
    assert np.array_equal(add, 0.5 * np.asarray(v, np.float64))
    add = oracle_mod.self_aug(q, k, v, np.array([[1.0, 0.0]], np.float32))
    g = 1.0 / (1.0 + np.exp(-1.0))
    assert np.allclose(add, g * np.asarray(v, np.float64), rtol=1e-15, atol=0)


# --- per-tier Head RMSNorm and SiLU gate ----------------------------------------------------
# y = o / sqrt(mean(o^2) + eps) * w_tier(h) * SiLU(g) ("i14 and the Laplace 3B architecture":
# the per-head outputs pass through a Head RMSNorm per decay tier and are gated by SiLU(g_t)).

def _silu_one():
    """The gate value x with x * sigmoid(x) = 1, by bisection (SiLU is increasing on x > 0)."""
    lo, hi = 0.0, 4.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid / (1.0 + np.exp(-mid)) < 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _norm_case(seed, rows=6, H=4, dv=8):
    o = _rand(seed, 31, (rows, H, dv))
    g = _rand(seed, 32, (rows, H, dv))
    w = _rand(seed, 33, (2, dv), 0.5) + 1.0
    tier = np.array([0, 0, 1, 1][:H], np.int32)
    return o, g, w, tier


def test_norm_gate_unit_gain_and_gate_give_unit_rms(oracle_mod):
    # w = 1 and SiLU(g) = 1 everywhere, eps = 0: every output row has RMS exactly 1
    o, _, _, tier = _norm_case(41)
    g = np.full(o.shape, _silu_one(), np.float32)
    y = oracle_mod.head_norm_gate(o, g, np.ones((2, o.shape[2]), np.float32), tier, 0.0)
    assert np.allclose(np.sqrt(np.mean(y ** 2, axis=2)), 1.0, rtol=0, atol=1e-6)


def test_norm_gate_is_scale_invariant_in_o(oracle_mod):
    o, g, w, tier = _norm_case(42)
    y1 = oracle_mod.head_norm_gate(o, g, w, tier, 0.0)
    y2 = oracle_mod.head_norm_gate(np.float32(4.0) * o, g, w, tier, 0.0)
    assert np.allclose(y1, y2, rtol=1e-12, atol=0)


def test_norm_gate_zero_gate_is_zero_and_tier_gain_scales(oracle_mod):
    o, g, w, tier = _norm_case(43)
    assert np.array_equal(oracle_mod.head_norm_gate(o, np.zeros_like(g), w, tier, 1e-6), np.zeros(o.shape))
    # gains c_0 (tier 0) and c_1 (tier 1): the heads of each tier scale by their tier's gain only
    base = oracle_mod.head_norm_gate(o, g, np.ones_like(w), tier, 1e-6)
    y = oracle_mod.head_norm_gate(o, g, np.stack([np.full(w.shape[1], 2.0), np.full(w.shape[1], -3.0)]).astype(np.float32),
                                  tier, 1e-6)
    assert np.allclose(y[:, tier == 0], 2.0 * base[:, tier == 0], rtol=1e-14, atol=0)
    assert np.allclose(y[:, tier == 1], -3.0 * base[:, tier == 1], rtol=1e-14, atol=0)


def test_norm_gate_worked_example(oracle_mod):
    # o = (3, 4): mean square 12.5, eps = 0.5 -> rms 3.6055...; g = (0, 1): SiLU = (0, 1/(1+e^-1))
    o = np.array([[[3.0, 4.0]]], np.float32)
    g = np.array([[[0.0, 1.0]]], np.float32)
    w = np.array([[2.0, 0.5]], np.float32)
    y = oracle_mod.head_norm_gate(o, g, w, np.array([0], np.int32), 0.5)
    want = np.array([0.0, 4.0 / np.sqrt(13.0) * 0.5 / (1.0 + np.exp(-1.0))])
    assert np.allclose(y[0, 0], want, rtol=1e-15, atol=0)


# --- bf16-stored decode state -----------------------------------------------------------------
# Rounding to bf16 is fixed by the format (8 significant bits, ties to even); the bf16-state step
# is the fp32-state step followed by that rounding of the stored state.

def test_round_to_bf16_format_facts(oracle_mod):
    x = np.array([1.0, -3.5, 2.0 ** -40, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -9,
                  255.0, 257.0, 0.0, -0.0], np.float64)
    want = np.array([1.0, -3.5, 2.0 ** -40, 1.0, 1 + 2.0 ** -6, 1.0, 255.0, 256.0, 0.0, 0.0])
    assert np.array_equal(oracle_mod.round_to_bf16(x), want)
    r = np.asarray(gs.normal(51, 1, (4096,)), np.float64) * 1e3
    y = oracle_mod.round_to_bf16(r)
    assert np.all(np.abs(y - r) <= np.abs(r) * 2.0 ** -8 + 0)   # half an ulp of 8-bit precision
    assert np.array_equal(oracle_mod.round_to_bf16(y), y)       # idempotent
    # agrees with the input generator's independent fp32 bit-level rounding on fp32 values
    r32 = np.asarray(gs.normal(52, 1, (4096,)), np.float32)
    assert np.array_equal(oracle_mod.round_to_bf16(r32.astype(np.float64)), gs.bf16_round(r32).astype(np.float64))


def test_decode_bf16_state_is_rounded_fp32_step(oracle_mod):
    N, H = 3, 2
    q = _rand(61, 1, (N, H, 5))
    k = _rand(61, 2, (N, H, 5))
    v = _rand(61, 3, (N, H, 7))
    ll = np.log(np.array([0.9, 0.5], np.float32))
    s0 = oracle_mod.round_to_bf16(np.asarray(_rand(61, 4, (N, H, 5, 7), 0.5), np.float64))
    s_full = s0.copy()
    o_full = oracle_mod.decode_step(q, k, v, ll, 0.3, s_full)
    s_b = s0.copy()
    o_b = oracle_mod.decode_step_bf16_state(q, k, v, ll, 0.3, s_b)
    assert np.allclose(o_b, o_full, rtol=1e-14, atol=1e-15)
    assert np.array_equal(s_b, oracle_mod.round_to_bf16(s_full))


# ------------------------------------------------------------------------------------------
# MXFP8 decode state (OCP Microscaling MXFP8: E4M3 elements, one E8M0 scale per 32 elements)
# ------------------------------------------------------------------------------------------
def test_e4m3_values_match_torch_float8(oracle_mod):
    """All 256 E4M3 codes at scale 2^0 against PyTorch's float8_e4m3fn (OCP E4M3: bias 7, no
    infinities, S.1111.111 NaN, largest finite 448, subnormals m 2^-9)."""
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8).reshape(8, 32)
    x = oracle_mod.mxfp8_dequantize(codes, np.full((8, 1), 127, np.uint8))
    ref = torch.from_numpy(codes.reshape(-1).copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(x.reshape(-1)), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(x.reshape(-1)[ok], ref[ok].astype(np.float64))
    assert x.reshape(-1)[0x7E] == 448.0 and x.reshape(-1)[0x01] == 2.0 ** -9 and x.reshape(-1)[0x38] == 1.0


def test_e4m3_conversion_is_round_to_nearest_even(oracle_mod):
    """A block whose maximum sits in [256, 448] has scale 2^0, so its codes are plain E4M3
    conversions: random values, and every midpoint between neighbouring positive values (the
    ties, which go to the even mantissa), against PyTorch's float -> float8_e4m3fn."""
    torch = pytest.importorskip("torch")
    vals = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(3)
    pool = np.concatenate([mids, -mids, rng.uniform(-448, 448, 400), rng.normal(0, 1, 400) * 2.0 ** -7])
    pool = pool.astype(np.float32)
    n = (len(pool) + 30) // 31
    blocks = np.zeros((n, 32), np.float32)
    blocks[:, 0] = 300.0                           # sets the block's scale to 2^0
    blocks[:, 1:].reshape(-1)[:len(pool)] = pool
    codes, scales = oracle_mod.mxfp8_quantize(blocks)
    assert np.all(scales == 127)
    ref = torch.from_numpy(blocks).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    zero = blocks == 0                             # signed zeros may differ in the sign bit only
    assert np.array_equal(codes[~zero], ref[~zero])
    assert np.all((codes[zero] & 0x7F) == 0)


def test_mxfp8_scale_is_smallest_that_holds_the_block(oracle_mod):
    """The shared exponent is the smallest at which the block's largest magnitude fits E4M3's 448
    (never saturating): max = 2^k gives 2^(k-8) (the max encodes to 256 = 0x78); max = 1.25 2^k
    gives the same scale (320 = 0x7A); max = 1.9 2^k needs 2^(k-7) (243.2 -> 240 = 0x77).  An
    all-zero block takes the smallest scale, 2^-127."""
    for k in (-6, -1, 0, 3, 9):
        for mant, want_se, want_code in ((1.0, k - 8, 0x78), (1.25, k - 8, 0x7A), (1.9, k - 7, 0x77)):
            b = np.zeros((1, 32), np.float32)
            b[0, 5] = -mant * 2.0 ** k
            b[0, 9] = 2.0 ** (k - 3)
            codes, scales = oracle_mod.mxfp8_quantize(b)
            assert scales[0, 0] == want_se + 127, (k, mant)
            assert codes[0, 5] == 0x80 | want_code, (k, mant, hex(codes[0, 5]))
    codes, scales = oracle_mod.mxfp8_quantize(np.zeros((2, 64), np.float32))
    assert np.all(scales == 0) and np.all(codes & 0x7F == 0)


def test_mxfp8_round_trip_error_bound_and_idempotence(oracle_mod):
    x = np.concatenate([gs.normal(71, 1, (64, 192), 0.1), gs.normal(71, 2, (64, 192), 30.0),
                        gs.normal(71, 3, (64, 192), 1e-5)]).astype(np.float32)
    codes, scales = oracle_mod.mxfp8_quantize(x)
    y = oracle_mod.mxfp8_dequantize(codes, scales)
    se = scales.astype(np.int64).repeat(32, axis=1) - 127
    # half an E4M3 step: 2^-4 of the value in the normal range, 2^(se - 10) below 2^(se - 6)
    bound = np.maximum(np.abs(x.astype(np.float64)) * 2.0 ** -4, np.ldexp(1.0, se - 10))
    assert np.all(np.abs(y - x) <= bound)
    assert np.max(np.abs(y) / np.ldexp(1.0, se)) <= 448.0
    # quantising the dequantised values again reproduces them exactly (a block maximum that
    # rounded down to 224 2^se is then held as 448 2^(se-1), the same value)
    c2, s2 = oracle_mod.mxfp8_quantize(y.astype(np.float32))
    assert np.array_equal(oracle_mod.mxfp8_dequantize(c2, s2), y)


def test_decode_mxfp8_state_is_quantised_fp32_step(oracle_mod):
    """The MXFP8 step reads out exactly what the fp64 step reads out from the widened state, and
    stores the fp32-rounded update quantised block by block."""
    N, H, dk, dv = 3, 2, 5, 64
    q = _rand(62, 1, (N, H, dk))
    k = _rand(62, 2, (N, H, dk))
    v = _rand(62, 3, (N, H, dv))
    ll = np.log(np.array([0.9, 0.5], np.float32))
    codes, scales = oracle_mod.mxfp8_quantize(_rand(62, 4, (N, H, dk, dv), 0.5))
    s_full = oracle_mod.mxfp8_dequantize(codes, scales)
    o_full = oracle_mod.decode_step(q, k, v, ll, 0.3, s_full)
    c, sc = codes.copy(), scales.copy()
    o_m, pre = oracle_mod.decode_step_mxfp8_state(q, k, v, ll, 0.3, c, sc, return_pre=True)
    assert np.allclose(o_m, o_full, rtol=1e-14, atol=1e-15)
    assert np.array_equal(pre, s_full.astype(np.float32))
    want_c, want_s = oracle_mod.mxfp8_quantize(s_full.astype(np.float32))
    assert np.array_equal(c, want_c) and np.array_equal(sc, want_s)

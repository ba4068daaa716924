"""Out-of-bounds guards, checkpoint/resume and heavy-tailed inputs, on the GPU.

* Canary regions: outputs and workspaces are views into larger buffers whose head and tail
  (4 KB each) hold a known byte pattern; after each call the pattern must be intact, so a store
  past a sequence end, a partial chunk or a state tile shows up even where a later sequence's
  rows would have overwritten it.  Single-sequence calls at ragged lengths put the sequence end
  right against the tail guard.
* Packed offsets are read on the device; a decreasing pair (all offsets inside [0, T]) must be
  reported as GLA_ERR_SHAPE through the error word, with nothing written outside the buffers.
* Resume ("Optimizing inference on Trainium2": prefill writes each sequence's state page, decode
  reads it): a forward over T1 tokens, then over T2 more from h0 = its hT, equals the oracle's
  forward over T1 + T2; and a prefill followed by 16 decode steps on its hT equals the oracle's
  forward over T + 16 (fp32 and bf16 state pools).
* Inputs with planted 5.5 and 6 sigma values, forward and backward.
"""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from tests.gpu_helpers import BF16_TOL, F32_TOL, flat, host_chunk_inputs, rel_err, to_device

pytestmark = pytest.mark.gpu

PAT = 0xA5
GUARD = 4096  # bytes before and after each guarded tensor


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


class Guarded:
    """A contiguous tensor of `shape` inside a byte buffer with GUARD bytes of PAT on each side."""

    def __init__(self, shape, dtype):
        el = torch.tensor([], dtype=dtype).element_size()
        n = int(np.prod(shape))
        self.buf = torch.full((n * el + 2 * GUARD,), PAT, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + n * el].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD] == PAT).all()) and bool((self.buf[-GUARD:] == PAT).all())


def _fwd_ref(d):
    return oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE), h0=d["h0"],
                      cu_seqlens=d["cu"])


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("lens", [[5, 0, 200, 1, 128, 129, 77], [1], [63], [127], [129], [255], [300]])
def test_fwd_writes_nothing_outside_o_and_hT(bf16, lens):
    H = 3
    d = host_chunk_inputs(60 + sum(lens), lens, H, bf16, with_h0=True, packed=True)
    g = to_device(d, bf16, packed=True)
    dt = torch.bfloat16 if bf16 else torch.float32
    o = Guarded((sum(lens), H, 192), dt)
    hT = Guarded((len(lens), H, 96, 192), torch.float32)
    gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"],
                      cu_seqlens=g["cu_seqlens"], o=o.t, hT=hT.t)
    assert o.intact() and hT.intact()
    o_ref, hT_ref = _fwd_ref(d)
    tol = BF16_TOL if bf16 else F32_TOL
    cu = d["cu"]
    for n in range(len(lens)):
        if lens[n]:
            assert rel_err(flat(o.t, True)[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]], bf16) <= tol
        assert rel_err(hT.t[n].cpu().numpy(), hT_ref[n]) <= tol


def test_fwd_balanced_launch_writes_nothing_outside():
    """Fixed-length batch large enough for the balanced persistent launch (pairs split across CTA
    groups, final states handed over through hT), with a partial last chunk."""
    B, T, H = 12, 300, 16
    d = host_chunk_inputs(71, [T] * B, H, True, with_h0=True, packed=False)
    g = to_device(d, True, packed=False)
    o = Guarded((B, T, H, 192), torch.bfloat16)
    hT = Guarded((B, H, 96, 192), torch.float32)
    gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"], o=o.t,
                      hT=hT.t)
    assert o.intact() and hT.intact()
    o_ref, hT_ref = _fwd_ref(d)
    assert rel_err(flat(o.t, False), o_ref, True) <= BF16_TOL
    assert rel_err(hT.t.cpu().numpy(), hT_ref) <= BF16_TOL


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("lens", [[70, 0, 1, 200, 128], [129], [255]])
def test_bwd_writes_nothing_outside_its_outputs(bf16, lens):
    H = 2
    d = host_chunk_inputs(80 + sum(lens), lens, H, bf16, with_h0=True, packed=True, grad=True)
    g = to_device(d, bf16, packed=True)
    dt = torch.bfloat16 if bf16 else torch.float32
    Tt = sum(lens)
    dq, dk = Guarded((Tt, H, 96), dt), Guarded((Tt, H, 96), dt)
    dv = Guarded((Tt, H, 192), dt)
    dh0 = Guarded((len(lens), H, 96, 192), torch.float32)
    need = gla.gla_bwd_workspace_bytes(len(lens), Tt, H, True, 0 if bf16 else 1)
    ws = Guarded((need,), torch.uint8)
    res = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], float(gs.SCALE),
                            h0=g["h0"], dhT=g["dhT"], cu_seqlens=g["cu_seqlens"], workspace=ws.t,
                            dq=dq.t, dk=dk.t, dv=dv.t, dh0=dh0.t)
    for x in (dq, dk, dv, dh0, ws):
        assert x.intact()
    ref = oracle.bwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE), d["dO"], h0=d["h0"],
                     dhT=d["dhT"], cu_seqlens=d["cu"])
    tol = BF16_TOL if bf16 else F32_TOL
    cu = d["cu"]
    for x, r in zip(res[:3], ref[:3]):
        for n in range(len(lens)):
            if lens[n]:
                assert rel_err(flat(x, True)[cu[n]:cu[n + 1]], r[cu[n]:cu[n + 1]], bf16) <= tol
    assert rel_err(res[3].cpu().numpy(), ref[3]) <= tol


def test_split_forward_writes_nothing_outside_outputs_and_workspace():
    lens, H = [700, 0, 1, 389], 2
    d = host_chunk_inputs(90, lens, H, True, with_h0=True, packed=True)
    g = to_device(d, True, packed=True)
    import ctypes
    cu_h = np.asarray(d["cu"], np.int32)
    need = gla.load_library().gla_split_workspace_bytes(cu_h.ctypes.data_as(ctypes.c_void_p), len(lens),
                                                        H, 1)
    ws = Guarded((need,), torch.uint8)
    o = Guarded((sum(lens), H, 192), torch.bfloat16)
    hT = Guarded((len(lens), H, 96, 192), torch.float32)
    gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, seg_chunks=1,
                            scale=float(gs.SCALE), h0=g["h0"], o=o.t, hT=hT.t, workspace=ws.t)
    assert o.intact() and hT.intact() and ws.intact()
    o_ref, hT_ref = _fwd_ref(d)
    cu = d["cu"]
    for n in range(len(lens)):
        if lens[n]:
            assert rel_err(flat(o.t, True)[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]], True) <= BF16_TOL
    assert rel_err(hT.t.cpu().numpy(), hT_ref) <= BF16_TOL


@pytest.mark.parametrize("state_bf16", [False, True])
def test_decode_writes_nothing_outside_pool_and_o(state_bf16):
    N, H, P = 5, 3, 9
    sdt = torch.bfloat16 if state_bf16 else torch.float32
    pool = Guarded((P, H, 96, 192), sdt)
    pool.t.copy_(torch.from_numpy(gs.normal(95, 7, (P, H, 96, 192), 0.1)).to(sdt))
    o = Guarded((N, H, 192), torch.bfloat16)
    slot = torch.tensor([8, 0, 3, 7, 1], dtype=torch.int32, device="cuda")
    q = torch.from_numpy(gs.normal(95, 1, (N, H, 96), 0.1)).cuda().to(torch.bfloat16)
    k = torch.from_numpy(gs.normal(95, 2, (N, H, 96), 0.1)).cuda().to(torch.bfloat16)
    v = torch.from_numpy(gs.normal(95, 3, (N, H, 192))).cuda().to(torch.bfloat16)
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    untouched = pool.t[[2, 4, 5, 6]].clone()
    gla.gla_decode_step(q, k, v, ll, pool.t, float(gs.SCALE), slot=slot, o=o.t)
    assert pool.intact() and o.intact()
    assert torch.equal(pool.t[[2, 4, 5, 6]], untouched)   # rows no slot names stay as they were


def _decode_inputs(seed, N, H, dt):
    q = torch.from_numpy(gs.normal(seed, 1, (N, H, 96), 0.1)).cuda().to(dt)
    k = torch.from_numpy(gs.normal(seed, 2, (N, H, 96), 0.1)).cuda().to(dt)
    v = torch.from_numpy(gs.normal(seed, 3, (N, H, 192))).cuda().to(dt)
    return q, k, v, torch.from_numpy(gs.laplace_log_lambda(H)).cuda()


@pytest.mark.parametrize("bf16", [True, False])
def test_decode_norm_gate_writes_nothing_outside_pool_and_y(bf16):
    N, H, P = 5, 6, 9
    dt = torch.bfloat16 if bf16 else torch.float32
    pool = Guarded((P, H, 96, 192), torch.float32)
    pool.t.copy_(torch.from_numpy(gs.normal(96, 7, (P, H, 96, 192), 0.1)))
    y = Guarded((N, H, 192), dt)
    slot = torch.tensor([8, 0, 3, 7, 1], dtype=torch.int32, device="cuda")
    q, k, v, ll = _decode_inputs(96, N, H, dt)
    g = torch.from_numpy(gs.normal(96, 4, (N, H, 192), 2.0)).cuda().to(dt)
    wt = (1.0 + torch.from_numpy(gs.normal(96, 5, (3, 192), 0.3))).cuda()
    tier = torch.tensor([0, 0, 1, 1, 2, 2], dtype=torch.int32, device="cuda")
    untouched = pool.t[[2, 4, 5, 6]].clone()
    gla.gla_decode_step_norm_gate(q, k, v, ll, pool.t, g, wt, tier, scale=float(gs.SCALE), slot=slot, y=y.t)
    assert pool.intact() and y.intact()
    assert torch.equal(pool.t[[2, 4, 5, 6]], untouched)
    assert bool(torch.isfinite(y.t.float()).all())


def test_mxfp8_conversions_write_nothing_outside():
    """Seven state rows (84 blocks of 16 codes, 42 scale bytes: the scale array ends off a
    16-byte boundary) to MXFP8 and back."""
    rows = 7
    x = torch.from_numpy(gs.normal(97, 1, (rows, 192), 0.3)).cuda()
    codes, scales = Guarded((rows, 192), torch.uint8), Guarded((rows, 6), torch.uint8)
    back = Guarded((rows, 192), torch.float32)
    gla.gla_state_to_mxfp8(x, codes.t, scales.t)
    gla.gla_state_from_mxfp8(codes.t, scales.t, back.t)
    assert codes.intact() and scales.intact() and back.intact()
    assert bool(torch.isfinite(back.t).all())
    assert float((back.t - x).abs().max()) <= float(x.abs().max()) * 2 ** -3


def test_mxfp8_decode_writes_nothing_outside_pool_and_o():
    N, H, P = 5, 3, 9
    codes = Guarded((P, H, 96, 192), torch.uint8)
    scales = Guarded((P, H, 96, 6), torch.uint8)
    gla.gla_state_to_mxfp8(torch.from_numpy(gs.normal(98, 7, (P, H, 96, 192), 0.1)).cuda(), codes.t, scales.t)
    o = Guarded((N, H, 192), torch.bfloat16)
    slot = torch.tensor([8, 0, 3, 7, 1], dtype=torch.int32, device="cuda")
    q, k, v, ll = _decode_inputs(98, N, H, torch.bfloat16)
    keep_c, keep_s = codes.t[[2, 4, 5, 6]].clone(), scales.t[[2, 4, 5, 6]].clone()
    gla.gla_decode_step_mxfp8_state(q, k, v, ll, codes.t, scales.t, float(gs.SCALE), slot=slot, o=o.t)
    assert codes.intact() and scales.intact() and o.intact()
    assert torch.equal(codes.t[[2, 4, 5, 6]], keep_c) and torch.equal(scales.t[[2, 4, 5, 6]], keep_s)


@pytest.mark.parametrize("bf16", [True, False])
def test_head_norm_gate_writes_nothing_outside_y(bf16):
    rows, H = 3, 5
    dt = torch.bfloat16 if bf16 else torch.float32
    o = torch.from_numpy(gs.normal(99, 1, (rows, H, 192))).cuda().to(dt)
    g = torch.from_numpy(gs.normal(99, 2, (rows, H, 192), 2.0)).cuda().to(dt)
    wt = (1.0 + torch.from_numpy(gs.normal(99, 3, (2, 192), 0.3))).cuda()
    tier = torch.tensor([0, 1, 1, 0, 1], dtype=torch.int32, device="cuda")
    y = Guarded((rows, H, 192), dt)
    gla.gla_head_norm_gate(o, g, wt, tier, y=y.t)
    assert y.intact() and bool(torch.isfinite(y.t.float()).all())


def test_decreasing_offsets_are_reported_and_stay_in_bounds():
    """cu_seqlens = [0, 200, 100, 300] (every offset inside [0, T = 300], the middle pair
    decreasing): the kernels clamp sequence 1 to an empty range, record GLA_ERR_SHAPE, and write
    nothing outside the buffers; the next valid call on the same context is exact again."""
    H = 2
    lens_ok = [200, 0, 100]
    d = host_chunk_inputs(33, lens_ok, H, True, with_h0=True, packed=True, grad=True)
    g = to_device(d, True, packed=True)
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device="cuda")
    for bf16 in (True, False):
        dt = torch.bfloat16 if bf16 else torch.float32
        q, k, v, dO = (g[x].to(dt) for x in ("q", "k", "v", "dO"))
        o = Guarded((300, H, 192), dt)
        hT = Guarded((3, H, 96, 192), torch.float32)
        gla.gla_chunk_fwd(q, k, v, g["log_lambda"], float(gs.SCALE), h0=g["h0"], cu_seqlens=bad, o=o.t,
                          hT=hT.t)
        assert o.intact() and hT.intact()
        assert gla.gla_get_device_error() == -2
        dq, dk = Guarded((300, H, 96), dt), Guarded((300, H, 96), dt)
        dv, dh0 = Guarded((300, H, 192), dt), Guarded((3, H, 96, 192), torch.float32)
        gla.gla_chunk_bwd(q, k, v, g["log_lambda"], dO, float(gs.SCALE), h0=g["h0"], dhT=g["dhT"],
                          cu_seqlens=bad, dq=dq.t, dk=dk.t, dv=dv.t, dh0=dh0.t)
        for x in (dq, dk, dv, dh0):
            assert x.intact()
        assert gla.gla_get_device_error() == -2
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"],
                              cu_seqlens=g["cu_seqlens"])
    assert gla.gla_get_device_error() == 0
    o_ref, hT_ref = _fwd_ref(d)
    assert rel_err(flat(o, True)[:200], o_ref[:200], True) <= BF16_TOL
    assert rel_err(hT.cpu().numpy(), hT_ref) <= BF16_TOL


# ------------------------------------------------------------------------------------------
# resume
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("bf16", [True, False])
def test_forward_resumed_from_its_final_state(bf16):
    B, T1, T2, H = 2, 300, 257, 3
    d = host_chunk_inputs(44, [T1 + T2] * B, H, bf16, with_h0=True, packed=False)
    g = to_device(d, bf16, packed=False)
    o1, hT1 = gla.gla_chunk_fwd(g["q"][:, :T1].contiguous(), g["k"][:, :T1].contiguous(),
                                g["v"][:, :T1].contiguous(), g["log_lambda"], float(gs.SCALE), h0=g["h0"])
    o2, hT2 = gla.gla_chunk_fwd(g["q"][:, T1:].contiguous(), g["k"][:, T1:].contiguous(),
                                g["v"][:, T1:].contiguous(), g["log_lambda"], float(gs.SCALE), h0=hT1)
    o_ref, hT_ref = _fwd_ref(d)
    o_ref = o_ref.reshape(B, T1 + T2, H, 192)
    tol = BF16_TOL if bf16 else F32_TOL
    for n in range(B):
        assert rel_err(o1[n].float().cpu().numpy(), o_ref[n, :T1], bf16) <= tol
        assert rel_err(o2[n].float().cpu().numpy(), o_ref[n, T1:], bf16) <= tol
        assert rel_err(hT2[n].cpu().numpy(), hT_ref[n]) <= tol


@pytest.mark.parametrize("state_bf16", [False, True])
@pytest.mark.parametrize("bf16", [True, False])
def test_decode_continues_a_prefill(bf16, state_bf16):
    """Prefill T tokens with the chunked forward, then 16 decode steps on its final states (the
    pool): each step's output against the oracle's forward over T + 16 tokens at that position,
    and the pool after the last step against its final state.  A bf16 pool is compared with the
    oracle's bf16-state steps started from the oracle prefill's state rounded to bf16."""
    B, T, H, steps = 3, 290, 2, 16
    d = host_chunk_inputs(55, [T + steps] * B, H, bf16, with_h0=True, packed=False)
    g = to_device(d, bf16, packed=False)
    _, pool = gla.gla_chunk_fwd(g["q"][:, :T].contiguous(), g["k"][:, :T].contiguous(),
                                g["v"][:, :T].contiguous(), g["log_lambda"], float(gs.SCALE), h0=g["h0"])
    if state_bf16:
        pool = pool.to(torch.bfloat16)
    o_ref, hT_ref = _fwd_ref(d)
    o_ref = o_ref.reshape(B, T + steps, H, 192)
    q4 = d["q"].reshape(B, T + steps, H, 96)
    k4 = d["k"].reshape(B, T + steps, H, 96)
    v4 = d["v"].reshape(B, T + steps, H, 192)
    if state_bf16:
        _, hT_pre = oracle.fwd(q4[:, :T].reshape(-1, H, 96), k4[:, :T].reshape(-1, H, 96),
                               v4[:, :T].reshape(-1, H, 192), d["log_lambda"], float(gs.SCALE),
                               h0=d["h0"], cu_seqlens=gs.cu_seqlens_of([T] * B))
        ref_state = oracle.round_to_bf16(hT_pre)
    tol = BF16_TOL if (bf16 or state_bf16) else F32_TOL
    for t in range(steps):
        q, k, v = (g[x][:, T + t].contiguous() for x in ("q", "k", "v"))
        o = gla.gla_decode_step(q, k, v, g["log_lambda"], pool, float(gs.SCALE))
        if state_bf16:
            ref = oracle.decode_step_bf16_state(q4[:, T + t], k4[:, T + t], v4[:, T + t],
                                                d["log_lambda"], float(gs.SCALE), ref_state)
        else:
            ref = o_ref[:, T + t]
        assert rel_err(o.float().cpu().numpy(), ref, bf16) <= tol, t
    if state_bf16:
        assert rel_err(pool.float().cpu().numpy(), ref_state, True) <= tol
    else:
        assert rel_err(pool.cpu().numpy(), hT_ref) <= tol


# ------------------------------------------------------------------------------------------
# planted outliers
# ------------------------------------------------------------------------------------------
def _plant(x, sigma, seed, count=24):
    """Sets `count` seeded positions of x to +-5.5 or +-6 sigma (bf16-exact multiples)."""
    rng = np.random.default_rng(seed)
    flat_x = x.reshape(-1)
    idx = rng.choice(flat_x.size, count, replace=False)
    flat_x[idx] = gs.bf16_round((rng.choice([5.5, 6.0], count) * rng.choice([-1.0, 1.0], count)
                                 * sigma).astype(np.float32))
    return x


def test_planted_outliers_forward_and_backward():
    lens, H = [300, 129, 64], 3
    d = host_chunk_inputs(66, lens, H, True, with_h0=True, packed=True, grad=True)
    qs = float(1 / np.sqrt(96))
    for name, sig, seed in (("q", qs, 1), ("k", qs, 2), ("v", 1.0, 3), ("dO", 1.0, 4)):
        _plant(d[name], sig, seed)
    g = to_device(d, True, packed=True)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"],
                              cu_seqlens=g["cu_seqlens"])
    res = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], float(gs.SCALE),
                            h0=g["h0"], dhT=g["dhT"], cu_seqlens=g["cu_seqlens"])
    o_ref, hT_ref = _fwd_ref(d)
    ref = oracle.bwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE), d["dO"], h0=d["h0"],
                     dhT=d["dhT"], cu_seqlens=d["cu"])
    cu = d["cu"]
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        assert rel_err(flat(o, True)[a:b], o_ref[a:b], True) <= BF16_TOL, ("o", n)
        for name, x, r in zip(("dq", "dk", "dv"), res[:3], ref[:3]):
            e = rel_err(flat(x, True)[a:b], r[a:b], True)
            assert e <= BF16_TOL, f"{name} of sequence {n}: {e:.3e}"
    assert rel_err(hT.cpu().numpy(), hT_ref) <= BF16_TOL
    assert rel_err(res[3].cpu().numpy(), ref[3]) <= BF16_TOL

"""GPU parity of gla_chunk_fwd / gla_chunk_bwd against the fp64 oracle, element by element.

Small cases are compared in full, per sequence (each sequence against the oracle run on its own
inputs); the full-size workloads are compared on sampled (sequence, head) units that the oracle
computes one by one.  Bar: max |gpu - oracle| / rms(oracle) per output tensor <= 2e-2 in bf16
mode (bf16 operands, fp32 accumulation and state), <= 1e-4 in fp32 mode."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from glasynth import workloads as wl
from tests.gpu_helpers import (BF16_TOL, F32_TOL, flat, host_chunk_inputs, rel_err, to_device,
                               within_one_bf16_rounding)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


def _check_fwd(d, o_gpu, hT_gpu, packed, tol):
    bf = o_gpu.dtype == torch.bfloat16
    o_ref, hT_ref = oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], d["scale"], h0=d["h0"],
                               cu_seqlens=d["cu"])
    o = flat(o_gpu, packed)
    assert np.all(np.isfinite(o))
    cu = d["cu"]
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b > a:
            e = rel_err(o[a:b], o_ref[a:b], bf)
            assert e <= tol, f"o of sequence {n} (len {b - a}): {e:.3e}"
        if hT_gpu is not None:
            e = rel_err(hT_gpu[n].cpu().numpy(), hT_ref[n])
            assert e <= tol, f"hT of sequence {n}: {e:.3e}"


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 127, 128, 129, 255, 300])
def test_fwd_fixed_length(bf16, T):
    B, H = 2, 3
    d = host_chunk_inputs(100 + T, [T] * B, H, bf16, with_h0=(T % 2 == 1), packed=False)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=False)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"])
    _check_fwd(d, o, hT, False, BF16_TOL if bf16 else F32_TOL)


def test_fwd_tiny_workload_fp32():
    """The tiny fp32 workload (B=1, T=256, H=2, lambda in {0.97, 0.999}, seed 0), all outputs."""
    w = wl.tiny()
    import torch
    g = w.device_inputs()
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale)
    torch.cuda.synchronize()
    for h in range(w.H):
        u = w.host_unit(0, h)
        o_ref, hT_ref = oracle.fwd(u["q"], u["k"], u["v"], u["log_lambda"], w.scale)
        assert rel_err(o[0, :, h].cpu().numpy(), o_ref[:, 0]) <= F32_TOL
        assert rel_err(hT[0, h].cpu().numpy(), hT_ref[0, 0]) <= F32_TOL


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("lens", [[5, 0, 200, 1, 128, 129, 77], [300], [0, 0], [1000, 3, 257]])
def test_fwd_varlen_per_sequence(bf16, lens):
    H = 2
    d = host_chunk_inputs(7 + len(lens), lens, H, bf16, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=True)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"],
                              cu_seqlens=g["cu_seqlens"])
    _check_fwd(d, o, hT, True, BF16_TOL if bf16 else F32_TOL)
    # a length-0 sequence passes h0 through unchanged
    for n, L in enumerate(lens):
        if L == 0:
            assert np.array_equal(hT[n].cpu().numpy(), d["h0"][n])


def test_fwd_varlen_equals_fixed_bitwise():
    """The same kernel on a packed batch of equal lengths and on the [B, T] layout gives the same
    bits: the schedule changes which CTA runs when, never the arithmetic."""
    import torch
    lens = [200] * 4
    d = host_chunk_inputs(5, lens, 2, True, with_h0=True, packed=True)
    g = to_device(d, True, packed=True)
    o1, h1 = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 0.1, h0=g["h0"],
                               cu_seqlens=g["cu_seqlens"])
    o2, h2 = gla.gla_chunk_fwd(g["q"].view(4, 200, 2, 96), g["k"].view(4, 200, 2, 96),
                               g["v"].view(4, 200, 2, 192), g["log_lambda"], 0.1, h0=g["h0"])
    assert torch.equal(o1.view(4, 200, 2, 192), o2) and torch.equal(h1, h2)


def test_fwd_output_alignment_16_vs_32_bitwise():
    """Output rows are written with 32-byte stores when o is 32-byte aligned and with 16-byte stores
    when it is only 16-byte aligned (the minimum the ABI asks for); both give the same bits."""
    import torch
    B, T, H = 2, 200, 2
    d = host_chunk_inputs(11, [T] * B, H, True, with_h0=True, packed=False)
    g = to_device(d, True, packed=False)
    n = B * T * H * 192
    o32 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    raw = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    o16 = raw[8:].view(n)  # 16 bytes past a 256-byte aligned allocation
    assert o32.data_ptr() % 32 == 0 and o16.data_ptr() % 32 == 16
    o32, o16 = o32.view(B, T, H, 192), o16.view(B, T, H, 192)
    gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 0.1, h0=g["h0"], o=o32)
    gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 0.1, h0=g["h0"], o=o16)
    assert torch.equal(o32, o16)


def test_fwd_pages_decay_schedule_no_overflow():
    """Half-life schedule 1..2048 tokens: head 0 has lambda = 0.5, so lambda^127 is 2^-127."""
    H = 16
    d = host_chunk_inputs(9, [384] * 2, H, True, with_h0=True, packed=False,
                          log_lambda=gs.halflife_log_lambda(H))
    d["scale"] = float(gs.SCALE)
    g = to_device(d, True, packed=False)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"])
    _check_fwd(d, o, hT, False, BF16_TOL)


def test_fwd_empty_and_degenerate():
    import torch
    ll = torch.zeros(2, device="cuda")
    q = torch.zeros(3, 0, 2, 96, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(3, 0, 2, 192, device="cuda", dtype=torch.bfloat16)
    h0 = torch.randn(3, 2, 96, 192, device="cuda")
    o, hT = gla.gla_chunk_fwd(q, q, v, ll, 0.1, h0=h0)
    assert o.numel() == 0 and torch.equal(hT, h0)
    o, hT = gla.gla_chunk_fwd(q, q, v, ll, 0.1)
    assert torch.count_nonzero(hT) == 0
    q = torch.zeros(0, 4, 2, 96, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(0, 4, 2, 192, device="cuda", dtype=torch.bfloat16)
    o, hT = gla.gla_chunk_fwd(q, q, v, ll, 0.1)
    assert hT.shape == (0, 2, 96, 192)


def test_fwd_persistent_units_with_h0():
    """Equal-length batches run persistent CTAs (one per SM) that take several (sequence, head,
    d_v tile) units each: 7 x 16 x 3 = 336 units put two or three units on every CTA, so the
    per-unit decay tables, initial-state loads and final-state stores rotate through their
    buffers.  T = 300 also ends every unit on a partial chunk.  Compared in full."""
    B, H, T = 7, 16, 300
    d = host_chunk_inputs(31, [T] * B, H, True, with_h0=True, packed=False)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, True, packed=False)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"])
    _check_fwd(d, o, hT, False, BF16_TOL)


@pytest.mark.parametrize("B,H,T", [(5, 10, 1000), (1, 51, 200), (3, 17, 129), (2, 40, 640)])
def test_fwd_balanced_ranges(B, H, T):
    """Equal-length batches with an hT output and at least as many (sequence, head) pairs as
    groups of three SMs run balanced chunk ranges: pairs straddling two ranges are split into a
    tail piece and a head piece handed over through the pair's hT tile.  These shapes put the
    range boundaries at varied chunk offsets, including ranges about one pair long, a single
    sequence with many heads, and partial last chunks.  Compared in full."""
    d = host_chunk_inputs(40 + B * H + T, [T] * B, H, True, with_h0=(T % 2 == 1), packed=False)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, True, packed=False)
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"])
    _check_fwd(d, o, hT, False, BF16_TOL)


def test_fwd_persistent_empty_sequences():
    """T = 0 with many units per persistent CTA: every unit passes its initial state through as
    the final state, bit for bit."""
    import torch
    B, H = 7, 16
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    q = torch.zeros(B, 0, H, 96, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(B, 0, H, 192, device="cuda", dtype=torch.bfloat16)
    h0 = torch.randn(B, H, 96, 192, device="cuda")
    o, hT = gla.gla_chunk_fwd(q, q, v, ll, 0.1, h0=h0)
    assert o.numel() == 0 and torch.equal(hT, h0)


def _sampled_units(w, units, o, hT, tol):
    import torch
    torch.cuda.synchronize()
    for n, h in units:
        u = w.host_unit(n, h)
        o_ref, hT_ref = oracle.fwd(u["q"], u["k"], u["v"], u["log_lambda"], w.scale, h0=u["h0"])
        a, b = int(w.cu[n]), int(w.cu[n + 1])
        og = (o[a:b, h] if w.packed else o[n, :, h]).float().cpu().numpy()
        assert np.all(np.isfinite(og))
        assert rel_err(og, o_ref[:, 0], bf16_out=True) <= tol, (n, h)
        assert rel_err(hT[n, h].cpu().numpy(), hT_ref[0, 0]) <= tol, (n, h)


def test_fwd_layer_workload_sampled():
    """B=8, T=2048, H=16 bf16 (the benchmark's forward launch), 6 sampled (sequence, head) units."""
    w = wl.layer()
    g = w.device_inputs()
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale)
    _sampled_units(w, [(0, 0), (7, 15), (3, 5), (5, 10), (1, 1), (6, 14)], o, hT, BF16_TOL)


def test_fwd_layer_workload_sampled_fp32_mode():
    """The all-fp32 mode at the benchmark's shapes (its fwd_fp32 launch: the layer workload's values
    in fp32), 4 sampled units at the fp32 bar."""
    w = wl.layer()
    g = w.device_inputs()
    q, k, v = (g[x].float() for x in ("q", "k", "v"))
    o, hT = gla.gla_chunk_fwd(q, k, v, g["log_lambda"], w.scale)
    torch.cuda.synchronize()
    for n, h in [(0, 0), (7, 15), (2, 9), (5, 4)]:
        u = w.host_unit(n, h)
        o_ref, hT_ref = oracle.fwd(u["q"], u["k"], u["v"], u["log_lambda"], w.scale, h0=u["h0"])
        og = o[n, :, h].cpu().numpy()
        assert np.all(np.isfinite(og))
        assert rel_err(og, o_ref[:, 0]) <= F32_TOL, (n, h)
        assert rel_err(hT[n, h].cpu().numpy(), hT_ref[0, 0]) <= F32_TOL, (n, h)


def test_fwd_varlen_workload_sampled():
    """32 packed sequences, lengths U[128, 16384], h0 ~ N(0, 0.1): longest, shortest, others."""
    w = wl.varlen()
    g = w.device_inputs()
    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale, h0=g["h0"],
                              cu_seqlens=g["cu_seqlens"])
    lens = np.array(w.lengths)
    units = [(int(lens.argmax()), 15), (int(lens.argmin()), 0), (0, 7), (31, 3), (17, 11)]
    _sampled_units(w, units, o, hT, BF16_TOL)


# ------------------------------------------------------------------------------------------
# Backward
# ------------------------------------------------------------------------------------------
def _check_bwd(d, res, packed, tol):
    dq, dk, dv, dh0 = res
    bf = dq.dtype == torch.bfloat16
    ref = oracle.bwd(d["q"], d["k"], d["v"], d["log_lambda"], d["scale"], d["dO"], h0=d["h0"],
                     dhT=d["dhT"], cu_seqlens=d["cu"])
    cu = d["cu"]
    got = [flat(dq, packed), flat(dk, packed), flat(dv, packed)]
    for name, x, r in zip(("dq", "dk", "dv"), got, ref[:3]):
        assert np.all(np.isfinite(x)), name
        for n in range(len(cu) - 1):
            a, b = cu[n], cu[n + 1]
            if b > a:
                e = rel_err(x[a:b], r[a:b], bf)
                assert e <= tol, f"{name} of sequence {n}: {e:.3e}"
    for n in range(len(cu) - 1):
        e = rel_err(dh0[n].cpu().numpy(), ref[3][n])
        assert e <= tol, f"dh0 of sequence {n}: {e:.3e}"


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T", [1, 64, 129, 300])
def test_bwd_fixed_length(bf16, T):
    d = host_chunk_inputs(200 + T, [T] * 2, 2, bf16, with_h0=True, packed=False, grad=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=False)
    res = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], d["scale"], h0=g["h0"],
                            dhT=g["dhT"])
    _check_bwd(d, res, False, BF16_TOL if bf16 else F32_TOL)


@pytest.mark.parametrize("bf16", [True, False])
def test_bwd_varlen_per_sequence(bf16):
    lens = [70, 0, 1, 200, 128]
    d = host_chunk_inputs(31, lens, 2, bf16, with_h0=True, packed=True, grad=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=True)
    res = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], d["scale"], h0=g["h0"],
                            dhT=g["dhT"], cu_seqlens=g["cu_seqlens"])
    _check_bwd(d, res, True, BF16_TOL if bf16 else F32_TOL)
    assert np.array_equal(res[3][1].cpu().numpy(), d["dhT"][1])


def test_bwd_layer_workload_sampled():
    """Backward at B=8, T=2048, H=16 bf16 with dO ~ N(0,1), dhT ~ N(0, 0.01); sampled units."""
    import torch
    w = wl.layer(with_grad=True)
    g = w.device_inputs()
    dq, dk, dv, dh0 = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], w.scale,
                                        dhT=g["dhT"])
    torch.cuda.synchronize()
    for n, h in [(0, 0), (7, 15), (4, 8)]:
        u = w.host_unit(n, h)
        ref = oracle.bwd(u["q"], u["k"], u["v"], u["log_lambda"], w.scale, u["dO"], dhT=u["dhT"])
        for x, r in zip((dq, dk, dv), ref[:3]):
            xs = x[n, :, h].float().cpu().numpy()
            assert np.all(np.isfinite(xs))
            assert rel_err(xs, r[:, 0], bf16_out=True) <= BF16_TOL, (n, h)
        assert rel_err(dh0[n, h].cpu().numpy(), ref[3][0, 0]) <= BF16_TOL, (n, h)


def test_bwd_layer_workload_sampled_fp32_mode():
    """The all-fp32 mode's backward at the benchmark's shapes (its bwd_fp32 launch), sampled units
    at the fp32 bar."""
    w = wl.layer(with_grad=True)
    g = w.device_inputs()
    q, k, v, dO = (g[x].float() for x in ("q", "k", "v", "dO"))
    dq, dk, dv, dh0 = gla.gla_chunk_bwd(q, k, v, g["log_lambda"], dO, w.scale, dhT=g["dhT"])
    torch.cuda.synchronize()
    for n, h in [(0, 0), (7, 15), (3, 6)]:
        u = w.host_unit(n, h)
        ref = oracle.bwd(u["q"], u["k"], u["v"], u["log_lambda"], w.scale, u["dO"], dhT=u["dhT"])
        for name, x, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref[:3]):
            xs = x[n, :, h].cpu().numpy()
            assert np.all(np.isfinite(xs))
            assert rel_err(xs, r[:, 0]) <= F32_TOL, (name, n, h)
        assert rel_err(dh0[n, h].cpu().numpy(), ref[3][0, 0]) <= F32_TOL, (n, h)


@pytest.mark.parametrize("bf16", [True, False])
def test_bwd_pages_decay_schedule(bf16):
    """Backward with the half-life schedule (lambda from 0.5 to 0.9997) on ragged lengths."""
    H = 16
    lens = [384, 257]
    d = host_chunk_inputs(91, lens, H, bf16, with_h0=True, packed=True, grad=True,
                          log_lambda=gs.halflife_log_lambda(H))
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=True)
    res = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], d["scale"], h0=g["h0"],
                            dhT=g["dhT"], cu_seqlens=g["cu_seqlens"])
    _check_bwd(d, res, True, BF16_TOL if bf16 else F32_TOL)


def test_run_to_run_reproducibility():
    """The forward (balanced persistent launch with hand-overs, and packed varlen), dv and dh0 of
    the backward, and the decode step give the same bits on every run; dq and dk (fp32 partial sums
    added in arrival order) differ by at most one bf16 rounding, element by element."""
    d = host_chunk_inputs(901, [300] * 12, 16, True, with_h0=True, packed=False, grad=True)
    g = to_device(d, True, packed=False)
    s = float(gs.SCALE)
    runs = [gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], s, h0=g["h0"]) for _ in range(3)]
    for o, hT in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(hT, runs[0][1])
    dv_ = host_chunk_inputs(902, [5, 0, 200, 1, 128, 129, 77], 3, True, with_h0=True, packed=True)
    gv = to_device(dv_, True, packed=True)
    runs = [gla.gla_chunk_fwd(gv["q"], gv["k"], gv["v"], gv["log_lambda"], s, h0=gv["h0"],
                              cu_seqlens=gv["cu_seqlens"]) for _ in range(3)]
    for o, hT in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(hT, runs[0][1])
    grads = [gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], s, h0=g["h0"], dhT=g["dhT"])
             for _ in range(3)]
    for r in grads[1:]:
        assert torch.equal(r[2], grads[0][2]) and torch.equal(r[3], grads[0][3])
        for x, y in zip(r[:2], grads[0][:2]):
            assert within_one_bf16_rounding(x.float().cpu().numpy(), y.float().cpu().numpy())
    pool0 = torch.from_numpy(gs.normal(903, 7, (5, 16, 96, 192), 0.1)).cuda()
    q1, k1 = (torch.from_numpy(gs.normal(903, i, (5, 16, 96), 0.1)).cuda().to(torch.bfloat16) for i in (1, 2))
    v1 = torch.from_numpy(gs.normal(903, 3, (5, 16, 192))).cuda().to(torch.bfloat16)
    outs = []
    for _ in range(2):
        pool = pool0.clone()
        outs.append((gla.gla_decode_step(q1, k1, v1, g["log_lambda"], pool, s), pool))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])

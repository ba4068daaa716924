"""GPU parity of the MXFP8 decode state (gla_decode_step_mxfp8_state, gla_state_to_mxfp8,
gla_state_from_mxfp8) against the oracle.

Quantisation and dequantisation are integer work on fp32 inputs: GPU codes and scales must equal
the oracle's bit for bit, and dequantised values exactly.  In the decode step the quantisation
decisions are taken on each side's own fp32 update (the kernel's fp32 fma chain, the oracle's
fp64 update rounded to fp32), which can differ in the last fp32 bit; a code or scale may then
differ where the oracle's value lies within that distance of an E4M3 rounding boundary (or the
block maximum of a scale boundary).  Each such difference is checked to be one of those near-ties,
and the test then writes the oracle's state into the GPU pool, so that every step starts from the
same state on both sides and its readout is compared at the parity bar."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from glasynth import workloads as wl
from tests.gpu_helpers import BF16_TOL, F32_TOL, rel_err

pytestmark = pytest.mark.gpu

# The two sides' fp32 updates differ by at most a few fp32 roundings of the operands: the
# kernel's lambda is fp32 (the oracle's fp64), its update one fma, the oracle's the fp64 update
# rounded once; so |x_gpu - x_oracle| <= 2^-22 (|lambda s| + |k v|), s the widened state before
# the step.  A code or scale may be decided apart only within that distance of a boundary
# (checked with room to spare).
NEAR = 2.0 ** -20


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


def _e4m3_table():
    codes = np.arange(128, dtype=np.uint8).reshape(4, 32)
    return oracle.mxfp8_dequantize(codes, np.full((4, 1), 127, np.uint8)).reshape(-1)


E4M3 = _e4m3_table()   # magnitudes of codes 0x00 .. 0x7F (0x7F NaN)


def _mixed_rows(seed, rows):
    """fp32 rows of 192 with blocks of many magnitudes, zeros, ties and tiny values."""
    x = gs.normal(seed, 1, (rows, 192), 1.0).astype(np.float64)
    x *= np.exp2(np.round(gs.normal(seed, 2, (rows, 6), 8.0))).repeat(32, axis=1)
    x[0] = 0.0
    x[1, :32] = -0.0
    x[2, :32] = gs.normal(seed, 3, (32,), 1e-39)              # fp32 subnormals
    mids = (E4M3[1:0x7F] + E4M3[:0x7E]) / 2                   # ties at scale 2^0
    x[3, :] = 0.0
    x[3, 0] = 300.0
    x[3, 1:32] = mids[::4][:31]
    x[4, :32] = 448.0 * 2.0 ** -20                            # block maximum exactly 448 2^se
    x[5, :32] = 1.75 * 2.0 ** 3                               # significand exactly 1.75
    x[5, 32:64] = np.nextafter(np.float32(1.75 * 2.0 ** 3), np.float32(100))
    return x.astype(np.float32)


def test_quantise_matches_oracle_bitwise_and_dequantise_is_exact():
    x = _mixed_rows(81, 4096)
    codes, scales = gla.gla_state_to_mxfp8(torch.from_numpy(x).cuda())
    c_ref, s_ref = oracle.mxfp8_quantize(x)
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    y = gla.gla_state_from_mxfp8(codes, scales)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), oracle.mxfp8_dequantize(c_ref, s_ref))


def test_dequantise_all_codes_and_scales():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, (512, 192)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                    # no NaN codes
    scales = rng.integers(0, 247, (512, 6)).astype(np.uint8)  # 448 2^(b - 127) within fp32
    y = gla.gla_state_from_mxfp8(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    assert np.array_equal(y.cpu().numpy().astype(np.float64), oracle.mxfp8_dequantize(codes, scales))


def _operand_size(s_prev, k, v, log_lambda):
    """|lambda s| + |k v| per state element ([N, H, dk, dv]): the scale of the update's rounding."""
    lam = np.exp(np.asarray(log_lambda, np.float64))[None, :, None, None]
    return (np.abs(lam * s_prev) + np.abs(np.asarray(k, np.float64)[..., :, None]
                                          * np.asarray(v, np.float64)[..., None, :]))


def _near_tie_differences(c_gpu, s_gpu, c_ref, s_ref, pre, size):
    """Differences between the GPU's and the oracle's quantised update, each checked to be a
    decision taken apart within NEAR * size of a boundary of the oracle's fp32 value `pre`;
    returns their count."""
    n = 0
    cols = c_ref.shape[-1]
    cg, cr = c_gpu.reshape(-1, cols), c_ref.reshape(-1, cols)
    sg, sr = s_gpu.reshape(-1, cols // 32), s_ref.reshape(-1, cols // 32)
    x = pre.reshape(-1, cols).astype(np.float64)
    sz = size.reshape(-1, cols)
    for r, b in zip(*np.nonzero(sg != sr)):                 # scale decided apart: the block maximum
        blk = np.abs(x[r, 32 * b:32 * b + 32])              # at a power of two or at 1.75 2^e
        m = np.max(blk)
        e = np.floor(np.log2(m))
        dist = min(abs(m - 2.0 ** e), abs(m - 1.75 * 2.0 ** e), abs(m - 2.0 ** (e + 1)))
        assert dist <= NEAR * np.max(sz[r, 32 * b:32 * b + 32]), (r, b, m)
        n += 1
    same_scale = (sg == sr).repeat(32, axis=1)
    for r, c in zip(*np.nonzero((cg != cr) & same_scale)):
        a, b = int(cg[r, c]), int(cr[r, c])
        if (a & 0x7F) == (b & 0x7F) == 0:                   # +0 against -0 of a value that rounds to zero
            continue
        assert ((a ^ b) & 0x80) == 0, (r, c, hex(a), hex(b))
        assert abs((a & 0x7F) - (b & 0x7F)) == 1, (r, c, hex(a), hex(b))
        scl = 2.0 ** (int(sr[r, c // 32]) - 127)
        mid = (E4M3[a & 0x7F] + E4M3[b & 0x7F]) / 2 * scl
        assert abs(abs(x[r, c]) - mid) <= NEAR * sz[r, c], (r, c)
        n += 1
    return n


def _run_steps(N, H, P, steps, bf16, aug_on, seed):
    rnd = gs.bf16_round if bf16 else (lambda x: x)
    dt = torch.bfloat16 if bf16 else torch.float32
    ll = gs.laplace_log_lambda(H)
    aug = gs.normal(seed, 9, (H, 96), 10.0) if aug_on else None
    slot_h = (np.arange(N) * 3 + 1) % P
    c0, s0 = oracle.mxfp8_quantize(gs.normal(seed, 7, (P, H, 96, 192), 0.1))
    codes, scales = torch.from_numpy(c0).cuda(), torch.from_numpy(s0).cuda()
    tol = BF16_TOL if bf16 else F32_TOL
    flips = 0
    for t in range(steps):
        q = rnd(gs.normal(seed, 100 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        k = rnd(gs.normal(seed, 101 + 3 * t, (N, H, 96), 1 / np.sqrt(96)))
        v = rnd(gs.normal(seed, 102 + 3 * t, (N, H, 192)))
        ref_c = codes.cpu().numpy()[slot_h].copy()
        ref_s = scales.cpu().numpy()[slot_h].copy()
        size = _operand_size(oracle.mxfp8_dequantize(ref_c, ref_s), k, v, ll)
        o = gla.gla_decode_step_mxfp8_state(*(torch.from_numpy(x).cuda().to(dt) for x in (q, k, v)),
                                            torch.from_numpy(ll).cuda(), codes, scales, float(gs.SCALE),
                                            slot=torch.from_numpy(slot_h.astype(np.int32)).cuda(),
                                            aug=None if aug is None else torch.from_numpy(aug).cuda())
        o_ref, pre = oracle.decode_step_mxfp8_state(q, k, v, ll, float(gs.SCALE), ref_c, ref_s, return_pre=True)
        if aug is not None:
            o_ref = o_ref + oracle.self_aug(q, k, v, aug)
        e = rel_err(o.float().cpu().numpy(), o_ref, bf16)
        assert e <= tol, f"step {t}: {e:.3e}"
        flips += _near_tie_differences(codes.cpu().numpy()[slot_h], scales.cpu().numpy()[slot_h], ref_c, ref_s,
                                       pre, size)
        idx = torch.from_numpy(slot_h).cuda()
        codes[idx] = torch.from_numpy(ref_c).cuda()       # both sides start the next step alike
        scales[idx] = torch.from_numpy(ref_s).cuda()
    untouched = [r for r in range(P) if r not in slot_h]
    assert np.array_equal(codes.cpu().numpy()[untouched], c0[untouched])
    return flips, steps * N * H * 96 * 192


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("aug_on", [False, True])
def test_decode_mxfp8_matches_oracle_step_by_step(bf16, aug_on):
    flips, total = _run_steps(5, 3, 8, 10, bf16, aug_on, 83)
    assert flips <= 1e-3 * total


def test_decode_mxfp8_bad_slot_is_reported_and_skipped():
    H = 2
    c0, s0 = oracle.mxfp8_quantize(gs.normal(84, 7, (3, H, 96, 192), 0.1))
    codes, scales = torch.from_numpy(c0).cuda(), torch.from_numpy(s0).cuda()
    q = k = torch.full((2, H, 96), 0.1, dtype=torch.bfloat16, device="cuda")
    v = torch.ones((2, H, 192), dtype=torch.bfloat16, device="cuda")
    slot = torch.tensor([5, 1], dtype=torch.int32, device="cuda")
    gla.gla_decode_step_mxfp8_state(q, k, v, torch.zeros(H, device="cuda"), codes, scales, slot=slot)
    assert gla.gla_get_device_error() == -2
    assert np.array_equal(codes.cpu().numpy()[[0, 2]], c0[[0, 2]])
    assert not np.array_equal(codes.cpu().numpy()[1], c0[1])


def test_decode_mxfp8_workload_sampled():
    """The benchmark's pool (1,280 sequences x 24 layers x 16 heads) quantised on the GPU from its
    fp32 states (bit-exact against the oracle's quantisation on the sampled states), then 16
    steps; 10 sampled (pool row, head) states compared with the oracle's step at every step."""
    w = wl.DecodeWorkload()
    rows_total = w.N * w.H * 96
    codes = torch.empty((w.N, w.H, 96, 192), dtype=torch.uint8, device="cuda")
    scales = torch.empty((w.N, w.H, 96, 6), dtype=torch.uint8, device="cuda")
    chunk = 2048   # pool rows per conversion (2048 x 16 x 72 KB = 2.4 GB of fp32 at a time)
    from glasynth.device import normal as dnormal
    for r0 in range(0, w.N, chunk):
        r1 = min(w.N, r0 + chunk)
        x = dnormal((r1 - r0, w.H, 96, 192), w.seed, gs.TID["state"], w.state_sigma, torch.float32,
                    start=r0 * w.H * 96 * 192)
        gla.gla_state_to_mxfp8(x, codes[r0:r1], scales[r0:r1])
        del x
    assert rows_total == codes.numel() // 192
    ll = torch.from_numpy(w.log_lambda).cuda()
    rng = np.random.default_rng(8)
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, w.N, 8), rng.integers(0, w.H, 8))]
    rows += [(0, 0), (w.N - 1, w.H - 1)]
    ri = torch.tensor([r for r, _ in rows], device="cuda")
    hi = torch.tensor([h for _, h in rows], device="cuda")
    ref_c, ref_s = oracle.mxfp8_quantize(w.host_state(rows))       # [n, 96, 192], [n, 96, 6]
    assert np.array_equal(codes[ri, hi].cpu().numpy(), ref_c)
    assert np.array_equal(scales[ri, hi].cpu().numpy(), ref_s)
    bufs = w.device_step(0)
    worst, flips = 0.0, 0
    for step in range(16):
        w.device_step(step, out=bufs)
        o = gla.gla_decode_step_mxfp8_state(bufs["q"], bufs["k"], bufs["v"], ll, codes, scales, w.scale)
        og = o[ri, hi].float().cpu().numpy()
        q, k, v = w.host_step(step, rows)
        lls = np.array([w.log_lambda[h] for _, h in rows], np.float32)
        c_step, s_step = ref_c[:, None].copy(), ref_s[:, None].copy()
        size = np.stack([_operand_size(oracle.mxfp8_dequantize(c_step[i:i + 1], s_step[i:i + 1]),
                                       k[i:i + 1, None], v[i:i + 1, None], lls[i:i + 1])[0, 0]
                         for i in range(len(rows))])
        o_ref = np.zeros((len(rows), 192))
        pre = np.zeros((len(rows), 1, 96, 192), np.float32)
        for i in range(len(rows)):
            ci, si = c_step[i:i + 1].copy(), s_step[i:i + 1].copy()
            oi, pi = oracle.decode_step_mxfp8_state(q[i:i + 1, None], k[i:i + 1, None], v[i:i + 1, None],
                                                    lls[i:i + 1], w.scale, ci, si, return_pre=True)
            o_ref[i], pre[i] = oi[0, 0], pi[0]
            c_step[i], s_step[i] = ci[0], si[0]
        worst = max(worst, rel_err(og, o_ref, bf16_out=True))
        flips += _near_tie_differences(codes[ri, hi].cpu().numpy(), scales[ri, hi].cpu().numpy(),
                                       c_step[:, 0], s_step[:, 0], pre[:, 0], size)
        ref_c, ref_s = c_step[:, 0], s_step[:, 0]
        codes[ri, hi] = torch.from_numpy(ref_c).cuda()
        scales[ri, hi] = torch.from_numpy(ref_s).cuda()
    assert worst <= BF16_TOL, worst
    assert flips <= 1e-3 * 16 * len(rows) * 96 * 192

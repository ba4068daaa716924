"""GPU parity of the sequence-split forward (gla_chunk_fwd_split) against the fp64 oracle run on
the unsplit sequences: the segments, the scan that chains their states and the second pass must
reproduce the per-token recurrence ("Beyond the KV cache", section "Challenge 1": only the
state's advance between chunks is sequential).  Bars as for gla_chunk_fwd."""
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


def _check(d, o, hT, tol, aug=None):
    bf = o.dtype == torch.bfloat16
    o_ref, hT_ref = oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], d["scale"], h0=d["h0"],
                               cu_seqlens=d["cu"])
    if aug is not None:
        o_ref = o_ref + oracle.self_aug(d["q"], d["k"], d["v"], aug)
    x = flat(o, True)
    cu = d["cu"]
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b > a:
            e = rel_err(x[a:b], o_ref[a:b], bf)
            assert e <= tol, f"o of sequence {n} (len {b - a}): {e:.3e}"
        e = rel_err(hT[n].cpu().numpy(), hT_ref[n])
        assert e <= tol, f"hT of sequence {n}: {e:.3e}"


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("seg_chunks", [1, 3, 16])
def test_split_long_sequence(bf16, seg_chunks):
    lens = [5000]
    d = host_chunk_inputs(1100 + seg_chunks, lens, 4, bf16, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=True)
    o, hT = gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, seg_chunks=seg_chunks,
                                    scale=d["scale"], h0=g["h0"])
    _check(d, o, hT, BF16_TOL if bf16 else F32_TOL)


@pytest.mark.parametrize("bf16", [True, False])
def test_split_mixed_lengths_with_empty_sequences(bf16):
    lens = [300, 0, 1000, 129, 1, 0, 256]
    d = host_chunk_inputs(1120, lens, 3, bf16, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=True)
    o, hT = gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, seg_chunks=2,
                                    scale=d["scale"], h0=g["h0"])
    _check(d, o, hT, BF16_TOL if bf16 else F32_TOL)


def test_split_without_h0_with_aug():
    lens = [2000, 700]
    H = 5
    d = host_chunk_inputs(1130, lens, H, True, with_h0=False, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, True, packed=True)
    aug = gs.normal(1131, 9, (H, 96), 10.0)
    o, hT = gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, seg_chunks=4,
                                    scale=d["scale"], aug=torch.from_numpy(aug).cuda())
    _check(d, o, hT, BF16_TOL, aug=aug)


def test_split_one_segment_per_sequence_matches_plain_forward_bitwise():
    """Segments as long as the sequences: step 1's states are the sequences' final states and
    step 3 is the plain forward; the outputs equal gla_chunk_fwd's bit for bit."""
    lens = [700, 129, 2048]
    d = host_chunk_inputs(1140, lens, 4, True, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, True, packed=True)
    o, hT = gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, seg_chunks=16,
                                    scale=d["scale"], h0=g["h0"])
    o2, hT2 = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"],
                                cu_seqlens=g["cu_seqlens"])
    assert torch.equal(o, o2)
    assert rel_err(hT.cpu().numpy(), hT2.cpu().numpy()) <= 1e-6


def test_split_automatic_segment_length_cuts_a_long_sequence():
    """seg_chunks = 0 on one long sequence with short ones: the library cuts it (the chosen length
    is below the longest sequence's 157 chunks) and the result still matches the oracle."""
    lens = [20000, 300, 0]
    H = 4
    L = gla.gla_split_choose_seg_chunks(lens, H)
    assert 1 <= L < 157
    d = host_chunk_inputs(1150, lens, H, True, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, True, packed=True)
    o, hT = gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, scale=d["scale"],
                                    h0=g["h0"])
    _check(d, o, hT, BF16_TOL)


@pytest.mark.parametrize("bf16", [True, False])
def test_split_automatic_on_a_balanced_batch_is_the_plain_forward(bf16):
    """seg_chunks = 0 where no split pays off (more units than SMs several times over, none much
    longer than the rest): the call is gla_chunk_fwd, bit for bit."""
    lens = [640] * 10 + [300, 129, 0]
    assert gla.gla_split_choose_seg_chunks(lens, 8) == 0
    d = host_chunk_inputs(1160, lens, 8, bf16, with_h0=True, packed=True)
    d["scale"] = float(gs.SCALE)
    g = to_device(d, bf16, packed=True)
    o, hT = gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, scale=d["scale"],
                                    h0=g["h0"])
    o2, hT2 = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"],
                                cu_seqlens=g["cu_seqlens"])
    assert torch.equal(o, o2)
    assert torch.equal(hT, hT2)

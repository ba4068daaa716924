"""gla_chunk_fwd_host: the forward on host buffers, copies pipelined with the compute inside the
library.  Its results must equal the device call's on the same values, bit for bit: pieces of
whole sequences run the same kernels on the same rows, and parts of a sequence cut at chunk
boundaries start from exactly the state the uncut scan carries across the cut."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    yield
    assert gla.gla_get_device_error() == 0


def _inputs(seed, B, T, H, bf16, pinned=True):
    dt = torch.bfloat16 if bf16 else torch.float32
    q = torch.from_numpy(gs.normal(seed, 1, (B, T, H, 96), 96 ** -0.5)).to(dt)
    k = torch.from_numpy(gs.normal(seed, 2, (B, T, H, 96), 96 ** -0.5)).to(dt)
    v = torch.from_numpy(gs.normal(seed, 3, (B, T, H, 192))).to(dt)
    h0 = torch.from_numpy(gs.normal(seed, 4, (B, H, 96, 192), 0.1))
    if pinned:
        q, k, v, h0 = (x.pin_memory() for x in (q, k, v, h0))
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    return q, k, v, h0, ll


def _device_call(q, k, v, h0, ll):
    o, hT = gla.gla_chunk_fwd(q.cuda(), k.cuda(), v.cuda(), ll, float(gs.SCALE),
                              h0=None if h0 is None else h0.cuda())
    return o.cpu(), hT.cpu()


@pytest.mark.parametrize("pieces", [1, 2, 4, 8, 16, 64])
def test_pieces_equal_the_device_call(pieces):
    """4 sequences of 512 tokens: sub-batches (1, 2, 4 pieces), one piece per sequence (4), two
    or four 128-token-multiple parts per sequence (8, 16), and a request for 16 parts per sequence
    that 512 tokens cannot give in whole chunks (64: four parts)."""
    q, k, v, h0, ll = _inputs(31, 4, 512, 4, True)
    o, hT = gla.gla_chunk_fwd_host(q, k, v, ll, float(gs.SCALE), h0=h0, pieces=pieces)
    torch.cuda.synchronize()
    o_ref, hT_ref = _device_call(q, k, v, h0, ll)
    assert torch.equal(o, o_ref)
    assert torch.equal(hT, hT_ref)


def test_fp32_mode_and_no_h0():
    q, k, v, _, ll = _inputs(32, 2, 256, 2, False)
    o, hT = gla.gla_chunk_fwd_host(q, k, v, ll, float(gs.SCALE), pieces=4)
    torch.cuda.synchronize()
    o_ref, hT_ref = _device_call(q, k, v, None, ll)
    assert torch.equal(o, o_ref) and torch.equal(hT, hT_ref)


def test_ragged_length_keeps_sequences_whole_and_skips_hT():
    """T = 300 is no whole number of chunks for any cut: eight pieces requested for two
    sequences run as two whole-sequence pieces; no final state requested."""
    q, k, v, h0, ll = _inputs(33, 2, 300, 3, True)
    o, hT = gla.gla_chunk_fwd_host(q, k, v, ll, float(gs.SCALE), h0=h0, pieces=8, output_final_state=False)
    torch.cuda.synchronize()
    assert hT is None
    o_ref, _ = _device_call(q, k, v, h0, ll)
    assert torch.equal(o, o_ref)


def test_pageable_host_memory():
    q, k, v, h0, ll = _inputs(34, 2, 256, 2, True, pinned=False)
    o = torch.empty(v.shape, dtype=v.dtype)
    hT = torch.empty((2, 2, 96, 192), dtype=torch.float32)
    gla.gla_chunk_fwd_host(q, k, v, ll, float(gs.SCALE), h0=h0, o=o, hT=hT, pieces=4)
    torch.cuda.synchronize()
    o_ref, hT_ref = _device_call(q, k, v, h0, ll)
    assert torch.equal(o, o_ref) and torch.equal(hT, hT_ref)


def test_back_to_back_calls_reuse_the_pipeline():
    """Calls queued one after another on the stream (the events and streams of the pipeline are
    reused) each give their own batch's results."""
    a = _inputs(35, 2, 256, 2, True)
    b = _inputs(36, 2, 256, 2, True)
    ra = gla.gla_chunk_fwd_host(a[0], a[1], a[2], a[4], float(gs.SCALE), h0=a[3], pieces=4)
    rb = gla.gla_chunk_fwd_host(b[0], b[1], b[2], b[4], float(gs.SCALE), h0=b[3], pieces=4)
    torch.cuda.synchronize()
    for (o, hT), x in ((ra, a), (rb, b)):
        o_ref, hT_ref = _device_call(x[0], x[1], x[2], x[3], x[4])
        assert torch.equal(o, o_ref) and torch.equal(hT, hT_ref)
    assert np.isfinite(ra[0].float().numpy()).all()


def test_zero_length_passes_h0_through():
    """T = 0: no rows to copy (the empty host tensors may have no storage at all); each final
    state is its initial state."""
    q, k, v, h0, ll = _inputs(37, 3, 0, 2, True)
    o, hT = gla.gla_chunk_fwd_host(q, k, v, ll, float(gs.SCALE), h0=h0, pieces=4)
    torch.cuda.synchronize()
    assert o.shape == (3, 0, 2, 192)
    assert torch.equal(hT, h0)

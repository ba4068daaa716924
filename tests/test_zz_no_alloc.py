"""The allocation-free forward, gla_chunk_fwd_noalloc, against gla_chunk_fwd.

Some callers cannot allocate device memory per call: a serving engine that gives all device memory
to its own pool at start-up, for one.  For them the library keeps the packed-sequence schedule in
a fixed device array of its own instead of a caller workspace.  These tests call the new entry
point through the C ABI, with every output preallocated here, and check it against the existing
entry point on two consecutive calls (the second reuses the array the first left behind).  This
file is collected last on purpose, so that a run stopping at the first failure has run the rest."""
import ctypes

import numpy as np
import pytest

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
from tests.gpu_helpers import BF16_TOL, host_chunk_inputs, rel_err, to_device

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, g, d, o, hT):
    import torch
    P = ctypes.c_void_p
    n_seq = len(d["cu"]) - 1
    T, H = g["q"].shape[0], g["q"].shape[1]
    rc = lib.gla_chunk_fwd_noalloc(P(g["q"].data_ptr()), P(g["k"].data_ptr()), P(g["v"].data_ptr()),
                                   P(g["log_lambda"].data_ptr()), P(g["h0"].data_ptr()),
                                   float(gs.SCALE), P(o.data_ptr()), P(hT.data_ptr()),
                                   P(g["cu_seqlens"].data_ptr()), n_seq, T, H, 96, 192, 0,
                                   P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, gla.gla_status_string(rc)


def test_noalloc_matches_workspace_forward_on_two_calls():
    import torch
    lib = gla.load_library()
    cases = [([200, 1, 0, 513, 128, 77], 3, 11), ([1000, 129, 5], 2, 12)]
    for lens, H, seed in cases:
        d = host_chunk_inputs(seed, lens, H, True, with_h0=True, packed=True)
        g = to_device(d, True, packed=True)
        o_ref, hT_ref = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE),
                                          h0=g["h0"], cu_seqlens=g["cu_seqlens"])
        o = torch.empty_like(o_ref)
        hT = torch.empty_like(hT_ref)
        _call_noalloc(lib, g, d, o, hT)
        torch.cuda.synchronize()
        assert gla.gla_get_device_error() == 0
        cu = d["cu"]
        on, orf = o.float().cpu().numpy(), o_ref.float().cpu().numpy()
        for n in range(len(cu) - 1):
            a, b = cu[n], cu[n + 1]
            if b > a:
                assert rel_err(on[a:b], orf[a:b], bf16_out=True) <= BF16_TOL
            assert rel_err(hT[n].cpu().numpy(), hT_ref[n].cpu().numpy()) <= BF16_TOL


def test_noalloc_rejects_too_many_sequences_before_launch():
    lib = gla.load_library()
    P = ctypes.c_void_p
    A = 0x10000
    n = gla.NOALLOC_MAX_SEQS + 1
    rc = lib.gla_chunk_fwd_noalloc(P(A), P(A), P(A), P(A), None, 0.1, P(A), None, P(A), n, 4 * n, 2,
                                   96, 192, 0, None)
    assert rc == -6  # GLA_ERR_WORKSPACE: the library's fixed array is too small

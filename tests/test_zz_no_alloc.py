"""The allocation-free forward, gla_chunk_fwd_noalloc, against gla_chunk_fwd and the oracle.

Some callers cannot allocate device memory per call: a serving engine that gives all device memory
to its own pool at start-up, for one.  For them the library keeps the packed-sequence schedule in
a fixed device array of its own instead of a caller workspace.  These tests call the new entry
point through the C ABI, with every output preallocated here, and check it against the existing
entry point on two consecutive calls (the second reuses the array the first left behind): bit for
bit, since both run the same kernels with the same schedule, and against the fp64 oracle at the
parity bar.  Cases: bf16 and fp32 modes, packed sequences (cu_seqlens) and fixed-length batches
(no cu_seqlens: the balanced persistent launch, which needs no schedule array).  This file is
collected last on purpose, so that a run stopping at the first failure has run the rest."""
import ctypes

import numpy as np
import pytest

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from tests.gpu_helpers import BF16_TOL, F32_TOL, flat, host_chunk_inputs, rel_err, to_device

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, g, d, o, hT, packed, bf16):
    import torch
    P = ctypes.c_void_p
    n_seq = len(d["cu"]) - 1
    T = g["q"].shape[0] if packed else g["q"].shape[1]
    H = g["q"].shape[-2]
    h0 = P(g["h0"].data_ptr()) if g["h0"] is not None else None
    cu = P(g["cu_seqlens"].data_ptr()) if packed else None
    rc = lib.gla_chunk_fwd_noalloc(P(g["q"].data_ptr()), P(g["k"].data_ptr()), P(g["v"].data_ptr()),
                                   P(g["log_lambda"].data_ptr()), h0, float(gs.SCALE),
                                   P(o.data_ptr()), P(hT.data_ptr()), cu, n_seq, T, H, 96, 192,
                                   0 if bf16 else 1, P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, gla.gla_status_string(rc)


# (lengths, H, seed, packed): ragged packed batches with empty sequences, and fixed-length batches
# (H = 16, 12 sequences: at least as many (sequence, head) pairs as groups of three SMs, so the
# fixed-length forward takes its balanced launch)
CASES = [([200, 1, 0, 513, 128, 77], 3, 11, True), ([1000, 129, 5], 2, 12, True),
         ([300] * 12, 16, 13, False)]


@pytest.mark.parametrize("bf16", [True, False])
def test_noalloc_matches_workspace_forward_on_two_calls(bf16):
    import torch
    lib = gla.load_library()
    tol = BF16_TOL if bf16 else F32_TOL
    for lens, H, seed, packed in CASES:
        d = host_chunk_inputs(seed, lens, H, bf16, with_h0=True, packed=packed)
        g = to_device(d, bf16, packed=packed)
        o_ws, hT_ws = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE),
                                        h0=g["h0"], cu_seqlens=g["cu_seqlens"])
        o = torch.empty_like(o_ws)
        hT = torch.empty_like(hT_ws)
        _call_noalloc(lib, g, d, o, hT, packed, bf16)
        torch.cuda.synchronize()
        assert gla.gla_get_device_error() == 0
        assert torch.equal(o, o_ws), f"o differs from gla_chunk_fwd ({lens}, H={H})"
        assert torch.equal(hT, hT_ws), f"hT differs from gla_chunk_fwd ({lens}, H={H})"
        o_ref, hT_ref = oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE),
                                   h0=d["h0"], cu_seqlens=d["cu"])
        on, cu = flat(o, packed), d["cu"]
        for n in range(len(cu) - 1):
            a, b = cu[n], cu[n + 1]
            if b > a:
                e = rel_err(on[a:b], o_ref[a:b], bf16)
                assert e <= tol, f"o of sequence {n}: {e:.3e}"
            e = rel_err(hT[n].cpu().numpy(), hT_ref[n])
            assert e <= tol, f"hT of sequence {n}: {e:.3e}"


def test_noalloc_rejects_too_many_sequences_before_launch():
    lib = gla.load_library()
    P = ctypes.c_void_p
    A = 0x10000
    n = gla.NOALLOC_MAX_SEQS + 1
    rc = lib.gla_chunk_fwd_noalloc(P(A), P(A), P(A), P(A), None, 0.1, P(A), None, P(A), n, 4 * n, 2,
                                   96, 192, 0, None)
    assert rc == -6  # GLA_ERR_WORKSPACE: the library's fixed array is too small

"""The bounded-wait path of the tensor-core scans on a GPU, without a fault: a wait limit of 1 us
makes the first wait that genuinely blocks (a load, an MMA) give up.  The kernel must then drain
its copies and MMAs, free tensor memory, return, and report GLA_ERR_TIMEOUT through the device
error word; the context stays usable and the next call, with the default limit, is correct."""
import pytest

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
import oracle
from tests.gpu_helpers import BF16_TOL, flat, host_chunk_inputs, rel_err, to_device

pytestmark = pytest.mark.gpu

GLA_ERR_TIMEOUT = -8
DEFAULT_LIMIT_NS = 2_000_000_000


def _inputs():
    d = host_chunk_inputs(21, [2048], 1, True, with_h0=True, packed=False)
    d["scale"] = float(gs.SCALE)
    return d, to_device(d, True, packed=False)


def test_short_wait_limit_reports_timeout_and_the_context_survives():
    import torch
    gla.load_library()
    d, g = _inputs()
    assert gla.gla_get_device_error() == 0
    gla.gla_set_wait_limit_ns(1000)
    try:
        gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"])
        err = gla.gla_get_device_error()
    finally:
        gla.gla_set_wait_limit_ns(DEFAULT_LIMIT_NS)
    assert err == GLA_ERR_TIMEOUT
    assert gla.gla_get_device_error() == 0  # the word is cleared once read

    o, hT = gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], d["scale"], h0=g["h0"])
    torch.cuda.synchronize()
    assert gla.gla_get_device_error() == 0
    o_ref, hT_ref = oracle.fwd(d["q"], d["k"], d["v"], d["log_lambda"], d["scale"], h0=d["h0"],
                               cu_seqlens=d["cu"])
    assert rel_err(flat(o, False), o_ref, True) <= BF16_TOL
    assert rel_err(hT.cpu().numpy(), hT_ref) <= BF16_TOL


def test_short_wait_limit_in_the_backward_reports_timeout():
    """The backward's three scans (two on side streams) take the same path."""
    gla.load_library()
    d = host_chunk_inputs(22, [1024], 1, True, with_h0=True, packed=False, grad=True)
    g = to_device(d, True, packed=False)
    assert gla.gla_get_device_error() == 0
    gla.gla_set_wait_limit_ns(1000)
    try:
        gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], 0.1, h0=g["h0"],
                          dhT=g["dhT"])
        err = gla.gla_get_device_error()
    finally:
        gla.gla_set_wait_limit_ns(DEFAULT_LIMIT_NS)
    assert err == GLA_ERR_TIMEOUT
    dq, dk, dv, dh0 = gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], 0.1,
                                        h0=g["h0"], dhT=g["dhT"])
    assert gla.gla_get_device_error() == 0


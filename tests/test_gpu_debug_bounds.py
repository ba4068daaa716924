"""The hot path through the debug-bounds build (libgla_debug.so, compiled with GLA_DEBUG_BOUNDS).

That build checks, on the device, every computed global access of the chunk scans (state rows,
output and gradient rows, partial-sum rows, TMA coordinates, hand-over flags, the packed order)
and of the fp32 kernels and the split's chain (unit and chunk row ranges, segment lists): an
index outside its buffer records GLA_ERR_BOUNDS and the access is skipped.  It stands in for a
memory checker.  Each case runs the same call through both builds on ragged shapes (partial
chunks, empty sequences, the balanced persistent launch, many short sequences) and requires no
bounds error and the release build's results: bit for bit where the kernels are deterministic,
within a bf16 rounding for dq and dk (their fp32 partial sums are added in arrival order)."""
import numpy as np
import pytest
import torch

import glasynth as gs
import linear_attention_recurrence_simple_gb300 as gla
from tests.gpu_helpers import host_chunk_inputs, to_device, within_one_bf16_rounding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gla.load_library()
    with gla.debug_bounds_library():
        assert gla.gla_debug_bounds() == 1
    yield
    assert gla.gla_get_device_error() == 0


def both(fn):
    """fn() through the release build, then through the debug-bounds build (whose error word must
    stay clear); returns both results as CPU tensors."""
    def run():
        r = fn()
        r = r if isinstance(r, tuple) else (r,)
        torch.cuda.synchronize()
        return tuple(None if x is None else x.detach().cpu() for x in r)
    rel = run()
    assert gla.gla_get_device_error() == 0
    with gla.debug_bounds_library():
        dbg = run()
        err = gla.gla_get_device_error()
    assert err == 0, gla.gla_status_string(err)
    return rel, dbg


def same(a, b):
    for x, y in zip(a, b):
        if x is None:
            assert y is None
        else:
            assert torch.equal(x, y)


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("lens", [[5, 0, 200, 1, 128, 129, 77], [300], [1]])
def test_forward_packed(bf16, lens):
    d = host_chunk_inputs(700 + sum(lens), lens, 3, bf16, with_h0=True, packed=True)
    g = to_device(d, bf16, packed=True)
    same(*both(lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"],
                                         cu_seqlens=g["cu_seqlens"])))


def test_forward_balanced_launch_and_aug():
    """Equal lengths with a final state: the balanced persistent launch with hand-overs; and the
    self-augmentation mode on the same inputs."""
    d = host_chunk_inputs(711, [300] * 12, 16, True, with_h0=True, packed=False)
    g = to_device(d, True, packed=False)
    same(*both(lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"])))
    aug = torch.from_numpy(gs.normal(711, 9, (16, 96), 10.0)).cuda()
    same(*both(lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"],
                                         aug=aug)))


def test_forward_many_short_sequences():
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 41, 300)]
    d = host_chunk_inputs(712, lens, 2, True, with_h0=False, packed=True)
    g = to_device(d, True, packed=True)
    same(*both(lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE),
                                         cu_seqlens=g["cu_seqlens"])))


@pytest.mark.parametrize("bf16", [True, False])
def test_backward_packed(bf16):
    lens = [385, 1, 128, 0, 130]
    d = host_chunk_inputs(713, lens, 3, bf16, with_h0=True, packed=True, grad=True)
    g = to_device(d, bf16, packed=True)
    rel, dbg = both(lambda: gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], float(gs.SCALE),
                                              h0=g["h0"], dhT=g["dhT"], cu_seqlens=g["cu_seqlens"]))
    if bf16:  # dq, dk: fp32 partial sums added in arrival order, then rounded
        for x, y in zip(rel[:2], dbg[:2]):
            assert within_one_bf16_rounding(y.float().numpy(), x.float().numpy())
        same(rel[2:], dbg[2:])
    else:
        same(rel, dbg)


def test_split_forward():
    lens = [700, 0, 1, 389]
    d = host_chunk_inputs(714, lens, 2, True, with_h0=True, packed=True)
    g = to_device(d, True, packed=True)
    same(*both(lambda: gla.gla_chunk_fwd_split(g["q"], g["k"], g["v"], g["log_lambda"], lens, seg_chunks=1,
                                               scale=float(gs.SCALE), h0=g["h0"])))


def test_decode_steps():
    N, H, P = 5, 3, 9
    slot = torch.tensor([8, 0, 3, 7, 1], dtype=torch.int32, device="cuda")
    q = torch.from_numpy(gs.normal(715, 1, (N, H, 96), 0.1)).cuda().to(torch.bfloat16)
    k = torch.from_numpy(gs.normal(715, 2, (N, H, 96), 0.1)).cuda().to(torch.bfloat16)
    v = torch.from_numpy(gs.normal(715, 3, (N, H, 192))).cuda().to(torch.bfloat16)
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    s0 = torch.from_numpy(gs.normal(715, 7, (P, H, 96, 192), 0.1)).cuda()
    pools = []

    def step():
        pool = s0.clone()
        pools.append(pool)
        return gla.gla_decode_step(q, k, v, ll, pool, float(gs.SCALE), slot=slot)
    same(*both(step))
    assert torch.equal(pools[0], pools[1])


def test_decreasing_offsets_report_shape_not_bounds():
    """Offsets that need clamping are reported as GLA_ERR_SHAPE, and the clamped accesses stay
    inside the buffers: the debug-bounds build records nothing else first."""
    H = 2
    d = host_chunk_inputs(716, [200, 0, 100], H, True, with_h0=True, packed=True)
    g = to_device(d, True, packed=True)
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device="cuda")
    with gla.debug_bounds_library():
        gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], float(gs.SCALE), h0=g["h0"], cu_seqlens=bad)
        assert gla.gla_get_device_error() == -2
        assert gla.gla_get_device_error() == 0

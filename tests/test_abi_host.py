"""Host-only checks of the C ABI: the library builds and loads, exports exactly what
include/gla.h declares, and rejects bad arguments with the documented status before launching
anything.  None of these calls touches a GPU (validation runs before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

import linear_attention_recurrence_simple_gb300 as gla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gla.h")

OK, NULL, SHAPE, DTYPE, ALIGN, UNSUP, WS = 0, -1, -2, -3, -4, -5, -6


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gla_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return gla.load_library()


def test_header_declarations_match_binding():
    assert _declared() == sorted(gla.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", gla.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gla_[a-z_0-9]+)\b", out))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # nothing else with the gla_ prefix leaks out of the library
    assert exported == set(_declared())


def test_debug_bounds_build_exports_the_same_symbols_and_says_which_it_is(lib):
    """libgla_debug.so (GLA_DEBUG_BOUNDS: device index checks) exports the same C ABI; the two
    builds tell themselves apart without touching a GPU."""
    dbg = gla.load_library(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", gla.library_path(debug=True)], capture_output=True,
                         text=True, check=True).stdout
    assert set(re.findall(r"\bT (gla_[a-z_0-9]+)\b", out)) == set(_declared())
    assert lib.gla_debug_bounds() == 0 and dbg.gla_debug_bounds() == 1
    assert gla.gla_debug_bounds() == 0
    with gla.debug_bounds_library():
        assert gla.gla_debug_bounds() == 1
        assert gla.gla_status_string(-9).startswith("GLA_ERR_BOUNDS")
    assert gla.gla_debug_bounds() == 0


def test_library_needs_no_cuda_runtime_soname():
    out = subprocess.run(["readelf", "-d", gla.library_path()], capture_output=True, text=True,
                         check=True).stdout
    assert "libcudart" not in out  # static runtime: loads on hosts without a CUDA driver


def test_status_strings(lib):
    for code in (OK, NULL, SHAPE, DTYPE, ALIGN, UNSUP, WS, -7, -8):
        s = gla.gla_status_string(code)
        assert s.startswith("GLA_")
    assert gla.gla_status_string(123) == "unknown gla_status"


def test_workspace_bytes(lib):
    assert gla.gla_workspace_bytes(0, 16) == 256
    assert gla.gla_workspace_bytes(32, 16) == 512
    assert gla.gla_workspace_bytes(65, 16) == 256 + 512
    assert lib.gla_workspace_bytes(-1, 16) == 0


# Fake, never-dereferenced device addresses: validation must reject before any use.
A = 0x10000          # 16-byte aligned
MIS = 0x10004        # misaligned


def _fwd(lib, q=A, k=A, v=A, ll=A, h0=None, o=A, hT=None, cu=None, n=2, T=8, H=2, dk=96, dv=192,
         dt=0, ws=None, wsb=0):
    P = ctypes.c_void_p
    return lib.gla_chunk_fwd(P(q), P(k), P(v), P(ll), P(h0), 0.1, P(o), P(hT), P(cu), n, T, H, dk,
                             dv, dt, P(ws), wsb, None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, dt=7) == DTYPE
    assert _fwd(lib, dk=64) == UNSUP
    assert _fwd(lib, dv=128) == UNSUP
    assert _fwd(lib, n=-1) == SHAPE
    assert _fwd(lib, T=-3) == SHAPE
    assert _fwd(lib, H=0) == SHAPE
    assert _fwd(lib, q=None) == NULL
    assert _fwd(lib, ll=None) == NULL
    assert _fwd(lib, o=None) == NULL
    assert _fwd(lib, k=MIS) == ALIGN
    assert _fwd(lib, h0=MIS) == ALIGN
    assert _fwd(lib, hT=MIS) == ALIGN
    # packed calls need a big enough, aligned workspace
    assert _fwd(lib, cu=A, n=3, T=20) == WS
    assert _fwd(lib, cu=A, n=3, T=20, ws=A, wsb=16) == WS
    assert _fwd(lib, cu=A, n=3, T=20, ws=MIS, wsb=4096) == ALIGN
    assert _fwd(lib, cu=A + 2, n=3, T=20, ws=A, wsb=4096) == ALIGN
    # empty work is accepted without touching a device
    assert _fwd(lib, n=0) == OK
    assert _fwd(lib, n=0, q=None, k=None, v=None, o=None, ll=None) == OK


def test_aug_argument_errors(lib):
    P = ctypes.c_void_p

    def fwd_aug(aug=A, dk=96, n=2, o=A):
        return lib.gla_chunk_fwd_aug(P(A), P(A), P(A), P(A), None, 0.1, P(aug), P(o), None, None, n, 8,
                                     2, dk, 192, 0, None, 0, None)

    def dec_aug(aug=A, N=4):
        return lib.gla_decode_step_aug(P(A), P(A), P(A), P(A), 0.1, P(aug), P(A), None, 4, P(A), N, 2,
                                       96, 192, 0, None)
    assert fwd_aug(aug=None) == NULL
    assert fwd_aug(aug=MIS) == ALIGN
    assert fwd_aug(dk=64) == UNSUP
    assert fwd_aug(o=None) == NULL
    assert fwd_aug(n=0) == OK
    assert dec_aug(aug=None) == NULL
    assert dec_aug(aug=MIS) == ALIGN
    assert dec_aug(N=0) == OK


def test_head_norm_gate_argument_errors(lib):
    P = ctypes.c_void_p

    def ng(o=A, g=A, w=A, tier=A, nt=2, eps=1e-6, y=A, rows=4, H=2, dv=192, dt=0):
        return lib.gla_head_norm_gate(P(o), P(g), P(w), P(tier), nt, eps, P(y), rows, H, dv, dt, None)
    assert ng(dt=5) == DTYPE
    assert ng(dv=128) == UNSUP
    assert ng(rows=-1) == SHAPE
    assert ng(H=0) == SHAPE
    assert ng(nt=0) == SHAPE
    assert ng(nt=33, rows=0) == OK   # any number of tiers
    assert ng(H=5000) == UNSUP
    assert ng(eps=-1.0) == SHAPE
    assert ng(eps=float("nan")) == SHAPE
    assert ng(o=None) == NULL
    assert ng(tier=None) == NULL
    assert ng(y=MIS) == ALIGN
    assert ng(w=MIS) == ALIGN
    assert ng(tier=A + 2) == ALIGN
    assert ng(rows=0, o=None, y=None) == OK


def test_decode_bf16_state_argument_errors(lib):
    P = ctypes.c_void_p

    def dec(state=A, N=4, dk=96, dt=0, aug=None):
        return lib.gla_decode_step_bf16_state(P(A), P(A), P(A), P(A), 0.1, P(aug), P(state), None, 4, P(A),
                                              N, 2, dk, 192, dt, None)
    assert dec(dt=4) == DTYPE
    assert dec(dk=32) == UNSUP
    assert dec(state=None) == NULL
    assert dec(state=MIS) == ALIGN
    assert dec(aug=MIS) == ALIGN
    assert dec(N=0) == OK


def test_split_argument_errors(lib):
    import numpy as np
    P = ctypes.c_void_p
    cu = np.array([0, 300, 300, 1000], np.int32)
    cp = cu.ctypes.data_as(P)
    need = lib.gla_split_workspace_bytes(cp, 3, 2, 2)
    assert need > 0
    assert lib.gla_split_workspace_bytes(None, 3, 2, 2) == 0
    assert lib.gla_split_workspace_bytes(cp, 3, 2, -1) == 0
    assert lib.gla_split_workspace_bytes(cp, 3, 2, 0) > 0      # 0: the library chooses

    def sp(cu_p=cp, n=3, T=1000, seg=2, ws=A, wsb=None, dk=96):
        return lib.gla_chunk_fwd_split(P(A), P(A), P(A), P(A), None, 0.1, None, P(A), None, cu_p, n, T, 2, dk,
                                       192, 0, seg, P(ws), need if wsb is None else wsb, None)
    assert sp(dk=64) == UNSUP
    assert sp(seg=-1) == SHAPE
    assert sp(cu_p=None) == NULL
    assert sp(T=999) == SHAPE                     # cu[n_seq] must equal T
    bad = np.array([0, 300, 200, 1000], np.int32)
    assert sp(cu_p=bad.ctypes.data_as(P)) == SHAPE  # offsets must not decrease
    assert sp(ws=None) == WS
    assert sp(wsb=need - 1) == WS
    assert sp(ws=A + 16) == ALIGN                 # 256-byte aligned workspace
    assert sp(n=0) == OK


def test_split_choice_of_segment_length(lib):
    """The automatic segment length: one long sequence among few is cut (into pieces that fill
    whole waves of 152 SMs better than the plain forward's one CTA per unit), a batch whose units
    already outnumber the SMs several times over is not, and neither is anything too short."""
    import numpy as np
    from glasynth import varlen_lengths
    P = ctypes.c_void_p

    def choose(lens, H=16):
        cu = np.zeros(len(lens) + 1, np.int32)
        cu[1:] = np.cumsum(lens)
        return lib.gla_split_choose_seg_chunks(cu.ctypes.data_as(P), len(lens), H)
    L = choose([131072])              # 1,024 chunks on 48 units: cut
    assert 16 <= L <= 128
    assert choose([131072, 2048, 4096]) > 0   # one long sequence with short ones: cut
    # 192 units of 1,024 chunks: the plain forward's second wave is 40 units long; the split's two
    # passes (the states-only one about half a full pass) spread the work evenly instead (GB300:
    # 3.52 ms at the chosen 147-chunk segments against 3.60 ms plain)
    assert 64 <= choose([131072] * 4) <= 512
    assert choose([int(x) for x in varlen_lengths(3, 32, 128, 16384)]) == 0   # balanced by ordering
    assert choose([2048] * 8) == 0    # 384 units of 16 chunks
    assert choose([128]) == 0         # one chunk
    assert choose([]) == 0
    assert choose([0, 0]) == 0
    # workspace: a batch the library keeps whole needs no segment states (two fp32 state arrays
    # per segment otherwise)
    lens = [2048] * 8
    cu = np.zeros(9, np.int32)
    cu[1:] = np.cumsum(lens)
    cp = cu.ctypes.data_as(P)
    whole, cut = lib.gla_split_workspace_bytes(cp, 8, 16, 0), lib.gla_split_workspace_bytes(cp, 8, 16, 4)
    assert 0 < whole < 8 * 16 * 96 * 192 * 4
    assert cut >= 2 * 4 * 8 * 16 * 96 * 192 * 4   # 4 segments per sequence, U and S_in
    assert lib.gla_split_choose_seg_chunks(None, 1, 16) == NULL
    bad = np.array([0, 300, 200], np.int32)
    assert lib.gla_split_choose_seg_chunks(bad.ctypes.data_as(P), 2, 16) == SHAPE
    assert lib.gla_split_choose_seg_chunks(bad.ctypes.data_as(P), 1, 0) == SHAPE


def test_bwd_argument_errors(lib):
    P = ctypes.c_void_p

    def bwd(q=A, dO=A, dq=A, dh0=None, dt=0, dk=96, n=2, cu=None, ws=A, wsb=1 << 40):
        return lib.gla_chunk_bwd(P(q), P(A), P(A), P(A), None, 0.1, P(dO), None, P(dq), P(A), P(A),
                                 P(dh0), P(cu), n, 8, 2, dk, 192, dt, P(ws), wsb, None)
    assert bwd(dt=2) == DTYPE
    assert bwd(dk=95) == UNSUP
    assert bwd(n=-5) == SHAPE
    assert bwd(dO=None) == NULL
    assert bwd(dq=None) == NULL
    assert bwd(dh0=MIS) == ALIGN
    assert bwd(cu=A, wsb=16) == WS
    assert bwd(ws=None, wsb=0) == WS          # bf16 mode keeps fp32 partial sums in the workspace
    assert bwd(ws=MIS) == ALIGN
    assert bwd(n=0) == OK


def test_host_forward_argument_errors(lib):
    """gla_chunk_fwd_host validates before touching a device: dtype, sizes, pointers, workspace."""
    P = ctypes.c_void_p
    need = lib.gla_chunk_fwd_host_workspace_bytes(2, 256, 4, 0)

    def hf(q=A, k=A, v=A, ll=A, o=A, n=2, T=256, H=4, dk=96, dv=192, dt=0, pieces=4, ws=A, wsb=None):
        return lib.gla_chunk_fwd_host(P(q), P(k), P(v), P(ll), None, ctypes.c_float(0.1), P(o), None, n, T, H,
                                      dk, dv, dt, pieces, P(ws), need if wsb is None else wsb, None)
    assert hf(dt=7) == DTYPE
    assert hf(dk=64) == UNSUP
    assert hf(n=-1) == SHAPE
    assert hf(H=0) == SHAPE
    assert hf(pieces=0) == SHAPE
    assert hf(n=0, q=None, o=None) == OK
    assert hf(ll=None) == NULL
    assert hf(q=None) == NULL
    assert hf(ws=None) == WS
    assert hf(wsb=need - 1) == WS
    assert hf(ws=A + 16) == ALIGN   # the workspace is 256-byte aligned
    assert hf(ll=A + 4) == ALIGN


def test_host_forward_workspace_bytes(lib):
    """The staged batch (q, k, v, o, each rounded up to 256 bytes) and four state sets."""
    def r(x):
        return -(-x // 256) * 256
    rows = 2 * 256 * 4
    st = r(2 * 4 * 96 * 192 * 4)
    for dt, el in ((0, 2), (1, 4)):
        assert lib.gla_chunk_fwd_host_workspace_bytes(2, 256, 4, dt) == (
            2 * r(rows * 96 * el) + 2 * r(rows * 192 * el) + 4 * st)
    assert lib.gla_chunk_fwd_host_workspace_bytes(-1, 256, 4, 0) == 0
    assert lib.gla_chunk_fwd_host_workspace_bytes(2, 256, 4, 9) == 0


def test_bwd_workspace_bytes(lib):
    acc = 2 * 8 * 2048 * 16 * 96 * 4
    assert gla.gla_bwd_workspace_bytes(8, 2048, 16, False, 0) == 256 + acc
    assert gla.gla_bwd_workspace_bytes(8, 2048, 16, False, 1) == 0
    assert gla.gla_bwd_workspace_bytes(3, 1000, 2, True, 1) == gla.gla_workspace_bytes(3, 2)
    assert gla.gla_bwd_workspace_bytes(3, 1000, 2, True, 0) == gla.gla_workspace_bytes(3, 2) + 2 * 768000


def test_decode_argument_errors(lib):
    P = ctypes.c_void_p

    def dec(q=A, state=A, slot=None, pool=4, N=4, H=2, dk=96, dt=0, o=A):
        return lib.gla_decode_step(P(q), P(A), P(A), P(A), 0.1, P(state), P(slot), pool, P(o), N, H,
                                   dk, 192, dt, None)
    assert dec(dt=3) == DTYPE
    assert dec(dk=32) == UNSUP
    assert dec(N=-1) == SHAPE
    assert dec(pool=3) == SHAPE          # identity slots need pool_rows >= N
    assert dec(H=0) == SHAPE
    assert dec(state=None) == NULL
    assert dec(o=None) == NULL
    assert dec(q=MIS) == ALIGN
    assert dec(slot=A + 2) == ALIGN
    assert dec(N=0) == OK


def test_no_device_is_reported_not_faulted(lib):
    """With valid arguments on a host without a usable sm_103 device, the call fails cleanly."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    assert _fwd(lib) == UNSUP


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 8, 2, 96)
    v = torch.zeros(1, 8, 2, 192)
    with pytest.raises(ValueError):
        gla.gla_chunk_fwd(q, q, v, torch.zeros(2))


def test_noalloc_argument_errors(lib):
    """The allocation-free forward runs the same argument and size checks as gla_chunk_fwd, before
    anything is launched, including the 32-bit limits of the device indexing."""
    P = ctypes.c_void_p

    def na(q=A, k=A, v=A, ll=A, h0=None, o=A, hT=None, cu=None, n=2, T=8, H=2, dk=96, dv=192, dt=0):
        return lib.gla_chunk_fwd_noalloc(P(q), P(k), P(v), P(ll), P(h0), 0.1, P(o), P(hT), P(cu), n, T,
                                         H, dk, dv, dt, None)
    assert na(dt=9) == DTYPE
    assert na(dk=64) == UNSUP
    assert na(dv=96) == UNSUP
    assert na(n=-1) == SHAPE
    assert na(T=-1) == SHAPE
    assert na(H=0) == SHAPE
    # n_seq * H * 96 state rows, or the token count, at 2^31 or beyond: refused, as in gla_chunk_fwd
    assert na(n=1 << 20, T=1, H=32) == SHAPE
    assert _fwd(lib, n=1 << 20, T=1, H=32) == SHAPE
    assert na(n=1 << 16, T=1 << 15, H=1) == SHAPE
    assert _fwd(lib, n=1 << 16, T=1 << 15, H=1) == SHAPE
    assert na(cu=A, n=1 << 22, T=100, H=8) == SHAPE     # the size check comes before the array limit
    assert na(q=None) == NULL
    assert na(ll=None) == NULL
    assert na(o=None) == NULL
    assert na(v=MIS) == ALIGN
    assert na(h0=MIS) == ALIGN
    assert na(hT=MIS) == ALIGN
    assert na(cu=A + 2, n=3, T=20) == ALIGN
    assert na(n=0) == OK
    assert na(n=0, q=None, k=None, v=None, o=None, ll=None) == OK

"""The parity metric of the GPU tests, checked on the CPU.

Bound: max |x - ref| / rms(ref) <= 2e-2 (bf16 operands) or 1e-4 (fp32).  For outputs stored in
bf16 each element may also take half a bf16 ulp of ref, the rounding that the exact answer itself
takes in that format; without it the exactly rounded oracle output fails the bound (about 2.0e-2
on a 255-token case), so the bound would measure the storage format, not the kernel."""
import numpy as np

import glasynth as gs
from tests.gpu_helpers import BF16_TOL, half_ulp_bf16, host_chunk_inputs, rel_err


def test_exactly_rounded_answer_scores_zero(oracle_mod):
    d = host_chunk_inputs(355, [255, 255], 3, True, with_h0=True, packed=False)
    o, _ = oracle_mod.fwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE), h0=d["h0"],
                          cu_seqlens=d["cu"])
    ob = gs.bf16_round(o.astype(np.float32)).astype(np.float64)
    assert rel_err(ob, o) > 1.5e-2            # the plain metric charges the format's rounding
    assert rel_err(ob, o, bf16_out=True) <= 1e-7   # fp64 -> fp32 -> bf16 double rounding


def test_allowance_does_not_hide_real_errors(oracle_mod):
    d = host_chunk_inputs(356, [300], 2, True, with_h0=False, packed=False)
    o, _ = oracle_mod.fwd(d["q"], d["k"], d["v"], d["log_lambda"], float(gs.SCALE),
                          cu_seqlens=d["cu"])
    rms = np.sqrt(np.mean(o ** 2))
    bad = o.copy()
    bad[17, 1, 5] += 0.03 * rms               # one element off by 3% of rms
    assert rel_err(bad, o, bf16_out=True) > BF16_TOL
    assert np.all(half_ulp_bf16(o) <= np.abs(o) * 2.0 ** -8)

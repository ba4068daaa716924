"""The oracle against its stored fixture, and the input generator against independent checks."""
import json
import os

import numpy as np
import pytest

import glasynth as gs
from tests.golden import make_golden

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_reproduces_golden_fixture(oracle_mod):
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        gold = json.load(f)
    for name, c in make_golden.cases():
        o, hT = oracle_mod.fwd(c["q"], c["k"], c["v"], c["ll"], c["scale"], h0=c["h0"])
        g = gold[name]
        if name == "dyadic_T3":
            assert np.allclose(o, np.array(g["o"]), rtol=0, atol=1e-14)
            assert np.allclose(hT, np.array(g["hT"]), rtol=0, atol=1e-14)
        else:
            for key, val in g["o"].items():
                assert abs(o[eval(key)] - val) <= 1e-13 * max(1.0, abs(val))
            for key, val in g["hT"].items():
                assert abs(hT[eval(key)] - val) <= 1e-13 * max(1.0, abs(val))


def test_generator_is_deterministic_and_sliceable():
    a = gs.normal(5, 3, (4, 16, 96))
    b = gs.normal(5, 3, (4, 16, 96))
    assert np.array_equal(a, b)
    rows = gs.normal_rows(5, 3, (16, 96), [3, 1])
    assert np.array_equal(rows[0], a[3]) and np.array_equal(rows[1], a[1])
    assert not np.array_equal(gs.normal(5, 4, (4, 16, 96)), a)
    assert not np.array_equal(gs.normal(6, 3, (4, 16, 96)), a)


def test_generator_moments():
    x = gs.normal(0, 1, (1 << 20,), sigma=0.1).astype(np.float64)
    assert abs(x.mean()) < 1e-3
    assert abs(x.std() - 0.1) < 1e-3
    z = x / 0.1
    assert abs(np.mean(z ** 3)) < 0.02            # symmetric
    assert abs(np.mean(z ** 4) - 3.0) < 0.05      # normal kurtosis (Irwin-Hall(4) would give 2.7)


def test_generator_is_gaussian_in_distribution_and_tails():
    """Empirical CDF against the normal CDF (Kolmogorov-Smirnov distance; at n = 2^22 the 1 % point
    is 1.63 / sqrt(n) = 8e-4), and the tail mass beyond 4 and 5 sigma against 2 (1 - Phi(x)).
    A generator with cut tails (Irwin-Hall(4) ends at 3.46 sigma) fails the tail checks."""
    import math
    n = 1 << 22
    z = np.sort(gs.normal(3, 7, (n,)).astype(np.float64))
    phi = 0.5 * (1.0 + np.array([math.erf(t / math.sqrt(2.0)) for t in z[::64]]))
    ecdf_hi = (np.arange(0, n, 64) + 1) / n
    ecdf_lo = np.arange(0, n, 64) / n
    ks = max(np.max(ecdf_hi - phi), np.max(phi - ecdf_lo))
    assert ks < 1.63 / math.sqrt(n) + 64 / n, ks
    for t, lo, hi in ((4.0, 0.7, 1.3), (5.0, 0.3, 2.2)):
        expect = n * math.erfc(t / math.sqrt(2.0))
        got = int(np.sum(np.abs(z) > t))
        assert lo * expect <= got <= hi * expect, (t, got, expect)
    assert np.max(np.abs(z)) > 5.0


def test_generator_series_against_library_log_and_cos():
    """The series-evaluated logarithm and cosine (written so that host and device agree bit for
    bit) against numpy's log and cos, and at points where the value is exact."""
    a = np.concatenate([np.arange(0, 1 << 32, 65521, dtype=np.uint64),
                        np.array([0, 1, 2, (1 << 31) - 1, 1 << 31, (1 << 32) - 1], np.uint64)])
    ref = np.log((a.astype(np.float64) + 0.5) / 2.0 ** 32)
    assert np.max(np.abs(gs.ln_u1(a) - ref) / np.abs(ref)) < 2e-15
    c = gs.cos_2pi(a)
    assert np.max(np.abs(c - np.cos(2.0 * np.pi * (a.astype(np.float64) / 2.0 ** 32)))) < 2e-15
    q = np.array([0, 1 << 30, 1 << 31, 3 << 30], np.uint64)   # angles 0, pi/2, pi, 3 pi/2
    assert list(gs.cos_2pi(q)) == [1.0, 0.0, -1.0, 0.0]
    assert gs.ln_u1(np.array([(1 << 31) - 1], np.uint64))[0] == pytest.approx(np.log(0.5), abs=3e-10)


def test_splitmix64_reference_values():
    """SplitMix64 seeded with 0 (state += gamma, then mix): the first outputs of the published
    generator are 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F."""
    key = 0
    out = [gs._mix64_int(key + (i + 1) * gs.GAMMA) for i in range(3)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = gs.normal(1, 1, (1 << 16,), sigma=3.0)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 65504.0]  # ties to even
    ours = gs.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


def test_varlen_lengths_recipe():
    lens = gs.varlen_lengths()
    assert len(lens) == 32 and lens.min() >= 128 and lens.max() <= 16384
    cu = gs.cu_seqlens_of(lens)
    assert cu[0] == 0 and cu[-1] == lens.sum()

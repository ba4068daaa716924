"""Plant plausible mistakes in a copy of the oracle and check that the pins catch every one.

Each mutant is the oracle source with one edit (a dropped term, a wrong sign or index, a
transposed operand, a missing factor), compiled on the CPU into a temporary library.  The pin
tests of ``test_oracle_pins.py`` then run against it, and at least one of them must fail.  The
oracle itself is never modified.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

# (name, text to replace, replacement, which occurrence: 0 = first)
MUTANTS = [
    ("fwd: decay dropped",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];",
     "S[(size_t)a * dv + b] = S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];", 0),
    ("fwd: wrong sign of the write",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] - (double)kt[a] * (double)vt[b];", 0),
    ("fwd: k and v swapped in the write (dk == dv case only hides it)",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[b % dk] * (double)vt[a % dv];", 0),
    ("fwd: scale dropped", "sq[a] = scale * (double)qt[a];", "sq[a] = (double)qt[a];", 0),
    ("fwd: readout column index reversed",
     "for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * sq[a];",
     "for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + (dv - 1 - b)] * sq[a];", 0),
    ("fwd: readout row index reversed",
     "for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * sq[a];",
     "for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * sq[dk - 1 - a];", 0),
    ("fwd: h0 ignored", "    if (h0) {\n      const float* src = h0",
     "    if (false && h0) {\n      const float* src = h0", 0),
    ("fwd: readout before the update (off by one token)",
     "      // o_t = S_t^T (scale * q_t)\n",
     "      // o_t = S_t^T (scale * q_t)\n      for (size_t e = 0; e < S.size(); ++e) S[e] -= 0.0 * e;\n"
     "      for (int a = 0; a < dk; ++a) for (int b = 0; b < dv; ++b)"
     " S[(size_t)a * dv + b] -= (double)kt[a] * (double)vt[b];\n", 0),
    ("chunked: inter-chunk decay off by one", "const double inter = scale * std::pow(lam, i + 1);",
     "const double inter = scale * std::pow(lam, i);", 0),
    ("chunked: state decay uses L-j", "acc += std::pow(lam, L - 1 - j) * K(j, a) * V(j, b);",
     "acc += std::pow(lam, L - j) * K(j, a) * V(j, b);", 0),
    ("chunked: intra-chunk mask lets a row see the next token", "for (int j = 0; j <= i; ++j) {",
     "for (int j = 0; j <= i + 1 && j < L; ++j) {", 0),
    ("chunked: intra-chunk mask drops the diagonal", "for (int j = 0; j <= i; ++j) {",
     "for (int j = 0; j < i; ++j) {", 0),
    ("chunked: state not decayed across the chunk", "double acc = lamL * S[(size_t)a * dv + b];",
     "double acc = S[(size_t)a * dv + b];", 0),
    ("decode: decay dropped",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];",
     "S[(size_t)a * dv + b] = S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];", 1),
    ("bwd: dq scale dropped", "dqt[a] = scale * acc;", "dqt[a] = acc;", 0),
    ("bwd: dk contracts with dO instead of v",
     "for (int b = 0; b < dv; ++b) acc += G[(size_t)a * dv + b] * (double)vt[b];",
     "for (int b = 0; b < dv; ++b) acc += G[(size_t)a * dv + b] * (double)gt[b];", 0),
    ("bwd: carry not decayed", "for (size_t e = 0; e < DS; ++e) R[e] = lam * G[e];",
     "for (size_t e = 0; e < DS; ++e) R[e] = G[e];", 0),
    ("bwd: dhT ignored", "    if (dhT) {", "    if (false && dhT) {", 0),
    ("aug: gate without the balance", "g += (double)qt[c] * ((double)ah[c] * (double)kt[c]);",
     "g += (double)qt[c] * (double)kt[c];", 0),
    ("aug: gate uses q twice", "g += (double)qt[c] * ((double)ah[c] * (double)kt[c]);",
     "g += (double)qt[c] * ((double)ah[c] * (double)qt[c]);", 0),
    ("aug: sigmoid of the wrong sign", "const double gate = 1.0 / (1.0 + std::exp(-g));",
     "const double gate = 1.0 / (1.0 + std::exp(g));", 0),
    ("aug: gate not applied", "for (int b = 0; b < dv; ++b) out[b] = gate * (double)vt[b];",
     "for (int b = 0; b < dv; ++b) out[b] = (double)vt[b];", 0),
    ("aug: balance of the wrong head", "const float* ah = aug + (size_t)h * dk;",
     "const float* ah = aug + (size_t)(H - 1 - h) * dk;", 0),
    ("norm: mean square without the division by d_v", "const double inv = 1.0 / std::sqrt(ss / dv + eps);",
     "const double inv = 1.0 / std::sqrt(ss + eps);", 0),
    ("norm: eps dropped", "const double inv = 1.0 / std::sqrt(ss / dv + eps);",
     "const double inv = 1.0 / std::sqrt(ss / dv);", 0),
    ("norm: sigmoid instead of SiLU", "const double silu = gc / (1.0 + std::exp(-gc));",
     "const double silu = 1.0 / (1.0 + std::exp(-gc));", 0),
    ("norm: gain of tier 0 for every head", "const float* wt = w + (size_t)tier[h] * dv;",
     "const float* wt = w;", 0),
    ("bf16 state: 7 significant bits", "const double r = std::nearbyint(std::ldexp(m, 8));",
     "const double r = std::nearbyint(std::ldexp(m, 7));", 0),
    ("bf16 state: truncation instead of rounding", "const double r = std::nearbyint(std::ldexp(m, 8));",
     "const double r = std::trunc(std::ldexp(m, 8));", 0),
    ("bf16 state: state stored unrounded", "for (size_t e = 0; e < S.size(); ++e) St[e] = round_to_bf16(S[e]);",
     "for (size_t e = 0; e < S.size(); ++e) St[e] = S[e];", 0),
    ("mxfp8: E4M3 exponent bias 8", "std::ldexp(8.0 + m, e - 10)", "std::ldexp(8.0 + m, e - 11)", 0),
    ("mxfp8: truncation instead of rounding", "const double r = std::nearbyint(std::ldexp(a, 3 - E));",
     "const double r = std::trunc(std::ldexp(a, 3 - E));", 0),
    ("mxfp8: subnormal range one binade too deep", "const int E = std::max(ex - 1, -6);",
     "const int E = std::max(ex - 1, -7);", 0),
    ("mxfp8: scale not raised for a block maximum above 448", "if (std::ldexp(mx, -se) > 448.0) se += 1;",
     "", 0),
    ("mxfp8: scale from the block's first element", "for (int i = 0; i < n; ++i) mx = std::max(mx, std::fabs((double)x[i]));",
     "mx = std::fabs((double)x[0]);", 0),
    ("mxfp8 step: decay dropped", "S[(size_t)a * dv + b] = lam * s_ab + (double)kt[a] * (double)vt[b];",
     "S[(size_t)a * dv + b] = s_ab + (double)kt[a] * (double)vt[b];", 0),
    ("bwd: dv contracts with q instead of k",
     "for (int a = 0; a < dk; ++a) acc += G[(size_t)a * dv + b] * (double)kt[a];",
     "for (int a = 0; a < dk; ++a) acc += G[(size_t)a * dv + b] * (double)qt[a];", 0),
    ("bwd: dq read off the state before its token's write",
     "for (int b = 0; b < dv; ++b) acc += S[(size_t)a * dv + b] * (double)gt[b];",
     "for (int b = 0; b < dv; ++b) acc += (S[(size_t)a * dv + b] - (double)kt[a] * (double)vt[b]) * (double)gt[b];", 0),
    ("bwd: adjoint seed without the scale",
     "G[(size_t)a * dv + b] = R[(size_t)a * dv + b] + scale * (double)qt[a] * (double)gt[b];",
     "G[(size_t)a * dv + b] = R[(size_t)a * dv + b] + (double)qt[a] * (double)gt[b];", 0),
    ("bwd: carry decayed twice", "for (size_t e = 0; e < DS; ++e) R[e] = lam * G[e];",
     "for (size_t e = 0; e < DS; ++e) R[e] = lam * lam * G[e];", 0),
    ("bwd: forward state missing its decay",
     "S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];",
     "S[(size_t)a * dv + b] = S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];", 2),
]

PIN_TESTS = [
    lambda o: pins.test_fwd_matches_quadratic_and_closed_form(o, 17, True),
    lambda o: pins.test_fwd_matches_quadratic_and_closed_form(o, 1, False),
    pins.test_exact_rational_worked_example,
    pins.test_lambda_one_is_causal_linear_attention,
    pins.test_lambda_zero_keeps_only_current_token,
    lambda o: pins.test_chunk_size_invariance(o, 7),
    pins.test_decode_steps_equal_prefill,
    lambda o: pins.test_backward_matches_finite_differences(o, [6]),
    pins.test_backward_lambda_one_closed_form,
    pins.test_self_aug_zero_balance_is_half_the_value,
    pins.test_self_aug_opposite_balances_sum_to_the_value,
    pins.test_self_aug_single_channel_saturates_by_sign_of_q_times_k,
    pins.test_self_aug_gate_against_exact_value,
    pins.test_norm_gate_unit_gain_and_gate_give_unit_rms,
    pins.test_norm_gate_is_scale_invariant_in_o,
    pins.test_norm_gate_zero_gate_is_zero_and_tier_gain_scales,
    pins.test_norm_gate_worked_example,
    pins.test_round_to_bf16_format_facts,
    pins.test_decode_bf16_state_is_rounded_fp32_step,
    pins.test_e4m3_values_match_torch_float8,
    pins.test_e4m3_conversion_is_round_to_nearest_even,
    pins.test_mxfp8_scale_is_smallest_that_holds_the_block,
    pins.test_mxfp8_round_trip_error_bound_and_idempotence,
    pins.test_decode_mxfp8_state_is_quantised_fp32_step,
]


def _replace_nth(src, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = src.find(old, idx + 1)
        if idx < 0:
            raise AssertionError(f"mutation anchor not found (occurrence {n}): {old!r}")
    return src[:idx] + new + src[idx + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, occ):
    src = open(oracle.source_path()).read()
    mutated = _replace_nth(src, old, new, occ)
    assert mutated != src
    cpp = os.path.join(tmp_path, "mutant.cpp")
    so = os.path.join(tmp_path, "libmutant.so")
    with open(cpp, "w") as f:
        f.write(mutated)
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", cpp, "-o", so])
    variant = oracle.Variant(so)
    caught = []
    for pin in PIN_TESTS:
        try:
            pin(variant)
        except AssertionError:
            caught.append(pin)
    assert caught, f"no pin caught the planted mistake: {name}"

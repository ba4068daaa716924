"""Host-side arithmetic of bench.py: the algorithmic bytes and FLOPs each row divides by, the
roofline fractions, and the rule that a profiled DRAM traffic figure is reported only while the
kernel source it was measured on is unchanged.  No GPU needed."""
import bench


def test_forward_bytes_and_flops_of_the_layer_workload():
    """B=8, T=2048, H=16: q, k (2 x 96 x 2 B) and v, o (2 x 192 x 2 B) per token-head, plus the
    fp32 hT [8, 16, 96, 192]: 311,427,072 B; FLOPs 2 (C d_k + C d_v + 2 d_k d_v) = 147,456 per
    token-head with C = 128."""
    tokens = 8 * 2048
    assert bench.fwd_bytes(tokens, 8, False) == tokens * 16 * 1152 + 8 * 16 * 96 * 192 * 4 == 311_427_072
    assert bench.fwd_bytes(tokens, 8, True) == 311_427_072 + 8 * 16 * 96 * 192 * 4
    assert bench.fwd_flops(tokens) == tokens * 16 * 147_456 == 38_654_705_664


def test_backward_bytes_of_the_layer_workload():
    """q, k, dq, dk (4 x 96 x 2 B) and v, dO, dv (3 x 192 x 2 B) per token-head, plus dhT read and
    dh0 written: 522,190,848 B (no o is read)."""
    tokens = 8 * 2048
    assert bench.bwd_bytes(tokens, 8) == tokens * 16 * (4 * 96 + 3 * 192) * 2 + 2 * 8 * 16 * 96 * 192 * 4
    assert bench.bwd_bytes(tokens, 8) == 522_190_848


def test_roofline_fractions():
    peaks = {"hbm_gbs": 6771.5, "bf16_tflops": 1922.2, "source": "measured"}
    r = bench.roofline(311_427_072, 38_654_705_664, 90.5e-6, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 311_427_072 / 90.5e-6 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6771.5) < 1e-4
    assert abs(r["frac_of_datasheet"] - r["achieved"] / 7900.0) < 1e-4
    assert r["algorithmic_bytes"] == 311_427_072 and r["traffic"] is None
    a = bench.roofline(613_416_960, 1e12, 1e-3, peaks, bound="alu")
    assert a["bound"] == "alu" and a["unit"] == "TFLOP/s"
    assert abs(a["peak"] - 152 * 128 * 2 * 2.07e9 / 1e12) < 0.01   # fp32 FMA lanes x 2 flops x max SM clock
    assert abs(a["frac"] - (1e12 / 1e-3 / 1e12) / (152 * 128 * 2 * 2.07e9 / 1e12)) < 1e-3


def test_profiled_traffic_only_for_the_profiled_source(monkeypatch):
    """An entry whose recorded source hash differs from the file on disk gives None (the counters
    no longer describe the kernel); a matching one scales by the units processed."""
    path, sha, per_unit, note = bench.PROFILED_TRAFFIC["fwd"]
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "fwd", (path, "0" * 16, per_unit, note))
    assert bench.profiled_traffic("fwd") is None
    import hashlib
    import os
    with open(os.path.join(bench.ROOT, path), "rb") as f:
        real = hashlib.sha256(f.read()).hexdigest()[:16]
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "fwd", (path, real, 1000.0, note))
    assert bench.profiled_traffic("fwd") == 1000
    assert bench.profiled_traffic("fwd", 3) == 3000
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "fwd", ("no/such/file.cu", real, 1000.0, note))
    assert bench.profiled_traffic("fwd") is None


def test_profiled_traffic_near_the_algorithmic_bytes():
    """Each recorded traffic figure sits near its row's algorithmic bytes (DRAM counters can read a
    little under them, when outputs are still in L2 at the end of a launch, and above them by the
    re-reads the summaries explain), so a unit mix-up (per launch against per state) shows."""
    tokens = 8 * 2048
    algorithmic = {
        "fwd": bench.fwd_bytes(tokens, 8, False),
        "fwd_aug": bench.fwd_bytes(tokens, 8, False),
        "fwd_fp32": tokens * 16 * (2 * 96 * 4 + 2 * 192 * 4) + 8 * 16 * 96 * 192 * 4,
        "bwd_fp32": 2 * bench.bwd_bytes(tokens, 8) - 2 * 8 * 16 * 96 * 192 * 4,
        "norm_gate": 16384 * 16 * 192 * 2 * 3,
        "decode": 2 * 96 * 192 * 4,
        "decode_norm_gate": 2 * 96 * 192 * 4,
        "decode_bf16_state": 2 * 96 * 192 * 2,
        "decode_mxfp8_state": 2 * (96 * 192 + 96 * 6),
    }
    for row, (_, _, per_unit, _) in bench.PROFILED_TRAFFIC.items():
        ratio = per_unit / algorithmic[row]
        assert 0.85 <= ratio <= 2.0, (row, ratio)

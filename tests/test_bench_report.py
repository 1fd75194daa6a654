"""The bench's report helpers on the shapes of entries the full run produces (CPU only)."""
import json

import bench


def _entries():
    t = {"us_per_call": 5.0, "gbps": 1800.0, "tflops": 13.0, "variant": "k"}
    return {
        "gate_up_swiglu": {"workload": "w", "us_per_call": 15.5, "gbps": 4000.0, "copies": 7, "variant": "pair"},
        "down_gemv": dict(t),
        "verify_m2": dict(t),
        "verify_over_m1": {"M2": 1.12, "M4": 1.15, "M8": 1.18, "M16": 1.58},
        "mid_m64": dict(t),
        "prefill": {"us_per_call": 204.0, "gbps": 520.0, "tflops": 1180.0, "variant": "tc"},
        "headline_hot_l2": dict(t, label="hot"),
        "f32_prefill": dict(t),
    }


def test_secondary_lines_cover_every_entry():
    extras = _entries()
    lines = bench.secondary_lines(extras)
    assert len(lines) == len(extras)
    assert any(line.startswith("verify_over_m1: {") for line in lines)
    assert all("us/call" in line for line in lines if not line.startswith("verify_over_m1"))


def test_annotate_secondary():
    extras = bench.annotate_secondary(_entries(), hbm=6755.8, tc=1881.1, peak_src="measured")
    assert abs(extras["prefill"]["roofline"]["frac"] - 1180.0 / 1881.1) < 1e-12
    assert "hbm_frac" not in extras["prefill"] and "hbm_frac" not in extras["headline_hot_l2"]
    assert abs(extras["down_gemv"]["hbm_frac"] - 1800.0 / 6755.8) < 1e-12
    assert "hbm_frac" not in extras["verify_over_m1"]
    json.dumps(extras)  # the line stays serialisable

"""Host-side pieces of bench.py that need no GPU: the reference arm's JSON
line, the visible-pair share used for the key-padded workload's effective
TFLOP/s, and the lookup of recorded DRAM traffic by kernel source hash."""

import io
import json
import os
import sys
import types
from contextlib import redirect_stdout

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from io_aware_exact_fa_gb300 import workloads as W  # noqa: E402


def test_reference_line_contract(monkeypatch):
    """The reference arm prints one JSON line: the oracle's rate as value, the
    oracle as its own cpu_baseline, and an e2e with no host-device bytes."""
    calls = []

    def fake_sample(w, budget):
        calls.append(budget)
        return 2.0e9, 0.5, 3   # flops, seconds, heads

    monkeypatch.setattr(bench, "oracle_prefill_sample", fake_sample)
    monkeypatch.setenv("RANK", "0")
    args = types.SimpleNamespace(steps=2, warmup=1, gpus=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] == pytest.approx(2 * 2.0e9 / (2 * 0.5) / 1e12)
    assert d["ms_per_step"] == pytest.approx(500.0)
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == W.WORKLOADS[bench.PREFILL].name
    assert len(calls) == 1 + 2   # one warm-up sample, then one per step


def _visible_share_brute(wp, causal):
    keep = W.key_padding_keep(1, wp.H, wp.Nk, wp.pad_heads, wp.pad_from)[0, :, 0].numpy()   # [H, Nk]
    i = np.arange(wp.Nq)[:, None]
    j = np.arange(wp.Nk)[None, :]
    allowed = (j <= i + (wp.Nk - wp.Nq)) if causal else np.ones((wp.Nq, wp.Nk), dtype=bool)
    full = allowed.sum() * wp.H
    return sum((allowed & keep[h][None, :]).sum() for h in range(wp.H)) / full


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(8, 96, 96, 4, 72), (4, 40, 64, 1, 17), (6, 64, 32, 3, 8)])
def test_visible_pair_fraction_matches_brute_force(shape, causal):
    H, Nq, Nk, pad_heads, pad_from = shape
    wp = types.SimpleNamespace(H=H, Nq=Nq, Nk=Nk, pad_heads=pad_heads, pad_from=pad_from)
    assert bench.visible_pair_fraction(wp, causal) == pytest.approx(_visible_share_brute(wp, causal))


def test_visible_pair_fraction_workloads():
    assert bench.visible_pair_fraction(W.WORKLOADS["prefill_32k"], True) == 1.0
    # half the heads lose the last quarter of the keys: under the causal mask those keys pair only
    # with the last quarter of the rows, 1/16 of the causal pairs, so the padded heads keep 15/16
    share = bench.visible_pair_fraction(W.WORKLOADS["prefill_32k_pad"], True)
    wp = W.WORKLOADS["prefill_32k_pad"]
    n, f = wp.Nk, wp.pad_from
    full = n * (n + 1) / 2
    kept_padded = full - (n - f) * (n - f + 1) / 2
    expect = (wp.pad_heads * kept_padded + (wp.H - wp.pad_heads) * full) / (wp.H * full)
    assert share == pytest.approx(expect)


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.json"
    h = bench.kernel_hash("decode_sm103.cu")
    rec.write_text(json.dumps({
        "w_current": {"source_hash": h, "dram_bytes_per_launch": 1234},
        "w_stale": {"source_hash": "0" * 16, "dram_bytes_per_launch": 99},
    }))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(rec))
    assert bench.recorded_traffic("decode_sm103.cu", "w_current") == 1234
    assert bench.recorded_traffic("decode_sm103.cu", "w_stale") is None     # kernel changed since the capture
    assert bench.recorded_traffic("decode_sm103.cu", "w_missing") is None
    # each kernel source has its own hash (a record of one kernel never matches another)
    assert bench.kernel_hash("decode_grouped_sm103.cu") != bench.kernel_hash("decode_sm103.cu")


def test_whole_job_rate_and_peaks():
    assert bench.whole_job_rate(10.0, 4, 2.0, 8) == 160.0
    p = bench.measured_peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["source"] in ("measured", "fallback")

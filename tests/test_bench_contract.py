"""bench.py's JSON line on CPU: the reference arm (the oracle timed on the
host cores) runs without a GPU and prints one line with the keys both arms
share, the same config object as the GPU arm, and the reference-specific
fields (impl, cpu_baseline, an e2e with no copies)."""

import contextlib
import io
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_reference_arm_line(monkeypatch):
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main()
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "us/pass"
    assert d["higher_is_better"] is False and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1e3 - d["value"]) <= 1.0
    assert d["config"] == bench.workload_config(1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "us/pass", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_roofline_arithmetic():
    """The algorithmic counts the roofline fractions divide by, for the pass
    workload (N=32, B=16, V=152064, D=3584, R=512, H=1536): the readout reads
    W2 (R*V*2), base (rows*V*2) and the latent (rows*R*2) once; the pass adds
    the latent stage's weights and inputs and the latent's write."""
    import bench
    from speculative_decoding_gb300 import synth

    sh = synth.SERVE
    assert sh.rows == 480
    assert bench.readout_bytes(sh) == 155_713_536 + 145_981_440 + 491_520 == 302_186_496
    assert bench.readout_flops(sh) == 2.0 * 480 * 152064 * 512
    assert abs(bench.pass_bytes(sh) / 1e6 - 315.8) < 0.1
    assert abs(bench.pass_flops(sh) / 1e9 - 78.89) < 0.01
    # at the measured 6790.7 GB/s the pass is HBM-bound at 46.5 us
    assert abs(bench.pass_bytes(sh) / 6790.7 / 1e3 - 46.5) < 0.05

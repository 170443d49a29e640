"""CPU: bench.py's JSON contract on the paths that run without a GPU -- the reference arm (the
CPU oracle timed on one host core) prints one line with every key the contract names, the
other ranks of a multi-process launch print nothing, and the product arm refuses to run
without a CUDA device instead of falling back to the CPU."""
import contextlib
import io
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_line_has_every_contract_key():
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    lines = [l for l in out.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["metric"] == bench.METRIC
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_runs_on_rank_zero_only():
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args, world=2, rank=1) is None


def test_product_arm_needs_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(SystemExit) as e:
        bench.main(["--steps", "1", "--warmup", "3"])
    assert "GPU" in str(e.value)

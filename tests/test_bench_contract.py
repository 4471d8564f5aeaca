"""The benchmark's one-line JSON contract, on the tiny correctness workload
(N=64, D=256, V=4096): the reference arm (the FP64 oracle on host cores) runs
here on CPU; our arm runs on a GB300 (marked gpu)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BASE_KEYS = {"metric": str, "value": float, "unit": str, "n_gpus": int, "steps": int, "warmup": int,
             "ms_per_step": float, "higher_is_better": bool, "scaling": str, "dtype": str, "data": str,
             "config": dict}


def _run(*args, timeout=300):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                       timeout=timeout)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def _check_base(line, steps, warmup):
    for k, t in BASE_KEYS.items():
        assert k in line, k
        assert isinstance(line[k], t) or (t is float and isinstance(line[k], int)), (k, line[k])
    assert line["steps"] == steps and line["warmup"] >= warmup and line["n_gpus"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny"
    assert line["vs_baseline"] is None or line["vs_baseline"] > 0
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] >= 0 and e2e["d2h_bytes_per_step"] >= 0


def test_reference_arm_line():
    line = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1")
    _check_base(line, 2, 1)
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"] and cpu["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    line = _run("--workload", "tiny", "--steps", "3", "--warmup", "3", "--cpu-rows", "64")
    _check_base(line, 3, 3)
    assert line["dtype"] == "bf16" and line["scaling"] == "weak"
    roof = line["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["unit"] in ("GB/s", "TFLOP/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0 and abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert "traffic" in roof
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
    assert line["gpu_launches"] == 6 * 3  # six kernels per fwd+bwd step (the tiny case has a bias)
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    clocks = line["clocks"]
    assert "sm_mhz" in clocks and "sm_max_mhz" in clocks and isinstance(clocks["reasons"], list)


@pytest.mark.gpu
def test_row_subset_and_shard_modes_run():
    """The secondary measurement modes run and report what they time."""
    line = _run("--op", "indexed", "--workload", "tiny", "--select-frac", "0.25", "--steps", "2", "--warmup", "3")
    assert line["config"]["K"] == 16 and line["value"] > 0 and line["plain_same_rows_ms"] > 0
    line = _run("--op", "shards", "--workload", "tiny", "--shards", "2", "--steps", "2", "--warmup", "3")
    assert line["config"]["shards"] == 2 and line["ms_per_step"] > 0 and line["unsharded_ms"] > 0
    assert line["higher_is_better"] is False


def test_sources_hash_ignores_comments_only(tmp_path):
    """The recorded ncu traffic stays valid across comment edits, never across code edits."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// a kernel\n__global__ void k(int* p) { p[0] = 1; /* store */ }\n")
    base = bench.sources_sha(str(tmp_path))
    src.write_text("// the same kernel, reworded\n__global__ void k(int* p) {\n  p[0] = 1;  // one store\n}\n")
    assert bench.sources_sha(str(tmp_path)) == base
    src.write_text("// a kernel\n__global__ void k(int* p) { p[0] = 2; /* store */ }\n")
    assert bench.sources_sha(str(tmp_path)) != base

"""Host-side logic of bench.py (no GPU): the algorithmic byte counts the
metric divides by, the staleness guard on the committed ncu traffic ratios,
and the reference arm's JSON line."""
import hashlib
import io
import json
import os
import types
from contextlib import redirect_stdout

import numpy as np
import pytest

import bench


def _layout_bytes(M, N, K):
    """Bytes of the buffers one block-scaled GEMM reads and writes, from arrays
    shaped as the C ABI lays them out."""
    qa = np.empty((M, K), np.uint8)
    sa = np.empty((K // 128, M), np.float32)
    qw = np.empty((N, K), np.uint8)
    sw = np.empty((-(-N // 128), K // 128), np.float32)
    y = np.empty((M, N), np.uint16)  # BF16
    return qa.nbytes + sa.nbytes + qw.nbytes + sw.nbytes + y.nbytes


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 28672, 4096), (4, 272, 14336), (16, 6144, 4096)])
def test_gemm_bytes_are_the_buffers_it_touches(M, N, K):
    assert bench.gemm_bytes(M, N, K) == _layout_bytes(M, N, K)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 14336)])
def test_linear_bytes_add_the_bf16_input(M, N, K):
    x = np.empty((M, K), np.uint16)
    assert bench.linear_bytes(M, N, K) == _layout_bytes(M, N, K) + x.nbytes


def test_act_quant_bytes():
    M, K = 8192, 14336
    x = np.empty((M, K), np.uint16)
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    assert bench.act_quant_bytes(M, K) == x.nbytes + q.nbytes + s.nbytes


def _fake_root(tmp_path, ratio=1.25):
    src = tmp_path / "kernel.cu"
    src.write_text("// a kernel\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    entry = {"k": {"sources": ["kernel.cu"], "sha256": sha,
                   "captures": {"a": {"dram_bytes": 125, "algorithmic_bytes": 100, "ratio": ratio},
                                "b": {"dram_bytes": 75, "algorithmic_bytes": 100, "ratio": 0.75}}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entry))
    return src


def test_traffic_uses_the_mean_captured_ratio(tmp_path, monkeypatch):
    _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("k", 1000.0) == pytest.approx(1000.0)  # mean of 1.25 and 0.75


def test_traffic_is_null_once_the_source_changed(tmp_path, monkeypatch):
    src = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src.write_text("// a kernel, edited after the capture\n")
    assert bench._traffic("k", 1000.0) is None
    assert bench._traffic("unknown_kernel", 1000.0) is None


def test_committed_traffic_file_is_well_formed():
    """Every committed capture names existing sources, a SHA-256 and positive
    DRAM/algorithmic ratios (whether it is still current is the bench's check:
    it reports null traffic for a kernel edited since its capture)."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    assert entries
    for name, e in entries.items():
        assert all(os.path.exists(os.path.join(bench.ROOT, s)) for s in e["sources"]), name
        assert len(e["sha256"]) == 64 and int(e["sha256"], 16) >= 0, name
        for c in e["captures"].values():
            assert c["ratio"] > 0 and c["ratio"] == pytest.approx(c["dram_bytes"] / c["algorithmic_bytes"], abs=1e-4)


def test_reference_arm_line(monkeypatch):
    calls = []

    def fake(threads=None, ms=None, cols=None, min_seconds=0.0):
        calls.append(cols)
        return 0.25, "a sample", 0.1
    monkeypatch.setattr(bench, "oracle_decode_sample", fake)
    args = types.SimpleNamespace(gpus=1, steps=2, warmup=3)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.reference_arm(args)
    line = json.loads(out.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] == 0.25 and line["steps"] == 2 and line["warmup"] == 3
    assert line["config"]["workload"] == bench.decode_workload()
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["sample"] == "a sample"
    assert line["e2e"] == {"value": 0.25, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    host = line["cpu_baseline"]["host"]
    assert host["logical_cpus"] == os.cpu_count() and host["machine"] and isinstance(host["model"], str)
    # one calibration call on 512 columns, then warmup + steps calls on one column count
    assert calls[0] == 512 and len(calls) == 1 + 3 + 2 and len(set(calls[1:])) == 1


def test_reference_arm_sizes_steps_to_the_run_budget(monkeypatch):
    """A calibration at 512 columns taking 1 s gives steps of REF_TOTAL_S /
    (warmup + steps) seconds: the column count scales with it (whole 128-column
    blocks), and a budget above the full layer runs the full layer."""
    calls = []

    def fake(threads=None, ms=None, cols=None, min_seconds=0.0):
        calls.append(cols)
        return 0.25, "a sample", 1.0
    monkeypatch.setattr(bench, "oracle_decode_sample", fake)
    with redirect_stdout(io.StringIO()):
        bench.reference_arm(types.SimpleNamespace(gpus=1, steps=100, warmup=80))
    per_step = bench.REF_TOTAL_S / 180
    assert calls[1] == max(128, int(512 * per_step) // 128 * 128)
    calls.clear()
    with redirect_stdout(io.StringIO()):
        bench.reference_arm(types.SimpleNamespace(gpus=1, steps=1, warmup=0))
    assert calls[1] is None


def test_oracle_sample_runs_on_a_small_slice():
    gbps, desc, seconds = bench.oracle_decode_sample(2, ms=[1, 4], cols=256)
    assert gbps > 0 and seconds > 0
    assert "[256, 256, 256, 256]" in desc and "2 host thread(s)" in desc and "passes" not in desc


def test_oracle_sample_repeats_to_its_minimum_time():
    _, _, one = bench.oracle_decode_sample(1, ms=[1], cols=128)
    gbps, desc, seconds = bench.oracle_decode_sample(1, ms=[1], cols=128, min_seconds=2.5 * one)
    assert seconds >= 2.5 * one and gbps > 0
    assert "passes" in desc


def test_oracle_sample_threads_cover_every_column(monkeypatch):
    """The column split over threads covers each projection's columns once."""
    import oracle
    seen = []
    real = oracle.gemm_block

    def spy(qa, sa, qw, sw, **kw):
        seen.append(qw.shape[0])
        return real(qa, sa, qw, sw, **kw)
    monkeypatch.setattr(oracle, "gemm_block", spy)
    bench.oracle_decode_sample(3, ms=[1], cols=640)
    assert sum(seen) == 4 * 640 and all(n % 128 == 0 for n in seen)


def test_cpu_quant_times_cover_every_row_once():
    """The threaded CPU quantizer leg splits rows at whole blocks and covers
    each row exactly once."""
    import threading
    seen = {"w": [], "x": []}
    lock = threading.Lock()

    def spy(name):
        def fn(a, b):
            with lock:
                seen[name].append((a, b))
        return fn
    out = bench._cpu_quant_times([("w", spy("w"), 1000, 128), ("x", spy("x"), 7, 1)])
    assert set(out) == {"w", "x"} and all(v["us"] > 0 and v["threads"] >= 1 for v in out.values())
    assert sorted(r for a, b in seen["w"] for r in range(a, b)) == list(range(1000))
    assert sorted(r for a, b in seen["x"] for r in range(a, b)) == list(range(7))
    assert all(a % 128 == 0 for a, _ in seen["w"])

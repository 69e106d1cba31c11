"""Host logic of bench.py that needs no GPU: the GEMM traffic figure is taken
from the committed ncu summary only while the profiled GEMM source is
unchanged."""
import hashlib
import os

import bench


def test_gemm_traffic_tracks_the_profiled_source(tmp_path, monkeypatch):
    text = open(bench.GEMM_PROFILE).read()
    want = text.split("gemm_tc.cu sha256: ")[1].split()[0]
    have = hashlib.sha256(open(bench.GEMM_SOURCE, "rb").read()).hexdigest()
    n = bench.gemm_traffic()
    if have.startswith(want):
        # the committed summary was captured on the committed source
        assert isinstance(n, int) and 500e6 < n < 1.5e9
    else:
        # the kernel changed since the capture: no traffic figure
        assert n is None
    # any edit of the kernel source invalidates the figure
    edited = tmp_path / "gemm_tc.cu"
    edited.write_bytes(open(bench.GEMM_SOURCE, "rb").read() + b"\n// edited\n")
    monkeypatch.setattr(bench, "GEMM_SOURCE", str(edited))
    assert bench.gemm_traffic() is None
    monkeypatch.setattr(bench, "GEMM_SOURCE", os.path.join(str(tmp_path), "missing.cu"))
    assert bench.gemm_traffic() is None



def test_config_names_the_saved_set(monkeypatch):
    """The bench line says which saved set the filtered calls were given: the
    lean one (a, b, s recomputed) for Llama-style blocks unless --saved full."""
    s = bench.workloads.WORKLOADS[bench.WORKLOAD]
    monkeypatch.setattr(bench, "SAVED", "lean")
    assert bench.config_dict(s, "x")["saved_set"].startswith("lean")
    monkeypatch.setattr(bench, "SAVED", "full")
    assert bench.config_dict(s, "x")["saved_set"] == "full"
    phi = bench.workloads.WORKLOADS["phi15_layer"]
    monkeypatch.setattr(bench, "SAVED", "lean")
    assert bench.config_dict(phi, "x")["saved_set"] == "full"   # LayerNorm blocks: the whole set


def test_cli_accepts_the_saved_set_and_timeline(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py", "--case", "timeline", "--saved", "full", "--steps", "2"])
    a = bench.parse()
    assert a.case == "timeline" and a.saved == "full" and a.steps == 2
    monkeypatch.setattr("sys.argv", ["bench.py"])
    a = bench.parse()
    assert a.case == "layer" and a.saved == "lean" and a.gpus == 1

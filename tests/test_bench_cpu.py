"""bench.py contract checks that need no GPU: the reference arm (the CPU oracle on a
token slab) runs end to end and prints one JSON line with the contract's keys, and the
ncu traffic record parser reads a capture."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0


def test_traffic_record_parser(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    csv_text = "\n".join([
        '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
        '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"',
        '"0","1","p","h","void mx::mxf4_gemm_kernel<256, 4, 1>(GemmParams)","1","7","(320,1,1)","(148,1,1)","0","10.3",'
        '"Command line profiler metrics","dram__bytes_read.sum","Mbyte","50.5"',
        '"0","1","p","h","void mx::mxf4_gemm_kernel<256, 4, 1>(GemmParams)","1","7","(320,1,1)","(148,1,1)","0","10.3",'
        '"Command line profiler metrics","dram__bytes_write.sum","Mbyte","100.25"',
        '"1","1","p","h","void mx::rq_kernel<16, 1, 1, 0>(QuantParams)","1","7","(256,1,1)","(112,64,1)","0","10.3",'
        '"Command line profiler metrics","dram__bytes_read.sum","Gbyte","0.235"',
    ])
    src = tmp_path / "l.csv"
    src.write_text(csv_text)
    out_dir = tmp_path / "profiles"
    out_dir.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "mxfp4_precision_gemms_gb300" / "csrc")
    for f in {f for files in bench.KERNEL_SOURCES.values() for f in files}:
        (tmp_path / "mxfp4_precision_gemms_gb300" / "csrc" / f).write_text(f)
    bench.write_traffic([str(src)])
    rec = json.load(open(out_dir / "traffic_llama8b_linears_T8192.json"))
    assert rec["gemm"]["bytes_per_launch"] == 150750000 and rec["quant"]["bytes_per_launch"] == 235000000
    t = bench.measured_traffic()
    assert t == {"gemm": 150750000, "quant": 235000000}


def test_step_stats_percentiles():
    """The JSON line's step-time summary: median, nearest-rank 10th / 90th percentiles and
    the slowest step."""
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench_stats_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    ms = [1.50, 1.40, 1.60, 1.45, 1.55, 1.42, 1.48, 1.52, 1.58, 1.44, 1.46]
    st = bench.step_stats(ms)
    assert st == {"median": 1.48, "p10": 1.42, "p90": 1.58, "max": 1.60, "max_at": 2}
    assert bench.step_stats([]) is None
    assert bench.step_stats([2.0]) == {"median": 2.0, "p10": 2.0, "p90": 2.0, "max": 2.0, "max_at": 0}

"""bench.py's reference arm on the CPU: the JSON line it prints carries the
contract's keys, and under a two-process launch only rank 0 prints it."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-pages", "4"]


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, *ARGS], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_prints_once_under_two_ranks():
    pytest.importorskip("torch.distributed.run")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), *ARGS, "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


# Algorithmic bytes per unit of each kernel group the bench reports traffic for
# (the encoder and the refine read bf16 or planes and write planes, metadata or
# bf16; decode attention reads codes and metadata per token and KV head).
ALGORITHMIC = {"quantize": 3.15625, "refine": 3.15625, "dequant_anchor": 2.65625,
               "decode_attn_full": 296.0, "decode_attn_anchor": 168.0}


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_records_are_near_the_algorithmic_bytes():
    """Each committed DRAM capture moves within 10 % of the kernel's algorithmic
    bytes (far above would mean re-reads; far below, a capture of the wrong
    launch)."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = {k: v for k, v in json.load(f).items() if isinstance(v, dict)}
    assert set(recs) == set(ALGORITHMIC)
    for k, r in recs.items():
        assert r["bytes_per_unit"] > 0
        ratio = r["bytes_per_unit"] / ALGORITHMIC[k]
        assert 0.9 <= ratio <= 1.1, (k, ratio)
        assert "--clock-control none" in r["command"]


def test_measured_traffic_is_null_once_the_source_changes(tmp_path):
    bench = _bench_module()
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    import hashlib
    (tmp_path / "profiles").mkdir()
    rec = {"g": {"kernel": "k", "source": "k.cu", "sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
                 "unit": "element", "bytes_per_unit": 3.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    bench.ROOT = str(tmp_path)
    assert bench.measured_traffic("g", 2e9) == pytest.approx(6.0)      # GB per launch
    assert bench.measured_traffic("other", 2e9) is None
    src.write_text("__global__ void k() { }\n")                       # the kernel changed
    assert bench.measured_traffic("g", 2e9) is None

"""bench.py's reference arm (the fp64 oracle on the host cores) for every bench mode,
on CPU: one JSON line with the contract's keys, the oracle named as the baseline."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
        "cpu_baseline", "e2e"}


@pytest.mark.parametrize("args", [
    ["--workload", "deltanet_f32_b1h1t64d16c16"],
    ["--workload", "linear_bf16_b4h16t4096d128c64", "--ref-budget", "1"],
    ["--workload", "decode_f32_n64h8d64"],
    ["--bwd", "--workload", "gdn_f32_b2h4t1024d64c64", "--ref-budget", "1"],
    ["--bwd", "--bwd-path", "tokens", "--workload", "gdn_f32_b2h4t1024d64c64", "--ref-budget", "1"],
], ids=["forward", "linear", "decode", "backward", "backward-tokens-path"])
def test_reference_arm_prints_one_contract_line(args):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--steps", "1", "--warmup", "0"] + args
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == args[args.index("--workload") + 1]


def test_recorded_traffic_is_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    """bench.py reports an ncu capture's DRAM bytes only while the captured kernel's
    source file still has the recorded hash."""
    sys.path.insert(0, ROOT)
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    name, entry = next(iter(rec["workloads"].items()))
    (tmp_path / "profiles").mkdir()
    src = tmp_path / entry["source"]
    src.parent.mkdir(parents=True)
    src.write_bytes(open(os.path.join(ROOT, entry["source"]), "rb").read())
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    import hashlib
    if hashlib.sha256(src.read_bytes()).hexdigest() == entry["source_sha256"]:
        assert bench.measured_traffic(name) == entry["dram_read_bytes"] + entry["dram_write_bytes"]
    src.write_bytes(src.read_bytes() + b"\n// changed\n")
    assert bench.measured_traffic(name) is None
    assert bench.measured_traffic("no_such_workload") is None


def test_reference_arm_under_torchrun_two_gloo_ranks():
    """The launch the driver uses for N > 1 (torchrun, one process per rank), on CPU with
    gloo: rank 0 alone runs the oracle and prints the one line, rank 1 exits 0 without
    work, and the process group comes up and goes down cleanly."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "deltanet_f32_b1h1t64d16c16"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="2", CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert KEYS <= set(d) and d["impl"] == "reference" and d["n_gpus"] == 2

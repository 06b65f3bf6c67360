"""Multi-rank host logic of bench.py on the CPU (gloo, world size 2): the step
time is the max over ranks, ranks draw independent batches, and the
reference arm runs on rank 0 only while the other ranks exit without work."""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, tmp_path, timeout=240):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}"] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def test_max_over_ranks_and_independent_batches(tmp_path):
    r = _torchrun([os.path.join(ROOT, "tests", "_multirank_child.py"), str(tmp_path)], tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    res = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert all(x["ws"] == 2 for x in res)
    assert all(x["max"] == 2.5 for x in res)
    assert res[0]["digest"] != res[1]["digest"]


def test_reference_arm_prints_once(tmp_path):
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "0", "--config", "c1"], tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"

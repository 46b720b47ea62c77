"""bench.py's multi-rank plumbing on the CPU with the gloo backend, world size
2: the max-over-ranks time and summed work, the barrier, and the reference arm
under torchrun (rank 0 alone prints one JSON line).  No GPU is used."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
rank, world, local = bench.dist_init()
assert world == 2 and rank in (0, 1)
bench.barrier(world)
t, units = bench.reduce_max_sum(world, 1.5 + rank, 10.0 * (rank + 1))
print(json.dumps({{"rank": rank, "t": t, "units": units}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_max_over_ranks_and_summed_work(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=180) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    lines = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    for line in lines:
        assert line["t"] == 2.5          # the slower rank's time
        assert line["units"] == 30.0     # both ranks' work


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_key_ignores_comments_not_code(tmp_path):
    """The ncu traffic figures are keyed to a hash of the kernel source's code:
    comment and whitespace edits keep the key, a code edit (even inside a
    string literal that holds comment markers) changes it."""
    sys.path.insert(0, ROOT)
    import bench
    a = tmp_path / "a.cu"
    a.write_text('int x = 1; // one\n/* block */ asm("mov.u32 %0, 1; // in a string" : "=r"(x));\nchar c = \'\\\'\';\n')
    b = tmp_path / "b.cu"
    b.write_text('int x = 1;\n\n   asm("mov.u32 %0, 1; // in a string" : "=r"(x)); // another\nchar c = \'\\\'\';')
    c = tmp_path / "c.cu"
    c.write_text('int x = 1; // one\n/* block */ asm("mov.u32 %0, 2; // in a string" : "=r"(x));\nchar c = \'\\\'\';\n')
    assert bench._code_sha(str(a)) == bench._code_sha(str(b))
    assert bench._code_sha(str(a)) != bench._code_sha(str(c))

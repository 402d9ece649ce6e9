"""bench.py's multi-process logic on the CPU: the per-call time of an N-rank
run is the maximum over ranks (world_size 2 over gloo), and under torchrun the
reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks([10.0 * (rank + 1), 5.0 - rank, 7.0], dist, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got[0] == got[1] == [20.0, 5.0, 7.0]


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks([3, 4.5], None, "cpu") == [3.0, 4.5]


def _bench(args, env):
    e = dict(os.environ, **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=e, cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_runs_on_rank0_only():
    args = ["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "bs4_kv1024_bf16"]
    r1 = _bench(args, {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
    r0 = _bench(args, {"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("extra,suffix", [
    ([], ""),
    (["--q-len", "2"], "_q2"),
    (["--page-size", "64"], "_paged64"),
])
def test_reference_arm_times_the_same_form(extra, suffix):
    """--impl reference times the oracle on the workload in the form the GPU arm
    decodes it (several tokens per sequence, or through a page table) and names
    it the same way."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "bs4_kv1024_bf16", *extra],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["config"]["workload"] == "bs4_kv1024_bf16" + suffix
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the reference arm names the workload with the same config object as the GPU arm
    import bench
    assert line["config"] == bench.workload_config("bs4_kv1024_bf16", bench.parse(["--workload", "bs4_kv1024_bf16",
                                                                                    *extra]), 1)


def test_default_workload_is_the_largest():
    """The bench's headline is bs=64, kv_len=8192, e4m3 KV (the most KV bytes per call)."""
    import bench
    from mla_attention_decode_gb300 import synth
    args = bench.parse([])
    assert args.workload == "bs64_kv8192_fp8"
    assert max(synth.WORKLOAD_ORDER, key=bench.workload_kv_bytes) == args.workload
    cfg = bench.workload_config(args.workload, args, 1)
    assert cfg["kv_bytes_per_call"] == 64 * 8192 * 576 + 4 and cfg["batch"] == 64 and cfg["kv_len"] == 8192

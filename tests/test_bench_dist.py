"""The benchmark's multi-process path on the CPU (gloo, two ranks): the
max-over-ranks timing and the reference arm under torchrun, where rank 0 alone
runs and prints one JSON line and the other rank exits 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench._max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: [2.0, 10.0], 1: [2.0, 10.0]}


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_baseline_reports_all_threads_and_one_thread():
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from speculative_tree_verify_gb300 import synth

    D = synth.TINY
    model = synth.gen_model(D, 5)
    cache = synth.gen_cache(D, 64, 128, 6)
    tree = synth.tree_lattice(8, 4, D.vocab, 7)
    threads = oracle.num_threads()
    out = bench.cpu_baseline(oracle, model, cache, tree, 0.5)
    assert out["kind"] == "oracle" and out["cores"] == threads and out["value"] > 0
    assert out["value_1_thread"] > 0 and out["sample_1_thread"].startswith("1 thread")
    assert oracle.num_threads() == threads   # the thread count is put back

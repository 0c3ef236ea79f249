"""Multi-rank host logic on CPU (gloo): bench.py's timing over ranks (the slowest rank's time is
the job's time, throughput is summed over ranks, the reference arm prints from rank 0 only), and
the ring run over real ranks (send / recv of KV blocks) with its failure behaviour."""
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.reduce_max(10.0 + 5.0 * rank, torch.device("cpu"))
    v = bench.aggregate_tflops(world, 1e12, 4, t)
    out[rank] = (t, v)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0                  # slowest rank's time
    assert abs(out[0][1] - 2 * 4e12 / 15e-3 / 1e12) < 1e-9  # both ranks' work / that time


def test_reduce_max_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-rows", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


# ----------------------------------------------------------------------------- ring over ranks

def _ring_worker(rank, world, port, out, Sq, Skv, fail_rank):
    import datetime
    import numpy as np
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    import oracle
    from oracle.ring_ranks import ring_attention_ranks
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, Sq, 16, generator=g, dtype=torch.float64)
    k = torch.randn(2, Skv, 16, generator=g, dtype=torch.float64)
    v = torch.randn(2, Skv, 16, generator=g, dtype=torch.float64)
    q0, q1 = (rank * Sq) // world, ((rank + 1) * Sq) // world
    k0, k1 = oracle.chunk_bounds(Skv, world, rank)
    if rank == fail_rank:
        # a rank that dies before its first send: the others must fail, not wait forever
        os._exit(3)
    if rank == -fail_rank - 2:
        # a rank that stays alive but never sends (a dropped message): the receives time out
        import time
        time.sleep(14)
        os._exit(0)
    try:
        o, lse = ring_attention_ranks(q[:, q0:q1], k[:, k0:k1], v[:, k0:k1])
        o_ref, lse_ref = oracle.attention(q[:, q0:q1], k, v)
        out[rank] = ("ok", float(np.abs(o - o_ref).max()), float(np.abs(lse - lse_ref).max()))
    except Exception as e:   # noqa: BLE001 -- the failure path is what is tested
        out[rank] = ("error", type(e).__name__, str(e)[:200])


def _run_ring(world, Sq, Skv, fail_rank=-1):
    port = _free_port()
    out = mp.Manager().dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_ring_worker, args=(r, world, port, out, Sq, Skv, fail_rank))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    return dict(out), alive


def test_ring_over_gloo_ranks_equals_attention():
    """Three CPU ranks run the ring (KV blocks passed with send/recv, LSE merge per step) and
    each gets exact attention for its query block, ragged blocks included."""
    out, alive = _run_ring(3, Sq=31, Skv=50)
    assert not alive
    assert sorted(out) == [0, 1, 2]
    for r in range(3):
        status, do, dl = out[r]
        assert status == "ok" and do < 1e-12 and dl < 1e-12, out[r]


def test_ring_rank_failure_is_detected():
    """A rank that dies before its first send: the surviving ranks' receives end with an error
    within the process group's 10 s timeout instead of hanging."""
    out, alive = _run_ring(3, Sq=24, Skv=48, fail_rank=1)
    assert not alive, "a surviving rank hung"
    assert 1 not in out
    for r in (0, 2):
        assert r in out and out[r][0] == "error", out.get(r)


def test_ring_dropped_message_times_out():
    """A rank that stays up but never sends its block: the others' receives end with the
    process group's timeout (10 s) instead of waiting forever."""
    import time
    t0 = time.time()
    out, alive = _run_ring(3, Sq=24, Skv=48, fail_rank=-3)   # rank 1 goes silent
    assert not alive, "a surviving rank hung"
    for r in (0, 2):
        assert r in out and out[r][0] == "error", out.get(r)
    assert time.time() - t0 < 90

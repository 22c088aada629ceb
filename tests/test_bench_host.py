"""Host-side logic of bench.py for N > 1 ranks, on CPU: the timings are
reduced to the slowest rank over a gloo process group of two ranks, the
whole-job rate counts every rank's work, and only rank 0 of the reference arm
prints."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r measured (step, e2e, kernel) times; rank 1 is the slower one
        # in the first two, rank 0 in the third.
        mine = [1.0 + rank, 2.0 + 3 * rank, 5.0 - rank]
        q.put((rank, bench.max_over_ranks(mine, world, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 5.0, 5.0]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([1, 2.5], 1, "cpu") == [1.0, 2.5]


def test_job_rate_counts_every_rank():
    # 188.7 MB per rank in 0.2 ms: 0.9435 TB/s per rank, 4 ranks -> 3.774 TB/s.
    assert bench.job_rate(4, 188.7e6, 0.2) == pytest.approx(4 * 188.7e6 / 0.2e-3)
    assert bench.job_rate(1, 10.0, 1000.0) == pytest.approx(10.0)


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_work_accounting_matches_the_workload_figures():
    # Prefill layer at B=4, S=4096 (DeepSeek-V2 dims): the projections
    # 2 * 149,225,472 FLOP per token, the causal attention
    # B * H * S(S+1)/2 * 2 * ((d_nope + d_rope) + d_v), unabsorbed count.
    total, attn = bench.prefill_flops()
    T = 4 * 4096
    assert attn == 4 * 128 * (4096 * 4097 / 2) * 2 * (192 + 128)
    assert total - attn == 2 * 149_225_472 * T
    assert total == pytest.approx(7.64e12, rel=2e-3)
    # Small-model prefill (B=8, S=1024, d_model 512, 8 heads of 64, r_kv 256,
    # an uncompressed W_Q): the projections W_DKV, W_Q, W_UK, W_UV, W_O are
    # 917,504 MACs = 1.835 MFLOP per token; the attention
    # B * H * S(S+1)/2 * 2 * (64 + 64).
    import mla_synth as syn
    total, attn = bench.prefill_flops(syn.WORKLOADS["small_lm_prefill"])
    assert attn == 8 * 8 * (1024 * 1025 / 2) * 2 * (64 + 64)
    assert total - attn == 2 * 917_504 * 8 * 1024
    assert total == pytest.approx(23.6e9, rel=3e-3)
    # Decode: 1152 cache bytes per cached token (512 latent + 64 rope, bf16).
    import numpy as np
    assert bench.decode_bytes(np.array([1, 2, 3])) == 6 * 1152
    # The decode call adds W_UK and W_UV (128 heads x 128 x 512 bf16 each),
    # the queries (128 + 64 per head) and the output (128 per head).
    assert bench.decode_call_extra_bytes(64) == 2 * 128 * 128 * 512 * 2 + 64 * 128 * (192 + 128) * 2

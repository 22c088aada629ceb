"""Host logic of MLRA latent sub-head tensor parallelism, on the CPU.

Two gloo ranks each take their shard of a small MLRA layer (weights sliced by
``mlra_tp.shard_weights``, cache columns by ``shard_cache_columns``), compute
their partial decode step with the fp64 oracle run on that shard alone (a
layer of H/n heads, rank r/n in L/n blocks), and sum the partial outputs with
``mlra_tp.all_reduce_partial``.  The sum must equal the whole layer's output,
and each rank's per-head outputs the matching heads of the whole layer's.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import mla_synth as syn

W = syn.Workload("mlra_tp_small", syn.VARIANT_MLRA, syn.DTYPE_BF16, d_model=256, n_heads=8, d_nope=32,
                 d_rope=0, d_v=32, r_kv=128, r_q=0, n_latent_heads=4, batch=3, seq=40, mode="decode")
LENS = np.array([1, 17, 40], np.int32)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


class _Cfg:
    variant, n_heads, n_latent_heads, d_nope, d_v, r_kv = (W.variant, W.n_heads, W.n_latent_heads, W.d_nope,
                                                           W.d_v, W.r_kv)


def _inputs():
    wts = {k: e for k, (_, e) in syn.weights(W).items()}
    lat = np.zeros((W.batch, W.seq, W.r_kv))
    for b, L in enumerate(LENS):
        lat[b, :L] = syn.cache_rows(W, b, int(L))[1]
    _, x = syn.activations(W, W.batch)
    return wts, lat, x


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from head_latent_attention_gb300 import mlra_tp
        wts, lat, x = _inputs()
        full = oracle.decode(W, x, LENS, lat, None, wts, n_threads=1)
        tw = {k: torch.from_numpy(v) for k, v in wts.items()}
        sw = {k: v.numpy() for k, v in mlra_tp.shard_weights(tw, _Cfg, rank, world).items()}
        cols = mlra_tp.shard_cache_columns(_Cfg, rank, world)
        ws = W.replace(n_heads=W.n_heads // world, r_kv=W.r_kv // world, n_latent_heads=W.n_latent_heads // world)
        part = oracle.decode(ws, x, LENS, np.ascontiguousarray(lat[:, :, cols]), None, sw, n_threads=1)
        hs = W.n_heads // world
        o_err = float(np.max(np.abs(part["o"] - full["o"][:, rank * hs:(rank + 1) * hs])))
        y = torch.from_numpy(part["y"].copy())
        mlra_tp.all_reduce_partial(y)
        y_err = float(np.max(np.abs(y.numpy() - full["y"])) / np.max(np.abs(full["y"])))
        out[rank] = (o_err, y_err)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_mlra_shards_sum_to_layer(world, oracle_mod):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    for r in range(world):
        o_err, y_err = out[r]
        assert o_err < 1e-12 and y_err < 1e-12, (r, o_err, y_err)


def test_shard_checks():
    from head_latent_attention_gb300 import mlra_tp
    with pytest.raises(ValueError):
        mlra_tp.check_shardable(_Cfg, 3)
    assert mlra_tp.shard_cache_columns(_Cfg, 1, 4) == slice(32, 64)

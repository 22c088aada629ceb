"""MLRA latent sub-head tensor parallelism on one GPU: the shards of a layer
run one after another through shard handles, and the sum of their partial
outputs matches the fp64 oracle's whole-layer output ("frankenstein-
transformer", latent/mlra_attn.py, module docstring: each device loads 1/L of
the KV cache).  Each shard's cache append, queries and per-head outputs are
checked against the matching slices of the oracle's too."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_synth as syn
from gpu_util import compare, config_of, to_dev, to_f64, upload_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from head_latent_attention_gb300 import _build
    _build.build()
    import head_latent_attention_gb300 as m
    return m


@pytest.mark.parametrize("n_shards", [4, 2, 1])
def test_mlra_sharded_decode_step(mla, oracle_mod, n_shards):
    from head_latent_attention_gb300 import mlra_tp
    w = syn.WORKLOADS["mlra_decode"].replace(seq=1024)
    lens = [1, 100, 1024, 517, 257]
    B, H, d = len(lens), w.n_heads, w.d_nope
    dev_w, ex_w = upload_weights(w)
    cfg = config_of(w, B, w.seq)
    lat_s, lat_e = np.zeros((B, w.seq, w.r_kv), np.uint16), np.zeros((B, w.seq, w.r_kv))
    for b, L in enumerate(lens):
        lat_s[b, :L], lat_e[b, :L] = syn.cache_rows(w, b, L)
    xs, xe = syn.activations(w, B)
    rnd = lambda a: syn.store(a, w.dtype)[1]
    ref = oracle_mod.decode(w, xe, np.asarray(lens, np.int32), lat_e, None, ex_w, absorbed=True, store=rnd)
    x = to_dev(xs)
    seq = torch.arange(B, dtype=torch.int32, device="cuda")
    pos = torch.tensor([L - 1 for L in lens], dtype=torch.int32, device="cuda")
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    hs = H // n_shards
    y_sum = np.zeros((B, w.d_model))
    for s in range(n_shards):
        cols = mlra_tp.shard_cache_columns(cfg, s, n_shards)
        lay = mla.MlaLayer(cfg, mlra_tp.shard_weights(dev_w, cfg, s, n_shards), B, ws_max_len=0,
                           shard=(s, n_shards))
        assert lay.cfg.n_heads == hs and lay.cfg.r_kv == w.r_kv // n_shards
        lay.cache_lat.copy_(to_dev(np.ascontiguousarray(lat_s[:, :, cols])))
        qn, qr = lay.project_latent(x, seq, pos)
        assert qr is None
        o = lay.decode(qn, None, sl)
        y = lay.out_proj(o)
        torch.cuda.synchronize()
        assert lay.device_status() == (mla.MLA_OK, 0)
        heads = slice(s * hs, (s + 1) * hs)
        compare(to_f64(qn), ref["q"][:, heads], w.dtype, f"shard {s} q")
        rows = to_f64(lay.cache_lat)[np.arange(B), np.asarray(lens) - 1]
        compare(rows, ref["c_kv"][:, cols], w.dtype, f"shard {s} appended latent")
        compare(to_f64(o), ref["o"][:, heads], w.dtype, f"shard {s} o")
        y_sum += to_f64(y)
    compare(y_sum, ref["y"], w.dtype, f"sum of {n_shards} partial outputs")


def test_mlra_shard_arguments(mla):
    w = syn.WORKLOADS["mlra_decode"]
    cfg = config_of(w, 2, 64)
    for shard, n in ((0, 3), (4, 4), (-1, 2), (0, 0)):
        with pytest.raises(mla.MlaError) as e:
            mla.mla_create_shard(cfg, shard, n)
        assert e.value.status == mla.MLA_ERR_INVALID_ARG
    dec = config_of(syn.WORKLOADS["dsv2_decode"], 2, 64)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_create_shard(dec, 0, 1)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED

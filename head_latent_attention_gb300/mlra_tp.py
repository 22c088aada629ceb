"""MLRA latent sub-head tensor parallelism: the host-side layout of a shard.

Source: "frankenstein-transformer", latent/mlra_attn.py, module docstring and
MLRAAttention.forward.  With the latent split into L disjoint blocks of rank
r/L, head h reads only block h L / H (when H d / L is a multiple of d), so a
device that holds a contiguous range of blocks can run those heads alone and
needs only its blocks' columns of the cache (1/n of it on each of n
devices).  The heads' outputs meet only in the output projection, which is a
sum over heads' columns of W_O: each device computes its partial
y_s = W_O[:, its heads] o_s, and one all-reduce (sum) of [T, d_model] gives y.

This module slices the whole layer's weights into a shard's and wraps the
all-reduce; the shard's compute runs through the library's entry points on a
handle from ``mla_create_shard`` (see ``MlaLayer(shard=...)``).
"""
from __future__ import annotations

from typing import Dict

import torch

VARIANT_MLRA = 2


def check_shardable(cfg, n_shards: int):
    if cfg.variant != VARIANT_MLRA:
        raise ValueError("latent sub-head sharding applies to MLRA layers only")
    if n_shards < 1 or cfg.n_latent_heads % n_shards or cfg.n_heads % n_shards:
        raise ValueError(f"{n_shards} shards do not divide L = {cfg.n_latent_heads} blocks "
                         f"and H = {cfg.n_heads} heads")


def shard_weights(weights: Dict[str, torch.Tensor], cfg, shard: int, n_shards: int) -> Dict[str, torch.Tensor]:
    """The weights shard `shard` of `n_shards` holds, from the whole layer's
    (nn.Linear layout [out, in]; W_UK / W_UV as L stacked blocks):

    - W_Q: rows of its heads [H/n * d, d_model]
    - W_DKV: rows of its latent columns [r/n, d_model]
    - W_UK, W_UV: its L/n blocks [L/n, H d / L, r / L]
    - W_O: columns of its heads [d_model, H/n * d_v]
    """
    check_shardable(cfg, n_shards)
    H, L, d, dv, r = cfg.n_heads, cfg.n_latent_heads, cfg.d_nope, cfg.d_v, cfg.r_kv
    hs, ls, rs = H // n_shards, L // n_shards, r // n_shards
    h0, l0, r0 = shard * hs, shard * ls, shard * rs
    return {
        "W_Q": weights["W_Q"][h0 * d:(h0 + hs) * d].contiguous(),
        "W_DKV": weights["W_DKV"][r0:r0 + rs].contiguous(),
        "W_UK": weights["W_UK"][l0:l0 + ls].contiguous(),
        "W_UV": weights["W_UV"][l0:l0 + ls].contiguous(),
        "W_O": weights["W_O"][:, h0 * dv:(h0 + hs) * dv].contiguous(),
    }


def shard_cache_columns(cfg, shard: int, n_shards: int) -> slice:
    """The latent cache columns shard `shard` holds."""
    check_shardable(cfg, n_shards)
    rs = cfg.r_kv // n_shards
    return slice(shard * rs, (shard + 1) * rs)


def all_reduce_partial(y: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the shards' partial outputs in place across the process group (one
    all-reduce of [T, d_model]: NCCL between GPUs, gloo on the CPU)."""
    import torch.distributed as dist
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y

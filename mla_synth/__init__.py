"""Seeded synthetic inputs for Multi-Head Latent Attention workloads.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests.  It holds no attention arithmetic: it only draws numbers,
rounds them to a storage type and describes workload shapes.

Every tensor is drawn from numpy's PCG64 generator seeded with
``SeedSequence([seed, tensor_id, *sub])`` (``sub`` selects an independent
stream, e.g. one per sequence of a cache), as ``standard_normal`` in float64
scaled by ``std``.  Values are then rounded to the storage type: float32 by
round-to-nearest-even, bfloat16 by rounding to float32 and then to bfloat16,
both round-to-nearest-even.  The exact stored value, widened to float64, is
what the oracle receives.

Distributions follow the workload statements: activations and caches
``N(0, 1)``, weights ``N(0, 1/fan_in)``.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

# Fixed stream ids, one per tensor role.
TENSOR_IDS: Dict[str, int] = {
    "x": 0,
    "W_DQ": 1,
    "W_UQ": 2,
    "W_QR": 3,
    "W_DKV": 4,
    "W_KR": 5,
    "W_UK": 6,
    "W_UV": 7,
    "W_O": 8,
    "W_Q": 9,
    "cache_lat": 10,
    "cache_rope": 11,
    "lengths": 12,
    "q_nope": 13,
    "q_rope": 14,
    "o": 15,
}

VARIANT_DECOUPLED = 0
VARIANT_SMALL = 1
VARIANT_MLRA = 2

DTYPE_F32 = 0
DTYPE_BF16 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one workload.  Field names follow the pages' notation."""

    name: str
    variant: int
    dtype: int
    d_model: int
    n_heads: int
    d_nope: int          # per-head query/key width (the pages' d_head)
    d_rope: int          # decoupled rope width (0 unless decoupled)
    d_v: int
    r_kv: int
    r_q: int             # query compression rank (decoupled only, else 0)
    n_latent_heads: int  # L (1 unless MLRA)
    batch: int
    seq: int             # prefill: tokens per sequence; decode: max cache length
    mode: str            # "prefill" or "decode"
    len_lo: int = 0      # decode: per-sequence cache lengths ~ U[len_lo, len_hi]
    len_hi: int = 0
    rope_base: float = 10000.0
    seed: int = 0

    @property
    def np_dtype(self):
        return np.float32 if self.dtype == DTYPE_F32 else np.uint16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == DTYPE_F32 else 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the method's statement: a tiny fp32 prefill, a
# small-LM prefill (RoPE on the decompressed Q/K), a DeepSeek-V2-shaped decode
# and prefill, and an MLRA decode; plus a small-LM decode step (below).
WORKLOADS: Dict[str, Workload] = {
    "tiny_fp32_prefill": Workload(
        "tiny_fp32_prefill", VARIANT_DECOUPLED, DTYPE_F32, d_model=64, n_heads=4,
        d_nope=16, d_rope=8, d_v=16, r_kv=32, r_q=32, n_latent_heads=1,
        batch=2, seq=16, mode="prefill"),
    "small_lm_prefill": Workload(
        "small_lm_prefill", VARIANT_SMALL, DTYPE_BF16, d_model=512, n_heads=8,
        d_nope=64, d_rope=0, d_v=64, r_kv=256, r_q=0, n_latent_heads=1,
        batch=8, seq=1024, mode="prefill"),
    "dsv2_decode": Workload(
        "dsv2_decode", VARIANT_DECOUPLED, DTYPE_BF16, d_model=5120, n_heads=128,
        d_nope=128, d_rope=64, d_v=128, r_kv=512, r_q=1536, n_latent_heads=1,
        batch=64, seq=4096, mode="decode", len_lo=1024, len_hi=4096),
    "dsv2_prefill": Workload(
        "dsv2_prefill", VARIANT_DECOUPLED, DTYPE_BF16, d_model=5120, n_heads=128,
        d_nope=128, d_rope=64, d_v=128, r_kv=512, r_q=1536, n_latent_heads=1,
        batch=4, seq=4096, mode="prefill"),
    "mlra_decode": Workload(
        "mlra_decode", VARIANT_MLRA, DTYPE_BF16, d_model=2048, n_heads=16,
        d_nope=128, d_rope=0, d_v=128, r_kv=1024, r_q=0, n_latent_heads=4,
        batch=128, seq=8192, mode="decode", len_lo=8192, len_hi=8192),
    # A decode step of the small-LM layer (the shape of its prefill: 8
    # sequences of up to 1024 cached tokens), cache lengths ~ U[512, 1024].
    # The pages give no decode workload for this form; this one times the
    # per-step decompression that its RoPE placement forces.
    "small_lm_decode": Workload(
        "small_lm_decode", VARIANT_SMALL, DTYPE_BF16, d_model=512, n_heads=8,
        d_nope=64, d_rope=0, d_v=64, r_kv=256, r_q=0, n_latent_heads=1,
        batch=8, seq=1024, mode="decode", len_lo=512, len_hi=1024),
}


def normal(seed: int, tensor: str, shape: Sequence[int], std: float = 1.0,
           sub: Sequence[int] = ()) -> np.ndarray:
    """float64 N(0, std^2) draws for one tensor role (and optional sub-stream)."""
    ss = np.random.SeedSequence([int(seed), TENSOR_IDS[tensor], *[int(s) for s in sub]])
    g = np.random.Generator(np.random.PCG64(ss))
    a = g.standard_normal(size=tuple(int(s) for s in shape), dtype=np.float64)
    if std != 1.0:
        a *= std
    return a


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 -> float32 (RNE) -> bfloat16 (RNE); return uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float64 exactly."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def store(a: np.ndarray, dtype: int) -> Tuple[np.ndarray, np.ndarray]:
    """Round float64 values to the storage type.

    Returns ``(stored, exact)``: ``stored`` is float32 or uint16 (bfloat16 bits)
    ready for upload, ``exact`` the same values widened to float64.
    """
    if dtype == DTYPE_F32:
        s = np.ascontiguousarray(a, dtype=np.float32)
        return s, s.astype(np.float64)
    s = f64_to_bf16_bits(a)
    return s, bf16_bits_to_f64(s)


def weight_shapes(w: Workload) -> Dict[str, Tuple[int, ...]]:
    """nn.Linear layout [out, in]; MLRA up-projections are L stacked blocks."""
    H, dn, dr, dv = w.n_heads, w.d_nope, w.d_rope, w.d_v
    if w.variant == VARIANT_DECOUPLED:
        return {
            "W_DQ": (w.r_q, w.d_model),
            "W_UQ": (H * dn, w.r_q),
            "W_QR": (H * dr, w.r_q),
            "W_DKV": (w.r_kv, w.d_model),
            "W_KR": (dr, w.d_model),
            "W_UK": (H * dn, w.r_kv),
            "W_UV": (H * dv, w.r_kv),
            "W_O": (w.d_model, H * dv),
        }
    if w.variant == VARIANT_SMALL:
        return {
            "W_Q": (H * dn, w.d_model),
            "W_DKV": (w.r_kv, w.d_model),
            "W_UK": (H * dn, w.r_kv),
            "W_UV": (H * dv, w.r_kv),
            "W_O": (w.d_model, H * dv),
        }
    L = w.n_latent_heads
    return {
        "W_Q": (H * dn, w.d_model),
        "W_DKV": (w.r_kv, w.d_model),
        "W_UK": (L, H * dn // L, w.r_kv // L),
        "W_UV": (L, H * dv // L, w.r_kv // L),
        "W_O": (w.d_model, H * dv),
    }


def weights(w: Workload) -> Dict[str, Tuple[np.ndarray, np.ndarray]]:
    """All weights of a workload as ``name -> (stored, exact)``."""
    out = {}
    for name, shape in weight_shapes(w).items():
        fan_in = shape[-1]
        out[name] = store(normal(w.seed, name, shape, std=fan_in ** -0.5), w.dtype)
    return out


def activations(w: Workload, n_tokens: int) -> Tuple[np.ndarray, np.ndarray]:
    """Layer input x [n_tokens, d_model] ~ N(0, 1)."""
    return store(normal(w.seed, "x", (n_tokens, w.d_model)), w.dtype)


def lengths(w: Workload) -> np.ndarray:
    """Decode cache lengths (new token included) ~ U[len_lo, len_hi], int32."""
    ss = np.random.SeedSequence([int(w.seed), TENSOR_IDS["lengths"]])
    g = np.random.Generator(np.random.PCG64(ss))
    return g.integers(w.len_lo, w.len_hi + 1, size=w.batch).astype(np.int32)


def cache_rows(w: Workload, b: int, n_rows: Optional[int] = None,
               part: str = "cache_lat") -> Tuple[np.ndarray, np.ndarray]:
    """Rows 0..n_rows-1 of sequence ``b`` of a cache ~ N(0, 1).

    ``part`` is ``cache_lat`` (width r_kv) or ``cache_rope`` (width d_rope).
    Each sequence has its own stream, so one sequence can be regenerated alone.
    """
    width = w.r_kv if part == "cache_lat" else w.d_rope
    n = w.seq if n_rows is None else n_rows
    return store(normal(w.seed, part, (n, width), sub=(b,)), w.dtype)


def stage_inputs(w: Workload, name: str, shape: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """A stage-level input (``q_nope``, ``q_rope`` or ``o``) ~ N(0, 1)."""
    return store(normal(w.seed, name, shape), w.dtype)



# ---------------------------------------------------------------------------
# Compressed convolutional attention (CCA) and its grouped form (CCGQA)
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class CcaWorkload:
    """Shape of a CCA / CCGQA layer and its batch.  CCA is the case
    n_kv_heads == n_heads (q_latent == kv_latent)."""

    name: str
    d_model: int
    n_heads: int          # query heads
    n_kv_heads: int       # key/value heads (groups of n_heads / n_kv_heads)
    q_latent: int         # query latent width (n_heads * d_h)
    kv_latent: int        # key/value latent width (n_kv_heads * d_h)
    batch: int
    seq: int
    conv_layers: int = 2
    conv_kernel_seq: int = 4
    conv_kernel_ch: int = 3
    qk_mean: bool = True
    value_shift: bool = True
    key_temp: float = 0.0  # the learnable key temperature beta (the page initialises it to 0)
    rope_base: float = 10000.0
    seed: int = 0

    @property
    def d_h(self) -> int:
        return self.q_latent // self.n_heads

    def replace(self, **kw) -> "CcaWorkload":
        return dataclasses.replace(self, **kw)


CCA_TENSOR_IDS: Dict[str, int] = {"W_QK": 20, "W_V1": 21, "W_V2": 22, "W_V": 23, "conv0": 24, "conv1": 25,
                                  "W_O": 26, "x": 27}

# CCA at compression 4 (d_model 2048 -> latent 512, 8 heads of 64) and CCGQA
# with the page's default rates (query latent E/2 in 16 heads, key/value
# latent E/8 in 4 heads, d_h 64 for both).
CCA_WORKLOADS: Dict[str, CcaWorkload] = {
    "cca_prefill": CcaWorkload("cca_prefill", d_model=2048, n_heads=8, n_kv_heads=8, q_latent=512,
                               kv_latent=512, batch=4, seq=2048),
    "ccgqa_prefill": CcaWorkload("ccgqa_prefill", d_model=2048, n_heads=16, n_kv_heads=4, q_latent=1024,
                                 kv_latent=256, batch=4, seq=2048),
}


def cca_weight_shapes(w: CcaWorkload) -> Dict[str, Tuple[int, ...]]:
    """nn.Linear layout [out, in]; conv0 [channels, k_seq] (depth-wise),
    conv1 [channels, d_h, k_ch] (one group of d_h channels per head)."""
    P = w.q_latent + w.kv_latent
    out = {"W_QK": (P, w.d_model)}
    if w.value_shift:
        out["W_V1"] = (w.kv_latent // 2, w.d_model)
        out["W_V2"] = (w.kv_latent // 2, w.d_model)
    else:
        out["W_V"] = (w.kv_latent, w.d_model)
    if w.conv_layers >= 1:
        out["conv0"] = (P, w.conv_kernel_seq)
    if w.conv_layers >= 2:
        out["conv1"] = (P, w.d_h, w.conv_kernel_ch)
    out["W_O"] = (w.d_model, w.q_latent)
    return out


def _cca_normal(w: CcaWorkload, name: str, shape, std: float = 1.0) -> np.ndarray:
    ss = np.random.SeedSequence([int(w.seed), CCA_TENSOR_IDS[name]])
    a = np.random.Generator(np.random.PCG64(ss)).standard_normal(size=tuple(shape), dtype=np.float64)
    return a * std if std != 1.0 else a


def cca_weights(w: CcaWorkload) -> Dict[str, Tuple[np.ndarray, np.ndarray]]:
    """All CCA weights as ``name -> (stored bf16 bits, exact)``; std
    1/sqrt(fan_in) (a convolution's fan-in is its taps times its input
    channels per group)."""
    out = {}
    for name, shape in cca_weight_shapes(w).items():
        fan_in = shape[-1] if name != "conv1" else shape[1] * shape[2]
        out[name] = store(_cca_normal(w, name, shape, fan_in ** -0.5), DTYPE_BF16)
    return out


def cca_activations(w: CcaWorkload, n_tokens: int) -> Tuple[np.ndarray, np.ndarray]:
    """Layer input x [n_tokens, d_model] ~ N(0, 1), bf16."""
    return store(_cca_normal(w, "x", (n_tokens, w.d_model)), DTYPE_BF16)

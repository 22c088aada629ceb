"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function raises ``AssertionError`` when the oracle disagrees
with something other than itself: closed-form values worked out by hand
(``tests/golden``), a library routine (torch's scaled-dot-product attention in
float64, numpy/scipy matrix products), an invariant of the definitions, or a
special case that reduces to a textbook formula.  ``test_oracle_pins.py`` runs
each one; ``test_oracle_mutations.py`` plants mistakes in a copy of the oracle
and checks that some pin fails for each.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.linalg
import torch
import torch.nn.functional as F

import mla_synth as syn

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-11


def tiny(variant: int, **kw) -> syn.Workload:
    base = dict(name="tiny", variant=variant, dtype=syn.DTYPE_F32, d_model=24,
                n_heads=3, d_nope=8, d_rope=4 if variant == syn.VARIANT_DECOUPLED else 0,
                d_v=8, r_kv=12, r_q=10 if variant == syn.VARIANT_DECOUPLED else 0,
                n_latent_heads=1, batch=2, seq=7, mode="prefill", rope_base=100.0)
    base.update(kw)
    return syn.Workload(**base)


def rand_weights(w: syn.Workload, seed: int = 1):
    rng = np.random.default_rng(seed)
    return {k: rng.standard_normal(s) / np.sqrt(s[-1]) for k, s in syn.weight_shapes(w).items()}


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def close(a, b, tol=TOL, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} (scale {scale:.3e})"


def sdpa(q, k, v, scale):
    """torch's causal scaled-dot-product attention in float64; q/k/v [B,H,S,d]."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float64))
    return F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True,
                                          scale=scale).numpy()


def heads(a, H):
    """[B, S, H*d] -> [B, H, S, d]"""
    B, S, n = a.shape
    return a.reshape(B, S, H, n // H).transpose(0, 2, 1, 3)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def pin_rope_closed_form(orc):
    """Hand-derived rotations (tests/golden/rope_closed_form.json)."""
    g = json.load(open(os.path.join(GOLD, "rope_closed_form.json")))
    f = {"cos": math.cos, "sin": math.sin, "zero": lambda a: 0.0,
         "-2sin": lambda a: -2 * math.sin(a), "2cos": lambda a: 2 * math.cos(a)}
    for c in g["cases"]:
        x = np.array(c["x"], np.float64).reshape(1, 1, -1)
        y = orc.rope(x, [c["pos"]], c["base"], c["style"])[0, 0]
        exp = [f[k](a) for k, a in c["expect"]]
        close(y, exp, 1e-13, f"rope case {c}")


def pin_rope_invariants(orc):
    """Norm preservation, RoPE_0 = identity, relative-position property, and
    the half-split pairing equal to the interleaved one after a permutation."""
    for style in ("interleaved", "half"):
        for d in (2, 8, 64):
            x = rand((5, 3, d), d)
            pos = np.array([0, 1, 7, 1000, 4095], np.int32)
            y = orc.rope(x, pos, 10000.0, style)
            close(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), 1e-13,
                  f"norm {style} {d}")
            close(y[0], x[0], 0.0, f"identity at 0 {style} {d}")
            q = rand((1, 1, d), 100 + d)
            k = rand((1, 1, d), 200 + d)
            for m, n, delta in ((3, 1, 5), (0, 9, 100), (17, 17, 3)):
                a = np.dot(orc.rope(q, [m], 10000.0, style).ravel(),
                           orc.rope(k, [n], 10000.0, style).ravel())
                b = np.dot(orc.rope(q, [m + delta], 10000.0, style).ravel(),
                           orc.rope(k, [n + delta], 10000.0, style).ravel())
                close(a, b, 1e-12, f"relative {style} {d}")
    d = 16
    x = rand((4, 2, d), 7)
    pos = np.array([0, 3, 11, 250], np.int32)
    perm = np.empty(d, np.int64)
    perm[0::2] = np.arange(d // 2)
    perm[1::2] = np.arange(d // 2) + d // 2
    yh = orc.rope(x, pos, 500.0, "half")
    yi = orc.rope(x[..., perm], pos, 500.0, "interleaved")
    close(yh[..., perm], yi, 1e-13, "half == permuted interleaved")


# --------------------------------------------------------------------------
# Projections and linear maps
# --------------------------------------------------------------------------

def pin_linear(orc):
    """orc.linear is x W^T (nn.Linear layout), against numpy's product."""
    x = rand((5, 7), 1)
    W = rand((3, 7), 2)
    close(orc.linear(x, W, 2), x @ W.T, 1e-13, "linear")


def pin_projection_shapes(orc):
    """Shapes of the numpy sketch of DeepSeek MLA ("Multi-Head Latent Attention"
    gist, mla.py): B=2, S=8, embed 8, 4 heads of 8, rope 4, latent rank 2 give
    q/k widths 8 + 4 per head and a latent of width 2 per token."""
    w = tiny(syn.VARIANT_DECOUPLED, d_model=8, n_heads=4, d_nope=8, d_rope=4, d_v=8,
             r_kv=2, r_q=2, batch=2, seq=8)
    W = rand_weights(w)
    pr = orc.project(w, rand((16, 8), 3), np.tile(np.arange(8, dtype=np.int32), 2), W)
    assert pr["c_kv"].shape == (16, 2)
    assert pr["k_r"].shape == (16, 4)
    assert pr["q_nope"].shape == (16, 4, 8)
    assert pr["q_rope"].shape == (16, 4, 4)
    out = orc.prefill(w, rand((2, 8, 8), 4), W)
    assert out["y"].shape == (2, 8, 8)


# --------------------------------------------------------------------------
# Attention: textbook reductions and closed forms
# --------------------------------------------------------------------------

def pin_small_reduces_to_mha(orc):
    """Small-model MLA with r_kv = d_model, W_DKV = I and no rotation is
    standard causal multi-head attention with W_K = W_UK, W_V = W_UV
    (checked against torch's SDPA, scale 1/sqrt(d))."""
    w = tiny(syn.VARIANT_SMALL, r_kv=24)
    W = rand_weights(w, 5)
    W["W_DKV"] = np.eye(24)
    x = rand((2, 7, 24), 6)
    out = orc.prefill(w, x, W, use_rope=False)
    H, d = w.n_heads, w.d_nope
    o = sdpa(heads(x @ W["W_Q"].T, H), heads(x @ W["W_UK"].T, H), heads(x @ W["W_UV"].T, H),
             1 / math.sqrt(d))
    close(out["o"], o.transpose(0, 2, 1, 3), what="small == MHA (o)")
    close(out["y"], o.transpose(0, 2, 1, 3).reshape(2, 7, -1) @ W["W_O"].T, what="small == MHA (y)")


def pin_small_rope_positions(orc):
    """Small-model MLA with rotation: queries are rotated at their position,
    keys at theirs (half-split), then standard causal SDPA."""
    w = tiny(syn.VARIANT_SMALL)
    W = rand_weights(w, 7)
    B, S, H, d = 2, 7, w.n_heads, w.d_nope
    x = rand((B, S, w.d_model), 8)
    out = orc.prefill(w, x, W)
    c = x @ W["W_DKV"].T
    pos = np.tile(np.arange(S, dtype=np.int32), B)
    q = orc.rope((x @ W["W_Q"].T).reshape(B * S, H, d), pos, w.rope_base, "half")
    k = orc.rope((c @ W["W_UK"].T).reshape(B * S, H, d), pos, w.rope_base, "half")
    v = c @ W["W_UV"].T
    o = sdpa(heads(q.reshape(B, S, -1), H), heads(k.reshape(B, S, -1), H), heads(v, H),
             1 / math.sqrt(d))
    close(out["o"], o.transpose(0, 2, 1, 3), what="small with rope")


def pin_decoupled_reduces_to_sdpa(orc):
    """Decoupled MLA equals SDPA on q = [q_C ‖ RoPE(q_R)], k = [k_C ‖ RoPE(k_R)
    shared by all heads], scale 1/sqrt(d_nope + d_rope)."""
    w = tiny(syn.VARIANT_DECOUPLED)
    W = rand_weights(w, 9)
    B, S, H = 2, 7, w.n_heads
    x = rand((B, S, w.d_model), 10)
    out = orc.prefill(w, x, W)
    pos = np.tile(np.arange(S, dtype=np.int32), B)
    cq = x.reshape(B * S, -1) @ W["W_DQ"].T
    qc = (cq @ W["W_UQ"].T).reshape(B * S, H, w.d_nope)
    qr = orc.rope((cq @ W["W_QR"].T).reshape(B * S, H, w.d_rope), pos, w.rope_base)
    c = x.reshape(B * S, -1) @ W["W_DKV"].T
    kc = (c @ W["W_UK"].T).reshape(B * S, H, w.d_nope)
    kr = orc.rope((x.reshape(B * S, -1) @ W["W_KR"].T).reshape(B * S, 1, w.d_rope), pos,
                  w.rope_base)
    kr = np.broadcast_to(kr, (B * S, H, w.d_rope))
    q = np.concatenate([qc, qr], -1).reshape(B, S, -1)
    k = np.concatenate([kc, kr], -1).reshape(B, S, -1)
    v = (c @ W["W_UV"].T).reshape(B, S, -1)
    o = sdpa(heads(q, H), heads(k, H), heads(v, H), 1 / math.sqrt(w.d_nope + w.d_rope))
    close(out["o"], o.transpose(0, 2, 1, 3), what="decoupled == SDPA")
    close(out["y"], o.transpose(0, 2, 1, 3).reshape(B, S, -1) @ W["W_O"].T,
          what="decoupled y")


def pin_rope_only_scores(orc):
    """With W_UK = 0 the decoupled scores come from the rope term alone:
    softmax(RoPE(q_R) . RoPE(k_R) / sqrt(d_nope + d_rope)); with W_QR = 0 and
    W_KR = 0 they come from q_C . k_C alone, with the same scale."""
    w = tiny(syn.VARIANT_DECOUPLED)
    B, S, H = 1, 6, w.n_heads
    x = rand((B, S, w.d_model), 12)
    pos = np.arange(S, dtype=np.int32)
    scale = 1 / math.sqrt(w.d_nope + w.d_rope)
    W = rand_weights(w, 11)
    W["W_UK"] = np.zeros_like(W["W_UK"])
    out = orc.prefill(w, x, W)
    cq = x[0] @ W["W_DQ"].T
    qr = orc.rope((cq @ W["W_QR"].T).reshape(S, H, w.d_rope), pos, w.rope_base)
    kr = orc.rope((x[0] @ W["W_KR"].T).reshape(S, 1, w.d_rope), pos, w.rope_base)
    v = (x[0] @ W["W_DKV"].T) @ W["W_UV"].T
    o = sdpa(qr.transpose(1, 0, 2)[None], np.broadcast_to(kr.transpose(1, 0, 2), (H, S, w.d_rope))[None],
             heads(v[None], H), scale)
    close(out["o"], o.transpose(0, 2, 1, 3), what="rope-only scores")
    W = rand_weights(w, 13)
    W["W_QR"] = np.zeros_like(W["W_QR"])
    W["W_KR"] = np.zeros_like(W["W_KR"])
    out = orc.prefill(w, x, W)
    c = x[0] @ W["W_DKV"].T
    qc = (x[0] @ W["W_DQ"].T) @ W["W_UQ"].T
    o = sdpa(heads(qc[None], H), heads((c @ W["W_UK"].T)[None], H), heads((c @ W["W_UV"].T)[None], H),
             scale)
    close(out["o"], o.transpose(0, 2, 1, 3), what="latent-only scores")


def pin_single_token_closed_form(orc):
    """With one token the causal softmax puts weight 1 on it, so
    y = W_O V W_DKV x with V = W_UV (MLRA: the block-diagonal arrangement of
    the L blocks W_UV,i), for every variant."""
    for variant in (syn.VARIANT_DECOUPLED, syn.VARIANT_SMALL, syn.VARIANT_MLRA):
        kw = dict(n_heads=4, r_kv=12, n_latent_heads=4) if variant == syn.VARIANT_MLRA else {}
        w = tiny(variant, **kw)
        W = rand_weights(w, 20 + variant)
        x = rand((3, 1, w.d_model), 30 + variant)
        y = orc.prefill(w, x, W)["y"]
        Wuv = W["W_UV"] if variant != syn.VARIANT_MLRA else scipy.linalg.block_diag(*W["W_UV"])
        close(y[:, 0], x[:, 0] @ (W["W_O"] @ Wuv @ W["W_DKV"]).T, what=f"S=1 variant {variant}")


def pin_uniform_cache(orc):
    """When every cached latent (and rope key) is the same vector c, every
    weighting is uniform over the same value: o_h = (W_UV c)[head h] whatever
    the query."""
    for variant in (syn.VARIANT_DECOUPLED, syn.VARIANT_SMALL, syn.VARIANT_MLRA):
        kw = dict(n_heads=4, r_kv=12, n_latent_heads=2) if variant == syn.VARIANT_MLRA else {}
        w = tiny(variant, **kw)
        W = rand_weights(w, 40 + variant)
        S = 9
        c = rand((w.r_kv,), 50 + variant)
        cl = np.broadcast_to(c, (1, S, w.r_kv)).copy()
        cr = np.broadcast_to(rand((max(w.d_rope, 1),), 60)[:w.d_rope], (1, S, w.d_rope)).copy()
        q_pos = np.array([0, 3, 8], np.int32)
        q_b = np.zeros(3, np.int32)
        H = w.n_heads
        if variant == syn.VARIANT_DECOUPLED:
            q = {"q_nope": rand((3, H, w.d_nope), 1), "q_rope": rand((3, H, w.d_rope), 2)}
        else:
            q = {"q": rand((3, H, w.d_nope), 3)}
        o = orc.attend(w, q_b, q_pos, q, cl, cr, W, use_rope=False)
        Wuv = W["W_UV"] if variant != syn.VARIANT_MLRA else scipy.linalg.block_diag(*W["W_UV"])
        v = (Wuv @ c).reshape(H, w.d_v)
        close(o, np.broadcast_to(v, o.shape), what=f"uniform cache variant {variant}")


def pin_softmax_weights(orc):
    """Attention weights: each row sums to 1, masked (future) keys have weight
    exactly 0, and the query at position 0 puts weight exactly 1 on key 0."""
    for variant in (syn.VARIANT_DECOUPLED, syn.VARIANT_SMALL, syn.VARIANT_MLRA):
        kw = dict(n_heads=4, r_kv=12, n_latent_heads=2) if variant == syn.VARIANT_MLRA else {}
        w = tiny(variant, **kw)
        W = rand_weights(w, 70 + variant)
        S = 8
        cl = rand((2, S, w.r_kv), 71)
        cr = rand((2, S, w.d_rope), 72)
        q_b = np.array([0, 0, 1, 1, 1], np.int32)
        q_pos = np.array([0, 5, 0, 2, 7], np.int32)
        H = w.n_heads
        if variant == syn.VARIANT_DECOUPLED:
            q = {"q_nope": rand((5, H, w.d_nope), 73), "q_rope": rand((5, H, w.d_rope), 74)}
        else:
            q = {"q": rand((5, H, w.d_nope), 75)}
        _, p = orc.attend(w, q_b, q_pos, q, cl, cr, W, want_probs=True)
        close(p.sum(-1), np.ones((5, H)), 1e-14, "rows sum to 1")
        for i, pp in enumerate(q_pos):
            assert np.all(p[i, :, pp + 1:] == 0.0), "masked keys must be exactly 0"
            assert np.all(p[i, :, :pp + 1] > 0.0)
        assert np.all(p[0, :, 0] == 1.0) and np.all(p[2, :, 0] == 1.0)


# --------------------------------------------------------------------------
# Identities between forms and variants
# --------------------------------------------------------------------------

def pin_absorbed_equals_definition(orc):
    """Weight absorption (q . W_UK c = (W_UK^T q) . c, sum p W_UV c =
    W_UV sum p c) gives the definition's result: decoupled and MLRA."""
    for variant, kw in ((syn.VARIANT_DECOUPLED, {}),
                        (syn.VARIANT_MLRA, dict(n_heads=4, r_kv=12, n_latent_heads=4)),
                        (syn.VARIANT_MLRA, dict(n_heads=6, d_nope=4, d_v=4, r_kv=12,
                                                n_latent_heads=4))):
        w = tiny(variant, **kw)
        W = rand_weights(w, 80 + variant)
        S = 11
        cl = rand((3, S, w.r_kv), 81)
        cr = rand((3, S, w.d_rope), 82)
        q_b = np.array([0, 1, 1, 2, 2, 2], np.int32)
        q_pos = np.array([10, 0, 6, 3, 9, 10], np.int32)
        H = w.n_heads
        if variant == syn.VARIANT_DECOUPLED:
            q = {"q_nope": rand((6, H, w.d_nope), 83), "q_rope": rand((6, H, w.d_rope), 84)}
        else:
            q = {"q": rand((6, H, w.d_nope), 85)}
        a = orc.attend(w, q_b, q_pos, q, cl, cr, W)
        b = orc.attend(w, q_b, q_pos, q, cl, cr, W, absorbed=True)
        close(a, b, 1e-12, f"absorbed variant {variant} {kw}")


def pin_mlra_block_structure(orc):
    """MLRA equals the small-model form without rotation whose W_UK / W_UV are
    the block-diagonal arrangements of the L blocks; with L = 1 it equals the
    small-model form without rotation on the same matrices."""
    for L, H, d, r in ((4, 4, 8, 12), (1, 3, 8, 12), (2, 6, 4, 8), (4, 2, 8, 8)):
        w = tiny(syn.VARIANT_MLRA, n_heads=H, d_nope=d, d_v=d, r_kv=r, n_latent_heads=L)
        W = rand_weights(w, 90 + L)
        ws = tiny(syn.VARIANT_SMALL, n_heads=H, d_nope=d, d_v=d, r_kv=r)
        Ws = dict(W)
        Ws["W_UK"] = scipy.linalg.block_diag(*W["W_UK"])
        Ws["W_UV"] = scipy.linalg.block_diag(*W["W_UV"])
        x = rand((2, 6, w.d_model), 91)
        a = orc.prefill(w, x, W)["y"]
        b = orc.prefill(ws, x, Ws, use_rope=False)["y"]
        close(a, b, what=f"MLRA L={L} == block-diagonal small")


def pin_decode_matches_prefill(orc):
    """Decoding token t against the cache of tokens 0..t gives row t of the
    causal prefill; prefill in two chunks (start_pos > 0) gives the one-pass
    result."""
    for variant in (syn.VARIANT_DECOUPLED, syn.VARIANT_SMALL, syn.VARIANT_MLRA):
        kw = dict(n_heads=4, r_kv=12, n_latent_heads=2) if variant == syn.VARIANT_MLRA else {}
        w = tiny(variant, **kw)
        W = rand_weights(w, 100 + variant)
        B, S = 2, 7
        x = rand((B, S, w.d_model), 101)
        full = orc.prefill(w, x, W)
        for t in (0, 3, 6):
            dec = orc.decode(w, x[:, t], np.array([t + 1] * B, np.int32), full["cache_lat"],
                             full["cache_rope"], W)
            close(dec["y"], full["y"][:, t], what=f"decode t={t} variant {variant}")
        first = orc.prefill(w, x[:, :4], W, cache_lat=np.zeros((B, S, w.r_kv)),
                            cache_rope=np.zeros((B, S, w.d_rope)))
        second = orc.prefill(w, x[:, 4:], W, start_pos=[4, 4], cache_lat=first["cache_lat"],
                             cache_rope=first["cache_rope"])
        close(np.concatenate([first["y"], second["y"]], 1), full["y"],
              what=f"chunked prefill variant {variant}")


def pin_cache_bytes(orc):
    """Cache bytes per token for each workload equal (r_kv + d_rope) * dtype
    size (tests/golden/cache_bytes.json)."""
    g = json.load(open(os.path.join(GOLD, "cache_bytes.json")))
    for name, nbytes in g["expect_bytes_per_token"].items():
        assert orc.cache_bytes_per_token(syn.WORKLOADS[name]) == nbytes, name


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

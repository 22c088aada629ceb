"""Pins of the CCA / CCGQA oracle ("frankenstein-transformer",
latent/cca_attn.py) against what the page and the mathematics fix, each
independent of the oracle's own code: library routines (torch conv1d,
normalize, scaled_dot_product_attention), invariants (causality, degree-1
homogeneity, the value-shift direction) and exact reductions (q-k-mean as a
change of the projection weights; grouped heads as replicated heads)."""
from __future__ import annotations

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import mla_synth as syn
from oracle import cca, rope

SMALL = syn.CcaWorkload("cca_small", d_model=48, n_heads=4, n_kv_heads=4, q_latent=32, kv_latent=32,
                        batch=2, seq=13)
SMALL_GQA = SMALL.replace(name="ccgqa_small", n_heads=4, n_kv_heads=2, q_latent=32, kv_latent=16)


def weights(w, seed=3):
    rng = np.random.default_rng(seed)
    return {k: rng.standard_normal(s) / np.sqrt(s[-1] if k != "conv1" else s[1] * s[2])
            for k, s in syn.cca_weight_shapes(w).items()}


def x_of(w, seed=4):
    return np.random.default_rng(seed).standard_normal((w.seq, w.d_model))


def test_convolutions_match_torch_conv1d():
    rng = np.random.default_rng(0)
    S, C, dh = 11, 12, 4
    a = rng.standard_normal((S, C))
    w0 = rng.standard_normal((C, 4))
    w1 = rng.standard_normal((C, dh, 3))
    at = torch.from_numpy(a.T[None])  # (1, C, S)
    ref0 = F.conv1d(F.pad(at, (3, 0)), torch.from_numpy(w0[:, None, :]), groups=C)[0].numpy().T
    np.testing.assert_allclose(cca.causal_depthwise_conv(a, w0), ref0, rtol=0, atol=1e-12)
    ref1 = F.conv1d(F.pad(at, (2, 0)), torch.from_numpy(w1), groups=C // dh)[0].numpy().T
    np.testing.assert_allclose(cca.causal_grouped_conv(a, w1, dh), ref1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("w", [SMALL.replace(key_temp=0.4), SMALL_GQA.replace(key_temp=-0.3)])
def test_attention_core_matches_sdpa(w):
    # No convolutions, no q-k-mean, no value-shift: the layer is attention on
    # L2-normalised, rotated projections.
    w = w.replace(conv_layers=0, qk_mean=False, value_shift=False)
    W = weights(w)
    x = x_of(w)
    S, Hq, Hkv, dh = w.seq, w.n_heads, w.n_kv_heads, w.d_h
    qk = torch.from_numpy(x @ W["W_QK"].T)
    q = F.normalize(qk[:, :w.q_latent].reshape(S, Hq, dh), dim=-1) * np.sqrt(dh)
    k = F.normalize(qk[:, w.q_latent:].reshape(S, Hkv, dh), dim=-1) * np.sqrt(dh) * np.exp(w.key_temp)
    pos = np.arange(S, dtype=np.int32)
    q = torch.from_numpy(rope(q.numpy(), pos, w.rope_base, "half")).permute(1, 0, 2)
    k = torch.from_numpy(rope(k.numpy(), pos, w.rope_base, "half")).permute(1, 0, 2)
    v = torch.from_numpy(x @ W["W_V"].T).reshape(S, Hkv, dh).permute(1, 0, 2)
    gs = Hq // Hkv
    o = F.scaled_dot_product_attention(q, k.repeat_interleave(gs, 0), v.repeat_interleave(gs, 0), is_causal=True,
                                       scale=1.0 / np.sqrt(dh))
    y_ref = o.permute(1, 0, 2).reshape(S, w.q_latent).numpy() @ W["W_O"].T
    np.testing.assert_allclose(cca.forward_sequence(w, x, W), y_ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("w", [SMALL, SMALL_GQA])
def test_causal(w):
    W = weights(w)
    x = x_of(w)
    y = cca.forward_sequence(w, x, W)
    x2 = x.copy()
    x2[7:] = np.random.default_rng(9).standard_normal(x2[7:].shape)
    y2 = cca.forward_sequence(w, x2, W)
    np.testing.assert_array_equal(y2[:7], y[:7])
    assert np.abs(y2[7:] - y[7:]).max() > 1e-3


@pytest.mark.parametrize("w", [SMALL, SMALL_GQA])
def test_homogeneous_of_degree_one(w):
    # Normalisation removes the scale of q and k; v and W_O are linear.
    W = weights(w)
    x = x_of(w)
    np.testing.assert_allclose(cca.forward_sequence(w, 2.5 * x, W), 2.5 * cca.forward_sequence(w, x, W),
                               rtol=0, atol=1e-11)


def test_value_shift_takes_the_previous_token():
    # With the current-token projection zero, token 0 sees only its own value,
    # which is then the projection of the token before it: zero.
    w = SMALL
    W = weights(w)
    W["W_V1"] = np.zeros_like(W["W_V1"])
    x = x_of(w)
    y = cca.forward_sequence(w, x, W)
    assert np.all(y[0] == 0.0) and np.abs(y[1:]).max() > 1e-3


@pytest.mark.parametrize("w", [SMALL, SMALL_GQA])
def test_qk_mean_is_a_change_of_projection(w):
    # Without convolutions, q-k-mean is linear in the projections:
    # q_h = 1.5 Wq_h x + 0.5 Wk_g(h) x and k_g = 1.5 Wk_g x + 0.5 mean_{h in g} Wq_h x.
    w0 = w.replace(conv_layers=0)
    W = weights(w0)
    x = x_of(w0)
    Hq, Hkv, dh = w.n_heads, w.n_kv_heads, w.d_h
    gs = Hq // Hkv
    Wq = W["W_QK"][:w.q_latent].reshape(Hq, dh, -1)
    Wk = W["W_QK"][w.q_latent:].reshape(Hkv, dh, -1)
    Wq2 = 1.5 * Wq + 0.5 * np.repeat(Wk, gs, axis=0)
    Wk2 = 1.5 * Wk + 0.5 * Wq.reshape(Hkv, gs, dh, -1).mean(axis=1)
    W2 = dict(W, W_QK=np.concatenate([Wq2.reshape(w.q_latent, -1), Wk2.reshape(w.kv_latent, -1)]))
    np.testing.assert_allclose(cca.forward_sequence(w0, x, W),
                               cca.forward_sequence(w0.replace(qk_mean=False), x, W2), rtol=0, atol=1e-11)


def test_grouped_heads_equal_replicated_heads():
    # Without q-k-mean and value-shift, CCGQA equals CCA whose key/value heads
    # (projection rows and channel-convolution groups) repeat each group's.
    w = SMALL_GQA.replace(qk_mean=False, value_shift=False)
    W = weights(w)
    x = x_of(w)
    Hq, Hkv, dh = w.n_heads, w.n_kv_heads, w.d_h
    gs = Hq // Hkv
    rep = lambda a: np.repeat(a.reshape(Hkv, dh, *a.shape[1:]), gs, axis=0).reshape(Hq * dh, *a.shape[1:])
    Wk = W["W_QK"][w.q_latent:]
    W2 = {
        "W_QK": np.concatenate([W["W_QK"][:w.q_latent], rep(Wk)]),
        "W_V": rep(W["W_V"]),
        "conv0": np.concatenate([W["conv0"][:w.q_latent], rep(W["conv0"][w.q_latent:])]),
        "conv1": np.concatenate([W["conv1"][:w.q_latent], rep(W["conv1"][w.q_latent:])]),
        "W_O": W["W_O"],
    }
    w2 = w.replace(n_kv_heads=Hq, kv_latent=w.q_latent)
    np.testing.assert_allclose(cca.forward_sequence(w, x, W), cca.forward_sequence(w2, x, W2), rtol=0, atol=1e-11)

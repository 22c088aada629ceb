"""fp64 oracle for compressed convolutional attention (CCA) and its grouped
form (CCGQA) — TEST INFRASTRUCTURE ONLY (same rules as the rest of
``oracle/``: only tests, the smoke check and the benchmark's CPU legs may
use it; the library never does).

Source: "frankenstein-transformer", latent/cca_attn.py: ``CCAAttention``
and ``CCGQAAttention`` (their ``forward``), ``_apply_causal_convs`` and
``_apply_rope``.  CCA is CCGQA with as many key/value heads as query heads,
so one function computes both.  The steps follow the page's order:

 1. packed down-projection of q and k: ``qk = W_QK x`` (widths Lq, Lkv);
 2. causal convolutions over the sequence on the packed tensor: a
    depth-wise one (k_seq taps per channel), then a grouped one (one group
    of d_h channels per head, k_ch taps), both left-padded with zeros;
 3. q-k-mean: each query head adds the mean of its own pre-convolution
    query and its group's pre-convolution key; each key head adds the
    average of that over the query heads of its group;
 4. value projection; with value-shift, the first half of the value latent
    comes from the current token and the second half from the previous one
    (zero before the first token), the halves concatenated before the split
    into heads;
 5. L2-normalisation of every query and key head to norm sqrt(d_h) (norms
    clamped at 1e-6), keys times exp(beta);
 6. RoPE with half-split pairs at positions 0..S-1 in the latent;
 7. causal softmax attention with scale 1/sqrt(d_h), query head h reading
    key/value head h / (Hq / Hkv);
 8. output projection ``y = W_O o``.

Everything is float64 on the exact (stored) input values; the library's
intermediates are bfloat16/fp16, which the tolerance covers.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from . import rope as _rope


def causal_depthwise_conv(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """a [S, C], w [C, k]: out[t, c] = sum_j w[c, j] a[t - (k - 1) + j, c],
    with a[< 0] = 0 (a cross-correlation over a left-padded sequence)."""
    S, C = a.shape
    k = w.shape[1]
    out = np.zeros_like(a)
    for j in range(k):
        shift = k - 1 - j  # input row t - shift feeds output row t
        if shift < S:
            out[shift:] += a[:S - shift] * w[None, :, j]
    return out


def causal_grouped_conv(a: np.ndarray, w: np.ndarray, group: int) -> np.ndarray:
    """a [S, C], w [C, group, k] with C / group groups of `group` channels:
    out[t, g*group + o] = sum_i sum_j w[g*group + o, i, j] a[t - (k - 1) + j, g*group + i]."""
    S, C = a.shape
    k = w.shape[2]
    G = C // group
    ag = a.reshape(S, G, group)
    wg = w.reshape(G, group, group, k)  # [g, o, i, j]
    out = np.zeros((S, G, group))
    for j in range(k):
        shift = k - 1 - j
        if shift < S:
            out[shift:] += np.einsum("tgi,goi->tgo", ag[:S - shift], wg[..., j])
    return out.reshape(S, C)


def forward_sequence(w, x: np.ndarray, W: Dict[str, np.ndarray], rows: Optional[Sequence[int]] = None,
                     want: bool = False):
    """One sequence x [S, d_model] through the layer (causal).  ``rows``
    limits the outputs to those query positions (attention over the keys
    each sees); ``want`` also returns the intermediates."""
    x = np.asarray(x, np.float64)
    S = x.shape[0]
    Hq, Hkv, dh = w.n_heads, w.n_kv_heads, w.d_h
    Lq, Lkv = w.q_latent, w.kv_latent
    gs = Hq // Hkv
    # 1. packed down-projection
    qk = x @ W["W_QK"].T
    q_pre, k_pre = qk[:, :Lq], qk[:, Lq:]
    # 2. causal convolutions on the packed tensor
    c = qk
    if w.conv_layers >= 1:
        c = causal_depthwise_conv(c, W["conv0"])
    if w.conv_layers >= 2:
        c = causal_grouped_conv(c, W["conv1"], dh)
    q = c[:, :Lq].reshape(S, Hq, dh)
    k = c[:, Lq:].reshape(S, Hkv, dh)
    # 3. q-k-mean
    if w.qk_mean:
        kp = np.repeat(k_pre.reshape(S, Hkv, dh), gs, axis=1)          # key head of each query head
        mean_q = 0.5 * (q_pre.reshape(S, Hq, dh) + kp)
        mean_k = mean_q.reshape(S, Hkv, gs, dh).mean(axis=2)
        q = q + mean_q
        k = k + mean_k
    # 4. values (value-shift: the second half from the previous token)
    if w.value_shift:
        v1 = x @ W["W_V1"].T
        x_prev = np.vstack([np.zeros((1, x.shape[1])), x[:-1]])
        v2 = x_prev @ W["W_V2"].T
        v = np.concatenate([v1, v2], axis=1).reshape(S, Hkv, dh)
    else:
        v = (x @ W["W_V"].T).reshape(S, Hkv, dh)
    # 5. L2 normalisation to norm sqrt(d_h), key temperature
    qn = np.maximum(np.linalg.norm(q, axis=-1, keepdims=True), 1e-6)
    kn = np.maximum(np.linalg.norm(k, axis=-1, keepdims=True), 1e-6)
    q = q * (np.sqrt(dh) / qn)
    k = k * (np.sqrt(dh) / kn) * np.exp(w.key_temp)
    # 6. RoPE (half-split pairs) at positions 0..S-1
    pos = np.arange(S, dtype=np.int32)
    q = _rope(q, pos, w.rope_base, style="half")
    k = _rope(k, pos, w.rope_base, style="half")
    # 7. causal attention, query head h on key/value head h // gs
    rows = np.arange(S) if rows is None else np.asarray(rows)
    o = np.empty((len(rows), Hq, dh))
    scale = 1.0 / np.sqrt(dh)
    for n, t in enumerate(rows):
        for h in range(Hq):
            s = (k[:t + 1, h // gs] @ q[t, h]) * scale
            p = np.exp(s - s.max())
            p /= p.sum()
            o[n, h] = p @ v[:t + 1, h // gs]
    # 8. output projection
    y = o.reshape(len(rows), Lq) @ W["W_O"].T
    if want:
        return {"y": y, "o": o, "q": q, "k": k, "v": v, "qk": qk}
    return y


def forward(w, x: np.ndarray, W: Dict[str, np.ndarray], rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """x [B, S, d_model] -> y [B, len(rows) or S, d_model]."""
    return np.stack([forward_sequence(w, xb, W, rows) for xb in np.asarray(x, np.float64)])

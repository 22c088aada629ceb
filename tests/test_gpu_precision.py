"""Numerics at the edges of the workloads, CUDA path against the fp64 oracle.

- Sharp softmax in decode and prefill: scores of tens of log2 units, where the
  rounding of the operands (the bfloat16 absorbed query, the fp16 score
  partials that the two CTAs of a decode cluster exchange, the fp16 keys and
  values of prefill) is amplified by the exponential.
- The full-size prefill projections (T = 16384 tokens at the DeepSeek-V2
  shapes), checked on sampled token rows that include the first and last
  row tiles of the benchmark's launch.
- Inputs outside the fp16 range on the fp16 prefill path: saturated and
  flagged, never infinite.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_synth as syn
from gpu_util import compare, config_of, to_dev, to_f64, upload_weights

pytestmark = pytest.mark.gpu

W = syn.WORKLOADS
LOG2E = 1.0 / np.log(2.0)


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from head_latent_attention_gb300 import _build
    _build.build()
    import head_latent_attention_gb300 as m
    return m


_WEIGHTS = {}


def weights_of(w: syn.Workload):
    key = (w.variant, w.d_model, w.n_heads, w.d_nope, w.d_rope, w.r_kv, w.r_q, w.n_latent_heads, w.seed)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        _WEIGHTS[key] = upload_weights(w)
    return _WEIGHTS[key]


def scaled(w, name, shape, alpha):
    """A stage input ~ N(0, alpha^2), rounded to the storage type."""
    return syn.store(syn.normal(w.seed, name, shape) * alpha, w.dtype)


# ---------------------------------------------------------------------------
# Decode with a sharp softmax
# ---------------------------------------------------------------------------

def run_decode(mla, oracle_mod, w, lens, q, rope_q, lat_rows, rope_rows, check_b):
    """Decode B sequences with the given stored/exact queries and cache rows;
    compare the sequences in check_b with the oracle's absorbed form."""
    B = len(lens)
    dev_w, ex_w = weights_of(w)
    lay = mla.MlaLayer(config_of(w, B, max(lens)), dev_w, B, ws_max_len=0)
    for b in range(B):
        lay.cache_lat[b, :lens[b]] = to_dev(lat_rows[b][0])
        lay.cache_rope[b, :lens[b]] = to_dev(rope_rows[b][0])
    o = lay.decode(to_dev(q[0]), to_dev(rope_q[0]), torch.tensor(lens, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    st, bits = lay.device_status()
    assert st == 0 and bits == 0, (st, bits)
    got = to_f64(o)
    for b in check_b:
        L = int(lens[b])
        qq = {"q_nope": q[1][b:b + 1], "q_rope": rope_q[1][b:b + 1]}
        ref = oracle_mod.attend(w, [0], [L - 1], qq, lat_rows[b][1][None], rope_rows[b][1][None], ex_w,
                                absorbed=True)
        compare(got[b:b + 1], ref, w.dtype, f"decode b={b} L={L}")
    return got


def test_dsv2_decode_sharp_planted(mla, oracle_mod):
    """Keys aligned with one head's absorbed query reach 30..64 log2 units
    (several within 1.5 units of each other, so their weights all matter),
    at the tile edges, in the middle and at the new token; the sequences are
    split across many work ranges, so the merge sees the sharp rows too."""
    w = W["dsv2_decode"]
    lens = [97, 1000, 2500, 4096, 48]
    B, H = len(lens), w.n_heads
    _, ex_w = weights_of(w)
    qn = syn.stage_inputs(w, "q_nope", (B, H, w.d_nope))
    qr = syn.stage_inputs(w, "q_rope", (B, H, w.d_rope))
    scale = 1.0 / np.sqrt(w.d_nope + w.d_rope)
    W_UK = ex_w["W_UK"].reshape(H, w.d_nope, w.r_kv)
    lat_rows, rope_rows = [], []
    for b, L in enumerate(lens):
        ls, le = syn.cache_rows(w, b, L)
        ls, le = ls.copy(), le.copy()
        h = (37 * b + 5) % H
        qa = W_UK[h].T @ qn[1][b, h]                     # the head's absorbed query (fp64)
        u = qa / np.linalg.norm(qa)
        unit = np.linalg.norm(qa) * scale * LOG2E         # log2-unit score per unit of row norm
        spots = sorted({0, 47, 48, L // 2, L - 2, L - 1} & set(range(L)))
        targets = [64.0, 63.2, 62.5, 40.0, 63.6, 30.0]
        for j, t in zip(spots, targets):
            s, e = syn.store(u * (t / unit), w.dtype)
            ls[j], le[j] = s, e
        lat_rows.append((ls, le))
        rope_rows.append(syn.cache_rows(w, b, L, "cache_rope"))
        s_max = (le @ qa) * scale * LOG2E
        assert s_max.max() > 60.0                          # the sharp regime is reached
    run_decode(mla, oracle_mod, w, lens, qn, qr, lat_rows, rope_rows, check_b=range(B))


def test_dsv2_decode_sharp_scaled(mla, oracle_mod):
    """Queries scaled by 2: random scores with a standard deviation of
    ~2.9 log2 units and maxima of ~14 (the regime where rounding the
    absorbed query to bfloat16 still keeps the error inside the bound; its
    score error grows as |s| 2^-9, like that of any bfloat16 key), at the
    full benchmark batch with its ragged lengths."""
    w = W["dsv2_decode"]
    lens = [int(v) for v in syn.lengths(w)]
    B, H = len(lens), w.n_heads
    qn = scaled(w, "q_nope", (B, H, w.d_nope), 2.0)
    qr = scaled(w, "q_rope", (B, H, w.d_rope), 2.0)
    lat_rows = [syn.cache_rows(w, b, L) for b, L in enumerate(lens)]
    rope_rows = [syn.cache_rows(w, b, L, "cache_rope") for b, L in enumerate(lens)]
    run_decode(mla, oracle_mod, w, lens, qn, qr, lat_rows, rope_rows, check_b=[0, 9, 31, 63])


# ---------------------------------------------------------------------------
# Prefill with a sharp softmax
# ---------------------------------------------------------------------------

def test_dsv2_prefill_sharp_scaled(mla, oracle_mod):
    """Queries scaled by 8 (maxima of ~50 log2 units) through the fp16
    prefill path, ragged: sampled rows in the first, a middle and the last
    query tile, all heads of a subset."""
    w = W["dsv2_prefill"].replace(seq=1100)
    B, S, H = 2, 1100, w.n_heads
    dev_w, ex_w = weights_of(w)
    lay = mla.MlaLayer(config_of(w, B, S), dev_w, B * S)
    qn = scaled(w, "q_nope", (B * S, H, w.d_nope), 8.0)
    qr = scaled(w, "q_rope", (B * S, H, w.d_rope), 8.0)
    lat, rope = [], []
    for b in range(B):
        ls, le = syn.cache_rows(w, b, S)
        rs, re_ = syn.cache_rows(w, b, S, "cache_rope")
        lay.cache_lat[b, :S] = to_dev(ls)
        lay.cache_rope[b, :S] = to_dev(rs)
        lat.append(le)
        rope.append(re_)
    o = lay.prefill(to_dev(qn[0]), to_dev(qr[0]), B, S)
    torch.cuda.synchronize()
    st, bits = lay.device_status()
    assert st == 0 and bits == 0, (st, bits)
    got = to_f64(o)
    heads = np.array([0, 3, 64, 127])
    wsub = w.replace(n_heads=len(heads))
    Wsub = dict(ex_w)
    Wsub["W_UK"] = ex_w["W_UK"].reshape(H, w.d_nope, -1)[heads].reshape(len(heads) * w.d_nope, -1)
    Wsub["W_UV"] = ex_w["W_UV"].reshape(H, w.d_v, -1)[heads].reshape(len(heads) * w.d_v, -1)
    for b, rows in {0: [0, 5, 127, 128, 600, 1099], 1: [64, 1023, 1024, 1099]}.items():
        rows = np.asarray(rows, np.int32)
        t = b * S + rows
        q = {"q_nope": qn[1][t][:, heads], "q_rope": qr[1][t][:, heads]}
        ref = oracle_mod.attend(wsub, np.zeros(len(rows), np.int32), rows, q, lat[b][None], rope[b][None], Wsub)
        compare(got[b, rows][:, heads], ref, w.dtype, f"sharp prefill b={b}")


# ---------------------------------------------------------------------------
# Full-size prefill projections (the benchmark's launch configuration)
# ---------------------------------------------------------------------------

def sample_rows(T, rng):
    """Token rows of the first and last 128-row tiles, tile edges and a
    random spread: 64 rows in all."""
    fixed = [0, 1, 63, 126, 127, 128, 129, 4095, 4096, 8191, 8192, 12288, T - 129, T - 128, T - 2, T - 1]
    rest = rng.choice(np.setdiff1d(np.arange(T), fixed), 64 - len(fixed), replace=False)
    return np.sort(np.concatenate([fixed, rest])).astype(np.int64)


def test_dsv2_project_full_sampled(mla, oracle_mod):
    w = W["dsv2_prefill"]
    B, S = w.batch, w.seq
    T = B * S
    dev_w, ex_w = weights_of(w)
    lay = mla.MlaLayer(config_of(w), dev_w, T, ws_max_len=0)
    xs, xe = syn.activations(w, T)
    pos = np.tile(np.arange(S, dtype=np.int32), B)
    seq = np.repeat(np.arange(B, dtype=np.int32), S)
    qn, qr = lay.project_latent(to_dev(xs), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    st, bits = lay.device_status()
    assert st == 0 and bits == 0, (st, bits)
    rows = sample_rows(T, np.random.default_rng(5))
    ref = oracle_mod.project(w, xe[rows], pos[rows], ex_w)
    rows_t = torch.from_numpy(rows).cuda()
    compare(to_f64(qn[rows_t]), ref["q_nope"], w.dtype, "q_nope rows")
    compare(to_f64(qr[rows_t]), ref["q_rope"], w.dtype, "q_rope rows")
    sq, ps = torch.from_numpy(seq[rows]).cuda().long(), torch.from_numpy(pos[rows]).cuda().long()
    compare(to_f64(lay.cache_lat[sq, ps]), ref["c_kv"], w.dtype, "latent cache rows")
    compare(to_f64(lay.cache_rope[sq, ps]), ref["k_r"], w.dtype, "rope cache rows")


def test_dsv2_out_proj_full_sampled(mla, oracle_mod):
    w = W["dsv2_prefill"]
    T = w.batch * w.seq
    dev_w, ex_w = weights_of(w)
    lay = mla.MlaLayer(config_of(w, 1, 16), dev_w, T, ws_max_len=0)
    os_, oe = syn.stage_inputs(w, "o", (T, w.n_heads * w.d_v))
    y = lay.out_proj(to_dev(os_).view(T, w.n_heads, w.d_v))
    torch.cuda.synchronize()
    rows = sample_rows(T, np.random.default_rng(6))
    got = to_f64(y[torch.from_numpy(rows).cuda()])
    compare(got, oracle_mod.out_proj(oe[rows], ex_w), w.dtype, "W_O rows")


# ---------------------------------------------------------------------------
# fp16 range of the prefill path
# ---------------------------------------------------------------------------

def test_prefill_f16_range_flagged(mla):
    """bfloat16 values beyond fp16's largest finite value (65504) reach the
    fp16 operands of prefill attention through the query and through the key
    and value up-projection: they are saturated (outputs stay finite) and
    the range bit of the status word is raised; in-range inputs raise nothing."""
    for name in ("dsv2_prefill", "small_lm_prefill"):
        w = W[name].replace(seq=160)
        B, S, H = 1, 130, w.n_heads
        dev_w, _ = weights_of(w)
        lay = mla.MlaLayer(config_of(w, B, w.seq), dev_w, B * S)
        qn = to_dev(syn.stage_inputs(w, "q_nope", (B * S, H, w.d_nope))[0])
        qr = to_dev(syn.stage_inputs(w, "q_rope", (B * S, H, w.d_rope))[0]) if w.d_rope else None
        lay.cache_lat[0, :S] = to_dev(syn.cache_rows(w, 0, S)[0])
        if w.d_rope:
            lay.cache_rope[0, :S] = to_dev(syn.cache_rows(w, 0, S, "cache_rope")[0])
        lay.device_status()
        lay.prefill(qn, qr, B, S)
        torch.cuda.synchronize()
        assert lay.device_status() == (mla.MLA_OK, 0)
        # A query element beyond the fp16 range.
        q_big = qn.clone()
        q_big[7, 3, 5] = 1.0e5
        o = lay.prefill(q_big, qr, B, S)
        torch.cuda.synchronize()
        st, bits = lay.device_status()
        assert st == mla.MLA_ERR_DEVICE_DATA and bits == mla.STATUS_F16_RANGE, (name, st, bits)
        assert torch.isfinite(o.float()).all()
        # A cache row whose up-projected keys and values leave the fp16 range.
        lay.cache_lat[0, 11] = 4.0e4
        o = lay.prefill(qn, qr, B, S)
        torch.cuda.synchronize()
        st, bits = lay.device_status()
        assert st == mla.MLA_ERR_DEVICE_DATA and bits == mla.STATUS_F16_RANGE, (name, st, bits)
        assert torch.isfinite(o.float()).all()

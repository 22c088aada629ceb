"""CUDA path against the fp64 oracle, through the C ABI, on seeded inputs.

Reduced sizes keep every model dimension of the workload and span several
tiles with ragged tails; full sizes (the benchmark's launch configuration) are
checked on sampled outputs that the oracle computes one by one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_synth as syn
from gpu_util import compare, config_of, to_dev, to_f64, upload_weights

pytestmark = pytest.mark.gpu

W = syn.WORKLOADS


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
    key = (w.variant, w.dtype, w.d_model, w.n_heads, w.d_nope, w.d_rope, w.r_kv, w.r_q,
           w.n_latent_heads, w.seed)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        _WEIGHTS[key] = upload_weights(w)
    return _WEIGHTS[key]


def subset_heads(w: syn.Workload, Wx, heads):
    """Weights restricted to a subset of heads (heads attend independently)."""
    assert w.variant != syn.VARIANT_MLRA
    H = len(heads)
    out = dict(Wx)
    out["W_UK"] = Wx["W_UK"].reshape(w.n_heads, w.d_nope, -1)[heads].reshape(H * w.d_nope, -1)
    out["W_UV"] = Wx["W_UV"].reshape(w.n_heads, w.d_v, -1)[heads].reshape(H * w.d_v, -1)
    return out


def boundary(w: syn.Workload):
    """Rounding of the tensors the C ABI hands between calls (cache rows,
    projected queries, attention output) to the workload's storage type.
    The oracle feeds these stored values to its next stage and compares each
    GPU stage output with its own value before rounding, so the output's
    rounding to bfloat16 is counted once (a second, independent rounding of
    the reference could differ by one unit in the last place, 0.031 at
    magnitude 4)."""
    return lambda a: syn.store(a, w.dtype)[1]


def make_layer(mla, w, dev_w, max_tokens, max_batch=None, max_seq=None, ws_max_len=None):
    return mla.MlaLayer(config_of(w, max_batch, max_seq), dev_w, max_tokens, ws_max_len=ws_max_len)


# ---------------------------------------------------------------------------
# End-to-end prefill: x -> project_latent -> prefill -> out_proj
# ---------------------------------------------------------------------------

def run_prefill_e2e(mla, oracle_mod, w, B, S, start_pos=None, poison=False):
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, B * S, max_batch=B, max_seq=max(w.seq, S + max(start_pos or [0])))
    if poison:
        # Cache rows nobody writes hold NaN: they must not reach any output.
        lay.cache_lat.fill_(float("nan"))
        if w.d_rope:
            lay.cache_rope.fill_(float("nan"))
    xs, xe = syn.activations(w, B * S)
    sp = np.zeros(B, np.int32) if start_pos is None else np.asarray(start_pos, np.int32)
    pos = (sp[:, None] + np.arange(S)[None, :]).reshape(-1).astype(np.int32)
    seq = np.repeat(np.arange(B, dtype=np.int32), S)
    cache_lat_e = np.zeros((B, lay.cfg.max_seq, w.r_kv))
    cache_rope_e = np.zeros((B, lay.cfg.max_seq, w.d_rope)) if w.d_rope else None
    if start_pos is not None:
        # A cached prefix for chunked prefill: seeded rows before start_pos.
        for b in range(B):
            ls, le = syn.cache_rows(w, b, int(sp[b]))
            lay.cache_lat[b, :sp[b]] = to_dev(ls)
            cache_lat_e[b, :sp[b]] = le
            if w.d_rope:
                rs, re_ = syn.cache_rows(w, b, int(sp[b]), "cache_rope")
                lay.cache_rope[b, :sp[b]] = to_dev(rs)
                cache_rope_e[b, :sp[b]] = re_
    x = to_dev(xs)
    qn, qr = lay.project_latent(x, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda())
    o = lay.prefill(qn, qr, B, S, list(sp) if start_pos is not None else None)
    y = lay.out_proj(o)
    torch.cuda.synchronize()
    st, bits = lay.device_status()
    assert st == 0 and bits == 0
    ref = oracle_mod.prefill(w, xe.reshape(B, S, -1), ex_w, start_pos=sp, cache_lat=cache_lat_e,
                             cache_rope=cache_rope_e, store=boundary(w))
    dt = w.dtype
    compare(to_f64(qn), ref["q_nope" if w.variant == syn.VARIANT_DECOUPLED else "q"], dt, "q_nope")
    if qr is not None:
        compare(to_f64(qr), ref["q_rope"], dt, "q_rope")
    for b in range(B):
        rows = slice(int(sp[b]), int(sp[b]) + S)
        toks = slice(b * S, (b + 1) * S)
        compare(to_f64(lay.cache_lat[b, rows]), ref["c_kv"][toks], dt, f"cache_lat b={b}")
        if w.d_rope:
            compare(to_f64(lay.cache_rope[b, rows]), ref["k_r"][toks], dt, f"cache_rope b={b}")
    compare(to_f64(o), ref["o"], dt, "o")
    compare(to_f64(y).reshape(B, S, -1), ref["y"], dt, "y")


def test_tiny_fp32_prefill_e2e(mla, oracle_mod):
    run_prefill_e2e(mla, oracle_mod, W["tiny_fp32_prefill"], 2, 16)


def test_tiny_fp32_prefill_ragged(mla, oracle_mod):
    w = W["tiny_fp32_prefill"].replace(seq=80)
    run_prefill_e2e(mla, oracle_mod, w, 3, 67)


def test_small_lm_prefill_e2e(mla, oracle_mod):
    run_prefill_e2e(mla, oracle_mod, W["small_lm_prefill"], 2, 200)


def test_dsv2_prefill_e2e(mla, oracle_mod):
    run_prefill_e2e(mla, oracle_mod, W["dsv2_prefill"].replace(seq=256), 2, 130)


def test_chunked_prefill(mla, oracle_mod):
    # Queries appended after a cached prefix (start_pos > 0), ragged per sequence.
    run_prefill_e2e(mla, oracle_mod, W["dsv2_prefill"].replace(seq=512), 2, 70, start_pos=[37, 200])
    run_prefill_e2e(mla, oracle_mod, W["small_lm_prefill"].replace(seq=512), 2, 45, start_pos=[0, 129])


def test_chunked_prefill_unwritten_rows_nan(mla, oracle_mod):
    # Ragged chunks: the shorter sequence's last key tile reaches past its
    # written rows, which hold NaN here.
    run_prefill_e2e(mla, oracle_mod, W["dsv2_prefill"].replace(seq=512), 2, 70, start_pos=[37, 200],
                    poison=True)
    run_prefill_e2e(mla, oracle_mod, W["small_lm_prefill"].replace(seq=512), 2, 45, start_pos=[0, 129],
                    poison=True)


def test_mlra_prefill_e2e(mla, oracle_mod):
    run_prefill_e2e(mla, oracle_mod, W["mlra_decode"].replace(seq=256), 2, 100)


# ---------------------------------------------------------------------------
# Decode stage: synthetic q and caches -> o
# ---------------------------------------------------------------------------

def decode_stage(mla, oracle_mod, w, lens, check_b=None, heads=None, absorbed=True, poison=False):
    B = len(lens)
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, B, max_batch=B, ws_max_len=0)
    if poison:
        # Cache rows past each sequence's length hold NaN: they must reach no output.
        lay.cache_lat.fill_(float("nan"))
        if w.d_rope:
            lay.cache_rope.fill_(float("nan"))
    H = w.n_heads
    qs, qe = syn.stage_inputs(w, "q_nope", (B, H, w.d_nope))
    q_rope = None
    if w.d_rope:
        rs, re_ = syn.stage_inputs(w, "q_rope", (B, H, w.d_rope))
        q_rope = to_dev(rs)
    check_b = list(range(B)) if check_b is None else check_b
    lat_e, rope_e = {}, {}
    for b in range(B):
        ls, le = syn.cache_rows(w, b, int(lens[b]))
        lay.cache_lat[b, :lens[b]] = to_dev(ls)
        lat_e[b] = le
        if w.d_rope:
            rs2, re2 = syn.cache_rows(w, b, int(lens[b]), "cache_rope")
            lay.cache_rope[b, :lens[b]] = to_dev(rs2)
            rope_e[b] = re2
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = lay.decode(to_dev(qs), q_rope, sl)
    torch.cuda.synchronize()
    st, bits = lay.device_status()
    assert st == 0 and bits == 0
    got = to_f64(o)
    hsel = np.arange(H) if heads is None else np.asarray(heads)
    for b in check_b:
        L = int(lens[b])
        cl = lat_e[b][None]
        cr = rope_e[b][None] if w.d_rope else None
        Wsub = dict(ex_w)
        wsub = w
        if heads is not None and w.variant == syn.VARIANT_DECOUPLED:
            Wsub = subset_heads(w, ex_w, hsel)
            wsub = w.replace(n_heads=len(hsel))
        if w.variant == syn.VARIANT_DECOUPLED:
            q = {"q_nope": qe[b:b + 1, hsel], "q_rope": re_[b:b + 1, hsel]}
        else:
            q = {"q": qe[b:b + 1]}
        ref = oracle_mod.attend(wsub, [0], [L - 1], q, cl, cr, Wsub, absorbed=absorbed)
        g = got[b:b + 1, hsel] if w.variant == syn.VARIANT_DECOUPLED else got[b:b + 1]
        compare(g, ref, w.dtype, f"decode b={b} L={L}")
    return lay


def test_dsv2_decode_stage_definition_form(mla, oracle_mod):
    # Definition form (keys and values materialised) at short ragged lengths.
    decode_stage(mla, oracle_mod, W["dsv2_decode"], [1, 2, 127, 300], absorbed=False,
                 heads=list(range(0, 128, 9)))


def test_dsv2_decode_stage_ragged(mla, oracle_mod):
    decode_stage(mla, oracle_mod, W["dsv2_decode"], [1, 64, 65, 511, 513, 1500, 4096])


def test_small_lm_decode_stage(mla, oracle_mod):
    # The small-model form decodes by decompressing the cache each step.
    w = W["small_lm_prefill"].replace(seq=600)
    decode_stage(mla, oracle_mod, w, [1, 2, 63, 64, 65, 300, 600, 129], absorbed=False)


def test_small_lm_decode_stage_unwritten_rows_nan(mla, oracle_mod):
    # Only each sequence's rows up to its length are decompressed; the rest
    # (NaN here, several 128-row tiles of them for the short sequences) are
    # neither computed nor read.
    w = W["small_lm_decode"].replace(seq=700)
    decode_stage(mla, oracle_mod, w, [1, 129, 700, 255, 256, 257, 400, 5], absorbed=False, poison=True)


def test_dsv2_decode_stage_unwritten_rows_nan(mla, oracle_mod):
    decode_stage(mla, oracle_mod, W["dsv2_decode"].replace(seq=1000), [1, 47, 48, 49, 1000, 333],
                 poison=True)


def test_mlra_decode_stage(mla, oracle_mod):
    w = W["mlra_decode"].replace(seq=2048)
    decode_stage(mla, oracle_mod, w, [1, 2, 255, 257, 2048])
    decode_stage(mla, oracle_mod, w.replace(), [300, 40], absorbed=False)


def test_dsv2_decode_full_sampled(mla, oracle_mod):
    w = W["dsv2_decode"]
    lens = syn.lengths(w)
    decode_stage(mla, oracle_mod, w, list(lens), check_b=[0, 17, 40, 63])


def test_mlra_decode_full_sampled(mla, oracle_mod):
    w = W["mlra_decode"]
    decode_stage(mla, oracle_mod, w, list(syn.lengths(w)), check_b=[0, 77, 127])


# ---------------------------------------------------------------------------
# Decode end to end: x -> project_latent (append at L-1) -> decode -> out_proj
# ---------------------------------------------------------------------------

def run_decode_e2e(mla, oracle_mod, w, lens):
    B = len(lens)
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, B, max_batch=B, ws_max_len=0)
    lat_e = np.zeros((B, w.seq, w.r_kv))
    rope_e = np.zeros((B, w.seq, w.d_rope)) if w.d_rope else None
    for b in range(B):
        ls, le = syn.cache_rows(w, b, int(lens[b]))
        lay.cache_lat[b, :lens[b]] = to_dev(ls)
        lat_e[b, :lens[b]] = le
        if w.d_rope:
            rs, re_ = syn.cache_rows(w, b, int(lens[b]), "cache_rope")
            lay.cache_rope[b, :lens[b]] = to_dev(rs)
            rope_e[b, :lens[b]] = re_
    xs, xe = syn.activations(w, B)
    pos = torch.tensor([l - 1 for l in lens], dtype=torch.int32, device="cuda")
    seq = torch.arange(B, dtype=torch.int32, device="cuda")
    qn, qr = lay.project_latent(to_dev(xs), seq, pos)
    o = lay.decode(qn, qr, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    y = lay.out_proj(o)
    torch.cuda.synchronize()
    ref = oracle_mod.decode(w, xe, np.asarray(lens, np.int32), lat_e, rope_e, ex_w, absorbed=True,
                            store=boundary(w))
    compare(to_f64(o), ref["o"], w.dtype, "decode o")
    compare(to_f64(y), ref["y"], w.dtype, "decode y")


def test_dsv2_decode_e2e(mla, oracle_mod):
    run_decode_e2e(mla, oracle_mod, W["dsv2_decode"], [1, 33, 129, 1000, 4096])


def test_mlra_decode_e2e(mla, oracle_mod):
    run_decode_e2e(mla, oracle_mod, W["mlra_decode"].replace(seq=1024), [1, 100, 1024])


# ---------------------------------------------------------------------------
# Full-size prefill, sampled queries
# ---------------------------------------------------------------------------

def prefill_stage_sampled(mla, oracle_mod, w, samples, heads):
    B, S = w.batch, w.seq
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, B * S)
    H = w.n_heads
    qs, qe = syn.stage_inputs(w, "q_nope", (B * S, H, w.d_nope))
    q_rope = None
    if w.d_rope:
        rs, re_ = syn.stage_inputs(w, "q_rope", (B * S, H, w.d_rope))
        q_rope = to_dev(rs)
    lat_e, rope_e = [], []
    for b in range(B):
        ls, le = syn.cache_rows(w, b, S)
        lay.cache_lat[b, :S] = to_dev(ls)
        lat_e.append(le)
        if w.d_rope:
            rs2, re2 = syn.cache_rows(w, b, S, "cache_rope")
            lay.cache_rope[b, :S] = to_dev(rs2)
            rope_e.append(re2)
    o = lay.prefill(to_dev(qs), q_rope, B, S)
    torch.cuda.synchronize()
    got = to_f64(o)
    hsel = np.asarray(heads)
    for b, rows in samples.items():
        rows = np.asarray(rows, np.int32)
        wsub = w.replace(n_heads=len(hsel))
        Wsub = subset_heads(w, ex_w, hsel)
        t = b * S + rows
        if w.variant == syn.VARIANT_DECOUPLED:
            q = {"q_nope": qe[t][:, hsel], "q_rope": re_[t][:, hsel]}
        else:
            q = {"q": qe[t][:, hsel]}
        ref = oracle_mod.attend(wsub, np.zeros(len(rows), np.int32), rows, q, lat_e[b][None],
                                rope_e[b][None] if w.d_rope else None, Wsub)
        compare(got[b, rows][:, hsel], ref, w.dtype, f"prefill b={b}")


def test_dsv2_prefill_full_sampled(mla, oracle_mod):
    w = W["dsv2_prefill"]
    prefill_stage_sampled(mla, oracle_mod, w, {0: [0, 1, 127, 128, 2047, 4095], 3: [4000, 4095]},
                          heads=[0, 77])


def test_small_lm_prefill_full_sampled(mla, oracle_mod):
    w = W["small_lm_prefill"]
    prefill_stage_sampled(mla, oracle_mod, w, {0: [0, 63, 64, 1023], 7: [511, 1000]},
                          heads=list(range(8)))


# ---------------------------------------------------------------------------
# Decode-sized projections (one grouped GEMM per shared input on the tensor
# cores): cache rows scattered to (sequence, position) and the queries
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["dsv2_decode", "small_lm_prefill", "mlra_decode"])
def test_project_decode_sized(mla, oracle_mod, name):
    w = W[name]
    T, B, S = 37, 5, 300
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, T, max_batch=B, max_seq=S)
    xs, xe = syn.activations(w, T)
    rng = np.random.default_rng(7)
    seq = rng.integers(0, B, T).astype(np.int32)
    pos = rng.permutation(S)[:T].astype(np.int32)  # distinct positions, no two tokens share a row
    qn, qr = lay.project_latent(to_dev(xs), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert lay.device_status()[0] == mla.MLA_OK
    ref = oracle_mod.project(w, xe, pos, ex_w)
    lat = to_f64(lay.cache_lat)[seq, pos]
    compare(lat, ref["c_kv"], w.dtype, f"{name} latent rows")
    if w.variant == syn.VARIANT_DECOUPLED:
        compare(to_f64(lay.cache_rope)[seq, pos], ref["k_r"], w.dtype, f"{name} rope rows")
        compare(to_f64(qn), ref["q_nope"], w.dtype, f"{name} q_nope")
        compare(to_f64(qr), ref["q_rope"], w.dtype, f"{name} q_rope")
    else:
        compare(to_f64(qn), ref["q"], w.dtype, f"{name} q")


# ---------------------------------------------------------------------------
# Output projection stage and edge cases
# ---------------------------------------------------------------------------

def test_out_proj_stage(mla, oracle_mod):
    w = W["dsv2_decode"]
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, 300, max_batch=1, max_seq=16, ws_max_len=0)
    os_, oe = syn.stage_inputs(w, "o", (300, w.n_heads * w.d_v))
    y = lay.out_proj(to_dev(os_).view(300, w.n_heads, w.d_v))
    compare(to_f64(y), oracle_mod.out_proj(oe, ex_w), w.dtype, "out_proj")


def test_edge_cases(mla, oracle_mod):
    w = W["dsv2_decode"]
    dev_w, _ = weights_of(w)
    lay = make_layer(mla, w, dev_w, 8, max_batch=4, max_seq=256)
    L = mla.load_library()
    dt = torch.bfloat16
    H = w.n_heads
    e = torch.empty(0, w.d_model, dtype=dt, device="cuda")
    i0 = torch.empty(0, dtype=torch.int32, device="cuda")
    qn = torch.empty(0, H, w.d_nope, dtype=dt, device="cuda")
    qr = torch.empty(0, H, w.d_rope, dtype=dt, device="cuda")
    # Empty calls are no-ops.
    assert mla.mla_project_latent(lay.h, lay.w, e, i0, i0, lay.cache, qn, qr, lay.ws) == 0
    q1 = torch.zeros(4, H, w.d_nope, dtype=dt, device="cuda")
    r1 = torch.zeros(4, H, w.d_rope, dtype=dt, device="cuda")
    o1 = torch.empty(4, H, w.d_v, dtype=dt, device="cuda")
    sl = torch.tensor([1, 256, 0, 257], dtype=torch.int32, device="cuda")
    assert mla.mla_decode(lay.h, lay.w, q1[:0], r1[:0], lay.cache, sl, 0, o1, lay.ws) == 0
    # Workspace too small.
    assert mla.mla_decode(lay.h, lay.w, q1, r1, lay.cache, sl, 4, o1, lay.ws[:1024]) == 3
    # Misaligned bfloat16 pointer.
    bad = torch.zeros(4 * H * w.d_nope + 1, dtype=dt, device="cuda")[1:].view(4, H, w.d_nope)
    assert mla.mla_decode(lay.h, lay.w, bad, r1, lay.cache, sl, 4, o1, lay.ws) == 1
    # Batch above capacity.
    q5 = torch.zeros(5, H, w.d_nope, dtype=dt, device="cuda")
    assert mla.mla_decode(lay.h, lay.w, q5, r1, lay.cache, sl, 5, o1, lay.ws) == 1
    # Cache rows that are not whole 16-byte units: refused before any launch.
    odd = mla.MlaCache(lay.cache.lat, lay.cache.rope, w.r_kv + 1, lay.cache.rope_stride)
    n0 = mla.mla_launch_count()
    assert mla.mla_decode(lay.h, lay.w, q1, r1, odd, sl, 4, o1, lay.ws) == 1
    odd_r = mla.MlaCache(lay.cache.lat, lay.cache.rope, lay.cache.lat_stride, w.d_rope + 1)
    assert mla.mla_decode(lay.h, lay.w, q1, r1, odd_r, sl, 4, o1, lay.ws) == 1
    assert mla.mla_prefill(lay.h, lay.w, q1, r1, odd_r, 1, 1, [0], o1, lay.ws) == 1
    assert mla.mla_launch_count() == n0
    # Prefill beyond the cache.
    assert mla.mla_prefill(lay.h, lay.w, q1, r1, lay.cache, 1, 200, [100], o1, lay.ws) == 4
    # Device-side bad lengths (0 and max_seq + 1) are skipped and flagged.
    lay.device_status()
    assert mla.mla_decode(lay.h, lay.w, q1, r1, lay.cache, sl, 4, o1, lay.ws) == 0
    st, bits = lay.device_status()
    assert st == mla.MLA_ERR_DEVICE_DATA and bits & 4
    st, bits = lay.device_status()
    assert st == 0 and bits == 0
    # Out-of-range positions and sequence ids in the cache append are flagged.
    x = torch.zeros(2, w.d_model, dtype=dt, device="cuda")
    qa = torch.empty(2, H, w.d_nope, dtype=dt, device="cuda")
    qb = torch.empty(2, H, w.d_rope, dtype=dt, device="cuda")
    seq = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
    pos = torch.tensor([300, 0], dtype=torch.int32, device="cuda")
    assert mla.mla_project_latent(lay.h, lay.w, x, seq, pos, lay.cache, qa, qb, lay.ws) == 0
    st, bits = lay.device_status()
    assert st == mla.MLA_ERR_DEVICE_DATA and (bits & 1) and (bits & 2)
    # Small-model decode (no absorbed form): a length beyond max_seq is
    # skipped with a zero output and flagged, a rope query is refused.
    ws_ = W["small_lm_prefill"]
    dw, _ = weights_of(ws_)
    lay2 = make_layer(mla, ws_, dw, 4, max_batch=2, max_seq=64)
    qq = torch.zeros(2, ws_.n_heads, ws_.d_nope, dtype=dt, device="cuda")
    oo = torch.full_like(qq, float("nan"))
    assert mla.mla_decode(lay2.h, lay2.w, qq, qq, lay2.cache, sl[:2], 2, oo, lay2.ws) == 1
    assert mla.mla_decode(lay2.h, lay2.w, qq, None, lay2.cache, sl[:2], 2, oo, lay2.ws) == 0
    st, bits = lay2.device_status()
    assert st == mla.MLA_ERR_DEVICE_DATA and bits == 4
    assert torch.all(oo[1] == 0)


# ---------------------------------------------------------------------------
# Decode batches that stress the split-KV schedule and the merge
# ---------------------------------------------------------------------------

def decode_mixed(mla, oracle_mod, w, lens, max_seq, check_b):
    """Decode a batch whose lengths may be invalid (< 1 or > max_seq): valid
    sequences in check_b match the oracle, invalid ones come out zero and the
    length flag is raised."""
    B = len(lens)
    dev_w, ex_w = weights_of(w)
    lay = make_layer(mla, w, dev_w, B, max_batch=B, max_seq=max_seq, ws_max_len=0)
    H = w.n_heads
    qs, qe = syn.stage_inputs(w, "q_nope", (B, H, w.d_nope))
    rs, re_ = syn.stage_inputs(w, "q_rope", (B, H, w.d_rope))
    lat_h = np.zeros((B, max_seq, w.r_kv), np.uint16)
    rope_h = np.zeros((B, max_seq, w.d_rope), np.uint16)
    lat_e, rope_e = {}, {}
    for b in range(B):
        L = int(lens[b])
        if 1 <= L <= max_seq:
            ls, le = syn.cache_rows(w, b, L)
            rs2, re2 = syn.cache_rows(w, b, L, "cache_rope")
            lat_h[b, :L] = ls
            rope_h[b, :L] = rs2
            if b in check_b:
                lat_e[b], rope_e[b] = le, re2
    lay.cache_lat.copy_(to_dev(lat_h).view(lay.cache_lat.shape))
    lay.cache_rope.copy_(to_dev(rope_h).view(lay.cache_rope.shape))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    lay.device_status()
    o = lay.decode(to_dev(qs), to_dev(rs), sl)
    torch.cuda.synchronize()
    st, bits = lay.device_status()
    invalid = [b for b in range(B) if not 1 <= lens[b] <= max_seq]
    if invalid:
        assert st == mla.MLA_ERR_DEVICE_DATA and bits == 4, (st, bits)
    else:
        assert st == 0 and bits == 0
    got = to_f64(o)
    for b in invalid:
        assert np.all(got[b] == 0.0), f"invalid length at b={b} must give a zero output"
    for b in check_b:
        L = int(lens[b])
        if not 1 <= L <= max_seq:
            continue
        q = {"q_nope": qe[b:b + 1], "q_rope": re_[b:b + 1]}
        ref = oracle_mod.attend(w, [0], [L - 1], q, lat_e[b][None], rope_e[b][None], ex_w, absorbed=True)
        compare(got[b:b + 1], ref, w.dtype, f"decode b={b} L={L}")


def test_decode_mixed_batch(mla, oracle_mod):
    # 70 sequences: two groups of 64 in the absorption and merge kernels, the
    # second ragged; invalid lengths (0 and max_seq + 1) between valid ones,
    # one sequence of the full max_seq, several of one key.
    w = W["dsv2_decode"].replace(n_heads=16)
    rng = np.random.default_rng(7)
    lens = [int(v) for v in rng.integers(1, 301, 70)]
    lens[5], lens[33], lens[69], lens[2], lens[64] = 0, 301, 300, 1, 1
    decode_mixed(mla, oracle_mod, w, lens, 300, check_b=[0, 2, 5, 33, 40, 63, 64, 65, 69])


def test_decode_many_short_sequences(mla, oracle_mod):
    # Thousands of 1..3-key sequences: every work range holds more sequences
    # than the kernel's shared-memory window of prefix sums, and the merge
    # runs over many groups of 64.
    w = W["dsv2_decode"].replace(n_heads=8)
    rng = np.random.default_rng(11)
    B = 6000
    lens = [int(v) for v in rng.integers(1, 4, B)]
    decode_mixed(mla, oracle_mod, w, lens, 4, check_b=[0, 1, 63, 64, 2999, 4095, 5998, 5999])

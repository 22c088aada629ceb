"""CCA / CCGQA through the C ABI against the fp64 oracle ("frankenstein-
transformer", latent/cca_attn.py), on seeded inputs: reduced sizes that span
several 128-token tiles with a ragged tail (every output compared), every
option of the layer, and the full workloads on sampled token rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_synth as syn
from gpu_util import compare, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from head_latent_attention_gb300 import _build
    _build.build()
    import head_latent_attention_gb300 as m
    return m


def cfg_of(mla, w, max_seq=None):
    return mla.make_cca_config(w.d_model, w.n_heads, w.n_kv_heads, w.q_latent, w.kv_latent, w.conv_layers,
                               w.conv_kernel_seq, w.conv_kernel_ch, w.qk_mean, w.value_shift, w.rope_base,
                               w.key_temp, max_seq or w.seq)


def run(mla, w, rows=None, n_check=None):
    """Forward B sequences on the GPU; compare sequences [0, n_check) (rows of
    each, or all) with the oracle.  Returns the GPU output."""
    from oracle import cca
    W = syn.cca_weights(w)
    lay = mla.CcaLayer(cfg_of(mla, w), {k: to_dev(s) for k, (s, _) in W.items()}, w.batch)
    xs, xe = syn.cca_activations(w, w.batch * w.seq)
    y = lay.forward(to_dev(xs).view(w.batch, w.seq, w.d_model))
    torch.cuda.synchronize()
    assert lay.device_status() == (mla.MLA_OK, 0)
    got = to_f64(y)
    ex = {k: e for k, (_, e) in W.items()}
    xe = xe.reshape(w.batch, w.seq, w.d_model)
    for b in range(n_check or w.batch):
        ref = cca.forward_sequence(w, xe[b], ex, rows)
        g = got[b] if rows is None else got[b, rows]
        compare(g, ref, syn.DTYPE_BF16, f"{w.name} b={b}")
    return got


BASE = syn.CcaWorkload("cca_test", d_model=512, n_heads=4, n_kv_heads=4, q_latent=256, kv_latent=256, batch=2,
                       seq=200)
GQA = syn.CcaWorkload("ccgqa_test", d_model=512, n_heads=8, n_kv_heads=2, q_latent=512, kv_latent=128, batch=2,
                      seq=150)


@pytest.mark.parametrize("w", [
    BASE,
    GQA,
    BASE.replace(name="no_conv", conv_layers=0),
    BASE.replace(name="one_conv", conv_layers=1, conv_kernel_seq=3),
    BASE.replace(name="no_mean_no_shift", qk_mean=False, value_shift=False),
    GQA.replace(name="gqa_temp", key_temp=0.7, seed=1),
    syn.CcaWorkload("cca_dh128", d_model=1024, n_heads=4, n_kv_heads=4, q_latent=512, kv_latent=512, batch=1,
                    seq=300),
], ids=lambda w: w.name)
def test_cca_parity(mla, w):
    run(mla, w)


@pytest.mark.parametrize("w", [
    # Many sequence starts inside one 128-row tile: sequences shorter than
    # either convolution's filter, so both causal paddings and the row shifts
    # of every tap cross sequence starts.
    BASE.replace(name="short_seqs", batch=37, seq=3, conv_kernel_seq=5, conv_kernel_ch=4),
    BASE.replace(name="single_token", batch=9, seq=1),
    # The widest filters: 8 depth-wise taps; 4 channel taps in one pass at
    # d_h = 64 and in two passes (two taps each) at d_h = 128.
    BASE.replace(name="widest_filters", conv_kernel_seq=8, conv_kernel_ch=4, seed=2),
    syn.CcaWorkload("dh128_four_taps", d_model=512, n_heads=2, n_kv_heads=2, q_latent=256, kv_latent=256, batch=2,
                    seq=140, conv_kernel_ch=4),
    # An odd number of heads in all (3 query heads, 1 key/value head).
    syn.CcaWorkload("odd_heads", d_model=256, n_heads=3, n_kv_heads=1, q_latent=192, kv_latent=64, batch=2, seq=130,
                    value_shift=False),
], ids=lambda w: w.name)
def test_cca_edges(mla, w):
    run(mla, w)


@pytest.mark.parametrize("name", ["cca_prefill", "ccgqa_prefill"])
def test_cca_full_sampled(mla, name):
    w = syn.CCA_WORKLOADS[name]
    rows = [0, 1, 127, 128, 1000, 2046, 2047]
    run(mla, w, rows=rows, n_check=2)


def test_cca_arguments(mla):
    w = BASE
    assert mla.mla_cca_check_config(cfg_of(mla, w)) == mla.MLA_OK
    bad = [dict(n_kv_heads=3), dict(kv_latent=512), dict(conv_layers=3), dict(q_latent=250)]
    for kw in bad:
        assert mla.mla_cca_check_config(cfg_of(mla, w.replace(**kw))) == mla.MLA_ERR_INVALID_ARG, kw
    # d_h 32 is valid on the page but not run by these kernels.
    assert mla.mla_cca_check_config(cfg_of(mla, w.replace(q_latent=128, kv_latent=128))) == mla.MLA_ERR_UNSUPPORTED
    W = syn.cca_weights(w)
    lay = mla.CcaLayer(cfg_of(mla, w, max_seq=64), {k: to_dev(s) for k, (s, _) in W.items()}, 1)
    x = torch.zeros(1, 65, w.d_model, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    n0 = mla.mla_launch_count()
    assert mla.mla_cca_forward(lay.h, lay.w, x, 1, 65, y, lay.ws) == mla.MLA_ERR_CACHE_OVERFLOW
    x64, y64 = x[:, :64].contiguous(), y[:, :64].contiguous()
    assert mla.mla_cca_forward(lay.h, lay.w, x64, 1, 64, y64, lay.ws[:1024]) == mla.MLA_ERR_WORKSPACE
    assert mla.mla_launch_count() == n0

"""mla_out_proj_static, the output projection that allocates nothing, against
mla_out_proj on the same inputs (and against the oracle).

Its scratch is one fixed buffer that keeps the previous call's contents; two
calls in a row with different token counts and inputs check that a call never
reads what the one before left there.  The file name sorts last so that, in a
run that stops at the first failure, every other GPU test has run before it.
"""
from __future__ import annotations

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


@pytest.mark.parametrize("name", ["dsv2_decode", "mlra_decode"])
def test_static_out_proj_matches_workspace_entry_point(mla, oracle_mod, name):
    w = syn.WORKLOADS[name]
    dev_w, ex_w = upload_weights(w)
    lay = mla.MlaLayer(config_of(w, 1, 16), dev_w, 64, ws_max_len=0)
    K = w.n_heads * w.d_v
    dt = torch.bfloat16 if w.dtype == syn.DTYPE_BF16 else torch.float32
    # Two calls in a row with different token counts (a full decode batch and
    # a ragged one) and different inputs: the second must not see the first's
    # partial sums.
    for T, sub in ((64, 1), (37, 2)):
        o_stored, o_exact = syn.store(syn.normal(w.seed, "o", (T, K), sub=(sub,)), w.dtype)
        o = to_dev(o_stored)
        assert o.dtype == dt
        y_static = torch.full((T, w.d_model), float("nan"), dtype=dt, device="cuda")
        st = mla.mla_out_proj_static(lay.h, lay.w, o, y_static)
        assert st == mla.MLA_OK, mla.mla_status_string(st)
        y_ws = lay.out_proj(o)
        torch.cuda.synchronize()
        compare(to_f64(y_static), to_f64(y_ws), w.dtype, f"{name} static out_proj T={T}")
        compare(to_f64(y_static), oracle_mod.out_proj(o_exact, ex_w), w.dtype, f"{name} static vs oracle T={T}")
    assert lay.device_status()[0] == mla.MLA_OK


def test_static_out_proj_argument_checks(mla):
    w = syn.WORKLOADS["dsv2_decode"]
    dev_w, _ = upload_weights(w)
    lay = mla.MlaLayer(config_of(w, 1, 16), dev_w, 8, ws_max_len=0)
    K = w.n_heads * w.d_v
    o = torch.zeros(8, K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(8, w.d_model, dtype=torch.bfloat16, device="cuda")
    L = mla.load_library()
    assert L.mla_out_proj_static(lay.h.ptr, None, mla._ptr(o), 8, mla._ptr(y), None) == \
        mla.MLA_ERR_INVALID_ARG
    # A misaligned operand is refused before anything is launched.
    yb = torch.zeros(8 * w.d_model + 1, dtype=torch.bfloat16, device="cuda")[1:]
    assert mla.mla_out_proj_static(lay.h, lay.w, o, yb.view(8, w.d_model)) == mla.MLA_ERR_INVALID_ARG
    # No tokens: nothing to do.
    assert mla.mla_out_proj_static(lay.h, lay.w, o[:0], y[:0]) == mla.MLA_OK


def test_static_out_proj_refuses_beyond_buffer(mla):
    """A shape whose split-K partial sums would not fit the fixed 32 MiB
    buffer (T = 128 tokens, d_model = 10496, 512 heads of 128: the planner
    splits the 65536-long reduction into ~7 parts, ~36 MiB of partials) is
    refused with MLA_ERR_WORKSPACE before anything is launched.  The operands
    are real allocations of the full size all the same."""
    cfg = mla.make_config(mla.VARIANT_DECOUPLED, mla.DTYPE_BF16, 10496, 512, 128, 64, 128, 512, 1536, 1,
                          10000.0, 1, 16)
    h = mla.mla_create(cfg)
    K, N, T = 512 * 128, 10496, 128
    W_O = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    wts = mla.make_weights({"W_O": W_O})
    o = torch.zeros(T, K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(T, N, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    n0 = mla.mla_launch_count()
    assert mla.mla_out_proj_static(h, wts, o, y) == mla.MLA_ERR_WORKSPACE
    assert mla.mla_launch_count() == n0
    mla.mla_destroy(h)

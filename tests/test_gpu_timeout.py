"""The give-up path of the bounded device waits, made to run without a fault.

The projection GEMM's pipeline waits (TMA copies landing, MMAs freeing a
stage, the accumulator filling) give up after a host-settable number of SM
clock cycles.  With the limit set to one cycle a wait on a copy that is still
in flight gives up: the kernel stops issuing, lets the copies and MMAs it has
already issued complete, frees its tensor memory and raises the timeout bit.
Nothing here waits on a flag that could stay unset or touches memory out of
bounds; the copies and MMAs all complete normally, only the waits end early.
"""
from __future__ import annotations

import pytest
import torch

import mla_synth as syn
from gpu_util import config_of, to_dev, upload_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from head_latent_attention_gb300 import _build
    _build.build()
    import head_latent_attention_gb300 as m
    return m


@pytest.mark.parametrize("T", [64, 1024])
def test_gemm_wait_timeout_unwinds(mla, T):
    # T = 64: the decode step's split-K output projection (with its reduce
    # kernel); T = 1024: eight row tiles, no split.
    w = syn.WORKLOADS["dsv2_decode"]
    dev_w, _ = upload_weights(w)
    lay = mla.MlaLayer(config_of(w, 1, 16), dev_w, T, ws_max_len=0)
    K = w.n_heads * w.d_v
    o = to_dev(syn.store(syn.normal(w.seed, "o", (T, K), sub=(9,)), w.dtype)[0])
    y_ref = lay.out_proj(o)
    torch.cuda.synchronize()
    assert lay.device_status() == (mla.MLA_OK, 0)

    y = torch.empty_like(y_ref)
    assert mla.mla_set_wait_limit(1) == mla.MLA_OK
    try:
        st = mla.mla_out_proj(lay.h, lay.w, o, y, lay.ws)
        torch.cuda.synchronize()
    finally:
        assert mla.mla_set_wait_limit(0) == mla.MLA_OK
    assert st == mla.MLA_OK
    st, bits = lay.device_status()
    assert st == mla.MLA_ERR_TIMEOUT and bits & mla.STATUS_TIMEOUT, (st, bits)

    # The context is intact: the same call on a re-zeroed workspace gives the
    # same result as before, bit for bit.
    lay.ws.zero_()
    y2 = lay.out_proj(o)
    torch.cuda.synchronize()
    assert lay.device_status() == (mla.MLA_OK, 0)
    assert torch.equal(y2, y_ref)
    assert mla.mla_set_wait_limit(-1) == mla.MLA_ERR_INVALID_ARG

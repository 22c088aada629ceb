"""Helpers shared by the GPU tests: upload seeded inputs, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import mla_synth as syn

# Tolerances of the workload statement: float32 normwise max relative error
# <= 1e-4; bfloat16 relative L2 error <= 1e-2 and max absolute error <= 3e-2
# on unit-scale outputs.  "Unit scale" is applied per output vector (the last
# axis: one head's output of one token, or one token's projected row): each
# vector is divided by the RMS of its reference.  Attention outputs that
# average many keys are much smaller than those of the first rows, so one
# global RMS would fail even an exactly computed output rounded to bfloat16.
F32_MAX_REL = 1e-4
BF16_REL_L2 = 1e-2
BF16_MAX_ABS_UNIT = 3e-2


def to_dev(stored: np.ndarray, device="cuda") -> torch.Tensor:
    if stored.dtype == np.uint16:
        return torch.from_numpy(stored.view(np.int16).copy()).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(stored, np.float32)).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(got, ref, dtype: int, what: str):
    """Assert got ~= ref under the workload tolerances; returns the metrics."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    if dtype == syn.DTYPE_F32:
        m = float(np.max(np.abs(diff)) / max(np.max(np.abs(ref)), 1e-300))
        assert m <= F32_MAX_REL, f"{what}: normwise max rel err {m:.3e} > {F32_MAX_REL}"
        return {"max_rel": m}
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    mabs = float(np.max(np.abs(diff) / np.maximum(rms, 1e-300))) if diff.size else 0.0
    assert l2 <= BF16_REL_L2, f"{what}: rel L2 {l2:.3e} > {BF16_REL_L2}"
    assert mabs <= BF16_MAX_ABS_UNIT, f"{what}: max abs (unit rms) {mabs:.3e} > {BF16_MAX_ABS_UNIT}"
    return {"rel_l2": l2, "max_abs_unit": mabs}


def config_of(w: syn.Workload, max_batch=None, max_seq=None):
    import head_latent_attention_gb300 as mla
    return mla.make_config(w.variant, w.dtype, w.d_model, w.n_heads, w.d_nope, w.d_rope, w.d_v,
                           w.r_kv, w.r_q, w.n_latent_heads, w.rope_base,
                           max_batch or w.batch, max_seq or w.seq)


def upload_weights(w: syn.Workload):
    """(device tensors, exact float64 values) of all weights."""
    dev, exact = {}, {}
    for name, (stored, ex) in syn.weights(w).items():
        dev[name] = to_dev(stored)
        exact[name] = ex
    return dev, exact

"""The C-ABI library on the host: it builds for sm_103a, loads without a GPU,
exports every entry point that include/mla.h declares, and validates
configurations and arguments before touching a device."""
import ctypes
import os
import re

import pytest

import mla_synth as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    from head_latent_attention_gb300 import _build
    _build.build()
    import head_latent_attention_gb300 as mla
    return mla


def declared_entry_points():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(mla_[a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert "mla_decode" in names and "mla_prefill" in names
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in include/ but not exported"
    assert set(lib.EXPORTS) <= set(names)


def cfg(lib, **kw):
    w = syn.WORKLOADS["dsv2_decode"]
    base = dict(variant=w.variant, dtype=w.dtype, d_model=w.d_model, n_heads=w.n_heads,
                d_nope=w.d_nope, d_rope=w.d_rope, d_v=w.d_v, r_kv=w.r_kv, r_q=w.r_q,
                n_latent_heads=w.n_latent_heads, rope_base=w.rope_base, max_batch=w.batch,
                max_seq=w.seq)
    base.update(kw)
    return lib.make_config(**base)


@pytest.mark.parametrize("name", sorted(syn.WORKLOADS))
def test_workload_configs_valid(lib, name):
    w = syn.WORKLOADS[name]
    c = lib.make_config(w.variant, w.dtype, w.d_model, w.n_heads, w.d_nope, w.d_rope, w.d_v,
                        w.r_kv, w.r_q, w.n_latent_heads, w.rope_base, w.batch, w.seq)
    assert lib.mla_check_config(c) == lib.MLA_OK


@pytest.mark.parametrize("bad,code", [
    (dict(d_rope=63), 1),                      # rotated width must be even
    (dict(r_kv=5120), 1),                      # latent rank below d_model (deepseek-mla asserts)
    (dict(r_q=6000), 1),
    (dict(d_v=64), 1),                         # d_v == d_nope
    (dict(n_heads=0), 1),
    (dict(max_seq=0), 1),
    (dict(rope_base=0.0), 1),
    (dict(dtype=7), 1),
    (dict(variant=9), 1),
    (dict(n_latent_heads=2), 1),               # L only for MLRA
    (dict(d_rope=128), 2),                     # RoPE groups wider than the kernels' 64
])
def test_decoupled_config_errors(lib, bad, code):
    assert lib.mla_check_config(cfg(lib, **bad)) == code


def test_small_and_mlra_config_errors(lib):
    small = dict(variant=1, d_model=512, n_heads=8, d_nope=64, d_rope=0, d_v=64, r_kv=256, r_q=0,
                 n_latent_heads=1)
    assert lib.mla_check_config(cfg(lib, **small)) == 0
    # mla_attn __init__: hidden_size divisible by num_heads, head_dim = hidden / heads.
    assert lib.mla_check_config(cfg(lib, **{**small, "n_heads": 7})) == 1
    assert lib.mla_check_config(cfg(lib, **{**small, "d_rope": 8})) == 1
    mlra = dict(variant=2, d_model=2048, n_heads=16, d_nope=128, d_rope=0, d_v=128, r_kv=1024,
                r_q=0, n_latent_heads=4)
    assert lib.mla_check_config(cfg(lib, **mlra)) == 0
    # mlra_attn __init__: L | latent rank, L | heads * head_dim.
    assert lib.mla_check_config(cfg(lib, **{**mlra, "n_latent_heads": 3})) == 1
    # A head spanning two latent blocks: defined (oracle) but not run by the kernels.
    odd = dict(variant=2, d_model=96, n_heads=3, d_nope=32, d_rope=0, d_v=32, r_kv=64, r_q=0,
               n_latent_heads=2)
    assert lib.mla_check_config(cfg(lib, **odd)) == 2


def test_create_rejects_bad_config_without_device(lib):
    out = ctypes.c_void_p(1234)
    st = lib.load_library().mla_create(ctypes.byref(cfg(lib, d_rope=3)), ctypes.byref(out))
    assert st == lib.MLA_ERR_INVALID_ARG
    assert not out.value
    assert lib.load_library().mla_check_config(None) == lib.MLA_ERR_INVALID_ARG


def test_null_handle_paths(lib):
    L = lib.load_library()
    assert L.mla_workspace_size(None, 1, 1, 1) == 0
    assert L.mla_project_latent(None, None, None, 1, None, None, None, None, None, None, 0,
                                None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_prefill(None, None, None, None, None, 1, 1, None, None, None, 0,
                         None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_decode(None, None, None, None, None, None, 1, None, None, 0,
                        None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_out_proj(None, None, None, 1, None, None, 0, None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_out_proj_static(None, None, None, 1, None, None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_copy(None, None, 16, None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_copy(None, None, 0, None) == lib.MLA_OK  # nothing to copy
    L.mla_destroy(None)


def test_status_strings(lib):
    for code in range(8):
        s = lib.mla_status_string(code)
        assert s and s != "unknown status"
    assert lib.mla_status_string(99) == "unknown status"


def test_profile_hook_arguments(lib):
    # Host-only bookkeeping: clearing any declared point is accepted, an
    # unknown point or a half-given pair is refused.
    L = lib.load_library()
    for which in (lib.MLA_PROFILE_DECODE_ATTENTION, lib.MLA_PROFILE_PREFILL_ATTENTION,
                  lib.MLA_PROFILE_DECODE_CALL):
        assert L.mla_set_profile_events(which, None, None) == lib.MLA_OK
    assert L.mla_set_profile_events(3, None, None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_set_profile_events(-1, None, None) == lib.MLA_ERR_INVALID_ARG
    assert L.mla_set_profile_events(0, ctypes.c_void_p(16), None) == lib.MLA_ERR_INVALID_ARG

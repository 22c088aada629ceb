"""fp64 oracle for Multi-Head Latent Attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library (``head_latent_attention_gb300``)
never imports, links or executes anything here, and nothing here imports the
library: the two share no code.  Inputs reach both sides from ``mla_synth``.

The arithmetic lives in ``mla_oracle.c`` (plain C, double precision, written
from the definitions on the pages; see that file's header for the sources).
This module compiles it with gcc, loads it with ctypes, and composes the
per-stage functions into whole forward passes with plain array indexing.

Pinned functions (tests/test_oracle_pins.py): RoPE (both pairings), the three
attention forms, the absorbed forms, the projections and the compositions
below.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

VARIANT_DECOUPLED, VARIANT_SMALL, VARIANT_MLRA = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class use_library:
    """Temporarily route every oracle call through another build of the C
    source (used by the tests that plant a mistake in a copy of the oracle)."""

    def __init__(self, path: str):
        self.path = path
        self.prev = None

    def __enter__(self):
        global _lib
        _load()
        self.prev = _lib
        _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


def _configure(lib):
    D = ctypes.POINTER(ctypes.c_double)
    I = ctypes.POINTER(ctypes.c_int)
    i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
    sig = {
        "orc_linear": [D, l, i, D, i, D, i],
        "orc_rope_interleaved": [D, l, i, i, I, d],
        "orc_rope_half": [D, l, i, i, I, d],
        "orc_decoupled_project": [i, i, i, i, i, i, d, l, D, I, D, D, D, D, D,
                                  D, D, D, D, i],
        "orc_small_project": [i, i, i, i, i, d, l, D, I, D, D, D, D, i],
        "orc_mlra_project": [i, i, i, i, l, D, D, D, D, D, i],
        "orc_decoupled_attend": [i, i, i, i, i, l, I, I, D, D, D, D, l, D, D, i,
                                 D, D],
        "orc_small_attend": [i, i, i, i, d, l, I, I, D, D, l, D, D, i, D, D],
        "orc_mlra_attend": [i, i, i, i, l, I, I, D, D, l, D, D, i, D, D],
        "orc_decoupled_attend_absorbed": [i, i, i, i, i, l, I, I, D, D, D, D, l,
                                          D, D, i, D],
        "orc_mlra_attend_absorbed": [i, i, i, i, l, I, I, D, D, l, D, D, i, D],
        "orc_max_threads": [],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int if name != "orc_linear" else None
    lib.orc_rope_interleaved.restype = None
    lib.orc_rope_half.restype = None
    return lib


def _d(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def default_threads() -> int:
    return int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))


# --------------------------------------------------------------------------
# Elementary steps
# --------------------------------------------------------------------------

def linear(x, W, n_threads: Optional[int] = None) -> np.ndarray:
    """y = x W^T (nn.Linear layout [out, in], no bias)."""
    x = _f64(x)
    W = _f64(W)
    lead = x.shape[:-1]
    x2 = x.reshape(-1, x.shape[-1])
    y = np.empty((x2.shape[0], W.shape[0]), np.float64)
    _load().orc_linear(_d(x2), x2.shape[0], x2.shape[1], _d(W), W.shape[0], _d(y),
                       n_threads or default_threads())
    return y.reshape(*lead, W.shape[0])


def rope(x, pos, base: float = 10000.0, style: str = "interleaved") -> np.ndarray:
    """Rotate the last axis of x [n_rows, n_groups, d] at positions pos [n_rows]."""
    y = _f64(x).copy()
    n_rows, n_groups, d = y.shape
    p = _i32(pos)
    assert p.shape == (n_rows,)
    f = _load().orc_rope_interleaved if style == "interleaved" else _load().orc_rope_half
    f(_d(y), n_rows, n_groups, d, _i(p), float(base))
    return y


def cache_bytes_per_token(w) -> int:
    """Bytes one token adds to the caches: the latent (r_kv) plus, for the
    decoupled variant, the shared rope key (d_rope), in the storage type."""
    per_elem = 4 if w.dtype == 0 else 2
    return (w.r_kv + (w.d_rope if w.variant == VARIANT_DECOUPLED else 0)) * per_elem


# --------------------------------------------------------------------------
# Projections (stage: latent projection + cache append, query path)
# --------------------------------------------------------------------------

def project(w, x, pos, Wts: Dict[str, np.ndarray], use_rope: bool = True,
            n_threads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Per-token projections of x [T, d_model] at positions pos [T].

    Returns ``c_kv`` [T, r_kv] and, per variant, ``k_r`` [T, d_rope] (rotated),
    ``q_nope`` [T, H, d_nope], ``q_rope`` [T, H, d_rope] (decoupled) or ``q``
    [T, H, d] (small-model, MLRA).
    """
    lib = _load()
    x = _f64(x)
    T = x.shape[0]
    pos = _i32(pos)
    nt = n_threads or default_threads()
    H = w.n_heads
    c_kv = np.empty((T, w.r_kv), np.float64)
    if w.variant == VARIANT_DECOUPLED:
        k_r = np.empty((T, w.d_rope), np.float64)
        qn = np.empty((T, H, w.d_nope), np.float64)
        qr = np.empty((T, H, w.d_rope), np.float64)
        _check(lib.orc_decoupled_project(
            w.d_model, H, w.d_nope, w.d_rope, w.r_kv, w.r_q, float(w.rope_base), T,
            _d(x), _i(pos), _d(_f64(Wts["W_DQ"])), _d(_f64(Wts["W_UQ"])),
            _d(_f64(Wts["W_QR"])), _d(_f64(Wts["W_DKV"])), _d(_f64(Wts["W_KR"])),
            _d(c_kv), _d(k_r), _d(qn), _d(qr), nt), "decoupled_project")
        return {"c_kv": c_kv, "k_r": k_r, "q_nope": qn, "q_rope": qr}
    q = np.empty((T, H, w.d_nope), np.float64)
    if w.variant == VARIANT_SMALL:
        _check(lib.orc_small_project(
            w.d_model, H, w.d_nope, w.r_kv, int(use_rope), float(w.rope_base), T,
            _d(x), _i(pos), _d(_f64(Wts["W_Q"])), _d(_f64(Wts["W_DKV"])), _d(c_kv),
            _d(q), nt), "small_project")
    else:
        _check(lib.orc_mlra_project(
            w.d_model, H, w.d_nope, w.r_kv, T, _d(x), _d(_f64(Wts["W_Q"])),
            _d(_f64(Wts["W_DKV"])), _d(c_kv), _d(q), nt), "mlra_project")
    return {"c_kv": c_kv, "q": q}


# --------------------------------------------------------------------------
# Attention over the cache (definition and absorbed forms)
# --------------------------------------------------------------------------

def attend(w, q_b, q_pos, q: Dict[str, np.ndarray], cache_lat, cache_rope,
           Wts: Dict[str, np.ndarray], use_rope: bool = True, absorbed: bool = False,
           want_probs: bool = False, n_threads: Optional[int] = None):
    """Causal attention of queries against the cache.

    q_b [n_q] / q_pos [n_q]: sequence and absolute position of each query (it
    sees keys 0..q_pos).  ``q`` holds ``q_nope``/``q_rope`` (decoupled) or
    ``q``.  cache_lat [B, S_max, r_kv], cache_rope [B, S_max, d_rope] or None.
    Returns o [n_q, H, d_v] (and the weights [n_q, H, S_max] if asked).
    """
    lib = _load()
    q_b, q_pos = _i32(q_b), _i32(q_pos)
    n_q = q_b.shape[0]
    nt = n_threads or default_threads()
    H = w.n_heads
    cl = _f64(cache_lat)
    S_max = cl.shape[1]
    o = np.empty((n_q, H, w.d_v), np.float64)
    probs = np.empty((n_q, H, S_max), np.float64) if want_probs else None
    if absorbed and want_probs:
        raise ValueError("the absorbed form does not report weights")
    if w.variant == VARIANT_DECOUPLED:
        qn, qr, cr = _f64(q["q_nope"]), _f64(q["q_rope"]), _f64(cache_rope)
        args = (H, w.d_nope, w.d_rope, w.d_v, w.r_kv, n_q, _i(q_b), _i(q_pos), _d(qn),
                _d(qr), _d(cl), _d(cr), S_max, _d(_f64(Wts["W_UK"])),
                _d(_f64(Wts["W_UV"])), nt, _d(o))
        if absorbed:
            _check(lib.orc_decoupled_attend_absorbed(*args), "decoupled_attend_absorbed")
        else:
            _check(lib.orc_decoupled_attend(*args, _d(probs)), "decoupled_attend")
    elif w.variant == VARIANT_SMALL:
        if absorbed:
            raise ValueError("RoPE sits between W_UK and the query: no absorbed form")
        _check(lib.orc_small_attend(
            H, w.d_nope, w.r_kv, int(use_rope), float(w.rope_base), n_q, _i(q_b),
            _i(q_pos), _d(_f64(q["q"])), _d(cl), S_max, _d(_f64(Wts["W_UK"])),
            _d(_f64(Wts["W_UV"])), nt, _d(o), _d(probs)), "small_attend")
    else:
        args = (H, w.d_nope, w.r_kv, w.n_latent_heads, n_q, _i(q_b), _i(q_pos),
                _d(_f64(q["q"])), _d(cl), S_max, _d(_f64(Wts["W_UK"])),
                _d(_f64(Wts["W_UV"])), nt, _d(o))
        if absorbed:
            _check(lib.orc_mlra_attend_absorbed(*args), "mlra_attend_absorbed")
        else:
            _check(lib.orc_mlra_attend(*args, _d(probs)), "mlra_attend")
    return (o, probs) if want_probs else o


def out_proj(o, Wts: Dict[str, np.ndarray], n_threads: Optional[int] = None) -> np.ndarray:
    """y = W_O [o_1 ‖ ... ‖ o_H] per token."""
    o = _f64(o)
    return linear(o.reshape(o.shape[0], -1), Wts["W_O"], n_threads)


# --------------------------------------------------------------------------
# Whole passes
# --------------------------------------------------------------------------

def _keep(a):
    return a


def prefill(w, x, Wts: Dict[str, np.ndarray], start_pos: Sequence[int] = None,
            cache_lat=None, cache_rope=None, use_rope: bool = True,
            n_threads: Optional[int] = None, store=None) -> Dict[str, np.ndarray]:
    """Causal prefill of x [B, S, d_model] appended at start_pos[b].

    Projects every token, writes c_KV (and rotated k_R) into the caches at
    (b, start_pos[b] + i), attends each query against keys
    0..start_pos[b] + i, and applies W_O.  Caches default to zeros of length
    max(start_pos) + S.

    ``store``, when given, is applied to every tensor that a staged
    implementation hands from one stage to the next in its storage type (the
    cache rows, the projected queries and the attention output), e.g. a
    rounding to bfloat16; all arithmetic stays in double precision.  The
    returned stage outputs (``c_kv``, ``k_r``, ``q*``, ``o``, ``y``) are the
    values before that rounding; the returned caches hold the stored values.
    """
    store = store or _keep
    x = _f64(x)
    B, S, _ = x.shape
    sp = np.zeros(B, np.int32) if start_pos is None else _i32(start_pos)
    need = int(sp.max()) + S
    if cache_lat is None:
        cache_lat = np.zeros((B, need, w.r_kv))
    cache_lat = _f64(cache_lat).copy()
    if w.variant == VARIANT_DECOUPLED:
        cache_rope = (np.zeros((B, cache_lat.shape[1], w.d_rope)) if cache_rope is None
                      else _f64(cache_rope).copy())
    pos = (sp[:, None] + np.arange(S, dtype=np.int32)[None, :]).astype(np.int32)
    pr = project(w, x.reshape(B * S, -1), pos.reshape(-1), Wts, use_rope, n_threads)
    st = {k: store(v) for k, v in pr.items()}
    q_b = np.repeat(np.arange(B, dtype=np.int32), S)
    for b in range(B):
        cache_lat[b, sp[b]:sp[b] + S] = st["c_kv"][b * S:(b + 1) * S]
        if w.variant == VARIANT_DECOUPLED:
            cache_rope[b, sp[b]:sp[b] + S] = st["k_r"][b * S:(b + 1) * S]
    o = attend(w, q_b, pos.reshape(-1), st, cache_lat, cache_rope, Wts, use_rope,
               n_threads=n_threads)
    y = out_proj(store(o), Wts, n_threads)
    return {"y": y.reshape(B, S, -1), "o": o.reshape(B, S, w.n_heads, w.d_v),
            "cache_lat": cache_lat, "cache_rope": cache_rope, **pr}


def decode(w, x, seq_lens, cache_lat, cache_rope, Wts: Dict[str, np.ndarray],
           absorbed: bool = False, n_threads: Optional[int] = None,
           store=None) -> Dict[str, np.ndarray]:
    """One decode step: the new token x[b] sits at position seq_lens[b] - 1
    (the length includes it); it is projected and appended, then attends keys
    0..seq_lens[b] - 1, and W_O is applied.  ``store`` as in ``prefill``."""
    store = store or _keep
    x = _f64(x)
    B = x.shape[0]
    sl = _i32(seq_lens)
    pos = (sl - 1).astype(np.int32)
    pr = project(w, x, pos, Wts, True, n_threads)
    st = {k: store(v) for k, v in pr.items()}
    cache_lat = _f64(cache_lat).copy()
    if w.variant == VARIANT_DECOUPLED:
        cache_rope = _f64(cache_rope).copy()
    for b in range(B):
        cache_lat[b, pos[b]] = st["c_kv"][b]
        if w.variant == VARIANT_DECOUPLED:
            cache_rope[b, pos[b]] = st["k_r"][b]
    q_b = np.arange(B, dtype=np.int32)
    o = attend(w, q_b, pos, st, cache_lat, cache_rope, Wts, absorbed=absorbed,
               n_threads=n_threads)
    y = out_proj(store(o), Wts, n_threads)
    return {"y": y, "o": o, "cache_lat": cache_lat, "cache_rope": cache_rope, **pr}

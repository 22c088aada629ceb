"""GB300 (sm_103a) Multi-Head Latent Attention: Python binding of the C ABI.

The functions here carry the same names as the entry points declared in
``include/mla.h`` and only marshal arguments: torch tensors become device
pointers, the current torch stream becomes the ``cudaStream_t``.  Every step
of the computation runs in the library's CUDA kernels (``libmla_gb300.so``,
built from ``csrc/`` by ``_build.build()``).  There is no fallback: if the
library is missing or cannot be loaded, importing the entry points raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_gb300.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CACHE_OVERFLOW = 4
MLA_ERR_CUDA = 5
MLA_ERR_TIMEOUT = 6
MLA_ERR_DEVICE_DATA = 7

# Bits of the device status word (mla_get_device_status).
STATUS_POS, STATUS_SEQ, STATUS_LEN, STATUS_TIMEOUT, STATUS_F16_RANGE = 1, 2, 4, 8, 16

VARIANT_DECOUPLED, VARIANT_SMALL, VARIANT_MLRA = 0, 1, 2
DTYPE_F32, DTYPE_BF16 = 0, 1
TORCH_DTYPE = {DTYPE_F32: torch.float32, DTYPE_BF16: torch.bfloat16}

# Entry points declared in include/mla.h.
EXPORTS = ("mla_check_config", "mla_create", "mla_destroy", "mla_workspace_size",
           "mla_project_latent", "mla_prefill", "mla_decode", "mla_out_proj",
           "mla_get_device_status", "mla_status_string", "mla_launch_count",
           "mla_set_profile_events", "mla_out_proj_static", "mla_set_wait_limit", "mla_create_shard",
           "mla_cca_check_config", "mla_cca_create", "mla_cca_destroy", "mla_cca_workspace_size",
           "mla_cca_forward", "mla_cca_get_device_status", "mla_copy")
MLA_PROFILE_DECODE_ATTENTION = 0
MLA_PROFILE_PREFILL_ATTENTION = 1
MLA_PROFILE_DECODE_CALL = 2


class MlaConfig(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("dtype", ctypes.c_int), ("d_model", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("d_nope", ctypes.c_int), ("d_rope", ctypes.c_int),
                ("d_v", ctypes.c_int), ("r_kv", ctypes.c_int), ("r_q", ctypes.c_int),
                ("n_latent_heads", ctypes.c_int), ("rope_base", ctypes.c_double),
                ("max_batch", ctypes.c_int), ("max_seq", ctypes.c_int)]


class MlaWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W_DQ", "W_UQ", "W_QR", "W_DKV", "W_KR", "W_UK", "W_UV", "W_O", "W_Q")]


class MlaCache(ctypes.Structure):
    _fields_ = [("lat", ctypes.c_void_p), ("rope", ctypes.c_void_p),
                ("lat_stride", ctypes.c_int64), ("rope_stride", ctypes.c_int64)]


class MlaCcaConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("d_model", "n_heads", "n_kv_heads", "q_latent", "kv_latent",
                                              "conv_layers", "conv_kernel_seq", "conv_kernel_ch", "qk_mean",
                                              "value_shift")] + \
               [("rope_base", ctypes.c_double), ("key_temp", ctypes.c_double), ("max_seq", ctypes.c_int)]


class MlaCcaWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W_QK", "W_V1", "W_V2", "W_V", "conv0", "conv1", "W_O")]


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {mla_status_string(status)} (status {status})")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "head_latent_attention_gb300._build.build()")
    lib = ctypes.CDLL(path)
    P, I, L, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "mla_check_config": (I, [P]),
        "mla_create": (I, [P, ctypes.POINTER(P)]),
        "mla_create_shard": (I, [P, I, I, ctypes.POINTER(P)]),
        "mla_destroy": (None, [P]),
        "mla_workspace_size": (S, [P, I, I, L]),
        "mla_project_latent": (I, [P, P, P, L, P, P, P, P, P, P, S, P]),
        "mla_prefill": (I, [P, P, P, P, P, I, I, P, P, P, S, P]),
        "mla_decode": (I, [P, P, P, P, P, P, I, P, P, S, P]),
        "mla_out_proj": (I, [P, P, P, L, P, P, S, P]),
        "mla_out_proj_static": (I, [P, P, P, L, P, P]),
        "mla_get_device_status": (I, [P, P, P, ctypes.POINTER(ctypes.c_uint32)]),
        "mla_status_string": (ctypes.c_char_p, [I]),
        "mla_launch_count": (ctypes.c_uint64, []),
        "mla_set_profile_events": (I, [I, P, P]),
        "mla_set_wait_limit": (I, [L]),
        "mla_copy": (I, [P, P, S, P]),
        "mla_cca_check_config": (I, [P]),
        "mla_cca_create": (I, [P, ctypes.POINTER(P)]),
        "mla_cca_destroy": (None, [P]),
        "mla_cca_workspace_size": (S, [P, I, I]),
        "mla_cca_forward": (I, [P, P, P, I, I, P, P, S, P]),
        "mla_cca_get_device_status": (I, [P, P, P, ctypes.POINTER(ctypes.c_uint32)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, what: str):
    if st != MLA_OK:
        raise MlaError(st, what)


def make_config(variant: int, dtype: int, d_model: int, n_heads: int, d_nope: int, d_rope: int,
                d_v: int, r_kv: int, r_q: int, n_latent_heads: int, rope_base: float,
                max_batch: int, max_seq: int) -> MlaConfig:
    return MlaConfig(variant, dtype, d_model, n_heads, d_nope, d_rope, d_v, r_kv, r_q,
                     n_latent_heads, float(rope_base), max_batch, max_seq)


def make_weights(w: Dict[str, torch.Tensor]) -> MlaWeights:
    """Device pointers of the weights present in ``w`` (the rest stay NULL)."""
    mw = MlaWeights()
    for name, _ in MlaWeights._fields_:
        t = w.get(name)
        setattr(mw, name, t.data_ptr() if t is not None else None)
    mw._keep = dict(w)
    return mw


def make_cache(lat: torch.Tensor, rope: Optional[torch.Tensor] = None) -> MlaCache:
    """Cache descriptor from [max_batch, max_seq, width] tensors (rows may be
    strided views of a packed buffer)."""
    for t in (lat, rope):
        if t is not None and t.stride(0) != t.shape[1] * t.stride(1):
            raise ValueError("cache rows of one sequence must be max_seq consecutive rows")
        if t is not None and t.stride(2) != 1:
            raise ValueError("cache rows must be contiguous")
    c = MlaCache(lat.data_ptr(), rope.data_ptr() if rope is not None else None,
                 lat.stride(1), rope.stride(1) if rope is not None else 0)
    c._keep = (lat, rope)
    return c


class Handle:
    """Owner of an ``mla_handle*``."""

    def __init__(self, ptr: ctypes.c_void_p, cfg: MlaConfig):
        self.ptr = ptr
        self.cfg = cfg

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.mla_destroy(self.ptr)
            self.ptr = None


def mla_status_string(status: int) -> str:
    return load_library().mla_status_string(int(status)).decode()


def mla_check_config(cfg: MlaConfig) -> int:
    return load_library().mla_check_config(ctypes.byref(cfg))


def mla_create(cfg: MlaConfig) -> Handle:
    out = ctypes.c_void_p()
    _check(load_library().mla_create(ctypes.byref(cfg), ctypes.byref(out)), "mla_create")
    return Handle(out, cfg)


def shard_config(cfg: MlaConfig, n_shards: int) -> MlaConfig:
    """The part of an MLRA layer that one of n_shards shards computes: H/n
    heads, rank r_kv/n in L/n latent blocks, the same d_model (the shape of a
    shard handle's weights, cache and outputs)."""
    return MlaConfig(cfg.variant, cfg.dtype, cfg.d_model, cfg.n_heads // n_shards, cfg.d_nope, cfg.d_rope,
                     cfg.d_v, cfg.r_kv // n_shards, cfg.r_q, cfg.n_latent_heads // n_shards, cfg.rope_base,
                     cfg.max_batch, cfg.max_seq)


def mla_create_shard(cfg: MlaConfig, shard: int, n_shards: int) -> Handle:
    """Handle for shard `shard` of `n_shards` of an MLRA layer (latent
    sub-head tensor parallelism); its cfg is the shard's own part."""
    out = ctypes.c_void_p()
    _check(load_library().mla_create_shard(ctypes.byref(cfg), int(shard), int(n_shards), ctypes.byref(out)),
           "mla_create_shard")
    return Handle(out, shard_config(cfg, n_shards))


def mla_destroy(h: Handle):
    if h.ptr:
        load_library().mla_destroy(h.ptr)
        h.ptr = None


def mla_workspace_size(h: Handle, batch: int, max_len: int, n_tokens: int) -> int:
    return load_library().mla_workspace_size(h.ptr, batch, max_len, n_tokens)


def mla_project_latent(h: Handle, w: MlaWeights, x: torch.Tensor, seq_idx: torch.Tensor,
                       pos: torch.Tensor, cache: MlaCache, q_nope: torch.Tensor,
                       q_rope: Optional[torch.Tensor], ws: torch.Tensor, stream=None) -> int:
    st = load_library().mla_project_latent(
        h.ptr, ctypes.byref(w), _ptr(x), x.shape[0], _ptr(seq_idx), _ptr(pos),
        ctypes.byref(cache), _ptr(q_nope), _ptr(q_rope), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream))
    return st


def mla_prefill(h: Handle, w: MlaWeights, q_nope: torch.Tensor, q_rope: Optional[torch.Tensor],
                cache: MlaCache, B: int, S: int, start_pos: Optional[Sequence[int]],
                o: torch.Tensor, ws: torch.Tensor, stream=None) -> int:
    sp = None
    if start_pos is not None:
        arr = (ctypes.c_int32 * B)(*[int(v) for v in start_pos])
        sp = ctypes.cast(arr, ctypes.c_void_p)
    return load_library().mla_prefill(
        h.ptr, ctypes.byref(w), _ptr(q_nope), _ptr(q_rope), ctypes.byref(cache), B, S, sp,
        _ptr(o), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def mla_decode(h: Handle, w: MlaWeights, q_nope: torch.Tensor, q_rope: Optional[torch.Tensor],
               cache: MlaCache, seq_lens: torch.Tensor, B: int, o: torch.Tensor,
               ws: torch.Tensor, stream=None) -> int:
    return load_library().mla_decode(
        h.ptr, ctypes.byref(w), _ptr(q_nope), _ptr(q_rope), ctypes.byref(cache), _ptr(seq_lens),
        B, _ptr(o), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def _check_out_proj_args(h: Handle, o: torch.Tensor, y: torch.Tensor):
    """o [T, H*d_v] and y [T, d_model], contiguous, in the handle's dtype:
    the C call trusts T and the row widths it derives from the config."""
    c = h.cfg
    dt = TORCH_DTYPE[c.dtype]
    T = o.shape[0]
    if o.dim() != 2 or o.shape[1] != c.n_heads * c.d_v:
        raise ValueError(f"o must be [T, {c.n_heads * c.d_v}], got {tuple(o.shape)}")
    if y.dim() != 2 or tuple(y.shape) != (T, c.d_model):
        raise ValueError(f"y must be [{T}, {c.d_model}], got {tuple(y.shape)}")
    for name, t in (("o", o), ("y", y)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor")


def mla_out_proj(h: Handle, w: MlaWeights, o: torch.Tensor, y: torch.Tensor, ws: torch.Tensor,
                 stream=None) -> int:
    _check_out_proj_args(h, o, y)
    return load_library().mla_out_proj(h.ptr, ctypes.byref(w), _ptr(o), o.shape[0], _ptr(y),
                                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def mla_out_proj_static(h: Handle, w: MlaWeights, o: torch.Tensor, y: torch.Tensor,
                        stream=None) -> int:
    """mla_out_proj without a workspace: for callers that cannot allocate
    device memory (the scratch is a fixed buffer owned by the library; see
    include/mla.h for its size limit and sharing rules)."""
    _check_out_proj_args(h, o, y)
    return load_library().mla_out_proj_static(h.ptr, ctypes.byref(w), _ptr(o), o.shape[0], _ptr(y),
                                              _stream(stream))


def mla_get_device_status(h: Handle, ws: Optional[torch.Tensor], stream=None):
    bits = ctypes.c_uint32(0)
    st = load_library().mla_get_device_status(h.ptr, _ptr(ws), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def mla_launch_count() -> int:
    return load_library().mla_launch_count()


def mla_copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> int:
    """Stream-ordered copy of src into dst (same byte size) by the SMs; either
    may be a CUDA tensor or a pinned CPU tensor."""
    for t in (dst, src):
        if not t.is_contiguous():
            raise ValueError("mla_copy needs contiguous tensors")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("mla_copy needs CUDA or pinned CPU tensors")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("mla_copy needs tensors of the same byte size")
    return load_library().mla_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                                   _stream(stream))


def mla_set_wait_limit(cycles: int) -> int:
    """Give-up limit (SM clock cycles) of the projection GEMM's bounded waits;
    0 restores the default (a test hook for the timeout path)."""
    return load_library().mla_set_wait_limit(int(cycles))


def mla_set_profile_events(which: int, begin: Optional[torch.cuda.Event],
                           end: Optional[torch.cuda.Event]) -> int:
    """Bracket every launch of one kernel with two torch CUDA events (None clears)."""
    b = ctypes.c_void_p(begin.cuda_event) if begin is not None else None
    e = ctypes.c_void_p(end.cuda_event) if end is not None else None
    return load_library().mla_set_profile_events(which, b, e)


class MlaLayer:
    """Convenience owner of a handle, its weights, caches and workspace.

    ``weights`` maps the mla_weights field names to device tensors in the
    configured dtype.  Caches are allocated packed (rope beside the latent)
    unless given.  The workspace covers prefill of ``ws_max_len`` keys per
    sequence (default max_seq; 0 for a decode-only layer) and projection of
    ``max_tokens`` tokens.  Each method raises ``MlaError`` on a non-OK status.
    """

    def __init__(self, cfg: MlaConfig, weights: Dict[str, torch.Tensor], max_tokens: int,
                 device: str = "cuda", cache_lat: Optional[torch.Tensor] = None,
                 cache_rope: Optional[torch.Tensor] = None, ws_max_len: Optional[int] = None,
                 shard: Optional[Sequence[int]] = None):
        # shard = (s, n): this layer is shard s of n of an MLRA layer (cfg
        # describes the whole layer; weights are the shard's, see
        # mla_create_shard), and its outputs of out_proj are partial sums.
        if shard is not None:
            self.h = mla_create_shard(cfg, shard[0], shard[1])
            cfg = self.h.cfg
        else:
            self.h = mla_create(cfg)
        self.cfg = cfg
        self.w = make_weights(weights)
        dt = TORCH_DTYPE[cfg.dtype]
        if cache_lat is None:
            width = cfg.r_kv + cfg.d_rope
            packed = torch.zeros(cfg.max_batch, cfg.max_seq, width, dtype=dt, device=device)
            cache_lat = packed[:, :, :cfg.r_kv]
            cache_rope = packed[:, :, cfg.r_kv:] if cfg.d_rope else None
        self.cache_lat, self.cache_rope = cache_lat, cache_rope
        self.cache = make_cache(cache_lat, cache_rope)
        n = mla_workspace_size(self.h, cfg.max_batch,
                               cfg.max_seq if ws_max_len is None else ws_max_len, max_tokens)
        self.ws = torch.zeros(n, dtype=torch.uint8, device=device)

    def project_latent(self, x, seq_idx, pos, stream=None):
        T, H = x.shape[0], self.cfg.n_heads
        dt = x.dtype
        q_nope = torch.empty(T, H, self.cfg.d_nope, dtype=dt, device=x.device)
        q_rope = (torch.empty(T, H, self.cfg.d_rope, dtype=dt, device=x.device)
                  if self.cfg.variant == VARIANT_DECOUPLED else None)
        _check(mla_project_latent(self.h, self.w, x, seq_idx, pos, self.cache, q_nope, q_rope,
                                  self.ws, stream), "mla_project_latent")
        return q_nope, q_rope

    def prefill(self, q_nope, q_rope, B, S, start_pos=None, stream=None):
        o = torch.empty(B, S, self.cfg.n_heads, self.cfg.d_v, dtype=q_nope.dtype,
                        device=q_nope.device)
        _check(mla_prefill(self.h, self.w, q_nope, q_rope, self.cache, B, S, start_pos, o,
                           self.ws, stream), "mla_prefill")
        return o

    def decode(self, q_nope, q_rope, seq_lens, stream=None):
        B = q_nope.shape[0]
        o = torch.empty(B, self.cfg.n_heads, self.cfg.d_v, dtype=q_nope.dtype, device=q_nope.device)
        _check(mla_decode(self.h, self.w, q_nope, q_rope, self.cache, seq_lens, B, o, self.ws,
                          stream), "mla_decode")
        return o

    def out_proj(self, o, stream=None):
        o2 = o.reshape(o.shape[0] if o.dim() == 3 else -1, self.cfg.n_heads * self.cfg.d_v)
        y = torch.empty(o2.shape[0], self.cfg.d_model, dtype=o.dtype, device=o.device)
        _check(mla_out_proj(self.h, self.w, o2, y, self.ws, stream), "mla_out_proj")
        return y

    def device_status(self, stream=None):
        return mla_get_device_status(self.h, self.ws, stream)


# ---------------------------------------------------------------------------
# Compressed convolutional attention (CCA / CCGQA)
# ---------------------------------------------------------------------------

def make_cca_config(d_model: int, n_heads: int, n_kv_heads: int, q_latent: int, kv_latent: int,
                    conv_layers: int = 2, conv_kernel_seq: int = 4, conv_kernel_ch: int = 3, qk_mean: bool = True,
                    value_shift: bool = True, rope_base: float = 10000.0, key_temp: float = 0.0,
                    max_seq: int = 4096) -> MlaCcaConfig:
    return MlaCcaConfig(d_model, n_heads, n_kv_heads, q_latent, kv_latent, conv_layers, conv_kernel_seq,
                        conv_kernel_ch, int(qk_mean), int(value_shift), float(rope_base), float(key_temp), max_seq)


class CcaHandle:
    """Owner of an ``mla_cca_handle*``."""

    def __init__(self, ptr: ctypes.c_void_p, cfg: MlaCcaConfig):
        self.ptr = ptr
        self.cfg = cfg

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.mla_cca_destroy(self.ptr)
            self.ptr = None


def mla_cca_check_config(cfg: MlaCcaConfig) -> int:
    return load_library().mla_cca_check_config(ctypes.byref(cfg))


def mla_cca_create(cfg: MlaCcaConfig) -> CcaHandle:
    out = ctypes.c_void_p()
    _check(load_library().mla_cca_create(ctypes.byref(cfg), ctypes.byref(out)), "mla_cca_create")
    return CcaHandle(out, cfg)


def mla_cca_workspace_size(h: CcaHandle, B: int, S: int) -> int:
    return load_library().mla_cca_workspace_size(h.ptr, B, S)


def make_cca_weights(w: Dict[str, torch.Tensor]) -> MlaCcaWeights:
    mw = MlaCcaWeights()
    for name, _ in MlaCcaWeights._fields_:
        t = w.get(name)
        setattr(mw, name, t.data_ptr() if t is not None else None)
    mw._keep = dict(w)
    return mw


def mla_cca_forward(h: CcaHandle, w: MlaCcaWeights, x: torch.Tensor, B: int, S: int, y: torch.Tensor,
                    ws: torch.Tensor, stream=None) -> int:
    c = h.cfg
    for name, t in (("x", x), ("y", y)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.numel() != B * S * c.d_model:
            raise ValueError(f"{name} must be a contiguous bfloat16 [B, S, d_model] tensor")
    return load_library().mla_cca_forward(h.ptr, ctypes.byref(w), _ptr(x), B, S, _ptr(y), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream))


def mla_cca_get_device_status(h: CcaHandle, ws: Optional[torch.Tensor], stream=None):
    bits = ctypes.c_uint32(0)
    st = load_library().mla_cca_get_device_status(h.ptr, _ptr(ws), _stream(stream), ctypes.byref(bits))
    return st, bits.value


class CcaLayer:
    """A CCA / CCGQA layer: handle, weights (bfloat16 device tensors named as
    in ``mla_cca_weights``) and a workspace for up to max_batch sequences of
    the config's max_seq tokens."""

    def __init__(self, cfg: MlaCcaConfig, weights: Dict[str, torch.Tensor], max_batch: int, device: str = "cuda"):
        self.cfg = cfg
        self.h = mla_cca_create(cfg)
        self.w = make_cca_weights(weights)
        self.ws = torch.zeros(mla_cca_workspace_size(self.h, max_batch, cfg.max_seq), dtype=torch.uint8,
                              device=device)

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        B, S = x.shape[0], x.shape[1]
        y = torch.empty_like(x)
        _check(mla_cca_forward(self.h, self.w, x, B, S, y, self.ws, stream), "mla_cca_forward")
        return y

    def device_status(self, stream=None):
        return mla_cca_get_device_status(self.h, self.ws, stream)

/*
 * mla.h — C ABI of the GB300 (sm_103a) Multi-Head Latent Attention library.
 *
 * The library computes the hot path of Multi-Head Latent Attention over a
 * compressed latent KV cache, in three forms taken from web pages on the
 * subject:
 *
 *  DECOUPLED  DeepSeek-V2-style MLA ("bird-of-paradise/deepseek-mla",
 *             src/mla.py, MultiHeadLatentAttention): c_Q = W_DQ x,
 *             q_C = W_UQ c_Q, q_R = RoPE(W_QR c_Q) per head, c_KV = W_DKV x,
 *             k_R = RoPE(W_KR x) shared by all heads; scores
 *             (q_C . W_UK c_KV + q_R . k_R) / sqrt(d_nope + d_rope), causal
 *             softmax, weighted sum of W_UV c_KV, output projection W_O.
 *             RoPE pairs elements (2i, 2i+1) (apply_rotary_emb).
 *  SMALL      small-model MLA ("frankenstein-transformer", latent/mla_attn.py,
 *             MLAAttention): q = W_Q x, k = W_UK c_KV, v = W_UV c_KV, RoPE on
 *             the decompressed q and k with half-split pairs (i, i + d/2)
 *             (_apply_rope), scale 1/sqrt(d).
 *  MLRA       multi-head low-rank attention ("frankenstein-transformer",
 *             latent/mlra_attn.py, MLRAAttention): the latent is split into L
 *             disjoint blocks of rank r_kv/L, each with its own up-projections;
 *             no RoPE, scale 1/sqrt(d).
 *
 * Readings of the pages that this ABI fixes: attention is always causal (the
 * query at absolute position p sees keys 0..p); positions are absolute and
 * 0-based for queries and cached keys alike; the rope-key cache holds k_R
 * after rotation; there are no biases and no dropout; d_v == d_nope.
 *
 * Conventions for every entry point
 *  - Tensors are caller-owned device memory, row-major, in the handle's
 *    dtype (float32 or bfloat16) unless stated.  Weights use the nn.Linear
 *    layout [out, in].  Index arrays are int32.  The library allocates
 *    nothing during compute calls: scratch comes from the caller's workspace
 *    `ws` (device memory, 256-byte aligned, at least mla_workspace_size()
 *    bytes, zero-filled once before first use).
 *  - Pointers handed to the tensor-core path must be 16-byte aligned and row
 *    strides multiples of 16 bytes; violations return MLA_ERR_INVALID_ARG.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream).  Host-side validation happens before anything is
 *    enqueued and returns synchronously; launch failures return MLA_ERR_CUDA.
 *    Bad index data that only the device can see (a position or length out
 *    of range) never traps: the kernel skips that row and sets a bit in the
 *    workspace status word, read with mla_get_device_status().
 *  - A handle is immutable after mla_create(); calls on different streams
 *    are safe when their output buffers and workspaces differ.
 *  - The tensor-core kernels are launched with programmatic dependent launch
 *    (each may start while the previous kernel on the stream finishes and
 *    waits for it before touching its results); setting the environment
 *    variable MLA_PDL=0 before the first call launches them in plain stream
 *    order.  Calls are captured into CUDA graphs as they are.
 *  - After MLA_ERR_TIMEOUT the workspace should be zero-filled again before
 *    reuse: an interrupted call can leave scratch state behind.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misalignment */
    MLA_ERR_UNSUPPORTED = 2,    /* dims or variant this build does not run */
    MLA_ERR_WORKSPACE = 3,      /* ws_bytes smaller than required */
    MLA_ERR_CACHE_OVERFLOW = 4, /* host-known position beyond max_seq */
    MLA_ERR_CUDA = 5,           /* a CUDA runtime or driver call failed */
    MLA_ERR_TIMEOUT = 6,        /* a bounded device wait gave up */
    MLA_ERR_DEVICE_DATA = 7     /* device-side index data was out of range */
} mla_status;

typedef enum {
    MLA_VARIANT_DECOUPLED = 0,
    MLA_VARIANT_SMALL = 1,
    MLA_VARIANT_MLRA = 2
} mla_variant;

typedef enum { MLA_DTYPE_F32 = 0, MLA_DTYPE_BF16 = 1 } mla_dtype;

/* Layer shape.  Field names follow the pages' notation.
 *  d_nope          per-head query/key width (the pages' d_head)
 *  d_rope          decoupled rope-key width (DECOUPLED only, even; else 0)
 *  d_v             per-head value width (== d_nope)
 *  r_kv            latent rank (the cached width)
 *  r_q             query compression rank (DECOUPLED only; else 0)
 *  n_latent_heads  L (MLRA only; 1 otherwise)
 *  rope_base       RoPE base (10000 on the pages)
 *  max_batch, max_seq  cache capacity: positions must lie in [0, max_seq)
 * Checks (mla_check_config): positive sizes; DECOUPLED r_kv < d_model and
 * r_q < d_model (deepseek-mla __init__ asserts) and even d_rope
 * (apply_rotary_emb); SMALL even d_nope; MLRA L | r_kv and L | H*d_nope
 * (MLRAAttention.__init__), and H*d_nope/L a multiple of d_nope so that each
 * head reads one latent block. */
typedef struct {
    int variant;    /* mla_variant */
    int dtype;      /* mla_dtype */
    int d_model, n_heads, d_nope, d_rope, d_v, r_kv, r_q, n_latent_heads;
    double rope_base;
    int max_batch, max_seq;
} mla_config;

/* Device weight pointers, nn.Linear layout [out, in]; unused ones NULL.
 *  DECOUPLED: W_DQ [r_q, d_model], W_UQ [H*d_nope, r_q], W_QR [H*d_rope, r_q],
 *             W_DKV [r_kv, d_model], W_KR [d_rope, d_model],
 *             W_UK [H*d_nope, r_kv], W_UV [H*d_v, r_kv], W_O [d_model, H*d_v]
 *  SMALL:     W_Q [H*d_nope, d_model], W_DKV, W_UK, W_UV, W_O as above
 *  MLRA:      W_Q, W_DKV, W_O as above; W_UK [L, H*d_nope/L, r_kv/L] and
 *             W_UV [L, H*d_v/L, r_kv/L] (the L stacked block projections) */
typedef struct {
    const void *W_DQ, *W_UQ, *W_QR, *W_DKV, *W_KR, *W_UK, *W_UV, *W_O, *W_Q;
} mla_weights;

/* Caches (deepseek-mla __init__: cache_kv [max_batch, max_seq, d_c] and
 * cache_rk [max_batch, max_seq, d_rotate]).  lat: [max_batch, max_seq] rows
 * of lat_stride elements, the first r_kv used; rope: same with rope_stride
 * and d_rope used (DECOUPLED only, else NULL).  A packed layout with
 * rope == lat + r_kv and both strides r_kv + d_rope is allowed. */
typedef struct {
    void *lat;
    void *rope;
    int64_t lat_stride, rope_stride;
} mla_cache;

typedef struct mla_handle mla_handle;

/* Validate a configuration without touching any device.  Returns MLA_OK,
 * MLA_ERR_INVALID_ARG (sizes, null) or MLA_ERR_UNSUPPORTED. */
mla_status mla_check_config(const mla_config *cfg);

/* Create a handle on the current CUDA device: validates cfg and builds the
 * float32 RoPE cos/sin table for positions [0, max_seq) (angles evaluated in
 * double precision on the host).  *out is NULL on failure. */
mla_status mla_create(const mla_config *cfg, mla_handle **out);

/* A handle for one shard of MLRA latent sub-head tensor parallelism
 * ("frankenstein-transformer", latent/mlra_attn.py, module docstring: with
 * the latent split into L sub-heads, each device loads 1/L of the KV cache).
 * cfg describes the whole MLRA layer (H heads, latent rank r_kv split into
 * L blocks); shard s of n_shards (n_shards divides L and H) owns latent
 * blocks [s L/n, (s+1) L/n) and the heads that read them, [s H/n, (s+1) H/n)
 * (head h reads block h L / H).  Every entry point then works on the shard's
 * part, as for an MLRA layer of H/n heads, rank r_kv/n and L/n blocks with
 * the same d_model:
 *  - weights: W_Q rows of its heads [H/n * d_nope, d_model], W_DKV rows of
 *    its latent columns [r_kv/n, d_model], W_UK / W_UV its L/n stacked
 *    blocks, W_O the columns of its heads [d_model, H/n * d_v] (contiguous);
 *  - cache: its latent columns only (r_kv/n wide);
 *  - mla_out_proj gives the shard's partial output W_O,s o_s [T, d_model];
 *    the layer's output is the sum of the partials over all shards (an
 *    all-reduce across the devices, made by the caller).
 * Returns MLA_ERR_UNSUPPORTED for other variants, MLA_ERR_INVALID_ARG for a
 * bad shard index or count. */
mla_status mla_create_shard(const mla_config *cfg, int shard, int n_shards, mla_handle **out);

/* Release a handle and its table (NULL is allowed).  Synchronises nothing;
 * the caller must not destroy a handle with work still in flight. */
void mla_destroy(mla_handle *h);

/* Workspace bytes that any call on up to `batch` sequences of up to
 * `max_len` keys, or on up to `n_tokens` projected tokens, needs (a SMALL
 * decode step always needs room for max_seq rows per sequence).
 * Returns 0 if h is NULL or a size is negative. */
size_t mla_workspace_size(const mla_handle *h, int batch, int max_len,
                          int64_t n_tokens);

/* Latent projection, query projection and cache append, per token t of
 * sequence seq_idx[t] at absolute position pos[t] (deepseek-mla forward,
 * query path and use_cache branch; mla_attn / mlra_attn forward):
 *  DECOUPLED: cache.lat[seq, pos] = W_DKV x,  cache.rope[seq, pos] =
 *             RoPE_pos(W_KR x), q_nope = W_UQ W_DQ x  [T, H, d_nope],
 *             q_rope = RoPE_pos(W_QR W_DQ x) per head [T, H, d_rope]
 *  SMALL:     cache.lat[seq, pos] = W_DKV x, q_nope = RoPE_half,pos(W_Q x)
 *             [T, H, d_nope]; q_rope must be NULL
 *  MLRA:      cache.lat[seq, pos] = W_DKV x, q_nope = W_Q x; q_rope NULL
 * x [T, d_model]; seq_idx, pos: device int32 [T].  T == 0 is a no-op.
 * Tokens whose seq_idx or pos is out of range are skipped (no cache row is
 * written; their query rows are zero) and flagged in the workspace status
 * word.  Workspace: the c_Q intermediate (DECOUPLED). */
mla_status mla_project_latent(mla_handle *h, const mla_weights *w, const void *x,
                              int64_t T, const int32_t *seq_idx, const int32_t *pos,
                              const mla_cache *cache, void *q_nope, void *q_rope,
                              void *ws, size_t ws_bytes, void *stream);

/* Causal prefill attention of S new queries per sequence against the cache
 * (deepseek-mla forward; mla_attn / mlra_attn forward in decoder mode).
 * Query i of sequence b sits at position start_pos[b] + i and sees cached
 * keys 0..start_pos[b] + i (which mla_project_latent must have written).
 * q_nope [B, S, H, d_nope], q_rope [B, S, H, d_rope] (DECOUPLED, else NULL),
 * o [B, S, H, d_v].  start_pos: HOST int32 [B] (NULL means all zero);
 * start_pos[b] + S > max_seq returns MLA_ERR_CACHE_OVERFLOW.  The keys and
 * values of every cached row in use are up-projected into the workspace.
 * bfloat16 runs both attention contractions with fp16 operands (finer
 * rounding than bfloat16, same tensor-core rate): query elements and
 * up-projected keys and values must lie within fp16's range (|v| < 65520);
 * larger ones are saturated to +-65504 and flagged (status bit 16). */
mla_status mla_prefill(mla_handle *h, const mla_weights *w, const void *q_nope,
                       const void *q_rope, const mla_cache *cache, int B, int S,
                       const int32_t *start_pos, void *o, void *ws, size_t ws_bytes,
                       void *stream);

/* One decode step for B sequences, weight-absorbed: the query of sequence b
 * sits at position seq_lens[b] - 1 and sees cached keys 0..seq_lens[b] - 1
 * (the length includes the new token, which mla_project_latent must have
 * appended).  DECOUPLED: q_abs = W_UK,h^T q_nope,h; scores q_abs . c_j +
 * q_rope,h . k_R,j over the latent cache; o_lat = softmax-weighted sum of c_j;
 * o_h = W_UV,h o_lat.  MLRA: the same per latent block.  SMALL: RoPE sits
 * between W_UK and the query, so there is no absorbed form; the keys and
 * values of every cache row up to max_seq are decompressed (keys rotated)
 * into the workspace each step and attended like a one-token prefill (the
 * workspace is then prefill-sized for max_seq rows, see
 * mla_workspace_size).  q_nope [B, H, d_nope], q_rope [B, H, d_rope] or NULL,
 * o [B, H, d_v]; seq_lens: DEVICE int32 [B], each in [1, max_seq] (others
 * are skipped, their output rows are zero, and the length bit is set in the
 * workspace status word).  B <= max_batch.  bfloat16 MLA/MLRA run on the
 * tensor cores: a scheduler kernel, the absorption, the split-KV attention
 * and one kernel that merges split sequences and applies W_UV. */
mla_status mla_decode(mla_handle *h, const mla_weights *w, const void *q_nope,
                      const void *q_rope, const mla_cache *cache,
                      const int32_t *seq_lens, int B, void *o, void *ws,
                      size_t ws_bytes, void *stream);

/* Output projection y = W_O [o_1 ‖ ... ‖ o_H] (deepseek-mla output_proj;
 * out_proj in mla_attn / mlra_attn).  o [T, H*d_v], y [T, d_model].  The
 * workspace holds split-K partial sums when T is small (decode). */
mla_status mla_out_proj(mla_handle *h, const mla_weights *w, const void *o, int64_t T,
                        void *y, void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, read and clear the status words of the workspace
 * (ws may be NULL) and of the handle (used by calls without a workspace).
 * *bits receives the flags OR-ed together (1: position out of range,
 * 2: sequence index out of range, 4: decode length out of range, 8: a bounded
 * device wait timed out and the kernel gave up, 16: a value that the
 * bfloat16 tensor-core prefill hands to its fp16 operands (a query element,
 * an up-projected key or value, or a rope key of a cache row some query
 * sees) lay beyond fp16's finite range, |v| >= 65520, and was saturated to
 * +-65504).  Returns MLA_OK when no flag was set, MLA_ERR_TIMEOUT when bit 8
 * was, MLA_ERR_DEVICE_DATA otherwise. */
mla_status mla_get_device_status(mla_handle *h, void *ws, void *stream, uint32_t *bits);

/* Output projection that allocates nothing: the same y = W_O [o_1 ‖ ... ‖ o_H]
 * as mla_out_proj (same arguments minus the workspace), for callers that can
 * neither allocate device memory nor hand the library a workspace — e.g. a
 * plugin inside an inference runtime that has reserved all device memory for
 * its own pool, or a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable.  The pages have no counterpart: this is
 * a deployment convenience, not part of the method.
 *  - Scratch (the split-K partial sums of small token counts) lives in one
 *    32 MiB buffer owned by the library (a static device array, held by every
 *    GPU that loads the library until the process exits).  A call whose
 *    partial sums would exceed it returns MLA_ERR_WORKSPACE; use mla_out_proj
 *    with a workspace then.
 *  - The first call on each device looks the buffer's device address up
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture on the device.
 *  - All calls on a device share the buffer, which keeps the previous call's
 *    contents (each call overwrites what it reads, so nothing needs clearing):
 *    calls whose executions overlap on the GPU (other streams or threads) race
 *    on it, and the caller must serialise them.
 *  - Device-side flags (timeouts) go to the handle's status word, read with
 *    mla_get_device_status(h, NULL, stream, &bits). */
mla_status mla_out_proj_static(mla_handle *h, const mla_weights *w, const void *o, int64_t T,
                               void *y, void *stream);

/* ---- Compressed convolutional attention (CCA) and its grouped form ----
 *
 * "frankenstein-transformer", latent/cca_attn.py (CCAAttention,
 * CCGQAAttention): q, k and v are down-projected into a compressed latent and
 * the whole attention runs there; only the output projection returns to
 * d_model.  Per token, in the page's order:
 *  - qk = W_QK x (query latent q_latent = n_heads * d_h, key latent
 *    kv_latent = n_kv_heads * d_h, packed);
 *  - causal convolutions over the sequence on the packed qk (conv_layers of
 *    them): depth-wise with conv_kernel_seq taps, then grouped (one group of
 *    d_h channels per head) with conv_kernel_ch taps, both left-padded;
 *  - q-k-mean (qk_mean != 0): query head h adds (q_pre,h + k_pre,g(h)) / 2,
 *    key head g the average of that over its query heads (g(h) = h / (n_heads
 *    / n_kv_heads));
 *  - values v = W_V x, or with value_shift != 0 [W_V1 x_t | W_V2 x_{t-1}]
 *    (x_{-1} = 0), the two halves concatenated before the split into heads;
 *  - q and k L2-normalised to norm sqrt(d_h) (norms clamped at 1e-6), k
 *    times exp(key_temp);
 *  - RoPE with half-split pairs at positions 0..S-1 in the latent;
 *  - causal softmax attention, scale 1/sqrt(d_h), query head h reading
 *    key/value head g(h); y = W_O o.
 * CCA is the case n_kv_heads == n_heads.  bfloat16 in and out; the grouped
 * convolution, the projections and the attention run on the tensor cores
 * (the convolution and the attention's keys and values with fp16 operands:
 * values beyond fp16's range saturate and set status bit 16), the
 * depth-wise convolution and the normalisation on the CUDA cores; d_h in
 * {64, 128}. */
typedef struct {
    int d_model, n_heads, n_kv_heads, q_latent, kv_latent;
    int conv_layers;      /* 0, 1 or 2 */
    int conv_kernel_seq;  /* depth-wise sequence convolution taps (1..8) */
    int conv_kernel_ch;   /* grouped channel convolution taps (1..4) */
    int qk_mean, value_shift;
    double rope_base;
    double key_temp;      /* the key temperature beta (its exponential scales k) */
    int max_seq;          /* longest sequence a forward call may take */
} mla_cca_config;

/* Device bfloat16 weights, nn.Linear layout [out, in]: W_QK [q_latent +
 * kv_latent, d_model]; value_shift: W_V1, W_V2 [kv_latent / 2, d_model],
 * otherwise W_V [kv_latent, d_model]; conv0 [q_latent + kv_latent,
 * conv_kernel_seq] (conv_layers >= 1); conv1 [q_latent + kv_latent, d_h,
 * conv_kernel_ch] (conv_layers == 2); W_O [d_model, q_latent].  Unused NULL. */
typedef struct {
    const void *W_QK, *W_V1, *W_V2, *W_V, *conv0, *conv1, *W_O;
} mla_cca_weights;

typedef struct mla_cca_handle mla_cca_handle;

/* Checks of the page's constructors: positive sizes; n_kv_heads | n_heads;
 * n_heads | q_latent, n_kv_heads | kv_latent, equal and even d_h;
 * kv_latent <= q_latent; conv_layers in {0, 1, 2}; value_shift needs even
 * n_kv_heads and kv_latent.  MLA_ERR_UNSUPPORTED for shapes the kernels do
 * not run (d_h not 64 or 128; latent widths, or the value halves, not
 * multiples of 64; more taps than the limits above). */
mla_status mla_cca_check_config(const mla_cca_config *cfg);

/* Handle on the current device: validates cfg and builds the float32 RoPE
 * table for positions [0, max_seq) (angles in double precision). */
mla_status mla_cca_create(const mla_cca_config *cfg, mla_cca_handle **out);
void mla_cca_destroy(mla_cca_handle *h);

/* Workspace bytes of a forward call on B sequences of S tokens (0 on bad
 * arguments). */
size_t mla_cca_workspace_size(const mla_cca_handle *h, int B, int S);

/* y = CCA(x) for B sequences of S tokens each (causal, positions from 0):
 * x [B, S, d_model], y [B, S, d_model], device bfloat16, 16-byte aligned.
 * S <= max_seq.  Scratch from ws (status word in its first 256 bytes, as for
 * the MLA calls); keys and values beyond fp16's range are saturated and
 * flagged (status bit 16).  Asynchronous on stream. */
mla_status mla_cca_forward(mla_cca_handle *h, const mla_cca_weights *w, const void *x, int B, int S, void *y,
                           void *ws, size_t ws_bytes, void *stream);

/* As mla_get_device_status, for a CCA workspace. */
mla_status mla_cca_get_device_status(mla_cca_handle *h, void *ws, void *stream, uint32_t *bits);

/* Static English text for a status code. */
const char *mla_status_string(mla_status s);

/* ---- Staging ----
 *
 * Copy `bytes` from src to dst on the stream, with the SMs rather than a copy
 * engine.  Either pointer may be device memory or pinned host memory
 * (cudaHostAlloc / cudaHostRegister), which a kernel reaches over the host
 * link through the same pointer under unified addressing; the copy is
 * launched like the library's other kernels (programmatic dependent launch),
 * so staging a step's inputs and reading back its result chain with the
 * step's kernels.  Any alignment; 16-byte aligned buffers copy as 16-byte
 * vectors.  Returns MLA_ERR_INVALID_ARG for a null pointer, a pointer no
 * kernel can reach (unregistered pageable host memory) or overlapping ranges,
 * MLA_ERR_CUDA if the launch fails.  Nothing is checked on the device. */
mla_status mla_copy(void *dst, const void *src, size_t bytes, void *stream);

/* ---- Diagnostics (used by the benchmark; not needed for computing) ---- */

/* Number of kernels this library has launched in this process so far. */
uint64_t mla_launch_count(void);

/* Test hook for the give-up path of the bounded device waits: the pipeline
 * waits of the projection GEMM (used by every bfloat16 projection, the
 * prefill key/value up-projection and mla_out_proj) give up after `cycles`
 * SM clock cycles instead of the default of about one second; 0 restores the
 * default.  A wait that gives up stops the kernel's issue, lets the copies and
 * MMAs it already issued complete, frees its tensor memory and sets the
 * timeout bit (mla_get_device_status then returns MLA_ERR_TIMEOUT and the
 * call's outputs are undefined).  Process-wide and read at each launch: set it
 * only while no other thread is calling into the library.  Negative values
 * return MLA_ERR_INVALID_ARG. */
mla_status mla_set_wait_limit(int64_t cycles);

typedef enum {
    MLA_PROFILE_DECODE_ATTENTION = 0,  /* the split-KV latent attention kernel */
    MLA_PROFILE_PREFILL_ATTENTION = 1, /* the causal flash attention kernel */
    MLA_PROFILE_DECODE_CALL = 2,       /* every launch of one mla_decode call (absorption, split-KV
                                          attention, merge, W_UV), from the first to the last */
    MLA_PROFILE_COUNT = 3
} mla_profile_point;

/* Process-wide timing hook: while set, every launch of the kernel named by
 * `which` is bracketed by records of `begin` and `end` on the stream of the
 * call that launches it (inside stream capture they are recorded as external
 * events, i.e. event-record nodes of the graph the caller can time).  begin/end are cudaEvent_t handles
 * owned by the caller; NULL clears the hook.  Not thread-safe: set it only
 * while no other thread is calling into the library. */
mla_status mla_set_profile_events(int which, void *begin, void *end);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */

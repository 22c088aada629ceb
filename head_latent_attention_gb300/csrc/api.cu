// C ABI entry points: argument validation, workspace layout, kernel dispatch.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "mla_internal.cuh"

using namespace mla;

namespace mla {

static unsigned long long g_launches = 0;
static cudaEvent_t g_prof_begin[MLA_PROFILE_COUNT] = {};
static cudaEvent_t g_prof_end[MLA_PROFILE_COUNT] = {};

bool pdl_enabled()
{
    static const bool on = [] {
        const char *v = getenv("MLA_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}

void note_launch(int n) { __atomic_fetch_add(&g_launches, (unsigned long long)n, __ATOMIC_RELAXED); }

static long long g_gemm_wait_cycles = 0;  // 0: the default limit
long long gemm_wait_cycles()
{
    const long long v = __atomic_load_n(&g_gemm_wait_cycles, __ATOMIC_RELAXED);
    return v > 0 ? v : ptx_default_wait_cycles();
}

// Inside stream capture the record is made external, so that it becomes an
// event-record node of the graph the caller can time; outside capture it is a
// plain record.  A failed diagnostic record must not surface as the error of
// the next launch, so its error state is cleared.
static void profile_record(cudaEvent_t ev, cudaStream_t s)
{
    if (!ev) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        e = cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else
        e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) (void)cudaGetLastError();
}

void profile_begin(int which, cudaStream_t s) { profile_record(g_prof_begin[which], s); }

void profile_end(int which, cudaStream_t s) { profile_record(g_prof_end[which], s); }

}  // namespace mla

namespace {

constexpr int kDecodeChunk = 512;  // keys per split of the CUDA-core decode
// Estimated cost of one extra segment of the tensor-core MLA decode, in keys:
// a sequence boundary inside a range (segment-end stores, the next query
// load, the pipeline refill) costs about 15,000 cycles against about 1,850
// per 48-key tile, i.e. about eight tiles.
constexpr int kSegmentCostKeys = 384;
constexpr double kLog2e = 1.4426950408889634;

size_t esize(const mla_config &c) { return c.dtype == MLA_DTYPE_F32 ? 4 : 2; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int rope_dim_of(const mla_config &c)
{
    if (c.variant == MLA_VARIANT_DECOUPLED) return c.d_rope;
    if (c.variant == MLA_VARIANT_SMALL) return c.d_nope;
    return 0;
}

// Latent width one head attends over, and heads that share one latent block.
int r_lat_of(const mla_config &c) { return c.r_kv / c.n_latent_heads; }
int heads_per_block_of(const mla_config &c) { return c.n_heads / c.n_latent_heads; }

int decode_splits(const mla_config &c) { return (c.max_seq + kDecodeChunk - 1) / kDecodeChunk; }

// Workspace regions, each 256-byte aligned, after the status header.
struct ProjectWs { size_t cq, split, end; };
struct OutProjWs { size_t split, end; };
struct DecodeWs { size_t q_abs, o_lat, o_part, ml_part, prefix, end; };
struct PrefillWs { size_t start_pos, k, v, kr, end; };

// The projection GEMMs of one call, in the shapes mla_project_latent runs
// them (used both to size and to launch; the pointers are filled in later).
struct ProjGemms {
    GemmArgs g[5];
    int n = 0;
};

// The projection GEMMs of mla_project_latent, as they are launched (the
// pointers may be null when only the workspace is being sized).  Products
// that read the same input form one segment list; a decode-sized bfloat16
// call launches each list as one grouped weight-streaming GEMM, any other
// call one GEMM per product.
ProjGemms project_gemms(const mla_handle *h, int64_t T, bool allow_group, const mla_weights *w = nullptr,
                        const void *x = nullptr, const int32_t *seq_idx = nullptr, const int32_t *pos = nullptr,
                        const mla_cache *cache = nullptr, void *q_nope = nullptr, void *q_rope = nullptr,
                        void *cq = nullptr)
{
    const mla_config &c = h->cfg;
    const int M = (int)T, H = c.n_heads;
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    Epilogue e_lat;
    e_lat.out = cache ? cache->lat : nullptr;
    e_lat.ldc = cache ? cache->lat_stride : c.r_kv;
    e_lat.row_seq = seq_idx; e_lat.row_pos = pos; e_lat.seq_rows = c.max_seq;
    e_lat.max_batch = c.max_batch; e_lat.max_seq = c.max_seq;
    Epilogue e_rope = e_lat;
    e_rope.out = cache ? cache->rope : nullptr;
    e_rope.ldc = cache ? cache->rope_stride : c.d_rope;
    e_rope.rope_mode = kRopeInterleaved; e_rope.rope_dim = c.d_rope;
    e_rope.rope_table = h->rope_table; e_rope.rope_pos = pos;
    Epilogue e_cq;
    e_cq.out = cq; e_cq.ldc = c.r_q;
    Epilogue e_qn;
    e_qn.out = q_nope; e_qn.ldc = (int64_t)H * c.d_nope;
    Epilogue e_qr;
    e_qr.out = q_rope; e_qr.ldc = (int64_t)H * c.d_rope;
    e_qr.rope_mode = kRopeInterleaved; e_qr.rope_dim = c.d_rope;
    e_qr.rope_table = h->rope_table; e_qr.rope_pos = pos; e_qr.max_seq = c.max_seq;
    if (c.variant == MLA_VARIANT_SMALL) {
        e_qn.rope_mode = kRopeHalf; e_qn.rope_dim = c.d_nope;
        e_qn.rope_table = h->rope_table; e_qn.rope_pos = pos; e_qn.max_seq = c.max_seq;
    }
    auto seg = [](const void *W, int N, int K, const Epilogue &e) {
        GemmSegment s;
        s.B = Mat2D{W, N, K, K};
        s.epi = e;
        s.N = N;
        return s;
    };
    GemmSegment lists[2][kMaxSeg];
    int nl[2] = {0, 0};
    lists[0][nl[0]++] = seg(w ? w->W_DKV : nullptr, c.r_kv, c.d_model, e_lat);
    if (dec) {
        lists[0][nl[0]++] = seg(w ? w->W_KR : nullptr, c.d_rope, c.d_model, e_rope);
        lists[0][nl[0]++] = seg(w ? w->W_DQ : nullptr, c.r_q, c.d_model, e_cq);
        lists[1][nl[1]++] = seg(w ? w->W_UQ : nullptr, H * c.d_nope, c.r_q, e_qn);
        lists[1][nl[1]++] = seg(w ? w->W_QR : nullptr, H * c.d_rope, c.r_q, e_qr);
    } else {
        lists[0][nl[0]++] = seg(w ? w->W_Q : nullptr, H * c.d_nope, c.d_model, e_qn);
    }
    const void *inputs[2] = {x, cq};
    const int in_cols[2] = {c.d_model, c.r_q};
    ProjGemms r;
    for (int l = 0; l < 2; ++l) {
        if (!nl[l]) continue;
        GemmArgs g;
        g.A = Mat2D{inputs[l], M, in_cols[l], in_cols[l]};
        g.M = M;
        g.K = in_cols[l];
        g.nseg = nl[l];
        for (int i = 0; i < nl[l]; ++i) g.seg[i] = lists[l][i];
        if (allow_group && c.dtype == MLA_DTYPE_BF16 && M <= 128 && nl[l] > 1 && gemm_tc_supported(g)) {
            r.g[r.n++] = g;
            continue;
        }
        for (int i = 0; i < nl[l]; ++i) {
            GemmArgs one;
            one.A = g.A;
            one.M = M;
            one.K = g.K;
            one.B = lists[l][i].B;
            one.N = lists[l][i].N;
            one.epi = lists[l][i].epi;
            r.g[r.n++] = one;
        }
    }
    return r;
}

size_t split_bytes(const mla_handle *h, const GemmArgs &g)
{
    return h->cfg.dtype == MLA_DTYPE_BF16 ? gemm_tc_workspace(g, h->num_sms) : 0;
}

ProjectWs project_ws(const mla_handle *h, int64_t T)
{
    const mla_config &c = h->cfg;
    ProjectWs w;
    w.cq = kWsHeader;
    size_t n = c.variant == MLA_VARIANT_DECOUPLED ? (size_t)T * c.r_q * esize(c) : 0;
    w.split = round_up(w.cq + n, 256);
    size_t sb = 0;
    if (T > 0 && T <= INT32_MAX) {
        // Either launch form may run (grouping depends on the caller's strides).
        for (bool grouped : {false, true}) {
            const ProjGemms pg = project_gemms(h, T, grouped);
            for (int i = 0; i < pg.n; ++i) sb = std::max(sb, split_bytes(h, pg.g[i]));
        }
    }
    w.end = round_up(w.split + sb, 256);
    return w;
}

OutProjWs out_proj_ws(const mla_handle *h, int64_t T)
{
    const mla_config &c = h->cfg;
    OutProjWs w;
    w.split = kWsHeader;
    size_t sb = 0;
    if (T > 0 && T <= INT32_MAX) {
        const int K = c.n_heads * c.d_v;
        GemmArgs g;
        g.A = Mat2D{nullptr, T, K, K};
        g.B = Mat2D{nullptr, c.d_model, K, K};
        g.M = (int)T; g.N = c.d_model; g.K = K;
        sb = split_bytes(h, g);
    }
    w.end = round_up(w.split + sb, 256);
    return w;
}

bool use_tc_decode(const mla_handle *h)
{
    const mla_config &c = h->cfg;
    // The kernel reads the absorbed queries in the head-interleaved layout
    // that only the absorption kernel writes.
    return c.dtype == MLA_DTYPE_BF16 && c.variant == MLA_VARIANT_DECOUPLED && h->decode_clusters > 0 &&
           decode_tc_supported(c.n_heads, c.r_kv, c.d_rope) && absorb_supported(r_lat_of(c), c.d_nope);
}

bool use_mlra_tc(const mla_handle *h)
{
    const mla_config &c = h->cfg;
    return c.dtype == MLA_DTYPE_BF16 && c.variant == MLA_VARIANT_MLRA &&
           mlra_tc_supported(c.n_heads, c.n_latent_heads, c.r_kv, c.d_rope);
}

DecodeWs decode_ws(const mla_handle *h, int B)
{
    const mla_config &c = h->cfg;
    DecodeWs w;
    size_t lat = (size_t)B * c.n_heads * r_lat_of(c);
    // The tensor-core MLA decode reads the absorbed query head-interleaved,
    // 128 head rows per chunk.
    size_t qsz = use_tc_decode(h) ? (size_t)B * kQChunks * kQRows * 8 : lat;
    size_t parts = use_tc_decode(h)  ? (size_t)(h->decode_clusters + B) * c.n_heads
                   : use_mlra_tc(h) ? (size_t)(mlra_tc_ctas() + B) * c.n_heads
                                     : (size_t)B * decode_splits(c) * c.n_heads;
    w.q_abs = kWsHeader;
    w.o_lat = round_up(w.q_abs + qsz * esize(c), 256);
    w.o_part = round_up(w.o_lat + lat * esize(c), 256);
    w.ml_part = round_up(w.o_part + parts * r_lat_of(c) * 4, 256);
    w.prefix = round_up(w.ml_part + parts * 2 * 4, 256);
    // the split-KV schedule (at most one range per SM)
    w.end = round_up(w.prefix + decode_sched_bytes(B, h->num_sms), 256);
    return w;
}

PrefillWs prefill_ws(const mla_config &c, int B, int64_t kv_rows)
{
    PrefillWs w;
    size_t rows = (size_t)B * kv_rows * c.n_heads;
    w.start_pos = kWsHeader;
    w.k = round_up(w.start_pos + (size_t)B * 4, 256);
    w.v = round_up(w.k + rows * c.d_nope * esize(c), 256);
    w.kr = round_up(w.v + rows * c.d_v * esize(c), 256);
    w.end = round_up(w.kr + (size_t)B * kv_rows * c.d_rope * 2, 256);
    return w;
}

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

#define MLA_TRY_CUDA(expr)                              \
    do {                                                \
        cudaError_t _e = (expr);                        \
        if (_e != cudaSuccess) return MLA_ERR_CUDA;     \
    } while (0)

// Every tensor the library reads or writes must be 16-byte aligned when the
// dtype is bfloat16 (tensor-memory-access copies need it).
bool align_ok(const mla_config &c, std::initializer_list<const void *> ptrs)
{
    if (c.dtype != MLA_DTYPE_BF16) return true;
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return false;
    return true;
}

// y[M, N] = x[M, K] W^T with x, W row-major (W in nn.Linear layout [N, K]).
GemmArgs linear_args(const void *x, int64_t ldx, const void *W, int64_t ldw, int M, int N, int K,
                     void *out, int64_t ldc)
{
    GemmArgs g;
    g.A = Mat2D{x, M, K, ldx};
    g.B = Mat2D{W, N, K, ldw};
    g.M = M; g.N = N; g.K = K;
    g.epi.out = out; g.epi.ldc = ldc;
    return g;
}

// bfloat16 runs on the tensor cores, float32 on the CUDA cores.
mla_status run_gemm(const mla_handle *h, GemmArgs g, uint32_t *status, cudaStream_t s, float *split = nullptr)
{
    if (!g.epi.status) g.epi.status = status;
    for (int i = 0; i < g.nseg; ++i)
        if (!g.seg[i].epi.status) g.seg[i].epi.status = status;
    g.split_ws = split;
    if (h->cfg.dtype == MLA_DTYPE_BF16) {
        if (!gemm_tc_supported(g)) return MLA_ERR_UNSUPPORTED;
        return cuda_status(gemm_tc(g, h->num_sms, s));
    }
    return cuda_status(gemm_simt(MLA_DTYPE_F32, g, s));
}

#define MLA_TRY(expr)                       \
    do {                                    \
        mla_status _st = (expr);            \
        if (_st != MLA_OK) return _st;      \
    } while (0)

}  // namespace

extern "C" {

mla_status mla_check_config(const mla_config *c)
{
    if (!c) return MLA_ERR_INVALID_ARG;
    if (c->variant < MLA_VARIANT_DECOUPLED || c->variant > MLA_VARIANT_MLRA) return MLA_ERR_INVALID_ARG;
    if (c->dtype != MLA_DTYPE_F32 && c->dtype != MLA_DTYPE_BF16) return MLA_ERR_INVALID_ARG;
    if (c->d_model <= 0 || c->n_heads <= 0 || c->d_nope <= 0 || c->d_v <= 0 || c->r_kv <= 0 ||
        c->max_batch <= 0 || c->max_seq <= 0 || c->n_latent_heads <= 0 || !(c->rope_base > 0.0))
        return MLA_ERR_INVALID_ARG;
    if (c->d_v != c->d_nope) return MLA_ERR_INVALID_ARG;
    switch (c->variant) {
    case MLA_VARIANT_DECOUPLED:
        // deepseek-mla __init__: d_c < d_embed and d_c1 < d_embed;
        // apply_rotary_emb: the rotated width is even.
        if (c->d_rope <= 0 || c->d_rope % 2 || c->r_q <= 0 || c->n_latent_heads != 1)
            return MLA_ERR_INVALID_ARG;
        if (c->r_kv >= c->d_model || c->r_q >= c->d_model) return MLA_ERR_INVALID_ARG;
        break;
    case MLA_VARIANT_SMALL:
        // mla_attn __init__: head_dim = hidden_size / num_heads, divisible.
        if (c->d_rope != 0 || c->r_q != 0 || c->n_latent_heads != 1) return MLA_ERR_INVALID_ARG;
        if (c->d_model % c->n_heads || c->d_nope != c->d_model / c->n_heads || c->d_nope % 2)
            return MLA_ERR_INVALID_ARG;
        break;
    case MLA_VARIANT_MLRA:
        // mlra_attn __init__: L | latent_rank and L | num_heads * head_dim.
        if (c->d_rope != 0 || c->r_q != 0) return MLA_ERR_INVALID_ARG;
        if (c->d_model % c->n_heads || c->d_nope != c->d_model / c->n_heads) return MLA_ERR_INVALID_ARG;
        if (c->r_kv % c->n_latent_heads || (c->n_heads * c->d_nope) % c->n_latent_heads)
            return MLA_ERR_INVALID_ARG;
        // Each head must read exactly one latent block.
        if ((c->n_heads * c->d_nope / c->n_latent_heads) % c->d_nope) return MLA_ERR_UNSUPPORTED;
        break;
    }
    int rd = rope_dim_of(*c);
    if (rd > 0 && (rd > 64 || 64 % rd)) return MLA_ERR_UNSUPPORTED;
    if (c->d_v > 128 || c->d_nope + c->d_rope > 256) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

// A handle computing the layer described by cfg (already validated).
static mla_status create_handle(const mla_config *cfg, int shard, int n_shards, mla_handle **out)
{
    mla_handle *h = new (std::nothrow) mla_handle();
    if (!h) return MLA_ERR_CUDA;
    h->cfg = *cfg;
    h->shard = shard;
    h->n_shards = n_shards;
    h->rope_dim = rope_dim_of(*cfg);
    h->rope_table = nullptr;
    h->status = nullptr;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
        cudaMalloc(&h->status, 256) != cudaSuccess) {
        delete h;
        return MLA_ERR_CUDA;
    }
    if (cudaMemset(h->status, 0, 256) != cudaSuccess) {
        mla_destroy(h);
        return MLA_ERR_CUDA;
    }
    h->decode_clusters = 0;
    if (cfg->dtype == MLA_DTYPE_BF16 && cfg->variant == MLA_VARIANT_DECOUPLED &&
        decode_tc_supported(cfg->n_heads, cfg->r_kv, cfg->d_rope))
        h->decode_clusters = decode_tc_max_clusters();
    if (h->rope_dim > 0) {
        // cos/sin of pos * base^(-2i/d) (deepseek-mla precompute_freqs_cis,
        // mla_attn _apply_rope), evaluated in double and stored as float.
        int half = h->rope_dim / 2;
        std::vector<float2> tab((size_t)cfg->max_seq * half);
        for (int p = 0; p < cfg->max_seq; ++p)
            for (int i = 0; i < half; ++i) {
                double theta = pow(cfg->rope_base, -2.0 * i / (double)h->rope_dim);
                double a = (double)p * theta;
                tab[(size_t)p * half + i] = make_float2((float)cos(a), (float)sin(a));
            }
        if (cudaMalloc(&h->rope_table, tab.size() * sizeof(float2)) != cudaSuccess ||
            cudaMemcpy(h->rope_table, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
                cudaSuccess) {
            mla_destroy(h);
            return MLA_ERR_CUDA;
        }
    }
    *out = h;
    return MLA_OK;
}

mla_status mla_create(const mla_config *cfg, mla_handle **out)
{
    if (!out) return MLA_ERR_INVALID_ARG;
    *out = nullptr;
    mla_status st = mla_check_config(cfg);
    if (st != MLA_OK) return st;
    return create_handle(cfg, 0, 1, out);
}

mla_status mla_create_shard(const mla_config *cfg, int shard, int n_shards, mla_handle **out)
{
    if (!out) return MLA_ERR_INVALID_ARG;
    *out = nullptr;
    mla_status st = mla_check_config(cfg);
    if (st != MLA_OK) return st;
    if (cfg->variant != MLA_VARIANT_MLRA) return MLA_ERR_UNSUPPORTED;
    const int L = cfg->n_latent_heads;
    if (n_shards < 1 || shard < 0 || shard >= n_shards || L % n_shards || cfg->n_heads % n_shards)
        return MLA_ERR_INVALID_ARG;
    // mlra_attn module docstring: device i loads 1/L of the cache.  The shard
    // is the MLRA layer restricted to its latent blocks and the heads that
    // read them (contiguous ranges, since head h reads block h L / H); its
    // output projection takes W_O's columns of those heads, so the layer's
    // output is the sum of the shards' partial outputs.
    mla_config eff = *cfg;
    eff.n_heads = cfg->n_heads / n_shards;
    eff.r_kv = cfg->r_kv / n_shards;
    eff.n_latent_heads = L / n_shards;
    return create_handle(&eff, shard, n_shards, out);
}

void mla_destroy(mla_handle *h)
{
    if (!h) return;
    if (h->rope_table) cudaFree(h->rope_table);
    if (h->status) cudaFree(h->status);
    delete h;
}

size_t mla_workspace_size(const mla_handle *h, int batch, int max_len, int64_t n_tokens)
{
    if (!h || batch < 0 || max_len < 0 || n_tokens < 0) return 0;
    const mla_config &c = h->cfg;
    size_t need = kWsHeader;
    need = std::max(need, project_ws(h, n_tokens).end);
    need = std::max(need, out_proj_ws(h, n_tokens).end);
    if (c.variant != MLA_VARIANT_SMALL) need = std::max(need, decode_ws(h, batch).end);
    else need = std::max(need, prefill_ws(c, batch, c.max_seq).end);  // decode re-decompresses the cache
    need = std::max(need, prefill_ws(c, batch, max_len).end);
    return need;
}

mla_status mla_project_latent(mla_handle *h, const mla_weights *w, const void *x, int64_t T,
                              const int32_t *seq_idx, const int32_t *pos, const mla_cache *cache,
                              void *q_nope, void *q_rope, void *ws, size_t ws_bytes, void *stream)
{
    if (!h || !w || !cache || T < 0) return MLA_ERR_INVALID_ARG;
    if (T == 0) return MLA_OK;
    const mla_config &c = h->cfg;
    if (T > (int64_t)c.max_batch * c.max_seq || T > INT32_MAX) return MLA_ERR_INVALID_ARG;
    if (!x || !seq_idx || !pos || !q_nope || !ws || !cache->lat || !w->W_DKV) return MLA_ERR_INVALID_ARG;
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    if (dec) {
        if (!q_rope || !cache->rope || !w->W_DQ || !w->W_UQ || !w->W_QR || !w->W_KR) return MLA_ERR_INVALID_ARG;
        if (cache->rope_stride < c.d_rope) return MLA_ERR_INVALID_ARG;
    } else if (q_rope || !w->W_Q) {
        return MLA_ERR_INVALID_ARG;
    }
    if (cache->lat_stride < c.r_kv) return MLA_ERR_INVALID_ARG;
    if (!align_ok(c, {x, q_nope, q_rope, cache->lat, cache->rope, w->W_DQ, w->W_UQ, w->W_QR, w->W_DKV,
                      w->W_KR, w->W_Q, ws}))
        return MLA_ERR_INVALID_ARG;
    ProjectWs L = project_ws(h, T);
    if (ws_bytes < L.end) return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *status = (uint32_t *)ws;
    char *wsb = (char *)ws;
    float *split = (float *)(wsb + L.split);

    // Latent and (decoupled) rope key written straight into the caches, then
    // the query projections.
    const ProjGemms pg = project_gemms(h, T, true, w, x, seq_idx, pos, cache, q_nope, q_rope, dec ? wsb + L.cq : nullptr);
    for (int i = 0; i < pg.n; ++i) MLA_TRY(run_gemm(h, pg.g[i], status, s, split));
    return MLA_OK;
}

// Whether the prefill runs on the tensor-core path (bfloat16, supported head
// widths); its TMA reads of the rope cache need rows of whole 16-byte units.
static bool prefill_uses_tc(const mla_config &c)
{
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    return c.dtype == MLA_DTYPE_BF16 && prefill_tc_supported(c.d_nope, dec ? c.d_rope : 0, c.d_v);
}

// The prefill computation once the (device) start positions are in the
// workspace: up-projected keys and values of rows [0, kv_rows) of every
// sequence, then causal attention of S queries per sequence.  The caller has
// validated every argument.
static mla_status prefill_core(mla_handle *h, const mla_weights *w, const void *q_nope, const void *q_rope,
                               const mla_cache *cache, int B, int S, int64_t kv_rows, void *o, void *ws,
                               cudaStream_t s)
{
    const mla_config &c = h->cfg;
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    PrefillWs L = prefill_ws(c, B, kv_rows);
    char *wsb = (char *)ws;
    int32_t *d_sp = (int32_t *)(wsb + L.start_pos);
    void *kbuf = wsb + L.k, *vbuf = wsb + L.v;
    const int H = c.n_heads;
    const int64_t ldk = (int64_t)H * c.d_nope, ldv = (int64_t)H * c.d_v;

    // Keys and values of every cached row in use (deepseek-mla forward:
    // UK_proj / UV_proj of the cached latent; mla_attn: k is then rotated;
    // mlra_attn: block-wise up-projections concatenated per head).
    const bool tc = prefill_uses_tc(c);
    int nblk = c.variant == MLA_VARIANT_MLRA ? c.n_latent_heads : 1;
    int sub_rank = c.r_kv / nblk, sub_k = H * c.d_nope / nblk, sub_v = H * c.d_v / nblk;
    for (int blk = 0; blk < nblk; ++blk) {
        GemmArgs gk;
        gk.A = Mat2D{(const char *)cache->lat + (size_t)blk * sub_rank * esize(c),
                     (int64_t)c.max_batch * c.max_seq, sub_rank, cache->lat_stride};
        gk.a_row_batch = c.max_seq;
        gk.B = Mat2D{(const char *)w->W_UK + (size_t)blk * sub_k * sub_rank * esize(c), sub_k, sub_rank,
                     sub_rank};
        gk.M = (int)kv_rows; gk.N = sub_k; gk.K = sub_rank; gk.batch = B;
        gk.epi.out = (char *)kbuf + (size_t)blk * sub_k * esize(c);
        gk.epi.ldc = ldk;
        gk.epi.batch_stride = kv_rows * ldk;
        gk.epi.out_f16 = tc;
        gk.epi.range_start = d_sp;
        gk.epi.range_len = S;
        if (c.variant == MLA_VARIANT_SMALL) {
            gk.epi.rope_mode = kRopeHalf; gk.epi.rope_dim = c.d_nope;
            gk.epi.rope_table = h->rope_table; gk.epi.max_seq = c.max_seq;
        }
        MLA_TRY(run_gemm(h, gk, (uint32_t *)ws, s));
        GemmArgs gv = gk;
        gv.B = Mat2D{(const char *)w->W_UV + (size_t)blk * sub_v * sub_rank * esize(c), sub_v, sub_rank,
                     sub_rank};
        gv.N = sub_v;
        gv.epi = Epilogue();
        gv.epi.out = (char *)vbuf + (size_t)blk * sub_v * esize(c);
        gv.epi.ldc = ldv;
        gv.epi.batch_stride = kv_rows * ldv;
        gv.epi.out_f16 = tc;
        gv.epi.range_start = d_sp;
        gv.epi.range_len = S;
        MLA_TRY(run_gemm(h, gv, (uint32_t *)ws, s));
    }
    const float scale_log2 = (float)(kLog2e / sqrt((double)(c.d_nope + (dec ? c.d_rope : 0))));
    if (tc) {
        PrefillTcArgs t;
        t.B = B; t.S = S; t.H = H;
        t.d_nope = c.d_nope; t.d_rope = dec ? c.d_rope : 0; t.d_v = c.d_v;
        t.max_batch = c.max_batch; t.max_seq = c.max_seq;
        t.kv_rows = kv_rows;
        t.q_nope = q_nope; t.q_rope = dec ? q_rope : nullptr;
        t.k = kbuf; t.v = vbuf;
        t.rope = dec ? cache->rope : nullptr; t.rope_stride = cache->rope_stride;
        t.k_rope16 = wsb + L.kr;
        t.start_pos = d_sp;
        t.scale_log2 = scale_log2;
        t.o = o;
        t.status = (uint32_t *)ws;
        MLA_TRY_CUDA(prefill_tc(t, s));
        return MLA_OK;
    }
    PrefillArgs p;
    p.dtype = c.dtype;
    p.B = B; p.S = S; p.H = H;
    p.d_qk_nope = c.d_nope; p.d_rope = dec ? c.d_rope : 0; p.d_v = c.d_v;
    p.q_nope = q_nope; p.q_rope = dec ? q_rope : nullptr;
    p.k = kbuf; p.v = vbuf; p.kv_rows = kv_rows;
    p.rope = dec ? cache->rope : nullptr; p.rope_stride = cache->rope_stride;
    p.max_seq = c.max_seq;
    p.start_pos = d_sp;
    p.scale_log2 = scale_log2;
    p.o = o;
    MLA_TRY_CUDA(prefill_simt(p, s));
    return MLA_OK;
}

mla_status mla_prefill(mla_handle *h, const mla_weights *w, const void *q_nope, const void *q_rope,
                       const mla_cache *cache, int B, int S, const int32_t *start_pos, void *o,
                       void *ws, size_t ws_bytes, void *stream)
{
    if (!h || !w || !cache || B < 0 || S < 0) return MLA_ERR_INVALID_ARG;
    if (B == 0 || S == 0) return MLA_OK;
    const mla_config &c = h->cfg;
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    if (B > c.max_batch) return MLA_ERR_INVALID_ARG;
    if (!q_nope || !o || !ws || !cache->lat || !w->W_UK || !w->W_UV) return MLA_ERR_INVALID_ARG;
    if (dec && (!q_rope || !cache->rope || cache->rope_stride < c.d_rope)) return MLA_ERR_INVALID_ARG;
    if (!dec && q_rope) return MLA_ERR_INVALID_ARG;
    if (cache->lat_stride < c.r_kv) return MLA_ERR_INVALID_ARG;
    if (!align_ok(c, {q_nope, q_rope, cache->lat, cache->rope, w->W_UK, w->W_UV, o, ws}))
        return MLA_ERR_INVALID_ARG;
    if (dec && prefill_uses_tc(c) && (cache->rope_stride * 2) % 16) return MLA_ERR_INVALID_ARG;
    int64_t kv_rows = 0;
    for (int b = 0; b < B; ++b) {
        int sp = start_pos ? start_pos[b] : 0;
        if (sp < 0) return MLA_ERR_INVALID_ARG;
        if ((int64_t)sp + S > c.max_seq) return MLA_ERR_CACHE_OVERFLOW;
        kv_rows = std::max<int64_t>(kv_rows, (int64_t)sp + S);
    }
    PrefillWs L = prefill_ws(c, B, kv_rows);
    if (ws_bytes < L.end) return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t *d_sp = (int32_t *)((char *)ws + L.start_pos);
    if (start_pos) MLA_TRY_CUDA(cudaMemcpyAsync(d_sp, start_pos, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s));
    else MLA_TRY_CUDA(cudaMemsetAsync(d_sp, 0, sizeof(int32_t) * B, s));
    return prefill_core(h, w, q_nope, q_rope, cache, B, S, kv_rows, o, ws, s);
}

// The launches of a validated absorbed-form decode call: absorption, the
// split-KV schedule and attention, the merge and W_UV.
static mla_status decode_launch(mla_handle *h, const mla_weights *w, const void *q_nope, const void *q_rope,
                                const mla_cache *cache, const int32_t *seq_lens, int B, void *o, void *ws,
                                const DecodeWs &L, bool tc_mla, bool tc_mlra, cudaStream_t s)
{
    const mla_config &c = h->cfg;
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    char *wsb = (char *)ws;
    const int H = c.n_heads, r_lat = r_lat_of(c);
    void *q_abs = wsb + L.q_abs, *o_lat = wsb + L.o_lat;

    // q_abs[b, h] = W_UK,h^T q_nope[b, h]: per head h, [B, d_nope] x [d_nope, r_lat].
    // (MLRA: the L stacked blocks [L, H*d/L, r/L] read as [H*d, r/L] rows.)
    const bool tc_split = tc_mla || tc_mlra;
    const int n_ranges = tc_mla ? h->decode_clusters : mlra_tc_ctas();
    const DecodeSched sc = decode_sched_at(wsb + L.prefix, B, n_ranges);
    if (tc_split) {
        // The split-KV schedule first: the attention kernel reads it (and
        // starts its cache loads) while the absorption kernel still runs.
        // The MLA kernel's ranges are balanced by estimated time, a
        // sequence start costing about as much as kSegmentCostKeys keys
        // (segment-end stores and the next query load); the MLRA kernel's
        // segments are cheap and its ranges uniform.
        decode_schedule(seq_lens, B, c.max_seq, n_ranges, tc_mla ? kSegmentCostKeys : 0, sc,
                        (uint32_t *)ws, s);
        MLA_TRY_CUDA(cudaGetLastError());
    }
    if (tc_split && absorb_supported(r_lat, c.d_nope)) {
        AbsorbArgs ab;
        ab.B = B; ab.H = H; ab.r_lat = r_lat; ab.d_nope = c.d_nope;
        ab.q_nope = q_nope;
        ab.W_UK = w->W_UK;
        ab.q_abs = q_abs;
        ab.interleave = tc_mla;  // the tensor-core MLA decode reads it head-interleaved
        ab.status = (uint32_t *)ws;
        MLA_TRY_CUDA(absorb(ab, s));
    } else {
        GemmArgs ga;
        ga.A = Mat2D{q_nope, B, (int64_t)H * c.d_nope, (int64_t)H * c.d_nope};
        ga.a_col_batch = c.d_nope;
        ga.B = Mat2D{w->W_UK, (int64_t)H * c.d_nope, r_lat, r_lat};
        ga.b_row_batch = c.d_nope;
        ga.trans_b = true;
        ga.M = B; ga.N = r_lat; ga.K = c.d_nope; ga.batch = H;
        ga.epi.out = q_abs; ga.epi.ldc = (int64_t)H * r_lat; ga.epi.batch_stride = r_lat;
        MLA_TRY(run_gemm(h, ga, (uint32_t *)ws, s));
    }

    const float scale_log2 = (float)(kLog2e / sqrt((double)(c.d_nope + (dec ? c.d_rope : 0))));
    // The tensor-core kernels leave split sequences as partials in slot order
    // (range + sequence); they are merged by the fused finish kernel or by
    // decode_combine before the value up-projection GEMM.
    if (tc_mla) {
        DecodeTcArgs t;
        t.B = B; t.H = H; t.r_kv = c.r_kv; t.d_rope = c.d_rope;
        t.max_batch = c.max_batch; t.max_seq = c.max_seq; t.n_clusters = h->decode_clusters;
        t.q_abs = q_abs; t.q_rope = q_rope;
        t.lat = cache->lat; t.lat_stride = cache->lat_stride;
        t.rope = cache->rope; t.rope_stride = cache->rope_stride;
        t.seq_lens = seq_lens;
        t.sc = sc;
        t.scale_log2 = scale_log2;
        t.o_lat = o_lat;
        t.o_part = (bf16 *)(wsb + L.o_part);
        t.ml_part = (float *)(wsb + L.ml_part);
        t.status = (uint32_t *)ws;
        MLA_TRY_CUDA(decode_tc(t, s));
    } else if (tc_mlra) {
        MlraTcArgs t;
        t.B = B; t.H = H; t.L = c.n_latent_heads; t.r_kv = c.r_kv;
        t.max_batch = c.max_batch; t.max_seq = c.max_seq; t.n_ctas = mlra_tc_ctas();
        t.q_abs = q_abs;
        t.lat = cache->lat; t.lat_stride = cache->lat_stride;
        t.seq_lens = seq_lens;
        t.prefix = sc.prefix;
        t.chunk = sc.chunk;
        t.scale_log2 = scale_log2;
        t.o_lat = o_lat;
        t.o_part = (bf16 *)(wsb + L.o_part);
        t.ml_part = (float *)(wsb + L.ml_part);
        t.status = (uint32_t *)ws;
        MLA_TRY_CUDA(mlra_tc(t, s));
    } else {
        DecodeArgs d;
        d.dtype = c.dtype;
        d.B = B; d.H = H; d.r_lat = r_lat; d.d_rope = dec ? c.d_rope : 0;
        d.heads_per_block_lat = heads_per_block_of(c);
        d.q_abs = q_abs; d.q_rope = dec ? q_rope : nullptr;
        d.lat = cache->lat; d.lat_stride = cache->lat_stride;
        d.rope = dec ? cache->rope : nullptr; d.rope_stride = cache->rope_stride;
        d.max_seq = c.max_seq;
        d.seq_lens = seq_lens;
        d.scale_log2 = scale_log2;
        d.o_part = (float *)(wsb + L.o_part);
        d.ml_part = (float *)(wsb + L.ml_part);
        d.n_split = decode_splits(c);
        d.chunk = kDecodeChunk;
        d.o_lat = o_lat;
        d.status = (uint32_t *)ws;
        MLA_TRY_CUDA(decode_simt(d, s));
    }

    if (tc_split && decode_finish_supported(r_lat, c.d_v)) {
        FinishArgs f;
        f.B = B; f.H = H; f.r_lat = r_lat; f.d_v = c.d_v;
        f.seq_fc = sc.seq_fc; f.seq_lc = sc.seq_lc;
        f.o_part = (const bf16 *)(wsb + L.o_part);
        f.ml_part = (float *)(wsb + L.ml_part);
        f.o_lat = o_lat;
        f.W_UV = w->W_UV;
        f.o = o;
        f.status = (uint32_t *)ws;
        MLA_TRY_CUDA(decode_finish(f, s));
        return MLA_OK;
    }
    if (tc_split) {
        decode_combine(sc, B, H, r_lat, (const bf16 *)(wsb + L.o_part), (float *)(wsb + L.ml_part), o_lat, s);
        MLA_TRY_CUDA(cudaGetLastError());
    }

    // o[b, h] = W_UV,h o_lat[b, h]: per head h, [B, r_lat] x [r_lat, d_v].
    GemmArgs gv;
    gv.A = Mat2D{o_lat, B, (int64_t)H * r_lat, (int64_t)H * r_lat};
    gv.a_col_batch = r_lat;
    gv.B = Mat2D{w->W_UV, (int64_t)H * c.d_v, r_lat, r_lat};
    gv.b_row_batch = c.d_v;
    gv.M = B; gv.N = c.d_v; gv.K = r_lat; gv.batch = H;
    gv.epi.out = o; gv.epi.ldc = (int64_t)H * c.d_v; gv.epi.batch_stride = c.d_v;
    MLA_TRY(run_gemm(h, gv, (uint32_t *)ws, s));
    return MLA_OK;
}

mla_status mla_decode(mla_handle *h, const mla_weights *w, const void *q_nope, const void *q_rope,
                      const mla_cache *cache, const int32_t *seq_lens, int B, void *o, void *ws,
                      size_t ws_bytes, void *stream)
{
    if (!h || !w || !cache || B < 0) return MLA_ERR_INVALID_ARG;
    const mla_config &c = h->cfg;
    if (B == 0) return MLA_OK;
    if (c.variant == MLA_VARIANT_SMALL) {
        // mla_attn decodes by re-decompressing the cached latent every step:
        // RoPE sits between W_UK and the query, so there is no absorbed form.
        // The prefill path with one query per sequence at position
        // seq_lens[b] - 1 computes exactly that (keys and values of every
        // cache row up to max_seq, causal attention).
        if (B > c.max_batch) return MLA_ERR_INVALID_ARG;
        if (!q_nope || !o || !ws || !seq_lens || !cache->lat || !w->W_UK || !w->W_UV || q_rope)
            return MLA_ERR_INVALID_ARG;
        if (cache->lat_stride < c.r_kv) return MLA_ERR_INVALID_ARG;
        if (!align_ok(c, {q_nope, cache->lat, w->W_UK, w->W_UV, o, ws})) return MLA_ERR_INVALID_ARG;
        const int64_t kv_rows = c.max_seq;
        PrefillWs L = prefill_ws(c, B, kv_rows);
        if (ws_bytes < L.end) return MLA_ERR_WORKSPACE;
        cudaStream_t s = (cudaStream_t)stream;
        profile_begin(MLA_PROFILE_DECODE_CALL, s);
        const mla_status st =
            positions_from_lengths(seq_lens, B, c.max_seq, (int32_t *)((char *)ws + L.start_pos), (uint32_t *)ws,
                                   s) == cudaSuccess
                ? prefill_core(h, w, q_nope, nullptr, cache, B, 1, kv_rows, o, ws, s)
                : MLA_ERR_CUDA;
        profile_end(MLA_PROFILE_DECODE_CALL, s);
        return st;
    }
    const bool dec = c.variant == MLA_VARIANT_DECOUPLED;
    if (B > c.max_batch) return MLA_ERR_INVALID_ARG;
    if (!q_nope || !o || !ws || !seq_lens || !cache->lat || !w->W_UK || !w->W_UV) return MLA_ERR_INVALID_ARG;
    if (dec && (!q_rope || !cache->rope || cache->rope_stride < c.d_rope)) return MLA_ERR_INVALID_ARG;
    if (!dec && q_rope) return MLA_ERR_INVALID_ARG;
    if (cache->lat_stride < c.r_kv) return MLA_ERR_INVALID_ARG;
    if (!align_ok(c, {q_nope, q_rope, cache->lat, cache->rope, w->W_UK, w->W_UV, o, ws}))
        return MLA_ERR_INVALID_ARG;
    // Every check comes before the first launch: a refused call leaves the
    // stream untouched.  The TMA paths need cache rows of whole 16-byte units.
    const bool tc_mla = use_tc_decode(h), tc_mlra = use_mlra_tc(h);
    if (tc_mla && ((cache->lat_stride * 2) % 16 || (cache->rope_stride * 2) % 16)) return MLA_ERR_INVALID_ARG;
    if (tc_mlra && (cache->lat_stride * 2) % 16) return MLA_ERR_INVALID_ARG;
    if (!tc_mla && !tc_mlra && decode_splits(c) > 64) return MLA_ERR_UNSUPPORTED;
    DecodeWs L = decode_ws(h, B);
    if (ws_bytes < L.end) return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    profile_begin(MLA_PROFILE_DECODE_CALL, s);
    const mla_status st = decode_launch(h, w, q_nope, q_rope, cache, seq_lens, B, o, ws, L, tc_mla, tc_mlra, s);
    profile_end(MLA_PROFILE_DECODE_CALL, s);
    return st;
}

mla_status mla_out_proj(mla_handle *h, const mla_weights *w, const void *o, int64_t T, void *y, void *ws,
                        size_t ws_bytes, void *stream)
{
    if (!h || !w || T < 0) return MLA_ERR_INVALID_ARG;
    if (T == 0) return MLA_OK;
    const mla_config &c = h->cfg;
    if (!o || !y || !w->W_O || !ws || T > INT32_MAX) return MLA_ERR_INVALID_ARG;
    if (!align_ok(c, {o, y, w->W_O, ws})) return MLA_ERR_INVALID_ARG;
    OutProjWs L = out_proj_ws(h, T);
    if (ws_bytes < L.end) return MLA_ERR_WORKSPACE;
    const int K = c.n_heads * c.d_v;
    GemmArgs g = linear_args(o, K, w->W_O, K, (int)T, c.d_model, K, y, c.d_model);
    return run_gemm(h, g, (uint32_t *)ws, (cudaStream_t)stream, (float *)((char *)ws + L.split));
}

mla_status mla_get_device_status(mla_handle *h, void *ws, void *stream, uint32_t *bits)
{
    if (!h) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v[2] = {0, 0};
    if (ws) MLA_TRY_CUDA(cudaMemcpyAsync(&v[0], ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    MLA_TRY_CUDA(cudaMemcpyAsync(&v[1], h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    MLA_TRY_CUDA(cudaStreamSynchronize(s));
    if (ws) MLA_TRY_CUDA(cudaMemsetAsync(ws, 0, sizeof(uint32_t), s));
    MLA_TRY_CUDA(cudaMemsetAsync(h->status, 0, sizeof(uint32_t), s));
    MLA_TRY_CUDA(cudaStreamSynchronize(s));
    const uint32_t all = v[0] | v[1];
    if (bits) *bits = all;
    if (all & kStatusTimeout) return MLA_ERR_TIMEOUT;
    return all ? MLA_ERR_DEVICE_DATA : MLA_OK;
}

uint64_t mla_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

mla_status mla_set_wait_limit(int64_t cycles)
{
    if (cycles < 0) return MLA_ERR_INVALID_ARG;
    __atomic_store_n(&g_gemm_wait_cycles, (long long)cycles, __ATOMIC_RELAXED);
    return MLA_OK;
}

mla_status mla_set_profile_events(int which, void *begin, void *end)
{
    if (which < 0 || which >= MLA_PROFILE_COUNT || (!begin) != (!end)) return MLA_ERR_INVALID_ARG;
    g_prof_begin[which] = (cudaEvent_t)begin;
    g_prof_end[which] = (cudaEvent_t)end;
    return MLA_OK;
}

const char *mla_status_string(mla_status st)
{
    switch (st) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or variant";
    case MLA_ERR_WORKSPACE: return "workspace too small";
    case MLA_ERR_CACHE_OVERFLOW: return "position beyond cache capacity";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "bounded device wait timed out";
    case MLA_ERR_DEVICE_DATA: return "device-side index data out of range";
    }
    return "unknown status";
}

}  // extern "C"

// Compressed convolutional attention (CCA) and its grouped form (CCGQA).
//
// "frankenstein-transformer", latent/cca_attn.py (CCAAttention,
// CCGQAAttention): attention runs inside a compressed latent.  The launches
// of one forward call, on B sequences of S tokens (T = B S rows):
//   1. the down-projections x -> [qk | v1 | W_V2 x] (tcgen05 GEMMs writing
//      column slices of one bf16 buffer);
//   2. cca_conv0_v_kernel: the depth-wise causal convolution of qk (fp32
//      out) and the values (value-shift reads the previous row's W_V2 x),
//      as fp16;
//   3. cca_qk_kernel: per (row tile, head) the grouped causal convolution,
//      q-k-mean, L2 normalisation, key temperature and half-split RoPE,
//      writing the query (bf16) and key (fp16) operands of the attention;
//   4. the causal flash prefill kernel (tcgen05) with grouped key/value
//      heads;
//   5. the output projection GEMM.
// The convolutions and the normalisation are small (a few hundred MACs per
// output) and run on the CUDA cores; the contractions on the tensor cores.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "mla_internal.cuh"
#include "ptx.cuh"

struct mla_cca_handle {
    mla_cca_config cfg;
    int device, num_sms, d_h;
    float2 *rope_table;  // [max_seq, d_h / 2] (cos, sin) of pos * base^(-2i/d_h)
    uint32_t *status;    // 256-byte device status word (unused by forward; kept for symmetry)
};

namespace mla {
namespace {

constexpr double kLog2eCca = 1.4426950408889634;
constexpr int kMaxTapsSeq = 8;
constexpr int kMaxTapsCh = 4;
constexpr int kRowsPerBlock = 32;  // token rows per cca_qk_kernel block

size_t cca_round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct CcaWs {
    size_t start_pos, pre, c0, q, k, v, o, split, end;
};

// x [M, K] W^T into columns [col, col + N) of out (row stride ldc).
GemmArgs cca_linear(const void *x, int64_t M, int K, const void *W, int N, void *out, int64_t ldc, int col,
                    uint32_t *status)
{
    GemmArgs g;
    g.A = Mat2D{x, M, K, K};
    g.B = Mat2D{W, N, K, K};
    g.M = (int)M; g.N = N; g.K = K;
    g.epi.out = (char *)out + (size_t)col * 2;
    g.epi.ldc = ldc;
    g.epi.status = status;
    return g;
}

// Split-K partial sums the largest of the call's GEMMs needs (few tokens).
size_t cca_split_bytes(const mla_cca_config &c, int64_t T, int num_sms)
{
    const int P = c.q_latent + c.kv_latent;
    const int n[4] = {P, c.kv_latent / 2, c.kv_latent, c.d_model};
    const int k[4] = {c.d_model, c.d_model, c.d_model, c.q_latent};
    size_t most = 0;
    for (int i = 0; i < 4; ++i) {
        GemmArgs g = cca_linear(nullptr, T, k[i], nullptr, n[i], nullptr, n[i], 0, nullptr);
        most = std::max(most, gemm_tc_workspace(g, num_sms));
    }
    return most;
}

// Scratch of one forward call: the projections [T, P + Lkv] (bf16), the
// depth-wise convolution [T, P] (fp32), the attention operands q (bf16), k
// and v (fp16), its output o (bf16) and the GEMMs' split-K partials.
CcaWs cca_ws(const mla_cca_config &c, int B, int S, int num_sms)
{
    const size_t T = (size_t)B * S, P = (size_t)c.q_latent + c.kv_latent;
    CcaWs w;
    w.start_pos = kWsHeader;
    w.pre = cca_round_up(w.start_pos + (size_t)B * 4, 256);
    w.c0 = cca_round_up(w.pre + T * (P + c.kv_latent) * 2, 256);
    w.q = cca_round_up(w.c0 + (c.conv_layers >= 1 ? T * P * 4 : 0), 256);
    w.k = cca_round_up(w.q + T * c.q_latent * 2, 256);
    w.v = cca_round_up(w.k + T * c.kv_latent * 2, 256);
    w.o = cca_round_up(w.v + T * c.kv_latent * 2, 256);
    w.split = cca_round_up(w.o + T * c.q_latent * 2, 256);
    w.end = cca_round_up(w.split + cca_split_bytes(c, (int64_t)T, num_sms), 256);
    return w;
}

__device__ __forceinline__ __half to_f16_sat(float v, bool &over)
{
    over |= ptx::beyond_f16(v);
    return __float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f));
}

// Columns [0, P) of each row: the depth-wise causal convolution of the packed
// qk (taps k0, left zero padding within the row's sequence), to fp32.
// Columns [P, P + Lkv): the values to fp16; with value-shift the second half
// is the previous row's W_V2 x (zero for a sequence's first token).  With no
// convolution only the value columns are run (col0 = P).
__global__ void __launch_bounds__(256)
    cca_conv0_v_kernel(const bf16 *__restrict__ pre, int64_t T, int S, int P, int Lkv, int col0, int k0,
                       const bf16 *__restrict__ w0, float *__restrict__ c0, __half *__restrict__ v, int value_shift,
                       uint32_t *status)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int Wp = P + Lkv, ncols = Wp - col0;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T * ncols) return;
    const int64_t r = i / ncols;
    const int c = (int)(i % ncols) + col0;
    const int t = (int)(r % S);
    if (c < P) {
        float acc = 0.f;
        for (int j = 0; j < k0; ++j) {
            const int back = k0 - 1 - j;  // row r - back feeds tap j
            if (t >= back) acc += __bfloat162float(w0[(int64_t)c * k0 + j]) * __bfloat162float(pre[(r - back) * Wp + c]);
        }
        c0[r * P + c] = acc;
        return;
    }
    const int cv = c - P;
    float val;
    if (value_shift && cv >= Lkv / 2) val = t >= 1 ? __bfloat162float(pre[(r - 1) * Wp + c]) : 0.f;
    else val = __bfloat162float(pre[r * Wp + c]);
    bool over = false;
    v[r * Lkv + cv] = to_f16_sat(val, over);
    if (over && status) atomicOr(status, kStatusF16Range);
}

struct CcaQkParams {
    const bf16 *pre;     // [T, P + Lkv] packed projections
    const float *c0;     // [T, P] after the depth-wise convolution, or null (none)
    const bf16 *w1;      // [P, d_h, k1] grouped convolution, or null
    int64_t T;
    int S, P, Lkv, Lq, Hq, gs, k1, conv_layers, qk_mean;
    float k_scale;       // exp(key temperature)
    const float2 *rope;  // [max_seq, d_h / 2]
    bf16 *q;             // [T, Lq]
    __half *k;           // [T, Lkv]
    uint32_t *status;
};

// One block per (kRowsPerBlock token rows, head g): query heads g < Hq, key
// heads after them.  The head's grouped-convolution weights are staged once
// in shared memory, transposed to [tap][in][out] so that the threads of a
// warp (consecutive output channels) read consecutive words.  Thread (o, y)
// produces channel o of rows y, y + kRowThreads, ...: the grouped causal
// convolution of the depth-wise output (one group of d_h channels per head),
// q-k-mean, the L2 normalisation over the head's channels to norm sqrt(d_h)
// (keys times exp(beta)), and RoPE with half-split pairs (o, o + d_h / 2) at
// the row's position.
constexpr int kRowThreads = 4;                            // thread rows per block
constexpr int kRowsPerThread = kRowsPerBlock / kRowThreads;

template <int DH>
struct QkSmem {
    static constexpr size_t kW = (size_t)kMaxTapsCh * DH * DH * 2;            // bf16 weights [tap][in][out]
    static constexpr size_t kIn = (size_t)(kRowsPerBlock + kMaxTapsCh - 1) * DH * 4;
    static constexpr size_t kVal = (size_t)kRowsPerBlock * DH * 4;
    static constexpr size_t kRed = (size_t)kRowsPerBlock * (DH / 32) * 4;
    static constexpr size_t kBytes = kW + kIn + kVal + kRed;
};

template <int DH>
__global__ void __launch_bounds__(DH * kRowThreads) cca_qk_kernel(CcaQkParams p)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    constexpr int R = kRowsPerBlock, RT = kRowsPerThread, half = DH / 2;
    using Sm = QkSmem<DH>;
    extern __shared__ __align__(16) uint8_t sm[];
    bf16 *wsm = reinterpret_cast<bf16 *>(sm);                               // [k1][DH in][DH out]
    float (*cin)[DH] = reinterpret_cast<float (*)[DH]>(sm + Sm::kW);       // rows r0 - halo + i
    float (*val)[DH] = reinterpret_cast<float (*)[DH]>(sm + Sm::kW + Sm::kIn);
    float (*red)[DH / 32] = reinterpret_cast<float (*)[DH / 32]>(sm + Sm::kW + Sm::kIn + Sm::kVal);
    const int o = threadIdx.x, y = threadIdx.y, tid = y * DH + o;
    const int g = blockIdx.y;
    const int64_t r0 = (int64_t)blockIdx.x * R;
    const int ch = g * DH + o;  // packed channel
    const int conv2 = p.conv_layers == 2;
    const int halo = conv2 ? p.k1 - 1 : 0;
    const int Wp = p.P + p.Lkv;
    if (conv2) {
        // w1[(g DH + out) DH + in][tap] -> wsm[tap][in][out]
        const bf16 *wg = p.w1 + (int64_t)g * DH * DH * p.k1;
        for (int e = tid; e < DH * DH * p.k1; e += DH * kRowThreads) {
            const int j = e % p.k1, i = (e / p.k1) % DH, oo = e / (p.k1 * DH);
            wsm[(j * DH + i) * DH + oo] = wg[e];
        }
    }
    for (int i = y; i < R + halo; i += kRowThreads) {
        const int64_t r = r0 - halo + i;
        float a = 0.f;
        if (r >= 0 && r < p.T) a = p.c0 ? p.c0[r * p.P + ch] : __bfloat162float(p.pre[r * Wp + ch]);
        cin[i][o] = a;
    }
    __syncthreads();
    float acc[RT];
    int tpos[RT];
#pragma unroll
    for (int k = 0; k < RT; ++k) {
        const int64_t r = r0 + y + k * kRowThreads;
        tpos[k] = r < p.T ? (int)(r % p.S) : 0;
        acc[k] = conv2 ? 0.f : cin[y + k * kRowThreads][o];
    }
    if (conv2) {
        // Tap j of row r reads row r - (k1 - 1 - j), within the row's sequence only.
        for (int j = 0; j < p.k1; ++j) {
            const int back = p.k1 - 1 - j;
            const bf16 *wj = wsm + (size_t)j * DH * DH + o;
#pragma unroll 4
            for (int i = 0; i < DH; ++i) {
                const float wv = __bfloat162float(wj[i * DH]);
#pragma unroll
                for (int k = 0; k < RT; ++k)
                    if (tpos[k] >= back) acc[k] += wv * cin[y + k * kRowThreads + j][i];
            }
        }
    }
#pragma unroll
    for (int k = 0; k < RT; ++k) {
        const int yy = y + k * kRowThreads;
        const int64_t r = r0 + yy;
        if (p.qk_mean && r < p.T) {
            // Query head g: (q_pre,g + k_pre of its group) / 2; key head j: the
            // average of that over its group's query heads.
            const bf16 *row = p.pre + r * Wp;
            if (g < p.Hq) {
                acc[k] += 0.5f * (__bfloat162float(row[g * DH + o]) + __bfloat162float(row[p.Lq + (g / p.gs) * DH + o]));
            } else {
                const int jh = g - p.Hq;
                float qs = 0.f;
                for (int h = jh * p.gs; h < (jh + 1) * p.gs; ++h) qs += __bfloat162float(row[h * DH + o]);
                acc[k] += 0.5f * (__bfloat162float(row[p.Lq + jh * DH + o]) + qs / (float)p.gs);
            }
        }
        float ss = acc[k] * acc[k];
#pragma unroll
        for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if ((o & 31) == 0) red[yy][o >> 5] = ss;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < RT; ++k) {
        const int yy = y + k * kRowThreads;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < DH / 32; ++w) tot += red[yy][w];
        float sc = sqrtf((float)DH) / fmaxf(sqrtf(tot), 1e-6f);
        if (g >= p.Hq) sc *= p.k_scale;
        val[yy][o] = acc[k] * sc;
    }
    __syncthreads();
    const int i = o < half ? o : o - half;
#pragma unroll
    for (int k = 0; k < RT; ++k) {
        const int yy = y + k * kRowThreads;
        const int64_t r = r0 + yy;
        if (r >= p.T) continue;
        const float2 cs = p.rope[(int64_t)tpos[k] * half + i];
        const float x0 = val[yy][i], x1 = val[yy][i + half];
        const float out = o < half ? x0 * cs.x - x1 * cs.y : x0 * cs.y + x1 * cs.x;
        if (g < p.Hq) {
            p.q[r * p.Lq + g * DH + o] = __float2bfloat16_rn(out);
        } else {
            bool over = false;
            p.k[r * p.Lkv + (g - p.Hq) * DH + o] = to_f16_sat(out, over);
            if (over && p.status) atomicOr(p.status, kStatusF16Range);
        }
    }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

mla_status mla_cca_check_config(const mla_cca_config *c)
{
    if (!c) return MLA_ERR_INVALID_ARG;
    if (c->d_model <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->q_latent <= 0 || c->kv_latent <= 0 ||
        c->max_seq <= 0 || !(c->rope_base > 0.0) || !isfinite(c->key_temp))
        return MLA_ERR_INVALID_ARG;
    // cca_attn constructors: heads divide the widths, equal and even d_h,
    // kv latent <= query latent, 0..2 convolutions, value-shift halves.
    if (c->n_heads % c->n_kv_heads || c->q_latent % c->n_heads || c->kv_latent % c->n_kv_heads)
        return MLA_ERR_INVALID_ARG;
    const int dh = c->q_latent / c->n_heads;
    if (c->kv_latent / c->n_kv_heads != dh || dh % 2 || c->kv_latent > c->q_latent) return MLA_ERR_INVALID_ARG;
    if (c->conv_layers < 0 || c->conv_layers > 2) return MLA_ERR_INVALID_ARG;
    if (c->conv_layers >= 1 && c->conv_kernel_seq < 1) return MLA_ERR_INVALID_ARG;
    if (c->conv_layers >= 2 && c->conv_kernel_ch < 1) return MLA_ERR_INVALID_ARG;
    if (c->value_shift && (c->n_kv_heads % 2 || c->kv_latent % 2)) return MLA_ERR_INVALID_ARG;
    // What the kernels run.
    if (dh != 64 && dh != 128) return MLA_ERR_UNSUPPORTED;
    if (c->q_latent % 64 || c->kv_latent % (c->value_shift ? 128 : 64) || c->d_model % 64) return MLA_ERR_UNSUPPORTED;
    if (c->conv_layers >= 1 && c->conv_kernel_seq > kMaxTapsSeq) return MLA_ERR_UNSUPPORTED;
    if (c->conv_layers >= 2 && c->conv_kernel_ch > kMaxTapsCh) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

mla_status mla_cca_create(const mla_cca_config *cfg, mla_cca_handle **out)
{
    if (!out) return MLA_ERR_INVALID_ARG;
    *out = nullptr;
    const mla_status st = mla_cca_check_config(cfg);
    if (st != MLA_OK) return st;
    mla_cca_handle *h = new (std::nothrow) mla_cca_handle();
    if (!h) return MLA_ERR_CUDA;
    h->cfg = *cfg;
    h->d_h = cfg->q_latent / cfg->n_heads;
    h->rope_table = nullptr;
    h->status = nullptr;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
        cudaMalloc(&h->status, 256) != cudaSuccess || cudaMemset(h->status, 0, 256) != cudaSuccess) {
        mla_cca_destroy(h);
        return MLA_ERR_CUDA;
    }
    // cos/sin of pos * base^(-2i/d_h) (cca_attn _apply_rope), in double.
    const int half = h->d_h / 2;
    std::vector<float2> tab((size_t)cfg->max_seq * half);
    for (int p = 0; p < cfg->max_seq; ++p)
        for (int i = 0; i < half; ++i) {
            const double a = (double)p * pow(cfg->rope_base, -2.0 * i / (double)h->d_h);
            tab[(size_t)p * half + i] = make_float2((float)cos(a), (float)sin(a));
        }
    if (cudaMalloc(&h->rope_table, tab.size() * sizeof(float2)) != cudaSuccess ||
        cudaMemcpy(h->rope_table, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
        mla_cca_destroy(h);
        return MLA_ERR_CUDA;
    }
    *out = h;
    return MLA_OK;
}

void mla_cca_destroy(mla_cca_handle *h)
{
    if (!h) return;
    if (h->rope_table) cudaFree(h->rope_table);
    if (h->status) cudaFree(h->status);
    delete h;
}

size_t mla_cca_workspace_size(const mla_cca_handle *h, int B, int S)
{
    if (!h || B < 0 || S < 0) return 0;
    return cca_ws(h->cfg, B, S, h->num_sms).end;
}

mla_status mla_cca_forward(mla_cca_handle *h, const mla_cca_weights *w, const void *x, int B, int S, void *y,
                           void *ws, size_t ws_bytes, void *stream)
{
    if (!h || !w || B < 0 || S < 0) return MLA_ERR_INVALID_ARG;
    if (B == 0 || S == 0) return MLA_OK;
    const mla_cca_config &c = h->cfg;
    if (S > c.max_seq) return MLA_ERR_CACHE_OVERFLOW;
    if (!x || !y || !ws || !w->W_QK || !w->W_O) return MLA_ERR_INVALID_ARG;
    if (c.value_shift ? (!w->W_V1 || !w->W_V2) : !w->W_V) return MLA_ERR_INVALID_ARG;
    if ((c.conv_layers >= 1 && !w->conv0) || (c.conv_layers >= 2 && !w->conv1)) return MLA_ERR_INVALID_ARG;
    const void *ptrs[] = {x, y, ws, w->W_QK, w->W_V1, w->W_V2, w->W_V, w->W_O};
    for (const void *p : ptrs)
        if ((uintptr_t)p & 15u) return MLA_ERR_INVALID_ARG;
    const int64_t T = (int64_t)B * S;
    if (T > INT32_MAX) return MLA_ERR_INVALID_ARG;
    const CcaWs L = cca_ws(c, B, S, h->num_sms);
    if (ws_bytes < L.end) return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char *wb = (char *)ws;
    uint32_t *status = (uint32_t *)ws;
    const int P = c.q_latent + c.kv_latent, Lkv = c.kv_latent, dh = h->d_h;
    const int Wp = P + Lkv;
    bf16 *pre = (bf16 *)(wb + L.pre);
    int32_t *d_sp = (int32_t *)(wb + L.start_pos);
    auto cuda = [](cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; };
    mla_status st;
    if ((st = cuda(cudaMemsetAsync(d_sp, 0, sizeof(int32_t) * B, s))) != MLA_OK) return st;

    // 1. Down-projections into column slices of pre: [W_QK x | W_V1 x | W_V2 x] (or [W_QK x | W_V x]).
    float *split = (float *)(wb + L.split);
    auto gemm = [&](GemmArgs g) -> mla_status {
        g.split_ws = split;  // GEMMs run one after another on the stream: one split region serves all
        if (!gemm_tc_supported(g)) return MLA_ERR_UNSUPPORTED;
        return cuda(gemm_tc(g, h->num_sms, s));
    };
    if ((st = gemm(cca_linear(x, T, c.d_model, w->W_QK, P, pre, Wp, 0, status))) != MLA_OK) return st;
    if (c.value_shift) {
        if ((st = gemm(cca_linear(x, T, c.d_model, w->W_V1, Lkv / 2, pre, Wp, P, status))) != MLA_OK) return st;
        if ((st = gemm(cca_linear(x, T, c.d_model, w->W_V2, Lkv / 2, pre, Wp, P + Lkv / 2, status))) != MLA_OK)
            return st;
    } else if ((st = gemm(cca_linear(x, T, c.d_model, w->W_V, Lkv, pre, Wp, P, status))) != MLA_OK) {
        return st;
    }

    // 2. Depth-wise convolution (fp32) and the values (fp16).
    float *c0 = c.conv_layers >= 1 ? (float *)(wb + L.c0) : nullptr;
    __half *v = (__half *)(wb + L.v);
    {
        const int col0 = c0 ? 0 : P;
        const int64_t n = T * (Wp - col0);
        st = cuda(launch_ex(cca_conv0_v_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, 1, (const bf16 *)pre,
                            T, S, P, Lkv, col0, c.conv_layers >= 1 ? c.conv_kernel_seq : 1, (const bf16 *)w->conv0, c0,
                            v, c.value_shift, status));
        note_launch();
        if (st != MLA_OK) return st;
    }

    // 3. Grouped convolution, q-k-mean, normalisation, temperature, RoPE.
    CcaQkParams q;
    q.pre = pre; q.c0 = c0; q.w1 = (const bf16 *)w->conv1;
    q.T = T; q.S = S; q.P = P; q.Lkv = Lkv; q.Lq = c.q_latent; q.Hq = c.n_heads;
    q.gs = c.n_heads / c.n_kv_heads;
    q.k1 = c.conv_layers >= 2 ? c.conv_kernel_ch : 1;
    q.conv_layers = c.conv_layers; q.qk_mean = c.qk_mean;
    q.k_scale = (float)exp(c.key_temp);
    q.rope = h->rope_table;
    q.q = (bf16 *)(wb + L.q);
    q.k = (__half *)(wb + L.k);
    q.status = status;
    {
        const dim3 grid((unsigned)((T + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)(c.n_heads + c.n_kv_heads));
        static std::atomic<int> smem64{-1}, smem128{-1};
        if (dh == 64) {
            st = cuda(smem_limit_once(smem64, (const void *)cca_qk_kernel<64>, (int)QkSmem<64>::kBytes));
            if (st == MLA_OK)
                st = cuda(launch_ex(cca_qk_kernel<64>, grid, dim3(64, kRowThreads), QkSmem<64>::kBytes, s, 1, q));
        } else {
            st = cuda(smem_limit_once(smem128, (const void *)cca_qk_kernel<128>, (int)QkSmem<128>::kBytes));
            if (st == MLA_OK)
                st = cuda(launch_ex(cca_qk_kernel<128>, grid, dim3(128, kRowThreads), QkSmem<128>::kBytes, s, 1, q));
        }
        note_launch();
        if (st != MLA_OK) return st;
    }

    // 4. Causal attention in the latent (query head h on key/value head h / gs).
    PrefillTcArgs a;
    a.B = B; a.S = S; a.H = c.n_heads;
    a.d_nope = dh; a.d_rope = 0; a.d_v = dh;
    a.max_batch = B; a.max_seq = S; a.kv_rows = S;
    a.q_nope = q.q; a.q_rope = nullptr;
    a.k = q.k; a.v = v;
    a.kv_group = q.gs;
    a.rope = nullptr; a.rope_stride = 0; a.k_rope16 = nullptr;
    a.start_pos = d_sp;
    a.scale_log2 = (float)(kLog2eCca / sqrt((double)dh));
    bf16 *o = (bf16 *)(wb + L.o);
    a.o = o;
    a.status = status;
    if ((st = cuda(prefill_tc(a, s))) != MLA_OK) return st;

    // 5. Output projection y = W_O o.
    return gemm(cca_linear(o, T, c.q_latent, w->W_O, c.d_model, y, c.d_model, 0, status));
}

mla_status mla_cca_get_device_status(mla_cca_handle *h, void *ws, void *stream, uint32_t *bits)
{
    if (!h) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v[2] = {0, 0};
    if (ws && cudaMemcpyAsync(&v[0], ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaMemcpyAsync(&v[1], h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (ws && cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaMemsetAsync(h->status, 0, sizeof(uint32_t), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return MLA_ERR_CUDA;
    const uint32_t all = v[0] | v[1];
    if (bits) *bits = all;
    if (all & kStatusTimeout) return MLA_ERR_TIMEOUT;
    return all ? MLA_ERR_DEVICE_DATA : MLA_OK;
}

}  // extern "C"

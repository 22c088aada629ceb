// Compressed convolutional attention (CCA) and its grouped form (CCGQA).
//
// "frankenstein-transformer", latent/cca_attn.py (CCAAttention,
// CCGQAAttention): attention runs inside a compressed latent.  The launches
// of one forward call, on B sequences of S tokens (T = B S rows):
//   1. the down-projections x -> [qk | v1 | W_V2 x] (one grouped tcgen05
//      GEMM writing column slices of one bf16 buffer);
//   2. cca_v_kernel: the values as fp16 (value-shift reads the previous
//      row's W_V2 x);
//   3. cca_qk_tc_kernel: per (128 token rows, head) the depth-wise causal
//      convolution, the grouped causal convolution on the tensor cores,
//      q-k-mean, L2 normalisation, key temperature and half-split RoPE,
//      writing the query (bf16) and key (fp16) operands of the attention;
//   4. the causal flash prefill kernel (tcgen05) with grouped key/value
//      heads;
//   5. the output projection GEMM.
// The depth-wise convolution and the normalisation run on the CUDA cores; the
// grouped convolution (K = d_h x taps per output) and the projections on the
// tensor cores.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include <cudaTypedefs.h>

#include "mla_internal.cuh"
#include "ptx.cuh"

struct mla_cca_handle {
    mla_cca_config cfg;
    int device, num_sms, d_h;
    float2 *rope_table;  // [max_seq, d_h / 2] (cos, sin) of pos * base^(-2i/d_h)
    uint32_t *status;    // 256-byte device status word (unused by forward; kept for symmetry)
};

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr double kLog2eCca = 1.4426950408889634;
constexpr int kMaxTapsSeq = 8;
constexpr int kMaxTapsCh = 4;

size_t cca_round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct CcaWs {
    size_t start_pos, pre, q, k, v, o, w1img, split, end;
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

// The down-projections as one grouped GEMM over x's rows: output columns
// [W_QK x | W_V1 x | W_V2 x] (or [W_QK x | W_V x]) of one [T, P + Lkv] buffer.
GemmArgs cca_down_proj(const mla_cca_config &c, const void *x, int64_t T, const mla_cca_weights *w, void *pre,
                       uint32_t *status)
{
    const int P = c.q_latent + c.kv_latent, Lkv = c.kv_latent, Wp = P + Lkv, K = c.d_model;
    GemmArgs g = cca_linear(x, T, K, nullptr, P, pre, Wp, 0, status);
    auto seg = [&](const void *W, int N, int col) {
        GemmSegment s;
        s.B = Mat2D{W, N, K, K};
        s.epi = g.epi;
        s.epi.out = (char *)pre + (size_t)col * 2;
        s.N = N;
        return s;
    };
    g.seg[0] = seg(w ? w->W_QK : nullptr, P, 0);
    if (c.value_shift) {
        g.nseg = 3;
        g.seg[1] = seg(w ? w->W_V1 : nullptr, Lkv / 2, P);
        g.seg[2] = seg(w ? w->W_V2 : nullptr, Lkv / 2, P + Lkv / 2);
    } else {
        g.nseg = 2;
        g.seg[1] = seg(w ? w->W_V : nullptr, Lkv, P);
    }
    return g;
}

// Split-K partial sums the larger of the call's two GEMMs needs (few tokens).
size_t cca_split_bytes(const mla_cca_config &c, int64_t T, int num_sms)
{
    const GemmArgs down = cca_down_proj(c, nullptr, T, nullptr, nullptr, nullptr);
    const GemmArgs out = cca_linear(nullptr, T, c.q_latent, nullptr, c.d_model, nullptr, c.d_model, 0, nullptr);
    return std::max(gemm_tc_workspace(down, num_sms), gemm_tc_workspace(out, num_sms));
}

// Scratch of one forward call: the projections [T, P + Lkv] (bf16), the
// attention operands q (bf16), k and v (fp16), its output o (bf16), the
// channel convolution's operand image (fp16, heads x taps x d_h x d_h) and
// the GEMMs' split-K partials.
CcaWs cca_ws(const mla_cca_config &c, int B, int S, int num_sms)
{
    const size_t T = (size_t)B * S, P = (size_t)c.q_latent + c.kv_latent;
    CcaWs w;
    w.start_pos = kWsHeader;
    w.pre = cca_round_up(w.start_pos + (size_t)B * 4, 256);
    w.q = cca_round_up(w.pre + T * (P + c.kv_latent) * 2, 256);
    w.k = cca_round_up(w.q + T * c.q_latent * 2, 256);
    w.v = cca_round_up(w.k + T * c.kv_latent * 2, 256);
    w.o = cca_round_up(w.v + T * c.kv_latent * 2, 256);
    const size_t dh = (size_t)c.q_latent / c.n_heads;
    const size_t k1 = c.conv_layers >= 2 ? (size_t)c.conv_kernel_ch : 1;
    w.w1img = cca_round_up(w.o + T * c.q_latent * 2, 256);
    w.split = cca_round_up(w.w1img + (size_t)(c.n_heads + c.n_kv_heads) * k1 * dh * dh * 2, 256);
    w.end = cca_round_up(w.split + cca_split_bytes(c, (int64_t)T, num_sms), 256);
    return w;
}

// The values to fp16: columns [P, P + Lkv) of each row, eight channels per
// thread.  With value-shift the second half is the previous row's W_V2 x
// (zero for a sequence's first token).
__global__ void __launch_bounds__(256)
    cca_v_kernel(const bf16 *__restrict__ pre, int64_t T, int S, int P, int Lkv, __half *__restrict__ v,
                 int value_shift, uint32_t *status)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int nc = Lkv / 8, Wp = P + Lkv;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T * nc) return;
    const int64_t r = i / nc;
    const int c = (int)(i % nc) * 8;
    const bool shifted = value_shift && c >= Lkv / 2;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (!shifted || r % S >= 1) w = *reinterpret_cast<const uint4 *>(pre + (r - (shifted ? 1 : 0)) * Wp + P + c);
    bool over = false;
    uint4 o;
    o.x = ptx::bf16x2_to_f16x2(w.x, over);
    o.y = ptx::bf16x2_to_f16x2(w.y, over);
    o.z = ptx::bf16x2_to_f16x2(w.z, over);
    o.w = ptx::bf16x2_to_f16x2(w.w, over);
    *reinterpret_cast<uint4 *>(v + r * Lkv + c) = o;
    if (over && status) atomicOr(status, kStatusF16Range);
}

struct CcaQkParams {
    const bf16 *pre;      // [T, P + Lkv] packed projections
    const bf16 *w0;       // [P, k0] depth-wise convolution, or null (none)
    const uint8_t *w1img; // per head, per tap: the channel convolution's operand image (cca_w1_image_kernel)
    int64_t T;
    int S, P, Lkv, Lq, Hq, gs, k0, k1, slots, qk_mean;
    float k_scale;        // exp(key temperature)
    const float2 *rope;   // [max_seq, d_h / 2]
    bf16 *q;              // [T, Lq]
    __half *k;            // [T, Lkv]
    uint32_t *status;
};

// One CTA per (128 token rows, head g): query heads g < Hq, key heads after
// them; 256 threads.  The grouped causal convolution (one
// group of d_h channels per head) is a contraction over (tap, input
// channel):
//   u[r, o] = sum_j sum_i a[r - (k1 - 1 - j), i] W1[g d_h + o, i, j],
// where a is the depth-wise causal convolution of the packed projections and
// rows before the sequence's first token are zero.  The steps:
//   - TMA copies the head's projection tile (the 128 rows, the channel
//     convolution's halo and the depth-wise one's, zero outside [0, T)) and a
//     bulk copy brings the tap weights W_j[o, i] (fp16, prepared once per
//     call as the MMA operand image);
//   - the threads compute a once per row from the tile and write each tap's
//     row-shifted copy A_j[n] = a[r0 + n - (k1 - 1 - j)] (fp16, zero where
//     the shift crosses the sequence start);
//   - one thread issues k1 * d_h / 16 MMAs (M = 128 rows, N = d_h output
//     channels, K = 16) accumulating into tensor memory; taps that do not fit
//     in shared memory at once run in passes;
//   - two threads per row read row m back from tensor-memory lane m, each
//     taking half of the RoPE pairs (o, o + d_h / 2), and apply q-k-mean, the
//     L2 normalisation to norm sqrt(d_h) (keys times exp(beta); the two
//     partial sums of squares meet in shared memory) and RoPE at the row's
//     position.
// Without the channel convolution W is the identity (k1 = 1); without the
// depth-wise convolution a is the projection itself.  Every wait is bounded.
constexpr int kQkRows = 128;
constexpr int kQkThreads = 256;  // two threads per row in the epilogue

template <int DH>
struct QkTc {
    static constexpr int kA = kQkRows * DH * 2;  // one shifted input copy
    static constexpr int kW = DH * DH * 2;       // one tap of the weights
    static constexpr int kMaxSlots = DH == 64 ? 4 : 2;  // taps resident at once
    static constexpr int kPosBytes = 160 * 4;            // tile rows' positions (at most 144 rows)
    static constexpr int kRedBytes = kQkRows * 2 * 4;    // per row, the two threads' partial squared norms
    // Rows of the projection tile (a multiple of 8: whole swizzle atoms): the
    // CTA's rows and both convolutions' halos.
    __host__ __device__ static int tile_rows(int k0, int k1)
    {
        return (kQkRows + (k1 - 1) + (k0 > 0 ? k0 - 1 : 0) + 7) / 8 * 8;
    }
    static size_t bytes(int slots, int k0, int k1)
    {
        return (size_t)slots * (kA + kW) + (size_t)tile_rows(k0, k1) * DH * 2 + (size_t)DH * kMaxTapsSeq * 4 +
               kPosBytes + kRedBytes + 64 + 1024;
    }
};

// Byte offset of 16-byte chunk c (channels 8c .. 8c + 7) of row n in a tile
// of `rows` rows laid out as the 128-byte swizzle places it (TMA copies, and
// K-major MMA operands): 64-channel column blocks of rows x 128 bytes, the
// chunk index XOR-ed with the row's position in its 8-row, 1024-byte atom.
__device__ __forceinline__ uint32_t sw128_offset(int rows, int n, int c)
{
    return (uint32_t)((c >> 3) * rows * 128 + n * 128 + (((c & 7) ^ (n & 7)) << 4));
}

__device__ __forceinline__ uint4 pack8_f16(const float (&a)[8], bool &over)
{
    uint4 o;
#pragma unroll
    for (int q = 0; q < 8; ++q) over |= ptx::beyond_f16(a[q]);
    o.x = ptx::pack_f16_satfinite(a[0], a[1]);
    o.y = ptx::pack_f16_satfinite(a[2], a[3]);
    o.z = ptx::pack_f16_satfinite(a[4], a[5]);
    o.w = ptx::pack_f16_satfinite(a[6], a[7]);
    return o;
}

__device__ __forceinline__ void unpack8_bf16(const uint4 &w, float (&a)[8])
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        a[2 * q] = __uint_as_float(u[q] << 16);
        a[2 * q + 1] = __uint_as_float(u[q] & 0xffff0000u);
    }
}

// The channel convolution's weights as the qk kernel copies them: per head g
// (grid y) and tap j, W_j[o, i] = W1[g d_h + o, i, j] in fp16 (the identity
// without the convolution) in the K-major 128-byte-swizzle operand layout.
template <int DH>
__global__ void __launch_bounds__(256) cca_w1_image_kernel(const bf16 *__restrict__ w1, int k1, uint8_t *img,
                                                           uint32_t *status)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    constexpr int kChunks = DH / 8, kPerTap = DH * kChunks;
    const int g = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= k1 * kPerTap) return;
    const int j = e / kPerTap, o = (e % kPerTap) / kChunks, c = e % kChunks;
    float a[8];
    if (w1) {
        const bf16 *src = w1 + ((int64_t)(g * DH + o) * DH + 8 * c) * k1 + j;
#pragma unroll
        for (int q = 0; q < 8; ++q) a[q] = __bfloat162float(src[q * k1]);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) a[q] = 8 * c + q == o ? 1.f : 0.f;
    }
    bool over = false;
    *reinterpret_cast<uint4 *>(img + ((size_t)g * k1 + j) * QkTc<DH>::kW + sw128_offset(DH, o, c)) = pack8_f16(a, over);
    if (over && status) atomicOr(status, kStatusF16Range);
}

template <int DH>
__global__ void __launch_bounds__(kQkThreads, DH == 64 ? 2 : 1)
    cca_qk_tc_kernel(const __grid_constant__ CUtensorMap tx, CcaQkParams p)
{
    using C = QkTc<DH>;
    constexpr int half = DH / 2, kChunks = DH / 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int slots = p.slots, k0 = p.k0, k1 = p.k1;
    const int halo = k1 - 1, halo0 = k0 > 0 ? k0 - 1 : 0;
    const int Ub = C::tile_rows(k0, k1);
    uint8_t *sA = smem;                                                   // slots x kA
    uint8_t *sW = sA + (size_t)slots * C::kA;                             // slots x kW
    uint8_t *sX = sW + (size_t)slots * C::kW;                             // Ub x DH projections
    float *sW0 = reinterpret_cast<float *>(sX + (size_t)Ub * DH * 2);     // [k0][DH]
    int *spos = reinterpret_cast<int *>(sW0 + DH * kMaxTapsSeq);          // [Ub] position in sequence, -1 outside
    float (*red)[2] = reinterpret_cast<float (*)[2]>(spos + C::kPosBytes / 4);
    uint64_t *x_full = reinterpret_cast<uint64_t *>(red + kQkRows);
    uint64_t *w_full = x_full + 1;
    uint64_t *mma_done = x_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(x_full + 3);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // Thread tid: row m = tid % 128 (tensor-memory lane m; warps w and w + 4
    // share a lane quarter) and half hf = tid / 128 of the row's RoPE pairs.
    const int tid = threadIdx.x, warp = tid / 32, m = tid % kQkRows, hf = tid / kQkRows;
    const int g = blockIdx.y, ch0 = g * DH;  // the head's first packed channel
    // Rows fit in 32 bits (the host checks T).
    const int T = (int)p.T;
    const int r0 = blockIdx.x * kQkRows, r = r0 + m;
    const int u0 = r0 - halo - halo0;        // global row of tile row 0
    const bool live = r < T;
    const int Wp = p.P + p.Lkv;
    const uint8_t *img = p.w1img + (size_t)g * k1 * C::kW;
    bool over = false;
    int w_loads = 0;  // weight copies issued (thread 0)

    if (tid == 0) {
        ptx::mbar_init(x_full, 1);
        ptx::mbar_init(w_full, 1);
        ptx::mbar_init(mma_done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tx);
    }
    // Depth-wise weights of the head's channels, [tap][channel] (immutable:
    // before the wait).
    for (int e = tid; e < DH * k0; e += kQkThreads)
        sW0[(e % k0) * DH + e / k0] = __bfloat162float(p.w0[(int64_t)ch0 * k0 + e]);
    for (int u = tid; u < Ub; u += kQkThreads) {
        const int row = u0 + u;
        spos[u] = row >= 0 && row < T ? row % p.S : -1;
    }
    __syncthreads();
    // The projections and the weight image come from earlier kernels.
    ptx::pdl_wait();
    if (warp == 0) ptx::tmem_alloc(tmem_slot, DH);
    if (tid == 0) {
        ptx::mbar_expect_tx(x_full, (uint32_t)(DH / 64) * Ub * 128);
        for (int kc = 0; kc < DH / 64; ++kc)
            ptx::tma_load_2d(sX + (size_t)kc * Ub * 128, &tx, x_full, ch0 + 64 * kc, u0);
        const int nt = min(slots, k1);
        ptx::mbar_expect_tx(w_full, (uint32_t)(nt * C::kW));
        ptx::bulk_load(sW, img, (uint32_t)(nt * C::kW), w_full);
        w_loads = 1;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = __syncthreads_and(ptx::mbar_wait(x_full, 0, abort_flag));

    int pass = 0;
    for (int j0 = 0; ok && j0 < k1; j0 += slots, ++pass) {
        const int nt = min(slots, k1 - j0);
        if (pass > 0) {
            // The slots are rewritten once the previous pass's MMAs have read them.
            ok = __syncthreads_and(ptx::mbar_wait(mma_done, (pass - 1) & 1, abort_flag));
            if (!ok) break;
            ptx::tc_fence_after();
            if (tid == 0) {
                ptx::mbar_expect_tx(w_full, (uint32_t)(nt * C::kW));
                ptx::bulk_load(sW, img + (size_t)j0 * C::kW, (uint32_t)(nt * C::kW), w_full);
                ++w_loads;
            }
        }
        // Depth-wise output a[s] for s = r0 - halo + i, i in [0, 128 + halo)
        // (tile row i + halo0),
        // once per (row, 8-channel chunk), written to every shifted copy it
        // feeds: A_j[n] = a[r0 + n - back_j] (back_j = k1 - 1 - j) at
        // n = i + back_j - halo, zero when row r0 + n lies fewer than back_j
        // rows into its sequence.  Consecutive threads take consecutive rows.
        const int n_rows = kQkRows + halo;
#pragma unroll 1
        for (int e = tid; e < n_rows * kChunks; e += kQkThreads) {
            const int i = e % n_rows, c = e / n_rows;
            const int u = i + halo0;  // tile row of s
            const int ts = spos[u];
            float a[8];
            if (k0 == 0) {
                unpack8_bf16(*reinterpret_cast<const uint4 *>(sX + sw128_offset(Ub, u, c)), a);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) a[q] = 0.f;
                // Tap jj reads row srow - (k0 - 1 - jj), within srow's sequence.
                for (int jj = 0; jj < k0; ++jj) {
                    const int b0 = k0 - 1 - jj;
                    if (ts < b0) continue;
                    float x[8];
                    unpack8_bf16(*reinterpret_cast<const uint4 *>(sX + sw128_offset(Ub, u - b0, c)), x);
                    const float4 wa = *reinterpret_cast<const float4 *>(sW0 + jj * DH + 8 * c);
                    const float4 wb = *reinterpret_cast<const float4 *>(sW0 + jj * DH + 8 * c + 4);
                    a[0] = fmaf(wa.x, x[0], a[0]);
                    a[1] = fmaf(wa.y, x[1], a[1]);
                    a[2] = fmaf(wa.z, x[2], a[2]);
                    a[3] = fmaf(wa.w, x[3], a[3]);
                    a[4] = fmaf(wb.x, x[4], a[4]);
                    a[5] = fmaf(wb.y, x[5], a[5]);
                    a[6] = fmaf(wb.z, x[6], a[6]);
                    a[7] = fmaf(wb.w, x[7], a[7]);
                }
            }
            const uint4 packed = pack8_f16(a, over);
            for (int s = 0; s < nt; ++s) {
                const int back = k1 - 1 - (j0 + s), n = i + back - halo;
                if (n < 0 || n >= kQkRows) continue;
                const bool in_seq = spos[n + halo + halo0] >= back;
                *reinterpret_cast<uint4 *>(sA + (size_t)s * C::kA + sw128_offset(kQkRows, n, c)) =
                    in_seq ? packed : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            if (ptx::mbar_wait(w_full, pass & 1, abort_flag)) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_f16(kQkRows, DH, false, false);
                for (int s = 0; s < nt; ++s) {
                    const uint32_t a0 = ptx::smem_u32(sA + (size_t)s * C::kA);
                    const uint32_t b0 = ptx::smem_u32(sW + (size_t)s * C::kW);
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        ptx::mma_bf16(tmem,
                                      ptx::sdesc_sw128(a0 + (kk >> 2) * (kQkRows * 128) + (kk & 3) * 32, 16, 1024),
                                      ptx::sdesc_sw128(b0 + (kk >> 2) * (DH * 128) + (kk & 3) * 32, 16, 1024), idesc,
                                      (j0 + s > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(mma_done);
            } else {
                *abort_flag = 1;
            }
        }
    }
    if (ok) ok = __syncthreads_and(ptx::mbar_wait(mma_done, (pass - 1) & 1, abort_flag));

    if (ok) {
        // This thread's columns: RoPE pairs i in [hf QH, hf QH + QH), i.e.
        // columns c0 + [0, QH) in v[0, QH) and c0 + half + [0, QH) in
        // v[QH, 2 QH).
        constexpr int QH = half / 2, kCq = QH / 8;
        const int c0 = hf * QH;
        ptx::tc_fence_after();
        float v[2 * QH];
        const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t w[QH];
            if constexpr (QH == 32) ptx::tmem_ld32(lane_base + c0 + part * half, w);
            else ptx::tmem_ld16(lane_base + c0 + part * half, w);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < QH; ++q) v[part * QH + q] = __uint_as_float(w[q]);
        }
        if (live && p.qk_mean) {
            // Query head g: + (q_g + k_(g / gs)) / 2 of the projections; key
            // head jh: + (k_jh + the mean of its group's query heads) / 2.
            const int u = m + halo + halo0;  // tile row of r
#pragma unroll
            for (int j = 0; j < 2 * kCq; ++j) {
                const int c = c0 / 8 + (j % kCq) + (j / kCq) * (half / 8);
                float a[8];
                unpack8_bf16(*reinterpret_cast<const uint4 *>(sX + sw128_offset(Ub, u, c)), a);
#pragma unroll
                for (int q = 0; q < 8; ++q) v[8 * j + q] = fmaf(0.5f, a[q], v[8 * j + q]);
            }
            const bool key = g >= p.Hq;
            const int other = key ? (g - p.Hq) * p.gs : p.Hq + g / p.gs;  // first partner head
            const int n_other = key ? p.gs : 1;
            const float w_other = 0.5f / (float)n_other;
            const uint4 *row = reinterpret_cast<const uint4 *>(p.pre + (int64_t)r * Wp);
#pragma unroll 1
            for (int h = other; h < other + n_other; ++h) {
                uint4 b[2 * kCq];
#pragma unroll
                for (int j = 0; j < 2 * kCq; ++j) b[j] = row[h * kChunks + c0 / 8 + (j % kCq) + (j / kCq) * (half / 8)];
#pragma unroll
                for (int j = 0; j < 2 * kCq; ++j) {
                    float x[8];
                    unpack8_bf16(b[j], x);
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[8 * j + q] = fmaf(w_other, x[q], v[8 * j + q]);
                }
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int o = 0; o < 2 * QH; ++o) ss = fmaf(v[o], v[o], ss);
        red[m][hf] = ss;
        __syncthreads();
        if (live) {
            const float tot = red[m][0] + red[m][1];
            float sc = sqrtf((float)DH) / fmaxf(sqrtf(tot), 1e-6f);
            if (g >= p.Hq) sc *= p.k_scale;
            const float4 *cs = reinterpret_cast<const float4 *>(p.rope + (int64_t)spos[m + halo + halo0] * half + c0);
#pragma unroll
            for (int i2 = 0; i2 < QH / 2; ++i2) {
                const float4 e = cs[i2];  // (cos, sin) of pairs c0 + 2 i2 and c0 + 2 i2 + 1
#pragma unroll
                for (int d = 0; d < 2; ++d) {
                    const int i = 2 * i2 + d;
                    const float cv = d ? e.z : e.x, sv = d ? e.w : e.y;
                    const float x0 = v[i] * sc, x1 = v[i + QH] * sc;
                    v[i] = x0 * cv - x1 * sv;
                    v[i + QH] = x0 * sv + x1 * cv;
                }
            }
            if (g < p.Hq) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.q + (int64_t)r * p.Lq + ch0);
#pragma unroll
                for (int j = 0; j < 2 * kCq; ++j)
                    dst[c0 / 8 + (j % kCq) + (j / kCq) * (half / 8)] =
                        make_uint4(ptx::pack_bf16(v[8 * j], v[8 * j + 1]), ptx::pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                                   ptx::pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                                   ptx::pack_bf16(v[8 * j + 6], v[8 * j + 7]));
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(p.k + (int64_t)r * p.Lkv + (ch0 - p.Lq));
#pragma unroll
                for (int j = 0; j < 2 * kCq; ++j) {
                    float a[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) a[q] = v[8 * j + q];
                    dst[c0 / 8 + (j % kCq) + (j / kCq) * (half / 8)] = pack8_f16(a, over);
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // Copies still in flight after a timeout land before the shared
        // memory is released.
        if (!ok && tid == 0) {
            volatile int never = 0;
            ptx::mbar_wait(x_full, 0, &never);
            if (w_loads > 0) ptx::mbar_wait(w_full, (w_loads - 1) & 1, &never);
        }
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, DH);
    }
    ptx::pdl_trigger();
    if (over && p.status) atomicOr(p.status, kStatusF16Range);
    if (tid == 0 && !ok && p.status) atomicOr(p.status, kStatusTimeout);
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

    // 1. Down-projections (one grouped GEMM) into column slices of pre:
    //    [W_QK x | W_V1 x | W_V2 x] (or [W_QK x | W_V x]).
    float *split = (float *)(wb + L.split);
    auto gemm = [&](GemmArgs g) -> mla_status {
        g.split_ws = split;  // GEMMs run one after another on the stream: one split region serves all
        if (!gemm_tc_supported(g)) return MLA_ERR_UNSUPPORTED;
        return cuda(gemm_tc(g, h->num_sms, s));
    };
    if ((st = gemm(cca_down_proj(c, x, T, w, pre, status))) != MLA_OK) return st;

    // 2. The values (fp16).
    __half *v = (__half *)(wb + L.v);
    {
        const int64_t n = T * (Lkv / 8);
        st = cuda(launch_ex(cca_v_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, 1, (const bf16 *)pre, T,
                            S, P, Lkv, v, c.value_shift, status));
        note_launch();
        if (st != MLA_OK) return st;
    }

    // 3. Both convolutions, q-k-mean, normalisation, temperature, RoPE.
    CcaQkParams q;
    q.pre = pre;
    q.w0 = c.conv_layers >= 1 ? (const bf16 *)w->conv0 : nullptr;
    q.w1img = (const uint8_t *)(wb + L.w1img);
    q.T = T; q.S = S; q.P = P; q.Lkv = Lkv; q.Lq = c.q_latent; q.Hq = c.n_heads;
    q.gs = c.n_heads / c.n_kv_heads;
    q.k0 = c.conv_layers >= 1 ? c.conv_kernel_seq : 0;
    q.k1 = c.conv_layers >= 2 ? c.conv_kernel_ch : 1;
    q.qk_mean = c.qk_mean;
    q.k_scale = (float)exp(c.key_temp);
    q.rope = h->rope_table;
    q.q = (bf16 *)(wb + L.q);
    q.k = (__half *)(wb + L.k);
    q.status = status;
    {
        const int heads = c.n_heads + c.n_kv_heads;
        const bf16 *w1 = c.conv_layers >= 2 ? (const bf16 *)w->conv1 : nullptr;
        uint8_t *img = (uint8_t *)(wb + L.w1img);
        const dim3 grid((unsigned)((T + kQkRows - 1) / kQkRows), (unsigned)heads);
        const dim3 igrid((unsigned)((q.k1 * dh * dh / 8 + 255) / 256), (unsigned)heads);
        static std::atomic<int> smem64{-1}, smem128{-1};
        auto run = [&](auto image_kernel, auto qk_kernel, auto cfg, std::atomic<int> &smem_set) -> mla_status {
            using Q = decltype(cfg);
            CUtensorMap tx;
            if (!make_tmap_bf16(&tx, pre, T, Wp, Wp, 64, Q::tile_rows(q.k0, q.k1))) return MLA_ERR_CUDA;
            mla_status r = cuda(launch_ex(image_kernel, igrid, dim3(256), 0, s, 1, w1, q.k1, img, status));
            note_launch();
            if (r != MLA_OK) return r;
            q.slots = std::min(q.k1, Q::kMaxSlots);
            r = cuda(smem_limit_once(smem_set, (const void *)qk_kernel,
                                     (int)Q::bytes(Q::kMaxSlots, kMaxTapsSeq, kMaxTapsCh)));
            if (r == MLA_OK)
                r = cuda(launch_ex(qk_kernel, grid, dim3(kQkThreads), Q::bytes(q.slots, q.k0, q.k1), s, 1, tx, q));
            note_launch();
            return r;
        };
        st = dh == 64 ? run(cca_w1_image_kernel<64>, cca_qk_tc_kernel<64>, QkTc<64>{}, smem64)
                      : run(cca_w1_image_kernel<128>, cca_qk_tc_kernel<128>, QkTc<128>{}, smem128);
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

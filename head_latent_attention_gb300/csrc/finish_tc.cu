// End of the weight-absorbed decode on the tensor cores: the log-sum-exp
// merge of the split-KV partials and the value up-projection, fused.
//
// deepseek-mla `MultiHeadLatentAttention.forward` (and mlra_attn per latent
// block) weights the up-projected values W_UV,h c_j by the softmax; by
// linearity o_h = W_UV,h (sum_j p_hj c_j), so the split-KV kernels attend in
// latent space and leave, per work range that covers only part of a
// sequence, its latent average (normalised by the range's own row sum, in
// bfloat16) with the range's reference max and row sum.  This kernel
// finishes the head:
//
// One CTA per (head h, group of 64 sequences):
//   1. TMA copies W_UV,h ([128, r_lat] bfloat16, K-major) into shared memory;
//   2. the eight warps merge the partials of each sequence of the group
//      (or read the latent average that a single range wrote directly) and
//      store the bfloat16 result as a K-major, 128-byte-swizzled operand;
//   3. one thread issues o_h^T[128, 64] = W_UV,h [128, r_lat] * o_lat^T
//      (tcgen05.mma M=128, N=64, accumulator in tensor memory);
//   4. the eight warps read the accumulator back and store o[b, h, :].
// The merged latent average never leaves the SM.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr int kTok = 64;        // sequences per CTA (MMA N)
constexpr int kDv = 128;        // value head width (MMA M)
constexpr int kThreads = 256;
constexpr int kWBlk = kDv * 128;   // one 64-column block of W_UV,h: 16 KB
constexpr int kOBlk = kTok * 128;  // one 64-column block of the latent operand: 8 KB

template <int R>
struct FinCfg {
    static constexpr int kBlocks = R / 64;
    static constexpr int kSmem = kBlocks * (kWBlk + kOBlk) + 1024 /*align*/ + 64 /*barriers*/;
};

struct FinParams {
    const int *seq_fc;     // [B] first range covering each sequence (-1: empty)
    const int *seq_lc;     // [B] last range covering each sequence
    int B, H;
    const bf16 *o_part;    // [(ranges + B), H, R] normalised partial averages
    const float *ml_part;  // [(ranges + B), H, 2] (max in log2 units, row sum)
    const bf16 *o_lat;     // [B, H, R] written directly for single-range sequences
    bf16 *o;               // [B, H, 128]
    uint32_t *status;
};

// Loads of up to four partial slots of one sequence (ranges c0 .. c0 + 3,
// clipped at lc): this lane's CPL columns of each normalised average and the
// slots' (max, row sum).
template <int R>
struct SlotGroup {
    uint4 v[4][R / 256];
    float2 ml[4];
};

template <int R>
__device__ __forceinline__ void load_group(const FinParams &p, int b, int h, int lane, int c0, int lc,
                                           SlotGroup<R> &g)
{
    constexpr int CPL = R / 32;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int c = c0 + u;
        if (c <= lc) {
            const int64_t slot = (int64_t)(c + b) * p.H + h;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.o_part + slot * R + lane * CPL);
#pragma unroll
            for (int j = 0; j < CPL / 8; ++j) g.v[u][j] = __ldcs(src + j);
            g.ml[u] = *reinterpret_cast<const float2 *>(p.ml_part + slot * 2);
        } else {
#pragma unroll
            for (int j = 0; j < CPL / 8; ++j) g.v[u][j] = make_uint4(0, 0, 0, 0);
            g.ml[u] = make_float2(-INFINITY, 0.f);
        }
    }
}

// Online merge of a group into (m, den, acc): slot c's average O_c
// (normalised by its row sum l_c) weighs 2^(m_c - m) l_c.
template <int R>
__device__ __forceinline__ void merge_group(const SlotGroup<R> &g, float &m, float &den, float (&acc)[R / 32])
{
    constexpr int CPL = R / 32;
    const float mg = fmaxf(fmaxf(g.ml[0].x, g.ml[1].x), fmaxf(g.ml[2].x, g.ml[3].x));
    const float m_new = fmaxf(m, mg);
    const float sc = exp2f(m - m_new);  // 0 on the first group (m = -inf)
    den *= sc;
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[i] *= sc;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float w = g.ml[u].y == 0.f ? 0.f : exp2f(g.ml[u].x - m_new) * g.ml[u].y;
        den += w;
#pragma unroll
        for (int j = 0; j < CPL / 8; ++j) {
            const uint32_t wd[4] = {g.v[u][j].x, g.v[u][j].y, g.v[u][j].z, g.v[u][j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[8 * j + 2 * q] += w * __uint_as_float(wd[q] << 16);
                acc[8 * j + 2 * q + 1] += w * __uint_as_float(wd[q] & 0xffff0000u);
            }
        }
    }
    m = m_new;
}

// Latent averages of sequences b and b + 1 (ranges fc[u] .. lc[u]), head h,
// columns [lane * CPL, lane * CPL + CPL) (CPL = R / 32), as bfloat16 pairs.
// The loads of both sequences go out before either is merged.
template <int R>
__device__ __forceinline__ void merged_pair(const FinParams &p, int b, const int (&fc)[2], const int (&lc)[2], int h,
                                           int lane, uint32_t (&out)[2][R / 64])
{
    constexpr int CPL = R / 32;
    SlotGroup<R> g[2];
    uint4 direct[2][CPL / 8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        if (fc[u] >= 0 && fc[u] == lc[u]) {
            const uint4 *src =
                reinterpret_cast<const uint4 *>(p.o_lat + ((int64_t)(b + u) * p.H + h) * R + lane * CPL);
#pragma unroll
            for (int i = 0; i < CPL / 8; ++i) direct[u][i] = src[i];
        } else if (fc[u] >= 0) {
            load_group<R>(p, b + u, h, lane, fc[u], lc[u], g[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int i = 0; i < CPL / 2; ++i) out[u][i] = 0u;
        if (fc[u] < 0) continue;  // empty or invalid length (or past the batch): zero
        if (fc[u] == lc[u]) {
#pragma unroll
            for (int i = 0; i < CPL / 8; ++i) {
                out[u][4 * i] = direct[u][i].x; out[u][4 * i + 1] = direct[u][i].y;
                out[u][4 * i + 2] = direct[u][i].z; out[u][4 * i + 3] = direct[u][i].w;
            }
            continue;
        }
        float m = -INFINITY, den = 0.f, acc[CPL];
#pragma unroll
        for (int i = 0; i < CPL; ++i) acc[i] = 0.f;
        merge_group<R>(g[u], m, den, acc);
        for (int c0 = fc[u] + 4; c0 <= lc[u]; c0 += 4) {  // more than four ranges: rare
            load_group<R>(p, b + u, h, lane, c0, lc[u], g[u]);
            merge_group<R>(g[u], m, den, acc);
        }
        const float inv = 1.f / den;
#pragma unroll
        for (int i = 0; i < CPL / 2; ++i) out[u][i] = ptx::pack_bf16(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1) decode_finish_kernel(const __grid_constant__ CUtensorMap tw,
                                                                    FinParams p)
{
    using C = FinCfg<R>;
    constexpr int CPL = R / 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sW = smem;
    uint8_t *sO = smem + C::kBlocks * kWBlk;
    uint64_t *w_full = (uint64_t *)(sO + C::kBlocks * kOBlk);
    uint64_t *mma_done = w_full + 1;
    uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int h = blockIdx.x, b0 = blockIdx.y * kTok;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        ptx::mbar_init(w_full, 1);
        ptx::mbar_init(mma_done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) ptx::tmem_alloc(tmem_slot, 64);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // 1. The weights of head h, in the background (they do not depend on
    // earlier kernels, so they go out before the wait for them).
    if (threadIdx.x == 0) {
        ptx::pdl_trigger();
        ptx::prefetch_tmap(&tw);
        ptx::mbar_expect_tx(w_full, C::kBlocks * kWBlk);
        const uint64_t evict_first = ptx::policy_evict_first();  // each weight byte is read once
#pragma unroll
        for (int kb = 0; kb < C::kBlocks; ++kb)
            ptx::tma_load_2d_hint(sW + kb * kWBlk, &tw, w_full, kb * 64, h * kDv, evict_first);
    }

    ptx::pdl_wait();
    // 2. Merged latent averages of the group's sequences: warp w takes
    //    sequences 8 w .. 8 w + 7, whose covering ranges its first lanes load
    //    in one round trip, then merges them two at a time.
    {
        constexpr int kPerWarp = kTok / (kThreads / 32);
        int fcv = -1, lcv = -1;
        if (lane < kPerWarp && b0 + warp * kPerWarp + lane < p.B) {
            fcv = p.seq_fc[b0 + warp * kPerWarp + lane];
            lcv = p.seq_lc[b0 + warp * kPerWarp + lane];
        }
#pragma unroll 1
        for (int i = 0; i < kPerWarp; i += 2) {
            const int t = warp * kPerWarp + i;
            int fc[2], lc[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                fc[u] = __shfl_sync(0xffffffffu, fcv, i + u);
                lc[u] = __shfl_sync(0xffffffffu, lcv, i + u);
            }
            uint32_t v[2][R / 64];
            merged_pair<R>(p, b0 + t, fc, lc, h, lane, v);
            // Columns [lane * CPL, +CPL) are CPL / 8 chunks of 16 bytes; chunk
            // g sits in 64-column block g / 8, at position (g % 8) ^ (row % 8)
            // of the row.
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int k = 0; k < CPL / 8; ++k) {
                    const int g = lane * (CPL / 8) + k, row = t + u;
                    uint8_t *dst = sO + (g >> 3) * kOBlk + row * 128 + (((g & 7) ^ (row & 7)) << 4);
                    *reinterpret_cast<uint4 *>(dst) =
                        make_uint4(v[u][4 * k], v[u][4 * k + 1], v[u][4 * k + 2], v[u][4 * k + 3]);
                }
        }
    }
    ptx::fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
    __syncthreads();

    // 3. o_h^T = W_UV,h * o_lat^T.
    if (warp == 0) {
        if (ptx::elect_one()) {
            if (ptx::mbar_wait(w_full, 0, abort_flag)) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16(kDv, kTok, false, false);
                const uint32_t w0 = ptx::smem_u32(sW), o0 = ptx::smem_u32(sO);
#pragma unroll
                for (int kb = 0; kb < C::kBlocks; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_bf16(tmem, ptx::sdesc_sw128(w0 + kb * kWBlk + k * 32, 16, 1024),
                                      ptx::sdesc_sw128(o0 + kb * kOBlk + k * 32, 16, 1024), idesc,
                                      (kb | k) != 0 ? 1u : 0u);
                ptx::mma_commit(mma_done);
            } else {
                *abort_flag = 1;
            }
        }
        __syncwarp();
    }

    // 4. Accumulator row d (tensor-memory lane d) holds o[b0 + t, h, d] in
    // column t; warps w and w + 4 share lane quadrant w % 4 and take token
    // halves.
    // (Warp-uniform outcome: the tensor-memory loads below are warp-wide.)
    if (__all_sync(0xffffffffu, ptx::mbar_wait(mma_done, 0, abort_flag))) {
        ptx::tc_fence_after();
        const int quad = warp % 4, half = warp / 4;
        const int d = quad * 32 + lane;
        uint32_t r[32];
        ptx::tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + half * 32, r);
        ptx::tmem_ld_wait();
        bf16 *dst = p.o + ((int64_t)(b0 + half * 32) * p.H + h) * kDv + d;
        const int nt = min(32, p.B - b0 - half * 32);
#pragma unroll
        for (int t = 0; t < 32; ++t)
            if (t < nt) dst[(int64_t)t * p.H * kDv] = __float2bfloat16_rn(__uint_as_float(r[t]));
    } else {
        *abort_flag = 1;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // A weight copy still in flight after a timeout must land before the
        // CTA's shared memory is released.
        if (*abort_flag) {
            volatile int never = 0;
            ptx::mbar_wait(w_full, 0, &never);
        }
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 64);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

template <int R>
cudaError_t launch_finish(const FinishArgs &a, cudaStream_t s)
{
    using C = FinCfg<R>;
    CUtensorMap tw;
    if (!make_tmap_bf16(&tw, a.W_UV, (int64_t)a.H * kDv, R, R, 64, kDv)) return cudaErrorInvalidValue;
    static std::atomic<int> smem_dev{-1};
    cudaError_t e = smem_limit_once(smem_dev, (const void *)decode_finish_kernel<R>, C::kSmem);
    if (e != cudaSuccess) return e;
    FinParams p;
    p.seq_fc = a.seq_fc; p.seq_lc = a.seq_lc;
    p.B = a.B; p.H = a.H;
    p.o_part = a.o_part; p.ml_part = a.ml_part;
    p.o_lat = (const bf16 *)a.o_lat;
    p.o = (bf16 *)a.o;
    p.status = a.status;
    e = launch_ex(decode_finish_kernel<R>, dim3(a.H, (a.B + kTok - 1) / kTok), dim3(kThreads), C::kSmem, s, 1, tw, p);
    note_launch();
    return e;
}

}  // namespace

bool decode_finish_supported(int r_lat, int d_v) { return d_v == kDv && (r_lat == 256 || r_lat == 512); }

cudaError_t decode_finish(const FinishArgs &a, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    if (!decode_finish_supported(a.r_lat, a.d_v)) return cudaErrorInvalidValue;
    return a.r_lat == 512 ? launch_finish<512>(a, s) : launch_finish<256>(a, s);
}

}  // namespace mla

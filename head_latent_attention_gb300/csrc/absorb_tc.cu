// Query absorption for the decode on the tensor cores.
//
// deepseek-mla `MultiHeadLatentAttention.forward` scores the query against the
// up-projected keys, q_C,h . (W_UK,h c_j); by associativity that equals
// (W_UK,h^T q_C,h) . c_j, so the decode attends over the cached latent with
// the absorbed query q_abs,h = W_UK,h^T q_C,h (mlra_attn: per head, the rows
// of its latent block's W_UK).  W_UK,h is rows [128 h, 128 h + 128) of W_UK
// viewed as [H * 128, r_lat], so q_abs,h[r] = sum_d q_C,h[d] W_UK[128 h + d, r].
//
// One CTA per (head h, group of 64 sequences), with the head's weights
// resident in shared memory:
//   - TMA copies W_UK,h (128 x r_lat, 128-byte swizzle; these copies go out
//     before the wait for the previous kernel, which does not write them) and
//     the group's q_C,h rows (64 x 128);
//   - q_abs,h^T [r_lat, 64] = W_UK,h^T [r_lat, 128] q_C,h^T: r_lat / 128 MMAs
//     chains of M = 128 latent columns, N = 64 sequences, K = 128, with
//     W_UK,h read as an MN-major A operand straight from its row-major copy;
//   - tensor-memory lane = latent column, column = sequence: the eight warps
//     read the accumulators back and store q_abs[b, h, :].
// Every wait is bounded.
#include <cudaTypedefs.h>

#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr int kTok = 64;           // sequences per CTA (MMA N)
constexpr int kD = 128;            // query head width (MMA K)
constexpr int kThreads = 256;
constexpr int kWBox = kD * 128;    // 64 latent columns x 128 rows of W_UK,h: 16 KB
constexpr int kQBox = kTok * 128;  // 64 query columns x 64 sequences: 8 KB

template <int R>
struct AbsCfg {
    static constexpr int kBoxes = R / 64;
    static constexpr int kChains = R / 128;
    static constexpr int kTmemCols = kChains * kTok;  // 256 or 128
    static constexpr int kSmem = kBoxes * kWBox + 2 * kQBox + 1024 /*align*/ + 64 /*barriers*/;
};

struct AbsParams {
    int B, H;
    bf16 *q_abs;  // [B, H, R], or head-interleaved (see AbsorbArgs)
    bool interleave;
    uint32_t *status;
};

template <int R>
__global__ void __launch_bounds__(kThreads, 1) absorb_kernel(const __grid_constant__ CUtensorMap tw,
                                                             const __grid_constant__ CUtensorMap tq, AbsParams p)
{
    using C = AbsCfg<R>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sW = smem;
    uint8_t *sQ = smem + C::kBoxes * kWBox;
    uint64_t *w_full = (uint64_t *)(sQ + 2 * kQBox);
    uint64_t *q_full = w_full + 1;
    uint64_t *mma_done = w_full + 2;
    uint32_t *tmem_slot = (uint32_t *)(w_full + 3);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int h = blockIdx.x, b0 = blockIdx.y * kTok;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        ptx::mbar_init(w_full, 1);
        ptx::mbar_init(q_full, 1);
        ptx::mbar_init(mma_done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        // The weights of head h: latent columns [64 i, 64 i + 64) in box i.
        ptx::prefetch_tmap(&tw);
        ptx::prefetch_tmap(&tq);
        ptx::mbar_expect_tx(w_full, C::kBoxes * kWBox);
        const uint64_t evict_first = ptx::policy_evict_first();  // each weight byte is read once
#pragma unroll
        for (int i = 0; i < C::kBoxes; ++i)
            ptx::tma_load_2d_hint(sW + i * kWBox, &tw, w_full, i * 64, h * kD, evict_first);
        // The queries come from the projection kernel.  The trigger comes after
        // the wait: the split-KV kernel that follows reads the scheduler's
        // output (written by the previous kernel) before its own wait.
        ptx::pdl_wait();
        ptx::pdl_trigger();
        ptx::mbar_expect_tx(q_full, 2 * kQBox);
        ptx::tma_load_2d(sQ, &tq, q_full, h * kD, b0);
        ptx::tma_load_2d(sQ + kQBox, &tq, q_full, h * kD + 64, b0);
    }
    if (warp == 0) ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::pdl_wait();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (ptx::elect_one()) {
            if (ptx::mbar_wait(w_full, 0, abort_flag) && ptx::mbar_wait(q_full, 0, abort_flag)) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16(128, kTok, true, false);
                const uint32_t w0 = ptx::smem_u32(sW), q0 = ptx::smem_u32(sQ);
#pragma unroll
                for (int m = 0; m < C::kChains; ++m)
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k)
                        // A: boxes 2m and 2m + 1 are the two 64-column atoms of
                        // the chain (LBO = one box); 16 rows of K = 2048 bytes.
                        ptx::mma_bf16(tmem + m * kTok,
                                      ptx::sdesc_sw128(w0 + 2 * m * kWBox + k * 2048, kWBox, 1024),
                                      ptx::sdesc_sw128(q0 + (k >> 2) * kQBox + (k & 3) * 32, 16, 1024), idesc,
                                      k != 0 ? 1u : 0u);
                ptx::mma_commit(mma_done);
            } else {
                *abort_flag = 1;
            }
        }
        __syncwarp();
    }

    // Chain m, tensor-memory lane l: latent column 128 m + l; column t of the
    // chain: sequence b0 + t.  Warps w and w + 4 share lane quadrant w % 4 and
    // take sequence halves.
    // (Warp-uniform outcome: the tensor-memory loads below are warp-wide.)
    if (__all_sync(0xffffffffu, ptx::mbar_wait(mma_done, 0, abort_flag))) {
        ptx::tc_fence_after();
        const int quad = warp % 4, half = warp / 4;
        const int nt = min(32, p.B - b0 - half * 32);
#pragma unroll 1
        for (int m = 0; m < C::kChains; ++m) {
            uint32_t r[32];
            ptx::tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + m * kTok + half * 32, r);
            ptx::tmem_ld_wait();
            const int col = m * 128 + quad * 32 + lane;  // latent column
            bf16 *dst = p.interleave
                            ? p.q_abs + (((int64_t)(b0 + half * 32) * kQChunks + col / 8) * kQRows + h) * 8 + col % 8
                            : p.q_abs + ((int64_t)(b0 + half * 32) * p.H + h) * R + col;
            const int64_t tstride = p.interleave ? (int64_t)kQChunks * kQRows * 8 : (int64_t)p.H * R;
#pragma unroll
            for (int t = 0; t < 32; ++t)
                if (t < nt) dst[(int64_t)t * tstride] = __float2bfloat16_rn(__uint_as_float(r[t]));
        }
    } else {
        *abort_flag = 1;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // Copies still in flight after a timeout land before the shared
        // memory is released.
        if (*abort_flag) {
            volatile int never = 0;
            ptx::mbar_wait(w_full, 0, &never);
            ptx::mbar_wait(q_full, 0, &never);
        }
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

template <int R>
cudaError_t launch_absorb(const AbsorbArgs &a, cudaStream_t s)
{
    using C = AbsCfg<R>;
    CUtensorMap tw, tq;
    if (!make_tmap_bf16(&tw, a.W_UK, (int64_t)a.H * kD, R, R, 64, kD) ||
        !make_tmap_bf16(&tq, a.q_nope, a.B, (int64_t)a.H * kD, (int64_t)a.H * kD, 64, kTok))
        return cudaErrorInvalidValue;
    static std::atomic<int> smem_dev{-1};
    cudaError_t e = smem_limit_once(smem_dev, (const void *)absorb_kernel<R>, C::kSmem);
    if (e != cudaSuccess) return e;
    AbsParams p;
    p.B = a.B; p.H = a.H;
    p.q_abs = (bf16 *)a.q_abs;
    p.interleave = a.interleave;
    p.status = a.status;
    e = launch_ex(absorb_kernel<R>, dim3(a.H, (a.B + kTok - 1) / kTok), dim3(kThreads), C::kSmem, s, 1, tw, tq, p);
    note_launch();
    return e;
}

}  // namespace

bool absorb_supported(int r_lat, int d_nope) { return d_nope == kD && (r_lat == 256 || r_lat == 512); }

cudaError_t absorb(const AbsorbArgs &a, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    if (!absorb_supported(a.r_lat, a.d_nope)) return cudaErrorInvalidValue;
    if (a.interleave && (a.r_lat != 512 || a.H > kQRows)) return cudaErrorInvalidValue;
    return a.r_lat == 512 ? launch_absorb<512>(a, s) : launch_absorb<256>(a, s);
}

}  // namespace mla

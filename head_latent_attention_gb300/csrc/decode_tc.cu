// Weight-absorbed split-KV latent attention for decode on tcgen05, one
// 2-CTA cluster per work range.
//
// Per sequence b the 128 heads attend over the latent cache rows c_j (r_kv =
// 512) and rope keys k_R,j (d_rope = 64): s_hj = q_abs,h . c_j + q_R,h . k_R,j,
// softmax over j, o_lat,h = sum_j p_hj c_j.  The fp32 accumulator o_lat for
// 128 heads x 512 latent columns is exactly one SM's tensor memory, so a
// cluster of two CTAs splits the latent: CTA r owns columns [256 r, 256 r +
// 256) (CTA 0 also the rope columns).  Each CTA
//   - streams only its own columns of each 64-key tile (TMA, 128-byte swizzle);
//   - computes a partial score tile S_r = Q_r K_r^T (M = 128 heads, N = 64
//     keys) into tensor memory;
//   - sends S_r to its peer through distributed shared memory and adds the
//     peer's partial, so both CTAs hold the same fp32 scores and take the
//     same online-softmax decisions;
//   - accumulates O_r += P V_r (M = 128, N = 256, K = 64 keys) with the same
//     shared-memory tile read as an MN-major operand.
// Warp roles per CTA: warp 0 TMA producer, warp 1 MMA issuer, warps 2..5
// softmax (one head row per thread).  The running max is only raised when
// it grows by more than 8 (log2 units), so the O rescale is rare; the final
// result is exact either way because the same stale max is used for P and
// for the running sum.
//
// Work: the concatenation of all sequences' keys is cut into one contiguous
// range per cluster (a device-side scheduler computes the prefix sums of
// the lengths); a cluster's range splits into one segment per sequence it
// touches.  A segment that covers a whole sequence writes o_lat directly;
// others write (O, m, l) partials that a combine kernel merges.
#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr int kH = 128;       // heads per CTA = MMA M
constexpr int kBKV = 64;      // keys per tile
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr int kXStride = 68;  // floats per exchange-buffer row (272 bytes: conflict-free v4 rows)
constexpr float kRescaleThreshold = 8.f;

template <int LA>  // latent atoms (64 columns) per CTA
struct DCfg {
    static constexpr int kQAtoms = LA + 1;
    static constexpr int kQBytes = kQAtoms * kH * 128;
    static constexpr int kAtomBytes = kBKV * 128;
    static constexpr int kStageBytes = kQAtoms * kAtomBytes;
    static constexpr int kPBytes = kH * 128;
    static constexpr int kXBytes = kH * kXStride * 4;
    static constexpr int kOffKV = kQBytes;
    static constexpr int kOffP = kOffKV + kStages * kStageBytes;
    static constexpr int kOffX = kOffP + kPBytes;
    static constexpr int kOffBar = kOffX + kXBytes;
    static constexpr int kSmem = kOffBar + 256 + 1024;
    static constexpr int kOCols = LA * 64;
    static constexpr int kSCol = kOCols;
    static constexpr int kRLat = 2 * LA * 64;
};

struct DecTcParams {
    int B, H, max_seq;
    const int *prefix;  // [B + 1] prefix sums of the valid lengths
    const int *chunk;   // keys per cluster
    float scale_log2;
    bf16 *o_lat;        // [B, H, r_kv]
    float *o_part;      // [slots, H, r_kv]
    float *ml_part;     // [slots, H, 2]
    uint32_t *status;
};

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full, pv_done, o_empty;
    uint64_t x_full, peer_free;
    int abort;
    uint32_t tmem;
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(const void *p, uint32_t peer)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(ptx::smem_u32(p)), "r"(peer));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t remote_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Segments of this cluster's key range [start, end) of the concatenated keys.
struct SegIter {
    const int *prefix;
    int B, start, end, b;
    __device__ void init(const int *pf, int nb, int cid, int chunk)
    {
        prefix = pf;
        B = nb;
        const int total = pf[nb];
        start = min(total, cid * chunk);
        end = min(total, start + chunk);
        int lo = 0, hi = nb - 1;  // first b with prefix[b + 1] > start
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            if (pf[mid + 1] > start) hi = mid;
            else lo = mid + 1;
        }
        b = (start < end) ? lo : nb;
    }
    // Next non-empty segment: sequence b, keys [k0, k1), whole-sequence flag.
    __device__ bool next(int &sb, int &k0, int &k1, bool &whole)
    {
        while (b < B && prefix[b] < end) {
            const int lo = prefix[b], hi = prefix[b + 1];
            const int gs = max(start, lo), ge = min(end, hi);
            const int cur = b++;
            if (gs < ge) {
                sb = cur;
                k0 = gs - lo;
                k1 = ge - lo;
                whole = (gs == lo && ge == hi);
                return true;
            }
        }
        return false;
    }
};

// Walks the tiles of this cluster's segments in order (g: global tile
// index, t: tile within segment nseg).
struct TileCursor {
    SegIter it;
    int b, k0, k1, nseg, t, ntiles, g;
    bool whole, valid;
    __device__ void init(const int *pf, int nb, int cid, int chunk)
    {
        it.init(pf, nb, cid, chunk);
        nseg = -1;
        g = 0;
        valid = true;
        next_segment();
    }
    __device__ void next_segment()
    {
        if (it.next(b, k0, k1, whole)) {
            ++nseg;
            t = 0;
            ntiles = (k1 - k0 + kBKV - 1) / kBKV;
        } else {
            valid = false;
        }
    }
    __device__ void step()
    {
        ++g;
        if (++t == ntiles) next_segment();
    }
};

template <int LA>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQR,
                     const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmR,
                     DecTcParams p)
{
    using C = DCfg<LA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + C::kOffKV;
    uint8_t *sP = smem + C::kOffP;
    float *sX = (float *)(smem + C::kOffX);
    Bars *bar = (Bars *)(smem + C::kOffBar);
    volatile int *abort_flag = &bar->abort;

    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int cid = (int)cluster_id();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nq_atoms = LA + (rank == 0 ? 1 : 0);

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar->q_full, 1);
        ptx::mbar_init(&bar->q_empty, 1);
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&bar->kv_full[i], 1);
            ptx::mbar_init(&bar->kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&bar->s_full[i], 1);
            ptx::mbar_init(&bar->s_empty[i], kH);
        }
        ptx::mbar_init(&bar->p_full, kH);
        ptx::mbar_init(&bar->pv_done, 1);
        ptx::mbar_init(&bar->o_empty, kH);
        ptx::mbar_init(&bar->x_full, kH);
        ptx::mbar_init(&bar->peer_free, kH);
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(&bar->tmem, 512);
    ptx::tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem = bar->tmem;
    const int chunk = *p.chunk;
    bool ok = true;
    auto fail = [&]() {
        ok = false;
        *abort_flag = 1;
        st_cluster_u32(map_peer((const void *)abort_flag, peer), 1u);
    };

    if (warp == 0) {
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&tmQ);
            ptx::prefetch_tmap(&tmQR);
            ptx::prefetch_tmap(&tmL);
            ptx::prefetch_tmap(&tmR);
            const uint64_t keep = ptx::policy_evict_last(), stream = ptx::policy_evict_first();
            SegIter it;
            it.init(p.prefix, p.B, cid, chunk);
            int b, k0, k1;
            bool whole;
            int nseg = 0, g = 0;
            int pending[kStages] = {-1, -1};
            int q_pending = -1;
            while (ok && it.next(b, k0, k1, whole)) {
                if (nseg > 0 && !ptx::mbar_wait(&bar->q_empty, (nseg - 1) & 1, abort_flag)) { fail(); break; }
                ptx::mbar_expect_tx(&bar->q_full, nq_atoms * kH * 128);
                for (int a = 0; a < LA; ++a)
                    ptx::tma_load_2d_hint(sQ + a * kH * 128, &tmQ, &bar->q_full, (int)rank * LA * 64 + a * 64,
                                          b * p.H, keep);
                if (rank == 0) ptx::tma_load_2d_hint(sQ + LA * kH * 128, &tmQR, &bar->q_full, 0, b * p.H, keep);
                q_pending = nseg & 1;
                ++nseg;
                const int ntiles = (k1 - k0 + kBKV - 1) / kBKV;
                for (int t = 0; t < ntiles; ++t, ++g) {
                    const int st = g & 1;
                    if (!ptx::mbar_wait(&bar->kv_empty[st], ((g >> 1) & 1) ^ 1, abort_flag)) { fail(); break; }
                    ptx::mbar_expect_tx(&bar->kv_full[st], nq_atoms * C::kAtomBytes);
                    const int row = b * p.max_seq + k0 + t * kBKV;
                    uint8_t *dst = sKV + st * C::kStageBytes;
                    for (int a = 0; a < LA; ++a)
                        ptx::tma_load_2d_hint(dst + a * C::kAtomBytes, &tmL, &bar->kv_full[st],
                                              (int)rank * LA * 64 + a * 64, row, stream);
                    if (rank == 0)
                        ptx::tma_load_2d_hint(dst + LA * C::kAtomBytes, &tmR, &bar->kv_full[st], 0, row, stream);
                    pending[st] = (g >> 1) & 1;
                }
            }
            volatile int never = 0;
            if (q_pending >= 0) ptx::mbar_wait(&bar->q_full, (uint32_t)q_pending, &never);
            for (int i = 0; i < kStages; ++i)
                if (pending[i] >= 0) ptx::mbar_wait(&bar->kv_full[i], (uint32_t)pending[i], &never);
        }
    } else if (warp == 1) {
        if (ptx::elect_one()) {
            // Non-blocking issue: poll both queues and issue whichever MMA
            // group is ready, P.V first (it frees a KV stage for the next
            // load); a QK^T waiting on its tile never holds back a P.V.
            constexpr uint32_t idesc_s = ptx::idesc_bf16(kH, kBKV, false, false);
            constexpr uint32_t idesc_o = ptx::idesc_bf16(kH, LA * 64, false, true);
            const uint32_t q0 = ptx::smem_u32(sQ), kv0 = ptx::smem_u32(sKV), p0 = ptx::smem_u32(sP);
            TileCursor qk, pv;
            qk.init(p.prefix, p.B, cid, chunk);
            pv.init(p.prefix, p.B, cid, chunk);
            long long last = clock64();
            while (ok && pv.valid) {
                bool progressed = false;
                if (pv.g < qk.g) {
                    bool ready = ptx::mbar_try_wait(ptx::smem_u32(&bar->p_full), pv.g & 1);
                    if (ready && pv.t == 0 && pv.nseg > 0)
                        ready = ptx::mbar_try_wait(ptx::smem_u32(&bar->o_empty), (pv.nseg - 1) & 1);
                    if (ready) {
                        ptx::tc_fence_after();
                        const int st = pv.g & 1;
                        const uint32_t vb = kv0 + st * C::kStageBytes;
#pragma unroll
                        for (int k = 0; k < kBKV / 16; ++k)
                            ptx::mma_bf16(tmem, ptx::sdesc_sw128(p0 + k * 32, 16, 1024),
                                          ptx::sdesc_sw128(vb + k * 2048, C::kAtomBytes, 1024), idesc_o,
                                          (pv.t == 0 && k == 0) ? 0u : 1u);
                        ptx::mma_commit(&bar->kv_empty[st]);
                        ptx::mma_commit(&bar->pv_done);
                        pv.step();
                        progressed = true;
                    }
                }
                if (qk.valid) {
                    const int st = qk.g & 1;
                    bool ready = qk.t > 0 || ptx::mbar_try_wait(ptx::smem_u32(&bar->q_full), qk.nseg & 1);
                    ready = ready && ptx::mbar_try_wait(ptx::smem_u32(&bar->kv_full[st]), (qk.g >> 1) & 1) &&
                            ptx::mbar_try_wait(ptx::smem_u32(&bar->s_empty[st]), ((qk.g >> 1) & 1) ^ 1);
                    if (ready) {
                        ptx::tc_fence_after();
                        const uint32_t kb = kv0 + st * C::kStageBytes;
                        const uint32_t d = tmem + C::kSCol + st * kBKV;
                        for (int a = 0; a < nq_atoms; ++a) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                ptx::mma_bf16(d, ptx::sdesc_sw128(q0 + a * kH * 128 + k * 32, 16, 1024),
                                              ptx::sdesc_sw128(kb + a * C::kAtomBytes + k * 32, 16, 1024),
                                              idesc_s, (a | k) != 0);
                        }
                        ptx::mma_commit(&bar->s_full[st]);
                        if (qk.t == qk.ntiles - 1) ptx::mma_commit(&bar->q_empty);
                        qk.step();
                        progressed = true;
                    }
                }
                if (progressed) last = clock64();
                else if (*abort_flag || clock64() - last > ptx::kWaitCycles) fail();
            }
        }
    } else {
        const int quad = warp % 4;
        const int h = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t peer_x = map_peer(sX + h * kXStride, peer);
        const uint32_t peer_xfull = map_peer(&bar->x_full, peer);
        const uint32_t peer_free = map_peer(&bar->peer_free, peer);
        float *my_x = sX + h * kXStride;
        uint8_t *prow = sP + h * 128;
        SegIter it;
        it.init(p.prefix, p.B, cid, chunk);
        int b, k0, k1;
        bool whole;
        int g = 0, s_cnt = 0, x_cnt = 0, p_cnt = 0;
        while (ok && it.next(b, k0, k1, whole)) {
            float m_run = -INFINITY, l_run = 0.f;
            const int len = k1 - k0;
            const int ntiles = (len + kBKV - 1) / kBKV;
            for (int t = 0; t < ntiles; ++t, ++g) {
                const int valid = min(kBKV, len - t * kBKV);
                const int sb = s_cnt & 1;
                if (!ptx::mbar_wait(&bar->s_full[sb], (s_cnt >> 1) & 1, abort_flag)) { fail(); break; }
                ptx::tc_fence_after();
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(tmem + lane_off + C::kSCol + sb * kBKV, r0);
                ptx::tmem_ld32(tmem + lane_off + C::kSCol + sb * kBKV + 32, r1);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar->s_empty[sb]);
                ++s_cnt;
                float s[64];
#pragma unroll
                for (int j = 0; j < 32; ++j) { s[j] = __uint_as_float(r0[j]); s[32 + j] = __uint_as_float(r1[j]); }
                // Exchange partial scores with the peer CTA.
                if (!ptx::mbar_wait_cluster(&bar->peer_free, (x_cnt & 1) ^ 1, abort_flag)) { fail(); break; }
#pragma unroll
                for (int j = 0; j < 64; j += 4) st_cluster_v4(peer_x + j * 4, s[j], s[j + 1], s[j + 2], s[j + 3]);
                arrive_remote(peer_xfull);
                if (!ptx::mbar_wait_cluster(&bar->x_full, x_cnt & 1, abort_flag)) { fail(); break; }
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(my_x + j);
                    // Same operand order in both CTAs: S_0 + S_1.
                    if (rank == 0) { s[j] += v.x; s[j + 1] += v.y; s[j + 2] += v.z; s[j + 3] += v.w; }
                    else { s[j] = v.x + s[j]; s[j + 1] = v.y + s[j + 1]; s[j + 2] = v.z + s[j + 2]; s[j + 3] = v.w + s[j + 3]; }
                }
                arrive_remote(peer_free);
                ++x_cnt;
                float mt = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s[j] = (j < valid) ? s[j] * p.scale_log2 : -INFINITY;
                    mt = fmaxf(mt, s[j]);
                }
                const bool resc = mt > m_run + kRescaleThreshold;
                const float m_new = resc ? mt : m_run;
                const float corr = exp2f(m_run - m_new);
                float psum = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float a0 = exp2f(s[2 * j] - m_new), a1 = exp2f(s[2 * j + 1] - m_new);
                    psum += a0 + a1;
                    pk[j] = ptx::pack_bf16(a0, a1);
                }
                l_run = l_run * corr + psum;
                m_run = m_new;
                // The previous PV must be done before P is overwritten or O rescaled.
                if (p_cnt > 0 && !ptx::mbar_wait(&bar->pv_done, (p_cnt - 1) & 1, abort_flag)) { fail(); break; }
                if (resc && t > 0) {
                    ptx::tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < C::kOCols; c += 32) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tmem + lane_off + c, o);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
                        ptx::tmem_st32(tmem + lane_off + c, o);
                    }
                    ptx::tmem_st_wait();
                }
                // P row (K-major, 128-byte swizzle: 16-byte chunk j at j ^ (h & 7)).
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4 *>(prow + ((j ^ (h & 7)) << 4)) =
                        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                if (valid < kBKV) {
                    // Rows past the segment may hold arbitrary cache contents;
                    // P is 0 there, but 0 * NaN is not 0: zero those rows.
                    uint8_t *stg = sKV + (g & 1) * C::kStageBytes;
                    const int nrow = kBKV - valid;
                    for (int i = h; i < LA * nrow * 8; i += kH) {
                        const int a = i / (nrow * 8), rr = (i / 8) % nrow, ch = i % 8;
                        *reinterpret_cast<uint4 *>(stg + a * C::kAtomBytes + (valid + rr) * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar->p_full);
                ++p_cnt;
            }
            if (!ok) break;
            // Segment done: read the accumulator once its last PV completed.
            if (!ptx::mbar_wait(&bar->pv_done, (p_cnt - 1) & 1, abort_flag)) { fail(); break; }
            ptx::tc_fence_after();
            const bool row_ok = h < p.H;
            const int slot = cid + b;
#pragma unroll 1
            for (int c = 0; c < C::kOCols; c += 32) {
                uint32_t o[32];
                ptx::tmem_ld32(tmem + lane_off + c, o);
                ptx::tmem_ld_wait();
                if (!row_ok) continue;
                const int col = (int)rank * C::kOCols + c;
                if (whole) {
                    const float inv = 1.f / l_run;
                    bf16 *dst = p.o_lat + ((int64_t)b * p.H + h) * C::kRLat + col;
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 w;
                        w.x = ptx::pack_bf16(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
                        w.y = ptx::pack_bf16(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                        w.z = ptx::pack_bf16(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
                        w.w = ptx::pack_bf16(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + j) = w;
                    }
                } else {
                    float *dst = p.o_part + ((int64_t)slot * p.H + h) * C::kRLat + col;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(dst + j) =
                            make_float4(__uint_as_float(o[j]), __uint_as_float(o[j + 1]),
                                        __uint_as_float(o[j + 2]), __uint_as_float(o[j + 3]));
                }
            }
            if (row_ok && !whole && rank == 0) {
                p.ml_part[((int64_t)slot * p.H + h) * 2] = m_run;
                p.ml_part[((int64_t)slot * p.H + h) * 2 + 1] = l_run;
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->o_empty);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

// Prefix sums of the valid lengths (invalid ones count as 0 and are flagged)
// and the per-cluster key range.
__global__ void __launch_bounds__(1024) decode_schedule_kernel(const int32_t *seq_lens, int B, int max_seq,
                                                               int n_clusters, int *prefix, int *chunk,
                                                               uint32_t *status)
{
    __shared__ int warp_sums[32];
    __shared__ int carry;
    if (threadIdx.x == 0) { carry = 0; prefix[0] = 0; }
    __syncthreads();
    for (int base = 0; base < B; base += 1024) {
        const int i = base + threadIdx.x;
        int L = 0;
        if (i < B) {
            L = seq_lens[i];
            if (L < 1 || L > max_seq) {
                atomicOr(status, kStatusLen);
                L = 0;
            }
        }
        int v = L;
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, off);
            if ((threadIdx.x & 31) >= off) v += n;
        }
        if ((threadIdx.x & 31) == 31) warp_sums[threadIdx.x >> 5] = v;
        __syncthreads();
        if (threadIdx.x < 32) {
            int w = warp_sums[threadIdx.x];
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, w, off);
                if (threadIdx.x >= off) w += n;
            }
            warp_sums[threadIdx.x] = w;
        }
        __syncthreads();
        const int incl = v + ((threadIdx.x >> 5) ? warp_sums[(threadIdx.x >> 5) - 1] : 0) + carry;
        if (i < B) prefix[i + 1] = incl;
        __syncthreads();
        if (threadIdx.x == 1023) carry = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int total = prefix[B];
        *chunk = max(128, (total + n_clusters - 1) / n_clusters);
    }
}

// o_lat[b, h] = sum_s 2^(m_s - m*) O_s / sum_s 2^(m_s - m*) l_s over the
// partial slots of sequence b (sequences handled by one cluster were written
// directly; invalid ones are zeroed).
__global__ void __launch_bounds__(128) decode_combine_tc_kernel(const int *prefix, const int *chunk_ptr, int B,
                                                                int H, int r_lat, const float *o_part,
                                                                const float *ml_part, bf16 *o_lat)
{
    const int h = blockIdx.x, b = blockIdx.y;
    const int lo = prefix[b], hi = prefix[b + 1], chunk = *chunk_ptr;
    bf16 *dst = o_lat + ((int64_t)b * H + h) * r_lat;
    if (hi <= lo) {
        for (int c = threadIdx.x; c < r_lat; c += blockDim.x) dst[c] = __float2bfloat16_rn(0.f);
        return;
    }
    const int fc = lo / chunk, lc = (hi - 1) / chunk;
    if (fc == lc) return;
    float m = -INFINITY;
    for (int c = fc; c <= lc; ++c) m = fmaxf(m, ml_part[((int64_t)(c + b) * H + h) * 2]);
    float den = 0.f;
    for (int c = fc; c <= lc; ++c) {
        const float *ml = ml_part + ((int64_t)(c + b) * H + h) * 2;
        den += exp2f(ml[0] - m) * ml[1];
    }
    const float inv = 1.f / den;
    for (int col = threadIdx.x; col < r_lat; col += blockDim.x) {
        float acc = 0.f;
        for (int c = fc; c <= lc; ++c) {
            const float w = exp2f(ml_part[((int64_t)(c + b) * H + h) * 2] - m);
            acc += w * o_part[((int64_t)(c + b) * H + h) * r_lat + col];
        }
        dst[col] = __float2bfloat16_rn(acc * inv);
    }
}

template <int LA>
cudaError_t launch_decode_tc(const DecodeTcArgs &a, cudaStream_t s)
{
    using C = DCfg<LA>;
    CUtensorMap tq, tqr, tl, tr;
    const int64_t q_rows = (int64_t)a.B * a.H;
    if (!make_tmap_bf16(&tq, a.q_abs, q_rows, 2 * LA * 64, 2 * LA * 64, 64, kH) ||
        !make_tmap_bf16(&tqr, a.q_rope, q_rows, 64, 64, 64, kH) ||
        !make_tmap_bf16(&tl, a.lat, (int64_t)a.max_batch * a.max_seq, 2 * LA * 64, a.lat_stride, 64, kBKV) ||
        !make_tmap_bf16(&tr, a.rope, (int64_t)a.max_batch * a.max_seq, 64, a.rope_stride, 64, kBKV))
        return cudaErrorInvalidValue;
    decode_schedule_kernel<<<1, 1024, 0, s>>>(a.seq_lens, a.B, a.max_seq, a.n_clusters, a.prefix, a.chunk,
                                              a.status);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_tc_kernel<LA>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    DecTcParams p;
    p.B = a.B; p.H = a.H; p.max_seq = a.max_seq;
    p.prefix = a.prefix; p.chunk = a.chunk;
    p.scale_log2 = a.scale_log2;
    p.o_lat = (bf16 *)a.o_lat;
    p.o_part = a.o_part;
    p.ml_part = a.ml_part;
    p.status = a.status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * a.n_clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    profile_begin(MLA_PROFILE_DECODE_ATTENTION, s);
    e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<LA>, tq, tqr, tl, tr, p);
    profile_end(MLA_PROFILE_DECODE_ATTENTION, s);
    note_launch();
    if (e != cudaSuccess) return e;
    decode_combine_tc_kernel<<<dim3(a.H, a.B), 128, 0, s>>>(a.prefix, a.chunk, a.B, a.H, 2 * LA * 64, a.o_part,
                                                            a.ml_part, (bf16 *)a.o_lat);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

int decode_tc_max_clusters()
{
    static int cached = -1;
    if (cached >= 0) return cached;
    using C = DCfg<4>;
    if (cudaFuncSetAttribute(decode_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
        cudaSuccess)
        return cached = 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<4>, &cfg) != cudaSuccess) n = 0;
    return cached = n;
}

bool decode_tc_supported(int H, int r_kv, int d_rope) { return H >= 1 && H <= kH && r_kv == 512 && d_rope == 64; }

cudaError_t decode_tc(const DecodeTcArgs &a, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    if (!decode_tc_supported(a.H, a.r_kv, a.d_rope) || a.n_clusters < 1) return cudaErrorInvalidValue;
    return launch_decode_tc<4>(a, s);
}

}  // namespace mla

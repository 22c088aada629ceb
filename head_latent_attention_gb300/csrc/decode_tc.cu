// Weight-absorbed split-KV latent attention for decode on tcgen05, one
// 2-CTA cluster per work range.
//
// Per sequence b the 128 heads attend over the latent cache rows c_j (r_kv =
// 512) and rope keys k_R,j (d_rope = 64): s_hj = q_abs,h . c_j + q_R,h . k_R,j,
// softmax over j, o_lat,h = sum_j p_hj c_j.  The fp32 accumulator o_lat for
// 128 heads x 512 latent columns is exactly one SM's tensor memory, so a
// cluster of two CTAs splits the columns: CTA r owns latent columns
// [256 r, 256 r + 256) and rope columns [32 r, 32 r + 32).  Each CTA
//   - keeps O (256 columns), its 288 query columns (the A operand of Q K^T)
//     and two 48-column score buffers in tensor memory;
//   - streams 48-key tiles of its own cache columns through a 6-stage ring
//     (TMA; 128-byte swizzle for the latent, 64-byte for rope);
//   - computes a partial score tile S_r = Q_r K_r^T (M = 128 heads, N = 48
//     keys, K = 288);
//   - scales S_r to log2 units, rounds it to fp16 and sends it to the peer
//     two tiles ahead of the softmax, one bulk copy per warp (distributed
//     shared memory moves ~12 bytes per clock per SM, so the exchange is
//     the scarce resource); both CTAs add the same two rounded partials and
//     so take bit-identical softmax decisions;
//   - writes P (bfloat16) to shared memory (K-major, no swizzle) and
//     accumulates O_r += P V_r (M = 128, N = 256, K = 48), V read as an
//     MN-major operand from the same shared-memory tile.
// Warp roles: warp 0 TMA producer (the first loads go out before the setup
// syncs), warp 1 MMA issuer (non-blocking polling of both queues), warps
// 2..9 softmax in two groups that take alternate tiles (two tiles in
// flight), one head row per thread.  The running reference max is raised
// only when a tile exceeds it by more than 8 (log2 units), so O is rarely
// rescaled; the groups hand it to each other tile by tile.  The result is
// exact either way because P and the row sums use the same reference.
//
// Work: the concatenation of all sequences' keys is cut into one contiguous
// range per cluster by a device-side scheduler that runs before the kernel
// preceding this one (ranges balanced by estimated time, a sequence start
// costing a few hundred keys); a range splits into one segment per sequence
// it touches.  A segment that covers a whole sequence writes o_lat
// directly; others write their normalised latent average (bf16) with its
// (m, l), merged later.  Warp roles: a Q K^T runs at most three tiles ahead
// of the next P.V, since the tensor pipe executes in order.
#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr int kH = 128;       // heads per CTA = MMA M
constexpr int kBKV = 48;      // keys per tile
constexpr int kStages = 6;    // KV ring
constexpr int kSBuf = 2;      // score buffers in tensor memory
constexpr int kSoftmaxThreads = 256;  // warps 2..9
constexpr int kThreads = 64 + kSoftmaxThreads;
constexpr float kRescaleThreshold = 8.f;
// Q K^T(g + 2) is read two tiles ahead by the group that owns tile g, and
// Q K^T(g + 3) by the other group at about the same time, so it may run
// three tiles ahead of P.V(g).
constexpr int kQKAhead = 3;
constexpr int kLA = 4;        // 64-column latent atoms per CTA (r_kv = 512)

// Shared memory (per CTA): the KV ring, the latent query, two exchange buffers.
constexpr int kAtom = kBKV * 128;                     // one 48x64 latent atom of a KV tile
constexpr int kStageBytes = kLA * kAtom + kBKV * 64;  // + 32 rope columns (64-byte rows)
constexpr int kXBuf = 2;                              // exchange buffers (partials travel two tiles ahead)
// Exchange buffer (fp16 scores): [head][48 keys], so each softmax warp's 32
// head rows are one contiguous block that the warp copies to the peer itself.
constexpr int kXRowBytes = kBKV * 2;
constexpr int kXWarpBytes = 32 * kXRowBytes;
constexpr int kXBytes = kH * kXRowBytes;
constexpr uint32_t kXTx = kXBytes;                    // one exchange = one bulk copy of a whole buffer
// Position of 16-byte chunk c within row `lane` of an exchange block.  Rows
// are 96 bytes (six chunks) apart, so eight consecutive rows would cover only
// four of the eight 16-byte bank groups; rotating the chunks of rows with
// lane % 8 >= 4 by one spreads every eight lanes over all eight.
__device__ __forceinline__ int xpos(int c, int lane)
{
    const int p = c + ((lane >> 2) & 1);
    return p >= kBKV / 8 ? p - kBKV / 8 : p;
}
constexpr int kOffX = kStages * kStageBytes;
// P (bf16, 128 heads x 48 keys) as the A operand of P.V: K-major without
// swizzle, 8-row x 16-byte core matrices, the six core matrices of an 8-row
// group adjacent (128 bytes apart), 8-row groups 768 bytes apart.
constexpr int kPBytes = kH * kBKV * 2;
constexpr int kPGroup = (kBKV / 8) * 128;
// A softmax group's P buffer also stages its outgoing partial: each warp's
// 32 rows occupy the same 3 KB in both layouts.
constexpr int kOffP = kOffX + kXBuf * kXBytes;
static_assert(kXWarpBytes == 4 * kPGroup, "a warp's staging block is its P rows");
constexpr int kOffRed = kOffP + 2 * kPBytes;          // reference maxima, segment-end (max, sum)
constexpr int kOffBar = kOffRed + 6 * kH * 4;
// The cluster's view of the schedule: its range [start, end) of the
// concatenated keys and the prefix sums of the sequences from the range's
// first one on (kWin + 1 entries; later ones are read from global memory).
constexpr int kWin = 63;
struct SchedWin {
    int start, end, b0, nwin;
    int pf[kWin + 1];
};
constexpr int kOffSched = kOffBar + 512;
constexpr int kSmem = kOffSched + (int)sizeof(SchedWin) + 1024;
static_assert(kOffP % 16 == 0, "P operand alignment");
static_assert(kSmem <= 232448, "shared memory per CTA");
// Tensor memory: O in [0, 256), the query (256 latent + 32 rope bf16 = 144
// columns) in [256, 400), two 48-column score buffers in [400, 496).
constexpr int kOCols = kLA * 64;
constexpr int kQCol = 256;
constexpr int kQRCol = kQCol + kOCols / 2;
constexpr int kSCol = kQRCol + 16;
static_assert(kSCol + kSBuf * kBKV <= 512, "tensor memory columns");
constexpr int kRLat = 2 * kLA * 64;
static_assert(kQRCol + 16 <= 512, "tensor memory columns");

struct DecTcParams {
    int B, H, max_seq;
    DecodeSched sc;     // prefix sums, range starts, first sequence of each range
    float scale_log2;
    bf16 *o_lat;        // [B, H, r_kv]
    bf16 *o_part;       // [slots, H, r_kv]
    float *ml_part;     // [slots, H, 2]
    uint32_t *status;
};

struct Bars {
    uint64_t q_full, q_empty;  // query written to tensor memory by the softmax warps; consumed
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[kSBuf], s_free[kSBuf];
    uint64_t p_full[2], pv_done[2];
    uint64_t o_empty;
    uint64_t x_full[kXBuf], x_free[kXBuf];
    // Softmax groups: reference-max handoff from group i, per lane quarter
    // (one arrival per thread of the producing warp), and the segment-end
    // meeting of the two warps of a lane quarter.
    uint64_t hand[2][4], seg[4];
    int abort;
    uint32_t tmem;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

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
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Shared-memory matrix descriptor without swizzle: 8-row x 16-byte core
// matrices, `lbo` bytes between core matrices along K, `sbo` bytes between
// 8-row groups.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version; layout type 0 = no swizzle
    return d;
}

// Bulk copy of `bytes` from this CTA's shared memory into the peer's, completing
// the bytes on the peer's mbarrier (both peer addresses already mapped).
__device__ __forceinline__ void bulk_to_peer(uint32_t peer_dst, const void *src, uint32_t bytes, uint32_t peer_bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t"
        "cp.async.bulk.commit_group;" ::"r"(peer_dst),
        "r"(ptx::smem_u32(src)), "r"(bytes), "r"(peer_bar)
        : "memory");
}
// The bulk copies this thread issued have finished reading their source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Arrive on the peer's mbarrier without ordering earlier memory operations
// (a release at cluster scope waits for this thread's outstanding remote
// stores, which costs thousands of cycles); callers order what they must
// with a barrier first.
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t remote_bar)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
// Two fp32 values to fp16 (round to nearest even, saturating at the largest
// finite value), the lower one in the low half.
__device__ __forceinline__ uint32_t pack_f16_sat(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float2 unpack_f16(uint32_t w)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

// Maximum and sum of a tile row as balanced trees (short dependency chains).
template <int N>
__device__ __forceinline__ float tree_max(const float (&v)[N])
{
    float t[N / 2];
#pragma unroll
    for (int j = 0; j < N / 2; ++j) t[j] = fmaxf(v[2 * j], v[2 * j + 1]);
#pragma unroll
    for (int w = N / 4; w >= 3; w /= 2)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
    return fmaxf(fmaxf(t[0], t[1]), t[2]);
}

// Segments of this cluster's key range [start, end) of the concatenated keys.
struct SegIter {
    const SchedWin *w;
    const int *prefix;
    int B, start, end, b;
    __device__ int pf(int i) const { return i - w->b0 <= w->nwin ? w->pf[i - w->b0] : prefix[i]; }
    __device__ void init(const SchedWin *win, const int *pfx, int nb)
    {
        w = win;
        prefix = pfx;
        B = nb;
        start = win->start;
        end = win->end;
        b = win->b0;
    }
    // Next non-empty segment: sequence b, keys [k0, k1), whole-sequence flag.
    __device__ bool next(int &sb, int &k0, int &k1, bool &whole)
    {
        while (b < B && pf(b) < end) {
            const int lo = pf(b), hi = pf(b + 1);
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

// The range of cluster cid and the prefix window from its first sequence,
// written by one warp (two rounds of independent loads) and read by every
// cursor of the CTA after a barrier.
__device__ void sched_window(SchedWin *w, const DecodeSched &sc, int nb, int cid, int lane)
{
    const int *pf = sc.prefix;
    const int start = sc.range_start[cid], end = sc.range_start[cid + 1], first = sc.range_b0[cid];
    const int b0 = (start < end) ? first : nb;
    const int nwin = min(kWin, nb - b0);
    for (int i = lane; i <= nwin; i += 32) w->pf[i] = pf[b0 + i];
    if (lane == 0) {
        w->start = start;
        w->end = end;
        w->b0 = b0;
        w->nwin = nwin;
    }
    __syncwarp();
}

// Walks the tiles of this cluster's segments in order (g: global tile
// index, t: tile within segment nseg).
struct TileCursor {
    SegIter it;
    int b, k0, k1, nseg, t, ntiles, g;
    bool whole, valid;
    __device__ void init(const SchedWin *win, const int *pf, int nb)
    {
        it.init(win, pf, nb);
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

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmR,
                     const bf16 *__restrict__ q_abs, const bf16 *__restrict__ q_rope, DecTcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sKV = smem;
    Bars *bar = (Bars *)(smem + kOffBar);
    SchedWin *win = (SchedWin *)(smem + kOffSched);
    volatile int *abort_flag = &bar->abort;

    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int cid = (int)cluster_id();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // KV loads are issued by thread 0: the first kStages right after the
    // barriers exist (before the CTA and cluster syncs, and before the wait
    // for the previous kernel, so the first HBM round trip overlaps both),
    // the rest from the producer loop.  The schedule and the cache rows are
    // complete when this kernel starts: the scheduler runs before the
    // kernel that precedes this one and does not let it start early, and it
    // waits for every earlier kernel itself.  Only the queries come from the
    // previous kernel.
    TileCursor ld;
    int pending[kStages];
    uint64_t evict_first = 0;
    auto issue_load = [&]() -> bool {
        const int st = ld.g % kStages;
        const uint32_t ph = (uint32_t)(ld.g / kStages) & 1;
        if (!ptx::mbar_wait(&bar->kv_empty[st], ph ^ 1, abort_flag)) return false;
        ptx::mbar_expect_tx(&bar->kv_full[st], kStageBytes);
        const int row = ld.b * p.max_seq + ld.k0 + ld.t * kBKV;
        uint8_t *dst = sKV + st * kStageBytes;
        for (int a = 0; a < kLA; ++a)
            ptx::tma_load_2d_hint(dst + a * kAtom, &tmL, &bar->kv_full[st], (int)rank * kLA * 64 + a * 64, row,
                                  evict_first);
        ptx::tma_load_2d_hint(dst + kLA * kAtom, &tmR, &bar->kv_full[st], (int)rank * 32, row, evict_first);
        pending[st] = (int)ph;
        ld.step();
        return true;
    };

    if (threadIdx.x == 0) {
        ptx::pdl_trigger();
        ptx::mbar_init(&bar->q_full, kSoftmaxThreads / 2);  // the group that sends a segment's first tile
        ptx::mbar_init(&bar->q_empty, 1);
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&bar->kv_full[i], 1);
            ptx::mbar_init(&bar->kv_empty[i], 1);
        }
        for (int i = 0; i < kSBuf; ++i) {
            ptx::mbar_init(&bar->s_full[i], 1);
            ptx::mbar_init(&bar->s_free[i], kSoftmaxThreads / 2);  // one softmax group per buffer
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&bar->p_full[i], kSoftmaxThreads / 2);
            ptx::mbar_init(&bar->pv_done[i], 1);
        }
        for (int i = 0; i < kXBuf; ++i) {
            ptx::mbar_init(&bar->x_full[i], 1);
            ptx::mbar_init(&bar->x_free[i], kSoftmaxThreads / 64);  // one arrival per warp of a peer group
        }
        ptx::mbar_init(&bar->o_empty, kSoftmaxThreads);
        for (int q = 0; q < 4; ++q) {
            ptx::mbar_init(&bar->hand[0][q], 32);
            ptx::mbar_init(&bar->hand[1][q], 32);
            ptx::mbar_init(&bar->seg[q], 64);
        }
        bar->abort = 0;
        ptx::fence_mbar_init();
        for (int i = 0; i < kXBuf; ++i) ptx::mbar_expect_tx(&bar->x_full[i], kXTx);  // arm every buffer
        ptx::prefetch_tmap(&tmL);
        ptx::prefetch_tmap(&tmR);
    }
    if (warp == 0) sched_window(win, p.sc, p.B, cid, lane);
    if (threadIdx.x == 0) {
        evict_first = ptx::policy_evict_first();
#pragma unroll
        for (int i = 0; i < kStages; ++i) pending[i] = -1;
        ld.init(win, p.sc.prefix, p.B);
        for (int i = 0; i < kStages && ld.valid; ++i) issue_load();  // fresh ring: no waits
        ptx::pdl_wait();
    }
    if (warp == 1) ptx::tmem_alloc(&bar->tmem, 512);
    ptx::tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before any remote arrive or store
    ptx::tc_fence_after();
    ptx::pdl_wait();
    const uint32_t tmem = bar->tmem;
    bool ok = true;
    auto fail = [&]() {
        ok = false;
        *abort_flag = 1;
        st_cluster_u32(map_peer((const void *)abort_flag, peer), 1u);
    };

    if (warp == 0) {
        if (threadIdx.x == 0) {
            while (ok && ld.valid)
                if (!issue_load()) { fail(); break; }
            // Copies still in flight land before the CTA may exit.
            volatile int never = 0;
            for (int i = 0; i < kStages; ++i)
                if (pending[i] >= 0) ptx::mbar_wait(&bar->kv_full[i], (uint32_t)pending[i], &never);
        }
    } else if (warp == 1) {
        if (ptx::elect_one()) {
            // Non-blocking issue (test_wait, never try_wait, which may suspend
            // the thread): poll both queues and issue whichever MMA group is
            // ready, P.V first (it frees a KV stage for the next load).
            constexpr uint32_t idesc_s = ptx::idesc_bf16(kH, kBKV, false, false);
            constexpr uint32_t idesc_o = ptx::idesc_bf16(kH, kLA * 64, false, true);
            const uint32_t kv0 = ptx::smem_u32(sKV), p0 = ptx::smem_u32(smem + kOffP);
            TileCursor qk, pv;
            qk.init(win, p.sc.prefix, p.B);
            pv.init(win, p.sc.prefix, p.B);
            long long last = clock64();
            while (ok && pv.valid) {
                bool progressed = false;
                if (pv.g < qk.g) {
                    bool ready = ptx::mbar_test(ptx::smem_u32(&bar->p_full[pv.g & 1]), (pv.g >> 1) & 1);
                    if (ready && pv.t == 0 && pv.nseg > 0)
                        ready = ptx::mbar_test(ptx::smem_u32(&bar->o_empty), (pv.nseg - 1) & 1);
                    if (ready) {
                        ptx::tc_fence_after();
                        const int st = pv.g % kStages;
                        const uint32_t vb = kv0 + st * kStageBytes;
                        const uint32_t pa = p0 + (pv.g & 1) * kPBytes;
#pragma unroll
                        for (int k = 0; k < kBKV / 16; ++k)
                            ptx::mma_bf16(tmem, sdesc_plain(pa + k * 256, 128, kPGroup),
                                          ptx::sdesc_sw128(vb + k * 2048, kAtom, 1024), idesc_o,
                                          (pv.t == 0 && k == 0) ? 0u : 1u);
                        ptx::mma_commit(&bar->kv_empty[st]);
                        ptx::mma_commit(&bar->pv_done[pv.g & 1]);
                        pv.step();
                        progressed = true;
                    }
                }
                // Q K^T runs at most kQKAhead tiles ahead of the next P.V: the
                // tensor pipe executes in issue order, and a Q K^T queued
                // early would delay the P.V that frees a KV stage.
                if (qk.valid && qk.g <= pv.g + kQKAhead) {
                    const int st = qk.g % kStages, sb = qk.g % kSBuf;
                    bool ready = qk.t > 0 || ptx::mbar_test(ptx::smem_u32(&bar->q_full), qk.nseg & 1);
                    ready = ready && ptx::mbar_test(ptx::smem_u32(&bar->kv_full[st]), (qk.g / kStages) & 1);
                    // Score buffer sb held tile g - 2: the softmax must have read it.
                    ready = ready && (qk.g < kSBuf ||
                                      ptx::mbar_test(ptx::smem_u32(&bar->s_free[sb]), ((qk.g / kSBuf) - 1) & 1));
                    if (ready) {
                        ptx::tc_fence_after();
                        const uint32_t kb = kv0 + st * kStageBytes;
                        const uint32_t d = tmem + kSCol + sb * kBKV;
                        // K steps 0..15: latent (keys in 128-byte swizzled
                        // atoms); 16..17: rope (keys 64-byte swizzled); the
                        // query is read from tensor memory.  (One straight-line
                        // burst: a runtime-indexed issue loop slows the MMAs.)
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            ptx::mma_f16_tmem_a(d, tmem + kQCol + k * 8,
                                                ptx::sdesc_sw128(kb + (k >> 2) * kAtom + (k & 3) * 32, 16, 1024),
                                                idesc_s, k != 0);
#pragma unroll
                        for (int k = 0; k < 2; ++k)
                            ptx::mma_f16_tmem_a(d, tmem + kQRCol + k * 8,
                                                ptx::sdesc_sw64(kb + kLA * kAtom + k * 32, 512), idesc_s, 1u);
                        ptx::mma_commit(&bar->s_full[sb]);
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
        // Softmax warps 2..9: warp w serves the tensor-memory lane quarter
        // w % 4 (head rows 32 (w % 4) + lane); warps 2..5 take the even tiles
        // and warps 6..9 the odd ones, each thread the whole row of its tile,
        // so two tiles are in flight.  The running reference max passes
        // from one group to the other tile by tile through shared memory,
        // ordered by a producer/consumer mbarrier per lane quarter.
        const int quad = warp % 4, grp = (warp - 2) / 4;
        const int h = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float *mslot = reinterpret_cast<float *>(smem + kOffRed);  // [2][kH] reference max after tile g (slot g & 1)
        uint32_t hand_in = 0, nseg_done = 0;                       // handoffs received, segments finished
        float *eslot = mslot + 2 * kH;                             // [2 groups][2][kH] (max, sum) at a segment end
        const int xblk = quad * kXWarpBytes;                       // this warp's block of an exchange buffer
        uint8_t *wstage = smem + kOffP + grp * kPBytes + xblk;
        uint32_t *my_stage = reinterpret_cast<uint32_t *>(wstage + lane * kXRowBytes);
        const uint32_t peer_xbuf = map_peer(smem + kOffX + grp * kXBytes + xblk, peer);
        const uint32_t peer_xfull = map_peer(&bar->x_full[grp], peer);
        const uint32_t peer_xfree = map_peer(&bar->x_free[grp], peer);
        // This CTA's 288 query columns of row h into tensor memory (lanes =
        // heads, bf16 pairs per 32-bit column, lower column in the low half,
        // which is how consecutive bf16 values sit in memory), written by the
        // group that sends the segment's first tile (part 0).  The first
        // segment's query is split between the groups, both idle at the
        // start: group 0 writes latent columns [0, 128) and the rope columns
        // (part 1), group 1 latent columns [128, 256) (part 2); they meet at a
        // named barrier before group 0 arrives on q_full for both.
        auto load_q = [&](int b, int nseg, int part) -> bool {
            if (nseg > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->q_empty, (nseg - 1) & 1, abort_flag)))
                return false;
            ptx::tc_fence_after();
            const bool row_ok = h < p.H;
            // q_abs is stored head-interleaved: 16-byte chunk c of row (b, h) at
            // ((b * kQChunks + c) * kQRows + h) * 16 bytes, so that a warp's
            // load of one chunk for its 32 heads is 512 contiguous bytes.
            const uint4 *src = reinterpret_cast<const uint4 *>(q_abs) + ((int64_t)b * kQChunks + rank * 32) * kQRows + h;
            const uint4 *rs = reinterpret_cast<const uint4 *>(q_rope + ((int64_t)b * p.H + h) * 64 + rank * 32);
            // Two 128-byte groups of the row in flight at a time.
            uint4 va[8], vb[8], vr[4];
            auto fetch = [&](uint4 (&v)[8], int c) {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = row_ok ? src[(int64_t)(c * 8 + i) * kQRows] : make_uint4(0, 0, 0, 0);
            };
            auto put = [&](const uint4 (&v)[8], int c) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w[4 * i] = v[i].x; w[4 * i + 1] = v[i].y; w[4 * i + 2] = v[i].z; w[4 * i + 3] = v[i].w;
                }
                ptx::tmem_st32(tmem + lane_off + kQCol + c * 32, w);
            };
            if (part != 2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) vr[i] = row_ok ? rs[i] : make_uint4(0, 0, 0, 0);
            }
            if (part == 0) {
                fetch(va, 0);
                fetch(vb, 1);
                put(va, 0);
                fetch(va, 2);
                put(vb, 1);
                fetch(vb, 3);
                put(va, 2);
                put(vb, 3);
            } else {
                const int c0 = part == 1 ? 0 : 2;
                fetch(va, c0);
                fetch(vb, c0 + 1);
                put(va, c0);
                put(vb, c0 + 1);
            }
            if (part != 2) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[4 * i] = vr[i].x; w[4 * i + 1] = vr[i].y; w[4 * i + 2] = vr[i].z; w[4 * i + 3] = vr[i].w;
                }
                ptx::tmem_st16(tmem + lane_off + kQRCol, w);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            if (part != 0) asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
            if (part != 2) ptx::mbar_arrive(&bar->q_full);
            return true;
        };
        // Row h of the partial scores of this group's tiles, scaled to log2
        // units and rounded to fp16: the current tile's and the one sent ahead.
        uint32_t own[kBKV / 2], own_next[kBKV / 2];
        // Read the partial of tile g into own_next, free its score buffer,
        // stage it and copy the warp's block into the peer's buffer grp.
        auto send = [&](int g) -> bool {
            const int sb = g % kSBuf;
            // (Warp-uniform outcome: the tensor-memory load below is warp-wide.)
            bool w = ptx::mbar_wait(&bar->s_full[sb], (g / kSBuf) & 1, abort_flag);
            w = w && ptx::mbar_wait_cluster(&bar->x_free[grp], ((g >> 1) & 1) ^ 1, abort_flag);
            if (!__all_sync(0xffffffffu, w)) return false;
            ptx::tc_fence_after();
            uint32_t r0[32], r1[16];
            ptx::tmem_ld32(tmem + lane_off + kSCol + sb * kBKV, r0);
            ptx::tmem_ld16(tmem + lane_off + kSCol + sb * kBKV + 32, r1);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->s_free[sb]);  // score buffer sb may take tile g + 2
#pragma unroll
            for (int j = 0; j < 16; ++j)
                own_next[j] = pack_f16_sat(__uint_as_float(r0[2 * j]) * p.scale_log2,
                                           __uint_as_float(r0[2 * j + 1]) * p.scale_log2);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                own_next[16 + j] = pack_f16_sat(__uint_as_float(r1[2 * j]) * p.scale_log2,
                                                __uint_as_float(r1[2 * j + 1]) * p.scale_log2);
            // Stage the row once the warp's previous copy has read its block,
            // then one lane copies the warp's block to the peer.
            if (lane == 0) bulk_wait_read();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < kBKV / 8; ++c)
                *reinterpret_cast<uint4 *>(my_stage + 4 * xpos(c, lane)) =
                    make_uint4(own_next[4 * c], own_next[4 * c + 1], own_next[4 * c + 2], own_next[4 * c + 3]);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) bulk_to_peer(peer_xbuf, wstage, kXWarpBytes, peer_xfull);
            return true;
        };
        TileCursor nx;  // the next tile of this group to send (sends run two tiles ahead)
        nx.init(win, p.sc.prefix, p.B);
        // Both groups take this branch or neither (the range is the CTA's),
        // and nothing in it can fail before the named barrier.
        if (nx.valid) load_q(nx.b, 0, grp + 1);
        if (grp == 1 && nx.valid) nx.step();
        if (ok && nx.valid) {
            if ((nx.t == 0 && nx.nseg > 0 && !load_q(nx.b, nx.nseg, 0)) || !send(nx.g)) fail();
#pragma unroll
            for (int j = 0; j < kBKV / 2; ++j) own[j] = own_next[j];
            nx.step();
            if (nx.valid) nx.step();
        }
        SegIter it;
        it.init(win, p.sc.prefix, p.B);
        int b, k0, k1;
        bool whole;
        int g = 0;
        while (ok && it.next(b, k0, k1, whole)) {
            // The reference max this group last used and its share of the
            // row sum (relative to that max).
            float m_grp = -INFINITY, l_grp = 0.f;
            const int len = k1 - k0;
            const int ntiles = (len + kBKV - 1) / kBKV;
            for (int t = 0; t < ntiles; ++t, ++g) {
                if ((g & 1) != grp) continue;
                const int valid = min(kBKV, len - t * kBKV);
                // 1. Scores of tile g: the two fp16-rounded partials, added
                //    identically in both CTAs.
                if (!ptx::mbar_wait_cluster(&bar->x_full[grp], (g >> 1) & 1, abort_flag)) { fail(); break; }
                float s[kBKV];
                float mt = -INFINITY;
                {
                    const uint32_t *xr =
                        reinterpret_cast<const uint32_t *>(smem + kOffX + grp * kXBytes + xblk + lane * kXRowBytes);
#pragma unroll
                    for (int c = 0; c < kBKV / 8; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(xr + 4 * xpos(c, lane));
                        const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 a = unpack_f16(own[4 * c + i]), bb = unpack_f16(pw[i]);
                            s[8 * c + 2 * i] = a.x + bb.x;
                            s[8 * c + 2 * i + 1] = a.y + bb.y;
                        }
                    }
                    if (valid < kBKV) {
#pragma unroll
                        for (int j = 0; j < kBKV; ++j) s[j] = (j < valid) ? s[j] : -INFINITY;
                    }
                    mt = tree_max<kBKV>(s);
                }
                // The warp's block of exchange buffer grp is read: the peer may
                // overwrite it once the group's four warps said so (the
                // group's first warp re-arms the buffer's barrier first).
                __syncwarp();
                if (lane == 0) {
                    if (h == 0) ptx::mbar_expect_tx(&bar->x_full[grp], kXTx);
                    arrive_remote_relaxed(peer_xfree);
                }
                // 2. Reference max after tile g: the previous tile's (from the
                //    other group) raised only when this tile exceeds it by
                //    more than the threshold.
                float m_prev = -INFINITY;
                if (t > 0) {
                    if (!ptx::mbar_wait(&bar->hand[grp ^ 1][quad], hand_in & 1, abort_flag)) { fail(); break; }
                    ++hand_in;
                    m_prev = mslot[((g - 1) & 1) * kH + h];
                }
                const float m_new = (mt > m_prev + kRescaleThreshold) ? mt : m_prev;
                mslot[(g & 1) * kH + h] = m_new;
                if (t + 1 < ntiles) ptx::mbar_arrive(&bar->hand[grp][quad]);
                // 3. The group's next tile: its query (at a segment boundary)
                //    and its partial, staged in P buffer grp once P.V(g - 2)
                //    has read P(g - 2) from it.  Each pv_done barrier is
                //    waited on phase by phase, never two phases behind
                //    (P.V(g) cannot finish before P(g) exists).
                if (g >= 2 && !ptx::mbar_wait(&bar->pv_done[grp], ((g >> 1) - 1) & 1, abort_flag)) { fail(); break; }
                if (nx.valid) {
                    if (nx.t == 0 && !load_q(nx.b, nx.nseg, 0)) { fail(); break; }
                    if (!send(nx.g)) { fail(); break; }
                    nx.step();
                    if (nx.valid) nx.step();
                }
                // 4. P = 2^(s - m_new) (bf16) and the group's row sum.
                uint32_t pk[kBKV / 2];
                float psum;
                {
                    float ps[kBKV / 2];
#pragma unroll
                    for (int j = 0; j < kBKV / 2; ++j) {
                        const float a0 = ptx::ex2(s[2 * j] - m_new), a1 = ptx::ex2(s[2 * j + 1] - m_new);
                        ps[j] = a0 + a1;
                        pk[j] = ptx::pack_bf16(a0, a1);
                    }
#pragma unroll
                    for (int w = kBKV / 4; w >= 3; w /= 2)
#pragma unroll
                        for (int j = 0; j < w; ++j) ps[j] += ps[j + w];
                    psum = (ps[0] + ps[1]) + ps[2];
                }
                l_grp = l_grp * ptx::ex2(m_grp - m_new) + psum;
                m_grp = m_new;
#pragma unroll
                for (int j = 0; j < kBKV / 2; ++j) own[j] = own_next[j];
                // Raised: O must hold every earlier P.V before it is rescaled
                // to the new reference.  The tensor-memory loads and stores
                // are warp-wide, so a warp rescales when any of its rows was
                // raised (the others multiply by 1).
                const bool raised = t > 0 && m_new != m_prev;
                if (__any_sync(0xffffffffu, raised)) {
                    const bool w = ptx::mbar_wait(&bar->pv_done[grp ^ 1], ((g - 1) >> 1) & 1, abort_flag);
                    if (!__all_sync(0xffffffffu, w)) { fail(); break; }
                    ptx::tc_fence_after();
                    const float corr = raised ? exp2f(m_prev - m_new) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < kOCols; c += 32) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tmem + lane_off + c, o);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
                        ptx::tmem_st32(tmem + lane_off + c, o);
                    }
                    ptx::tmem_st_wait();
                }
                // P over the staged partial once the warp's copy has read it.
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                {
                    uint8_t *prow = smem + kOffP + grp * kPBytes + (h >> 3) * kPGroup + (h & 7) * 16;
#pragma unroll
                    for (int c = 0; c < kBKV / 8; ++c)
                        *reinterpret_cast<uint4 *>(prow + c * 128) =
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                }
                if (valid < kBKV) {
                    // Rows past the segment may hold arbitrary cache contents;
                    // P is 0 there, but 0 * NaN is not 0: zero those rows.
                    uint8_t *stg = sKV + (g % kStages) * kStageBytes;
                    const int nrow = kBKV - valid;
                    for (int i = h; i < kLA * nrow * 8; i += kH) {
                        const int a = i / (nrow * 8), rr = (i / 8) % nrow, ch = i % 8;
                        *reinterpret_cast<uint4 *>(stg + a * kAtom + (valid + rr) * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                ptx::fence_proxy_async_smem();  // P and zeroed rows visible to the tensor core
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar->p_full[grp]);
            }
            if (!ok) break;
            // Segment done: the two groups' (max, sum) give the row sum
            // relative to the final reference max; then each group stores
            // half of the accumulator's columns once its last P.V completed.
            eslot[(grp * 2) * kH + h] = m_grp;
            eslot[(grp * 2 + 1) * kH + h] = l_grp;
            ptx::mbar_arrive(&bar->seg[quad]);
            if (!ptx::mbar_wait(&bar->seg[quad], nseg_done & 1, abort_flag)) { fail(); break; }
            ++nseg_done;
            const float m_o = eslot[((grp ^ 1) * 2) * kH + h], l_o = eslot[((grp ^ 1) * 2 + 1) * kH + h];
            const float m_fin = fmaxf(m_grp, m_o);
            const float l_tot = l_grp * exp2f(m_grp - m_fin) + (m_o == -INFINITY ? 0.f : l_o * exp2f(m_o - m_fin));
            const int gl = g - 1;  // last tile of the segment
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bar->pv_done[gl & 1], (gl >> 1) & 1, abort_flag))) { fail(); break; }
            ptx::tc_fence_after();
            const int slot = cid + b;
            // The normalised latent average in bfloat16, to o_lat for a whole
            // sequence or to the range's partial slot.  Each warp stages 32
            // rows x 64 bytes at a time in its own block of its group's P
            // buffer (free: every P.V of the segment has completed, and the
            // warp's last copy to the peer has read it), so the global stores
            // go out as 64-byte row pieces; the 16-byte pieces of a row are
            // rotated by (row / 2) % 4 against bank conflicts.  Two 32-column
            // chunks are read from tensor memory per wait.
            uint8_t *wst = smem + kOffP + grp * kPBytes + xblk;
            if (lane == 0) bulk_wait_read();
            __syncwarp();
            const int rd_row = lane >> 2, rd_piece = lane & 3;
            bf16 *dst_base = whole ? p.o_lat + (int64_t)b * p.H * kRLat : p.o_part + (int64_t)slot * p.H * kRLat;
            const float inv = 1.f / l_tot;
#pragma unroll 1
            for (int c2 = grp * (kOCols / 2); c2 < (grp + 1) * (kOCols / 2); c2 += 64) {
                uint32_t o[2][32];
                ptx::tmem_ld32(tmem + lane_off + c2, o[0]);
                ptx::tmem_ld32(tmem + lane_off + c2 + 32, o[1]);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c = c2 + 32 * half;
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        w[j] = ptx::pack_bf16(__uint_as_float(o[half][2 * j]) * inv,
                                              __uint_as_float(o[half][2 * j + 1]) * inv);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<uint4 *>(wst + lane * 64 + ((i ^ ((lane >> 1) & 3)) * 16)) =
                            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = rd_row + 8 * k;  // row within the warp
                        const int hr = quad * 32 + r;  // head
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(wst + r * 64 + ((rd_piece ^ ((r >> 1) & 3)) * 16));
                        if (hr < p.H)
                            *reinterpret_cast<uint4 *>(dst_base + (int64_t)hr * kRLat + (int)rank * kOCols + c +
                                                       rd_piece * 8) = v;
                    }
                    __syncwarp();
                }
            }
            const bool row_ok = h < p.H;
            if (row_ok && !whole && rank == 0 && grp == 0) {
                p.ml_part[((int64_t)slot * p.H + h) * 2] = m_fin;
                p.ml_part[((int64_t)slot * p.H + h) * 2 + 1] = l_tot;
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->o_empty);
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_all();  // copies into the peer have landed
    ptx::tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

// Prefix sums of the valid lengths (invalid ones count as 0 and are
// flagged), then the ranges (see DecodeSched) and each sequence's first and
// last range.
__device__ __forceinline__ int last_range_at_or_before(const int *range_start, int n, int x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (range_start[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Batches and range counts up to these sizes keep their prefix sums and
// range starts in shared memory for the binary searches below (each probe
// of a global copy would be a dependent L2 round trip; the scheduler sits
// between the query projection and the attention).
constexpr int kSchedSmemSeqs = 8192;
constexpr int kSchedSmemRanges = 1024;

__global__ void __launch_bounds__(1024) decode_schedule_kernel(const int32_t *seq_lens, int B, int max_seq, int n,
                                                               int seg_cost, DecodeSched sc, uint32_t *status)
{
    // The kernel after this one (the absorption) lets its own successor start
    // only after its wait for this kernel has returned, so the split-KV
    // kernel may read the schedule (and anything written before it) before
    // its own wait.
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ int s_prefix[kSchedSmemSeqs + 1];
    __shared__ int s_range[kSchedSmemRanges + 1];
    __shared__ int warp_sums[32];
    __shared__ int carry;
    const bool prefix_smem = B <= kSchedSmemSeqs, range_smem = n <= kSchedSmemRanges;
    int *prefix = sc.prefix;
    if (threadIdx.x == 0) {
        carry = 0;
        prefix[0] = 0;
        s_prefix[0] = 0;
    }
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
            const int nb = __shfl_up_sync(0xffffffffu, v, off);
            if ((threadIdx.x & 31) >= off) v += nb;
        }
        if ((threadIdx.x & 31) == 31) warp_sums[threadIdx.x >> 5] = v;
        __syncthreads();
        if (threadIdx.x < 32) {
            int w = warp_sums[threadIdx.x];
            for (int off = 1; off < 32; off <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, w, off);
                if (threadIdx.x >= off) w += nb;
            }
            warp_sums[threadIdx.x] = w;
        }
        __syncthreads();
        const int incl = v + ((threadIdx.x >> 5) ? warp_sums[(threadIdx.x >> 5) - 1] : 0) + carry;
        if (i < B) {
            prefix[i + 1] = incl;
            if (prefix_smem) s_prefix[i + 1] = incl;
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry = incl;
        __syncthreads();
    }
    // (A thread's global writes are visible to the block after the barrier
    // above when the sums do not fit in shared memory.)
    const int *pf = prefix_smem ? s_prefix : prefix;
    const int total = pf[B];
    const int chunk = max(128, (total + n - 1) / n);
    if (threadIdx.x == 0) *sc.chunk = chunk;
    // Range starts.  With a segment cost, cost position x of the sequence
    // walk C(b) = prefix[b] + b * seg_cost (seg_cost phantom keys before
    // each sequence) is cut into n equal parts.
    const long long tcost = (long long)total + (long long)seg_cost * B;
    for (int c = threadIdx.x; c <= n; c += blockDim.x) {
        int st;
        if (c == n) {
            st = total;
        } else if (seg_cost == 0) {
            st = (int)min((long long)total, (long long)c * chunk);
        } else {
            const long long x = tcost * c / n;
            int lo = 0, hi = B;  // last b with C(b) <= x
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if ((long long)pf[mid] + (long long)mid * seg_cost <= x) lo = mid;
                else hi = mid - 1;
            }
            if (lo >= B) {
                st = total;
            } else {
                const long long off = x - ((long long)pf[lo] + (long long)lo * seg_cost) - seg_cost;
                const int len = pf[lo + 1] - pf[lo];
                st = pf[lo] + (int)min((long long)len, max(0ll, off));
            }
        }
        sc.range_start[c] = st;
        if (range_smem) s_range[c] = st;
    }
    __syncthreads();
    const int *rs = range_smem ? s_range : sc.range_start;
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
        const int st = rs[c], en = rs[c + 1];
        int lo = 0, hi = B;  // first b with prefix[b + 1] > st
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (pf[mid + 1] > st) hi = mid;
            else lo = mid + 1;
        }
        sc.range_b0[c] = st < en ? lo : B;
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int lo = pf[b], hi = pf[b + 1];
        sc.seq_fc[b] = hi > lo ? last_range_at_or_before(rs, n, lo) : -1;
        sc.seq_lc[b] = hi > lo ? last_range_at_or_before(rs, n, hi - 1) : -1;
    }
}

// o_lat[b, h] = sum_s w_s O_s / sum_s w_s, w_s = 2^(m_s - m*) l_s, over the
// partial slots of sequence b (O_s normalised by its own row sum l_s;
// sequences handled by one range were written directly; invalid ones are
// zeroed).
__global__ void __launch_bounds__(128) decode_combine_tc_kernel(DecodeSched sc, int B, int H, int r_lat,
                                                                const bf16 *o_part, const float *ml_part,
                                                                bf16 *o_lat)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y;
    const int fc = sc.seq_fc[b], lc = sc.seq_lc[b];
    bf16 *dst = o_lat + ((int64_t)b * H + h) * r_lat;
    if (fc < 0) {
        for (int c = threadIdx.x; c < r_lat; c += blockDim.x) dst[c] = __float2bfloat16_rn(0.f);
        return;
    }
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
            const float *ml = ml_part + ((int64_t)(c + b) * H + h) * 2;
            acc += exp2f(ml[0] - m) * ml[1] * __bfloat162float(o_part[((int64_t)(c + b) * H + h) * r_lat + col]);
        }
        dst[col] = __float2bfloat16_rn(acc * inv);
    }
}

cudaError_t launch_decode_tc(const DecodeTcArgs &a, cudaStream_t s)
{
    CUtensorMap tl, tr;
    const int64_t c_rows = (int64_t)a.max_batch * a.max_seq;
    if (!make_tmap_bf16(&tl, a.lat, c_rows, kRLat, a.lat_stride, 64, kBKV) ||
        !make_tmap_bf16(&tr, a.rope, c_rows, 64, a.rope_stride, 32, kBKV))
        return cudaErrorInvalidValue;
    static std::atomic<int> smem_dev{-1};
    cudaError_t e = smem_limit_once(smem_dev, (const void *)decode_tc_kernel, kSmem);
    if (e != cudaSuccess) return e;
    DecTcParams p;
    p.B = a.B; p.H = a.H; p.max_seq = a.max_seq;
    p.sc = a.sc;
    p.scale_log2 = a.scale_log2;
    p.o_lat = (bf16 *)a.o_lat;
    p.o_part = a.o_part;
    p.ml_part = a.ml_part;
    p.status = a.status;
    profile_begin(MLA_PROFILE_DECODE_ATTENTION, s);
    e = launch_ex(decode_tc_kernel, dim3(2 * a.n_clusters), dim3(kThreads), kSmem, s, 2, tl, tr,
                  (const bf16 *)a.q_abs, (const bf16 *)a.q_rope, p);
    profile_end(MLA_PROFILE_DECODE_ATTENTION, s);
    note_launch();
    return e;
}

}  // namespace

size_t decode_sched_bytes(int B, int n) { return ((size_t)B + 1 + 1 + (n + 1) + n + 2 * (size_t)B) * sizeof(int); }

DecodeSched decode_sched_at(void *base, int B, int n)
{
    DecodeSched sc;
    sc.prefix = (int *)base;
    sc.chunk = sc.prefix + B + 1;
    sc.range_start = sc.chunk + 1;
    sc.range_b0 = sc.range_start + n + 1;
    sc.seq_fc = sc.range_b0 + n;
    sc.seq_lc = sc.seq_fc + B;
    return sc;
}

void decode_schedule(const int32_t *seq_lens, int B, int max_seq, int n_ranges, int seg_cost, const DecodeSched &sc,
                     uint32_t *status, cudaStream_t s)
{
    launch_ex(decode_schedule_kernel, dim3(1), dim3(1024), 0, s, 1, seq_lens, B, max_seq, n_ranges, seg_cost, sc,
              status);
    note_launch();
}

void decode_combine(const DecodeSched &sc, int B, int H, int r_lat, const bf16 *o_part, const float *ml_part,
                    void *o_lat, cudaStream_t s)
{
    launch_ex(decode_combine_tc_kernel, dim3(H, B), dim3(128), 0, s, 1, sc, B, H, r_lat, o_part, ml_part,
              (bf16 *)o_lat);
    note_launch();
}

int decode_tc_max_clusters()
{
    static int cached = -1;
    if (cached >= 0) return cached;
    if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
        return cached = 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) != cudaSuccess) n = 0;
    return cached = n;
}

bool decode_tc_supported(int H, int r_kv, int d_rope) { return H >= 1 && H <= kH && r_kv == 512 && d_rope == 64; }

cudaError_t decode_tc(const DecodeTcArgs &a, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    if (!decode_tc_supported(a.H, a.r_kv, a.d_rope) || a.n_clusters < 1) return cudaErrorInvalidValue;
    return launch_decode_tc(a, s);
}

}  // namespace mla

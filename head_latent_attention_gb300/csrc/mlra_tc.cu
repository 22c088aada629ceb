// Split-KV decode for Multi-head Low-Rank Attention (MLRA) on tcgen05.
//
// The latent is cut into L sub-heads of rank r = 256; head h reads only
// block i = h / (H / L) of every cached row, through its absorbed query
// q_abs,h (256 wide).  Per sequence and block the few heads of the block
// (4 at H = 16, L = 4) attend over the block's 256 latent columns, which
// serve as both keys and values.  With so few heads the keys take the
// MMA's M dimension:
//   S^T = K_i Q_i^T          M = 128 keys, N = 16 (heads, zero-padded), K = 256
//   O_i^T += V_i^T P^T        M = 2 x 128 latent columns, N = 16, K = 128 keys
// so one 128-key tile of one block (64 KB of cache) costs 32 MMAs, about
// half the time the SM's share of HBM bandwidth needs to deliver the tile.
//
// Work: the concatenated keys of all sequences are cut into one contiguous
// range per CTA (the decode scheduler's prefix sums); a range splits into
// segments (one per sequence it touches), and each segment into L units
// (one per block), streamed block by block so that every cached byte is
// read once.  Warp 0 issues TMA (query rows of the unit, then 128-key x
// 256-column tiles through a 3-stage ring), warp 1 the MMAs (non-blocking
// polling), warps 2..5 the softmax: thread j owns key j of a tile, keeps a
// running reference max per head (raised only when a tile exceeds it by
// more than 8 in log2 units, with the accumulator rescaled) and its own
// share of the row sums, reduced at the end of the unit.  A unit covering a
// whole sequence writes o_lat; the others write (O, m, l) partials for the
// decode combine kernel.
#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr int kKeys = 128;      // keys per tile = MMA M of S^T
constexpr int kR = 256;         // latent columns per block
constexpr int kNH = 16;         // heads per block, padded (MMA N)
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.f;
constexpr int kAtomK = kKeys * 128;              // one 128-key x 64-column atom of a tile (16 KB)
constexpr int kStageBytes = (kR / 64) * kAtomK;  // 64 KB
constexpr int kQAtom = kNH * 128;                // one 16-row x 64-column query atom (2 KB)
constexpr int kQBytes = (kR / 64) * kQAtom;      // 8 KB
constexpr int kPAtom = kNH * 128;                // P: 16 heads x 64 keys (2 KB)
constexpr int kPBytes = (kKeys / 64) * kPAtom;   // 4 KB
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffRed = kOffP + 2 * kPBytes;     // per-warp head maxima / sums
constexpr int kOffBar = kOffRed + 4 * kNH * 4;
constexpr int kSmem = kOffBar + 256 + 1024;
static_assert(kSmem <= 232448, "shared memory per CTA");
// Tensor memory: O^T (two 128-row halves of the 256 columns, 16 head columns
// each) in [0, 32), two S^T buffers in [32, 64).
constexpr int kOCol = 0;
constexpr int kSCol = 32;
constexpr int kTmemCols = 64;

struct MlraParams {
    int B, H, hpb, max_seq;
    const int *prefix;
    const int *chunk;
    float scale_log2;
    bf16 *o_lat;     // [B, H, 256]
    bf16 *o_part;    // [slots, H, 256] normalised partial averages
    float *ml_part;  // [slots, H, 2]
    uint32_t *status;
};

struct Bars {
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[2], pv_done[2];
    uint64_t o_empty;
    int abort;
    uint32_t tmem;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Segments of this CTA's key range [start, end) of the concatenated keys.
struct Segs {
    const int *prefix;
    int B, start, end, b;
    __device__ void init(const int *pf, int nb, int cta, int chunk)
    {
        prefix = pf;
        B = nb;
        const int total = pf[nb];
        start = min(total, cta * chunk);
        end = min(total, start + chunk);
        int lo = 0, hi = nb - 1;  // first b with prefix[b + 1] > start
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (pf[mid + 1] > start) hi = mid;
            else lo = mid + 1;
        }
        b = (start < end) ? lo : nb;
    }
    // Next non-empty segment: sequence sb, keys [k0, k1), whole-sequence flag.
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

// Walks the (segment, block, tile) sequence of this CTA: u counts units
// (segment x block), g counts tiles overall.
struct Cursor {
    Segs segs;
    int L;
    int b, k0, k1, blk, t, ntiles, u, g;
    bool whole, valid;
    __device__ void init(const int *pf, int nb, int cta, int chunk, int nblk)
    {
        segs.init(pf, nb, cta, chunk);
        L = nblk;
        u = -1;
        g = 0;
        valid = segs.next(b, k0, k1, whole);
        blk = 0;
        t = 0;
        ntiles = (k1 - k0 + kKeys - 1) / kKeys;
        if (valid) u = 0;
    }
    __device__ void step()
    {
        ++g;
        if (++t < ntiles) return;
        t = 0;
        ++u;
        if (++blk < L) return;
        blk = 0;
        valid = segs.next(b, k0, k1, whole);
        if (valid) ntiles = (k1 - k0 + kKeys - 1) / kKeys;
    }
};

__device__ __forceinline__ void softmax_vote(bool in, bool &any)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)in)
        : "memory");
    any = r != 0;
}
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
    mlra_tc_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmQ, MlraParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sKV = smem;
    uint8_t *sQ = smem + kOffQ;
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    Bars *bar = (Bars *)(smem + kOffBar);
    volatile int *abort_flag = &bar->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int L = p.H / p.hpb;

    if (threadIdx.x == 0) ptx::pdl_trigger();
    // Query and P rows beyond the block's heads stay zero for the whole kernel.
    for (int i = threadIdx.x; i < (kQBytes + 2 * kPBytes) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(sQ)[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&bar->kv_full[i], 1);
            ptx::mbar_init(&bar->kv_empty[i], 1);
        }
        ptx::mbar_init(&bar->q_full, 1);
        ptx::mbar_init(&bar->q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&bar->s_full[i], 1);
            ptx::mbar_init(&bar->s_free[i], kKeys);
            ptx::mbar_init(&bar->p_full[i], kKeys);
            ptx::mbar_init(&bar->pv_done[i], 1);
        }
        ptx::mbar_init(&bar->o_empty, kKeys);
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(&bar->tmem, kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::pdl_wait();  // the schedule, queries and cache come from earlier kernels
    const uint32_t tmem = bar->tmem;
    const int chunk = *p.chunk;
    const int cta = blockIdx.x;

    if (warp == 0) {
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&tmKV);
            ptx::prefetch_tmap(&tmQ);
            const uint64_t stream = ptx::policy_evict_first();
            Cursor c;
            c.init(p.prefix, p.B, cta, chunk, L);
            int pending[kStages];
#pragma unroll
            for (int i = 0; i < kStages; ++i) pending[i] = -1;
            int q_pending = -1;
            bool ok = true;
            while (ok && c.valid) {
                if (c.t == 0) {
                    // The unit's query rows, once every Q K^T of the previous unit completed.
                    if (c.u > 0 && !ptx::mbar_wait(&bar->q_empty, (c.u - 1) & 1, abort_flag)) { ok = false; break; }
                    ptx::mbar_expect_tx(&bar->q_full, (uint32_t)(kR * p.hpb * 2));
                    for (int a = 0; a < kR / 64; ++a)
                        ptx::tma_load_2d(sQ + a * kQAtom, &tmQ, &bar->q_full, a * 64, c.b * p.H + c.blk * p.hpb);
                    q_pending = c.u & 1;
                }
                const int st = c.g % kStages;
                const uint32_t ph = (uint32_t)(c.g / kStages) & 1;
                if (!ptx::mbar_wait(&bar->kv_empty[st], ph ^ 1, abort_flag)) { ok = false; break; }
                ptx::mbar_expect_tx(&bar->kv_full[st], kStageBytes);
                const int row = c.b * p.max_seq + c.k0 + c.t * kKeys;
                for (int a = 0; a < kR / 64; ++a)
                    ptx::tma_load_2d_hint(sKV + st * kStageBytes + a * kAtomK, &tmKV, &bar->kv_full[st],
                                          c.blk * kR + a * 64, row, stream);
                pending[st] = (int)ph;
                c.step();
            }
            if (!ok) *abort_flag = 1;
            volatile int never = 0;
            for (int i = 0; i < kStages; ++i)
                if (pending[i] >= 0) ptx::mbar_wait(&bar->kv_full[i], (uint32_t)pending[i], &never);
            if (q_pending >= 0) ptx::mbar_wait(&bar->q_full, (uint32_t)q_pending, &never);
        }
    } else if (warp == 1) {
        if (ptx::elect_one()) {
            constexpr uint32_t idesc_s = ptx::idesc_bf16(kKeys, kNH, false, false);
            constexpr uint32_t idesc_o = ptx::idesc_bf16(kKeys, kNH, true, false);
            const uint32_t kv0 = ptx::smem_u32(sKV), q0 = ptx::smem_u32(sQ), p0 = ptx::smem_u32(smem + kOffP);
            Cursor qk, pv;
            qk.init(p.prefix, p.B, cta, chunk, L);
            pv.init(p.prefix, p.B, cta, chunk, L);
            bool ok = true;
            long long last = clock64();
            while (ok && pv.valid) {
                bool progressed = false;
                if (pv.g < qk.g) {
                    bool ready = ptx::mbar_test(ptx::smem_u32(&bar->p_full[pv.g & 1]), (pv.g >> 1) & 1);
                    if (ready && pv.t == 0 && pv.u > 0)
                        ready = ptx::mbar_test(ptx::smem_u32(&bar->o_empty), (pv.u - 1) & 1);
                    if (ready) {
                        ptx::tc_fence_after();
                        const int st = pv.g % kStages;
                        const uint32_t vb = kv0 + st * kStageBytes;
                        const uint32_t pb = p0 + (pv.g & 1) * kPBytes;
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                            for (int k = 0; k < kKeys / 16; ++k)
                                ptx::mma_bf16(tmem + kOCol + mt * kNH,
                                              ptx::sdesc_sw128(vb + 2 * mt * kAtomK + k * 2048, kAtomK, 1024),
                                              ptx::sdesc_sw128(pb + (k >> 2) * kPAtom + (k & 3) * 32, 16, 1024),
                                              idesc_o, (pv.t == 0 && k == 0) ? 0u : 1u);
                        ptx::mma_commit(&bar->kv_empty[st]);
                        ptx::mma_commit(&bar->pv_done[pv.g & 1]);
                        pv.step();
                        progressed = true;
                    }
                }
                if (qk.valid) {
                    const int st = qk.g % kStages, sb = qk.g & 1;
                    bool ready = qk.t > 0 || ptx::mbar_test(ptx::smem_u32(&bar->q_full), qk.u & 1);
                    ready = ready && ptx::mbar_test(ptx::smem_u32(&bar->kv_full[st]), (qk.g / kStages) & 1);
                    ready = ready && (qk.g < 2 || ptx::mbar_test(ptx::smem_u32(&bar->s_free[sb]), ((qk.g >> 1) - 1) & 1));
                    if (ready) {
                        ptx::tc_fence_after();
                        const uint32_t kb = kv0 + st * kStageBytes;
#pragma unroll
                        for (int k = 0; k < kR / 16; ++k)
                            ptx::mma_bf16(tmem + kSCol + sb * kNH,
                                          ptx::sdesc_sw128(kb + (k >> 2) * kAtomK + (k & 3) * 32, 16, 1024),
                                          ptx::sdesc_sw128(q0 + (k >> 2) * kQAtom + (k & 3) * 32, 16, 1024),
                                          idesc_s, k != 0);
                        ptx::mma_commit(&bar->s_full[sb]);
                        if (qk.t == qk.ntiles - 1) ptx::mma_commit(&bar->q_empty);
                        qk.step();
                        progressed = true;
                    }
                }
                if (progressed) last = clock64();
                else if (*abort_flag || clock64() - last > ptx::kWaitCycles) ok = false;
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        // Softmax: thread j owns key j of every tile (tensor-memory lane j;
        // warp w reaches lanes 32 (w % 4) ...).
        const int quad = warp % 4;
        const int j = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int hpb = p.hpb;
        Cursor c;
        c.init(p.prefix, p.B, cta, chunk, L);
        bool ok = true;
        float m_ref[kNH], l_part[kNH];
        while (c.valid) {
            const int g = c.g, t = c.t;
            const int valid = min(kKeys, c.k1 - c.k0 - t * kKeys);
            if (t == 0) {
#pragma unroll
                for (int h = 0; h < kNH; ++h) { m_ref[h] = -INFINITY; l_part[h] = 0.f; }
            }
            // 1. This key's scores (log2 units; beyond the segment: -inf).
            float s[kNH];
            if (ok && ptx::mbar_wait(&bar->s_full[g & 1], (g >> 1) & 1, abort_flag)) {
                ptx::tc_fence_after();
                uint32_t r[16];
                ptx::tmem_ld16(tmem + lane_off + kSCol + (g & 1) * kNH, r);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar->s_free[g & 1]);
#pragma unroll
                for (int h = 0; h < kNH; ++h) s[h] = (j < valid && h < hpb) ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
            } else {
                ok = false;
#pragma unroll
                for (int h = 0; h < kNH; ++h) s[h] = -INFINITY;
            }
            bool raise_me = false;
#pragma unroll
            for (int h = 0; h < kNH; ++h) raise_me = raise_me || (s[h] > m_ref[h] + kRescaleThreshold);
            // Every softmax thread takes the same branch: a failure anywhere
            // ends the loop for all of them, and a raise is done by all.
            bool any_fail, any_raise;
            softmax_vote(!ok, any_fail);
            if (any_fail) break;
            softmax_vote(raise_me, any_raise);
            if (any_raise) {
                // Exact tile maximum per head (warp shuffles, then across warps).
                float mx[kNH];
#pragma unroll
                for (int h = 0; h < kNH; ++h) {
                    float v = s[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    mx[h] = v;
                }
                if (lane == 0)
#pragma unroll
                    for (int h = 0; h < kNH; ++h) red[(warp - 2) * kNH + h] = mx[h];
                softmax_bar();
                float corr[kNH];
                bool changed = false;
#pragma unroll
                for (int h = 0; h < kNH; ++h) {
                    const float tmax =
                        fmaxf(fmaxf(red[h], red[kNH + h]), fmaxf(red[2 * kNH + h], red[3 * kNH + h]));
                    const float m_new = fmaxf(m_ref[h], tmax);
                    corr[h] = (m_new == m_ref[h]) ? 1.f : ptx::ex2(m_ref[h] - m_new);
                    changed = changed || (m_new != m_ref[h] && t > 0);
                    m_ref[h] = m_new;
                    l_part[h] *= corr[h];
                }
                softmax_bar();  // red may be reused
                if (changed) {
                    // O holds every earlier P.V of the unit before it is rescaled.
                    // (Warp-uniform outcome: the tensor-memory accesses are warp-wide.)
                    if (!__all_sync(0xffffffffu,
                                    ptx::mbar_wait(&bar->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_flag))) {
                        ok = false;
                    } else {
                        ptx::tc_fence_after();
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            uint32_t o[16];
                            ptx::tmem_ld16(tmem + lane_off + kOCol + mt * kNH, o);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < kNH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * corr[h]);
                            ptx::tmem_st16(tmem + lane_off + kOCol + mt * kNH, o);
                        }
                        ptx::tmem_st_wait();
                    }
                }
            }
            // 2. P = 2^(s - m_ref) into P buffer g & 1 (once P.V(g - 2) has read it).
            float pv[kNH];
#pragma unroll
            for (int h = 0; h < kNH; ++h) {
                pv[h] = ptx::ex2(s[h] - m_ref[h]);
                if (h < hpb) l_part[h] += pv[h];
            }
            if (ok && g >= 2 && !ptx::mbar_wait(&bar->pv_done[g & 1], ((g >> 1) - 1) & 1, abort_flag)) ok = false;
            if (ok) {
                uint8_t *pb = smem + kOffP + (g & 1) * kPBytes + (j >> 6) * kPAtom;
                const int jj = j & 63;
                for (int h = 0; h < hpb; ++h) {
                    const int chunk16 = (jj >> 3) ^ (h & 7);
                    *reinterpret_cast<bf16 *>(pb + (h >> 3) * 1024 + (h & 7) * 128 + chunk16 * 16 + (jj & 7) * 2) =
                        __float2bfloat16_rn(pv[h]);
                }
                if (valid < kKeys && j >= valid) {
                    // Rows past the segment may hold arbitrary cache contents;
                    // P is 0 there, but 0 * NaN is not 0: zero the row.
                    uint8_t *stg = sKV + (g % kStages) * kStageBytes;
                    for (int a = 0; a < kR / 64; ++a)
                        for (int ch = 0; ch < 8; ++ch)
                            *reinterpret_cast<uint4 *>(stg + a * kAtomK + j * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->p_full[g & 1]);
            const bool last_tile = (t == c.ntiles - 1);
            const int b = c.b, blk = c.blk;
            const bool whole = c.whole;
            c.step();
            if (!last_tile) continue;

            // 3. Unit done: the heads' row sums, then O (lane j = latent
            //    columns j and 128 + j of the block) once the last P.V finished.
            float lsum[kNH];
#pragma unroll
            for (int h = 0; h < kNH; ++h) {
                float v = l_part[h];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                lsum[h] = v;
            }
            if (lane == 0)
#pragma unroll
                for (int h = 0; h < kNH; ++h) red[(warp - 2) * kNH + h] = lsum[h];
            softmax_bar();
#pragma unroll
            for (int h = 0; h < kNH; ++h) lsum[h] = (red[h] + red[kNH + h]) + (red[2 * kNH + h] + red[3 * kNH + h]);
            softmax_bar();
            bool any_fail2;
            const bool got = ok && ptx::mbar_wait(&bar->pv_done[g & 1], (g >> 1) & 1, abort_flag);
            softmax_vote(!got, any_fail2);
            if (any_fail2) { ok = false; break; }
            ptx::tc_fence_after();
            const int slot = cta + b;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                uint32_t o[16];
                ptx::tmem_ld16(tmem + lane_off + kOCol + mt * kNH, o);
                ptx::tmem_ld_wait();
                const int col = mt * 128 + j;
                for (int h = 0; h < hpb; ++h) {
                    const int head = blk * hpb + h;
                    bf16 *dst = whole ? p.o_lat + ((int64_t)b * p.H + head) * kR
                                      : p.o_part + ((int64_t)slot * p.H + head) * kR;
                    dst[col] = __float2bfloat16_rn(__uint_as_float(o[h]) / lsum[h]);
                }
            }
            if (!whole && j < hpb) {
                const int head = blk * hpb + j;
                float mj = m_ref[0], lj = lsum[0];
#pragma unroll
                for (int h = 1; h < kNH; ++h)
                    if (h == j) { mj = m_ref[h]; lj = lsum[h]; }
                p.ml_part[((int64_t)slot * p.H + head) * 2] = mj;
                p.ml_part[((int64_t)slot * p.H + head) * 2 + 1] = lj;
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->o_empty);
        }
        if (!ok) *abort_flag = 1;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

}  // namespace

bool mlra_tc_supported(int H, int L, int r_kv, int d_rope)
{
    return L >= 1 && H % L == 0 && H / L <= kNH && r_kv == L * kR && d_rope == 0;
}

int mlra_tc_ctas()
{
    static int cached = -1;
    if (cached >= 0) return cached;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return cached = sms;
}

cudaError_t mlra_tc(const MlraTcArgs &a, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    const int L = a.L, hpb = a.H / a.L;
    if (!mlra_tc_supported(a.H, a.L, a.r_kv, 0) || a.n_ctas < 1) return cudaErrorInvalidValue;
    CUtensorMap tkv, tq;
    if (!make_tmap_bf16(&tkv, a.lat, (int64_t)a.max_batch * a.max_seq, a.r_kv, a.lat_stride, 64, kKeys) ||
        !make_tmap_bf16(&tq, a.q_abs, (int64_t)a.B * a.H, kR, kR, 64, hpb))
        return cudaErrorInvalidValue;
    static std::atomic<int> smem_dev{-1};
    cudaError_t e = smem_limit_once(smem_dev, (const void *)mlra_tc_kernel, kSmem);
    if (e != cudaSuccess) return e;
    MlraParams p;
    p.B = a.B; p.H = a.H; p.hpb = hpb; p.max_seq = a.max_seq;
    p.prefix = a.prefix; p.chunk = a.chunk;
    p.scale_log2 = a.scale_log2;
    p.o_lat = (bf16 *)a.o_lat;
    p.o_part = a.o_part;
    p.ml_part = a.ml_part;
    p.status = a.status;
    (void)L;
    profile_begin(MLA_PROFILE_DECODE_ATTENTION, s);
    e = launch_ex(mlra_tc_kernel, dim3(a.n_ctas), dim3(kThreads), kSmem, s, 1, tkv, tq, p);
    profile_end(MLA_PROFILE_DECODE_ATTENTION, s);
    note_launch();
    return cudaGetLastError();
}

}  // namespace mla

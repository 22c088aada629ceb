// Causal flash-style prefill attention on tcgen05 (fp16 operands, fp32 softmax).
//
// One CTA per (pair of adjacent 128-query tiles, head, sequence); pairs with
// more keys launch first.  The two query tiles share every 64-key K/V tile
// (3-stage TMA ring) and have their own softmax warpgroup, so while one
// warpgroup turns scores into probabilities the tensor pipe runs the other
// tile's QK^T or P.V.  Per query tile q and key tile j:
//   S_q = Q_q K_j^T   tcgen05.mma M=128, N=64, K=d_qk into one of two
//                     tensor-memory score buffers of tile q;
//   softmax           one query row per thread: scale, causal mask (key <=
//                     query position), online max with a lazy rescale (only
//                     when the max grows by more than 8 in log2 units), exp2;
//                     P (fp16) is written back over its scores in tensor memory;
//   O_q += P V_j      tcgen05.mma with A = P from tensor memory and V read as
//                     an MN-major operand from its TMA tile (M=128, N=d_v).
// Warp 0 is the TMA producer, warp 1 issues the MMAs (non-blocking polling of
// both tiles' queues), warps 2..5 and 6..9 are the two softmax warpgroups.
// For the decoupled variant the key is [k_C ‖ k_R (shared by all heads)] and
// the query [q_nope ‖ q_rope].
// Both contractions run in fp16 (same tensor-core rate as bfloat16, 8x finer
// rounding): K and V come from an fp16 workspace, the bfloat16 query tiles are
// converted to fp16 in shared memory after their load (exact for |q| in fp16's
// normal range), and P is fp16 (values in [0, 256]).
#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {

bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

namespace {

constexpr int kQ = 128;
constexpr int kBN = 64;
constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.f;

template <int NQ, int NV>  // 64-column atoms of q/k (NQ) and of v (NV)
struct PCfg {
    static constexpr int kQBytes = NQ * kQ * 128;  // one query tile
    static constexpr int kAtom = kBN * 128;
    static constexpr int kStageBytes = (NQ + NV) * kAtom;
    static constexpr int kOffKV = 2 * kQBytes;
    static constexpr int kOffBar = kOffKV + kStages * kStageBytes;
    static constexpr int kSmem = kOffBar + 512 + 1024;
    // Tensor memory: O_0 at 0, O_1 at 128, score/P buffers (tile q, buffer i)
    // at 256 + 64 (2q + i).
    static constexpr int kOCol = 128;
    static constexpr int kSCol = 256;
};

struct PreTcParams {
    int B, S, H, max_seq, d_nope;
    int kv_group;              // query heads per key/value head (head h reads key/value head h / kv_group)
    int64_t kv_rows;
    bool rope;                 // decoupled: last q/k atom from q_rope / rope keys
    const int32_t *start_pos;  // device [B]
    float scale_log2;
    bf16 *o;                   // [B, S, H, d_v]
    int d_v;
    uint32_t *status;
};

struct PBars {
    uint64_t q_full[2], q_ready[2];
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2][2];
    uint64_t p_full[2], pv_done[2];
    int abort;
    uint32_t tmem;
};

template <int NQ, int NV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tQR,
                      const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tKR,
                      const __grid_constant__ CUtensorMap tV, PreTcParams p)
{
    using C = PCfg<NQ, NV>;
    ptx::pdl_trigger();
    ptx::pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sKV = smem + C::kOffKV;
    PBars *bar = (PBars *)(smem + C::kOffBar);
    volatile int *abort_flag = &bar->abort;

    const int n_qt = (p.S + kQ - 1) / kQ;
    const int n_pairs = (n_qt + 1) / 2;
    const int pi = n_pairs - 1 - (int)blockIdx.x;  // longest pairs first
    const int h = blockIdx.y, b = blockIdx.z;
    const int sp = p.start_pos[b];
    // Query tile q of this CTA covers rows [q0[q], q0[q] + nq[q]); nq = 0 if absent.
    int q0[2], nq[2], n_kt[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        q0[q] = (2 * pi + q) * kQ;
        nq[q] = max(0, min(kQ, p.S - q0[q]));
        n_kt[q] = nq[q] > 0 ? (sp + q0[q] + nq[q] - 1) / kBN + 1 : 0;
    }
    const int n_kt_all = max(n_kt[0], n_kt[1]);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nk_nope = p.rope ? NQ - 1 : NQ;  // q/k atoms from q_nope / the key workspace

    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            ptx::mbar_init(&bar->q_full[q], 1);
            ptx::mbar_init(&bar->q_ready[q], kQ);
            ptx::mbar_init(&bar->p_full[q], kQ);
            ptx::mbar_init(&bar->pv_done[q], 1);
            for (int i = 0; i < 2; ++i) ptx::mbar_init(&bar->s_full[q][i], 1);
        }
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&bar->kv_full[i], 1);
            ptx::mbar_init(&bar->kv_empty[i], 1);
        }
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(&bar->tmem, 512);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bar->tmem;
    bool ok = true;

    if (warp == 0) {
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&tQ);
            ptx::prefetch_tmap(&tK);
            ptx::prefetch_tmap(&tV);
            if (p.rope) {
                ptx::prefetch_tmap(&tQR);
                ptx::prefetch_tmap(&tKR);
            }
            bool q_pending[2] = {false, false};
            for (int q = 0; q < 2; ++q) {
                if (nq[q] == 0) continue;
                uint8_t *dq = smem + q * C::kQBytes;
                const int qrow = b * p.S + q0[q];
                ptx::mbar_expect_tx(&bar->q_full[q], C::kQBytes);
                for (int a = 0; a < nk_nope; ++a)
                    ptx::tma_load_2d(dq + a * kQ * 128, &tQ, &bar->q_full[q], h * p.d_nope + a * 64, qrow);
                if (p.rope) ptx::tma_load_2d(dq + (NQ - 1) * kQ * 128, &tQR, &bar->q_full[q], h * 64, qrow);
                q_pending[q] = true;
            }
            int pending[kStages] = {-1, -1, -1};
            for (int t = 0; t < n_kt_all; ++t) {
                const int st = t % kStages;
                const uint32_t ph = (t / kStages) & 1;
                if (!ptx::mbar_wait(&bar->kv_empty[st], ph ^ 1, abort_flag)) { ok = false; break; }
                ptx::mbar_expect_tx(&bar->kv_full[st], C::kStageBytes);
                uint8_t *dst = sKV + st * C::kStageBytes;
                const int krow = (int)(b * p.kv_rows) + t * kBN;
                for (int a = 0; a < nk_nope; ++a)
                    ptx::tma_load_2d(dst + a * C::kAtom, &tK, &bar->kv_full[st], (h / p.kv_group) * p.d_nope + a * 64,
                                     krow);
                if (p.rope) ptx::tma_load_2d(dst + (NQ - 1) * C::kAtom, &tKR, &bar->kv_full[st], 0, krow);
                for (int a = 0; a < NV; ++a)
                    ptx::tma_load_2d(dst + (NQ + a) * C::kAtom, &tV, &bar->kv_full[st], (h / p.kv_group) * p.d_v + a * 64,
                                     krow);
                pending[st] = (int)ph;
            }
            if (!ok) *abort_flag = 1;
            volatile int never = 0;
            for (int q = 0; q < 2; ++q)
                if (q_pending[q]) ptx::mbar_wait(&bar->q_full[q], 0, &never);
            for (int i = 0; i < kStages; ++i)
                if (pending[i] >= 0) ptx::mbar_wait(&bar->kv_full[i], (uint32_t)pending[i], &never);
        }
    } else if (warp == 1) {
        if (ptx::elect_one()) {
            // Four queues: QK^T and P.V of each query tile, issued as soon as
            // ready (test_wait polling, P.V first).  QK^T(q, j) overwrites the
            // buffer of P(q, j - 2): P.V(q, j - 2) must have been issued (the
            // tensor pipe keeps order).  The key tile's stage is released with
            // the last P.V that reads it (tile 1 reads every key tile tile 0 does).
            constexpr uint32_t idesc_s = ptx::idesc_f16(kQ, kBN, false, false);
            constexpr uint32_t idesc_o = ptx::idesc_f16(kQ, NV * 64, false, true);
            const uint32_t kv0 = ptx::smem_u32(sKV);
            int qk[2] = {0, 0}, pv[2] = {0, 0};
            bool qready[2] = {nq[0] == 0, nq[1] == 0};
            long long last = clock64();
            while (ok && (pv[0] < n_kt[0] || pv[1] < n_kt[1])) {
                bool progressed = false;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int j = pv[q];
                    if (j >= n_kt[q] || j >= qk[q]) continue;
                    // The stage is released by tile 1's P.V; it must come after tile 0's.
                    if (q == 1 && j < n_kt[0] && pv[0] <= j) continue;
                    if (!ptx::mbar_test(ptx::smem_u32(&bar->p_full[q]), j & 1)) continue;
                    ptx::tc_fence_after();
                    const int st = j % kStages;
                    const uint32_t vb = kv0 + st * C::kStageBytes + NQ * C::kAtom;
                    const uint32_t pa = tmem + C::kSCol + (2 * q + (j & 1)) * kBN;
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k)
                        ptx::mma_f16_tmem_a(tmem + q * C::kOCol, pa + k * 8,
                                            ptx::sdesc_sw128(vb + k * 2048, C::kAtom, 1024), idesc_o,
                                            (j > 0 || k > 0) ? 1u : 0u);
                    ptx::mma_commit(&bar->pv_done[q]);
                    const bool last_reader = (q == 1) || (j >= n_kt[1]);
                    if (last_reader) ptx::mma_commit(&bar->kv_empty[st]);
                    ++pv[q];
                    progressed = true;
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int j = qk[q];
                    if (j >= n_kt[q] || pv[q] < j - 1) continue;
                    if (!qready[q]) {
                        if (!ptx::mbar_test(ptx::smem_u32(&bar->q_ready[q]), 0)) continue;
                        qready[q] = true;
                    }
                    const int st = j % kStages;
                    if (!ptx::mbar_test(ptx::smem_u32(&bar->kv_full[st]), (j / kStages) & 1)) continue;
                    ptx::tc_fence_after();
                    const uint32_t qa = ptx::smem_u32(smem + q * C::kQBytes);
                    const uint32_t kb = kv0 + st * C::kStageBytes;
                    const uint32_t d = tmem + C::kSCol + (2 * q + (j & 1)) * kBN;
                    for (int a = 0; a < NQ; ++a) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            ptx::mma_bf16(d, ptx::sdesc_sw128(qa + a * kQ * 128 + k * 32, 16, 1024),
                                          ptx::sdesc_sw128(kb + a * C::kAtom + k * 32, 16, 1024), idesc_s,
                                          (a | k) != 0);
                    }
                    ptx::mma_commit(&bar->s_full[q][j & 1]);
                    ++qk[q];
                    progressed = true;
                }
                if (progressed) last = clock64();
                else if (*abort_flag || clock64() - last > ptx::kWaitCycles) ok = false;
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        const int q = (warp - 2) / 4;  // query tile of this softmax warpgroup
        const int quad = warp % 4;
        const int r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int my_pos = sp + q0[q] + r;
        uint8_t *sQ = smem + q * C::kQBytes;
        float m_run = -INFINITY, l_run = 0.f;
        if (nq[q] > 0) {
            // Query tile: bfloat16 -> fp16 in place (row r of every atom).
            if (!ptx::mbar_wait(&bar->q_full[q], 0, abort_flag)) ok = false;
            if (ok) {
                // Values beyond fp16's range saturate and raise the range flag.
                // The row's eight 16-byte chunks are visited in swizzled order
                // (chunk j sits at position j ^ (r % 8)): each is converted in
                // place, and a warp's 32 rows then spread over all banks
                // instead of all hitting the same four.
                bool over = false;
                for (int a = 0; a < NQ; ++a) {
                    uint4 *row = reinterpret_cast<uint4 *>(sQ + a * kQ * 128 + r * 128);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = jj ^ (r & 7);
                        uint4 w = row[j];
                        w.x = ptx::bf16x2_to_f16x2(w.x, over);
                        w.y = ptx::bf16x2_to_f16x2(w.y, over);
                        w.z = ptx::bf16x2_to_f16x2(w.z, over);
                        w.w = ptx::bf16x2_to_f16x2(w.w, over);
                        row[j] = w;
                    }
                }
                if (over && p.status) atomicOr(p.status, kStatusF16Range);
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&bar->q_ready[q]);
            }
        }
        for (int t = 0; ok && t < n_kt[q]; ++t) {
            const uint32_t sbuf = C::kSCol + (2 * q + (t & 1)) * kBN;
            // (Warp-uniform outcome: the tensor-memory loads below are warp-wide.)
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bar->s_full[q][t & 1], (t >> 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t r0[32], r1[32];
            ptx::tmem_ld32(tmem + lane_off + sbuf, r0);
            ptx::tmem_ld32(tmem + lane_off + sbuf + 32, r1);
            ptx::tmem_ld_wait();
            const int lim = my_pos - t * kBN;  // keys t*64 + j with j <= lim are visible
            // Raw scores; the scale is folded into the exponent below (it is
            // positive, so the maximum commutes with it).  Only the diagonal
            // tile needs the causal mask.
            float s[64];
            float mt = -INFINITY;
            if (lim >= kBN - 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = __uint_as_float(r0[j]);
                    s[32 + j] = __uint_as_float(r1[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = (j <= lim) ? __uint_as_float(r0[j]) : -INFINITY;
                    s[32 + j] = (32 + j <= lim) ? __uint_as_float(r1[j]) : -INFINITY;
                }
            }
            {
                // Balanced trees (short dependency chains) for the row max.
                float t[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) t[j] = fmaxf(s[j], s[32 + j]);
#pragma unroll
                for (int w = 16; w >= 1; w /= 2)
#pragma unroll
                    for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
                mt = t[0];
            }
            mt *= p.scale_log2;
            const bool resc = mt > m_run + kRescaleThreshold;
            const float m_new = resc ? mt : m_run;
            // Rows past the sequence end see no key; keep their state finite.
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float corr = (m_run == -INFINITY) ? 0.f : ptx::ex2(m_run - m_use);
            float psum;
            uint32_t pk[32];
            {
                float ps[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float a0 = ptx::ex2(fmaf(s[2 * j], p.scale_log2, -m_use));
                    const float a1 = ptx::ex2(fmaf(s[2 * j + 1], p.scale_log2, -m_use));
                    ps[j] = a0 + a1;
                    pk[j] = ptx::pack_f16(a0, a1);
                }
#pragma unroll
                for (int w = 16; w >= 1; w /= 2)
#pragma unroll
                    for (int j = 0; j < w; ++j) ps[j] += ps[j + w];
                psum = ps[0];
            }
            l_run = l_run * corr + psum;
            m_run = m_new;
            // P.V(t - 1) every tile: keeps the pv_done phases observed in
            // order, and O must hold it before a rescale.
            // (Warp-uniform outcome: the tensor-memory accesses below are warp-wide.)
            if (t > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->pv_done[q], (t - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            // The tensor-memory loads and stores are warp-wide: a warp
            // rescales when any of its rows needs it (the others multiply by 1).
            const bool do_resc = resc && t > 0 && corr != 1.f;
            if (__any_sync(0xffffffffu, do_resc)) {
                const float cf = do_resc ? corr : 1.f;
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < NV * 64; c += 32) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tmem + lane_off + q * C::kOCol + c, o);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * cf);
                    ptx::tmem_st32(tmem + lane_off + q * C::kOCol + c, o);
                }
            }
            // Key rows at or past the sequence's end (sp + S) may hold
            // arbitrary contents of unwritten cache rows; their P is 0, but
            // 0 * NaN is not 0: zero those rows of the V tile (both query
            // tiles write the same zeros before their own P.V).
            const int v0 = sp + p.S - t * kBN;
            if (v0 < kBN) {
                uint8_t *vt = sKV + (t % kStages) * C::kStageBytes + NQ * C::kAtom;
                const int r0 = max(v0, 0), nrow = kBN - r0;
                for (int i = r; i < NV * nrow * 8; i += kQ) {
                    const int a = i / (nrow * 8), rr = (i / 8) % nrow, ch = i % 8;
                    *reinterpret_cast<uint4 *>(vt + a * C::kAtom + (r0 + rr) * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                }
                ptx::fence_proxy_async_smem();
            }
            ptx::tmem_st32(tmem + lane_off + sbuf, pk);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->p_full[q]);
        }
        if (ok && n_kt[q] > 0) {
            if (__all_sync(0xffffffffu, ptx::mbar_wait(&bar->pv_done[q], (n_kt[q] - 1) & 1, abort_flag))) {
                ptx::tc_fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
                for (int c = 0; c < NV * 64; c += 32) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tmem + lane_off + q * C::kOCol + c, o);
                    ptx::tmem_ld_wait();
                    if (r < nq[q]) {
                        bf16 *dst = p.o + (((int64_t)b * p.S + q0[q] + r) * p.H + h) * p.d_v + c;
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            uint4 w;
                            w.x = ptx::pack_bf16(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
                            w.y = ptx::pack_bf16(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                            w.z = ptx::pack_bf16(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
                            w.w = ptx::pack_bf16(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
                            *reinterpret_cast<uint4 *>(dst + j) = w;
                        }
                    }
                }
            } else {
                ok = false;
            }
        }
        if (!ok) *abort_flag = 1;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

// Query positions of a one-token-per-sequence step from the cache lengths
// (the length includes the new token): start_pos[b] = seq_lens[b] - 1, or -1
// (no visible key: a zero output) for a length outside [1, max_seq], which
// is flagged.
__global__ void __launch_bounds__(256) positions_from_lengths_kernel(const int32_t *seq_lens, int B, int max_seq,
                                                                     int32_t *start_pos, uint32_t *status)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int L = seq_lens[b];
    const bool ok = L >= 1 && L <= max_seq;
    if (!ok) atomicOr(status, kStatusLen);
    start_pos[b] = ok ? L - 1 : -1;
}

// fp16 copy of the rope keys of rows [0, kv_rows) of every sequence.
__global__ void __launch_bounds__(256) rope_to_f16_kernel(const uint16_t *rope, int64_t stride, int max_seq,
                                                          int64_t kv_rows, int B, uint16_t *out,
                                                          const int32_t *start_pos, int S, uint32_t *status)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // one 8-element chunk
    const int64_t total = (int64_t)B * kv_rows * 8;
    if (i >= total) return;
    const int64_t row = i / 8, ch = i % 8;
    const int64_t b = row / kv_rows, j = row % kv_rows;
    const uint4 w = *reinterpret_cast<const uint4 *>(rope + (b * max_seq + j) * stride + ch * 8);
    bool over = false;
    *reinterpret_cast<uint4 *>(out + row * 64 + ch * 8) =
        make_uint4(ptx::bf16x2_to_f16x2(w.x, over), ptx::bf16x2_to_f16x2(w.y, over),
                   ptx::bf16x2_to_f16x2(w.z, over), ptx::bf16x2_to_f16x2(w.w, over));
    // Only rows that a query sees count (the others may hold anything).
    if (over && status && j < start_pos[b] + S) atomicOr(status, kStatusF16Range);
}

template <int NQ, int NV>
cudaError_t launch_prefill_tc(const PrefillTcArgs &a, cudaStream_t s)
{
    using C = PCfg<NQ, NV>;
    const int kvg = a.kv_group > 0 ? a.kv_group : 1;
    if (a.H % kvg) return cudaErrorInvalidValue;
    const int Hkv = a.H / kvg;
    CUtensorMap tq, tqr, tk, tkr, tv;
    const int64_t T = (int64_t)a.B * a.S;
    const int64_t KR = (int64_t)a.B * a.kv_rows;
    if (!make_tmap_bf16(&tq, a.q_nope, T, (int64_t)a.H * a.d_nope, (int64_t)a.H * a.d_nope, 64, kQ) ||
        !make_tmap_bf16(&tk, a.k, KR, (int64_t)Hkv * a.d_nope, (int64_t)Hkv * a.d_nope, 64, kBN) ||
        !make_tmap_bf16(&tv, a.v, KR, (int64_t)Hkv * a.d_v, (int64_t)Hkv * a.d_v, 64, kBN))
        return cudaErrorInvalidValue;
    if (a.d_rope) {
        if (!make_tmap_bf16(&tqr, a.q_rope, T, (int64_t)a.H * 64, (int64_t)a.H * 64, 64, kQ) ||
            !make_tmap_bf16(&tkr, a.k_rope16, KR, 64, 64, 64, kBN))
            return cudaErrorInvalidValue;
        cudaError_t e = launch_ex(rope_to_f16_kernel, dim3((unsigned)((KR * 64 / 8 + 255) / 256)), dim3(256), 0, s,
                                  1, (const uint16_t *)a.rope, a.rope_stride, a.max_seq, a.kv_rows, a.B,
                                  (uint16_t *)a.k_rope16, a.start_pos, a.S, a.status);
        note_launch();
        if (e != cudaSuccess) return e;
    } else {
        tqr = tq;
        tkr = tk;
    }
    static std::atomic<int> smem_dev{-1};
    cudaError_t e = smem_limit_once(smem_dev, (const void *)prefill_tc_kernel<NQ, NV>, C::kSmem);
    if (e != cudaSuccess) return e;
    PreTcParams p;
    p.B = a.B; p.S = a.S; p.H = a.H; p.max_seq = a.max_seq; p.d_nope = a.d_nope;
    p.kv_rows = a.kv_rows;
    p.kv_group = kvg;
    p.rope = a.d_rope != 0;
    p.start_pos = a.start_pos;
    p.scale_log2 = a.scale_log2;
    p.o = (bf16 *)a.o;
    p.d_v = a.d_v;
    p.status = a.status;
    dim3 grid(((a.S + kQ - 1) / kQ + 1) / 2, a.H, a.B);
    profile_begin(MLA_PROFILE_PREFILL_ATTENTION, s);
    e = launch_ex(prefill_tc_kernel<NQ, NV>, grid, dim3(kThreads), C::kSmem, s, 1, tq, tqr, tk, tkr, tv, p);
    profile_end(MLA_PROFILE_PREFILL_ATTENTION, s);
    note_launch();
    return e;
}

}  // namespace

cudaError_t positions_from_lengths(const int32_t *seq_lens, int B, int max_seq, int32_t *start_pos,
                                   uint32_t *status, cudaStream_t s)
{
    if (B == 0) return cudaSuccess;
    cudaError_t e = launch_ex(positions_from_lengths_kernel, dim3((B + 255) / 256), dim3(256), 0, s, 1, seq_lens, B,
                              max_seq, start_pos, status);
    note_launch();
    return e;
}

bool prefill_tc_supported(int d_nope, int d_rope, int d_v)
{
    return (d_nope == 128 && d_rope == 64 && d_v == 128) || (d_nope == 64 && d_rope == 0 && d_v == 64) ||
           (d_nope == 128 && d_rope == 0 && d_v == 128);
}

cudaError_t prefill_tc(const PrefillTcArgs &a, cudaStream_t s)
{
    if (a.B == 0 || a.S == 0) return cudaSuccess;
    if (a.d_nope == 128 && a.d_rope == 64 && a.d_v == 128) return launch_prefill_tc<3, 2>(a, s);
    if (a.d_nope == 64 && a.d_rope == 0 && a.d_v == 64) return launch_prefill_tc<1, 1>(a, s);
    if (a.d_nope == 128 && a.d_rope == 0 && a.d_v == 128) return launch_prefill_tc<2, 2>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace mla

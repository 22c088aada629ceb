// Projection GEMM on the 5th-generation tensor cores (tcgen05), bfloat16 in,
// fp32 accumulation in tensor memory, with the RoPE / cache-append epilogue.
//
// C[M, N] = A[M, K] B^T per batch entry.  Persistent kernel, one CTA per SM:
//   warp 0      TMA producer: 128x64 A tiles and BNx64 B tiles into a ring of
//               128-byte-swizzled shared-memory stages;
//   warp 1      MMA issuer: tcgen05.mma M=128, N=BN, K=16 into one of two
//               tensor-memory accumulators (so the epilogue of one tile
//               overlaps the main loop of the next);
//   warps 2..9  epilogue: tcgen05.ld of the accumulator rows (one row per
//               thread; the two warps of a lane quadrant take half of the
//               tile's columns each), RoPE on column pairs, bfloat16
//               conversion, and the store to the output or to the
//               (sequence, position) cache row.
// Every mbarrier wait is bounded: on timeout the CTA raises the status word's
// timeout bit, stops issuing, drains its own copies and frees tensor memory.
#include <cudaTypedefs.h>

#include <algorithm>

#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kEpiWarps = 8;  // two per tensor-memory lane quadrant, each half of a tile's columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kGroupM = 16;  // raster: 16 M-tiles share each sweep over N (L2 reuse)

struct TcGemmParams {
    int M, N, K, batch;
    int64_t a_row_batch, a_col_batch, b_row_batch, b_col_batch;
    int tiles_m, tiles_n;
    int splits, kb_per_split;  // split-K: unit u = (tile u % tiles, K slice u / tiles)
    float *partial;            // split-K partial sums [splits, M, N] (fp32), or null
    int nseg;                  // column segments: [seg_n0[i], seg_n0[i + 1]) uses epi[i]
    int seg_n0[kMaxSeg + 1];
    Epilogue epi[kMaxSeg];
    uint32_t *status;
    long long wait_cycles;     // give-up limit of the pipeline waits
    int tma_store;             // epilogue writes through the output tensor maps (staged 32 x 64 chunks)
};

template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kEpiBytes = kEpiWarps * 4096;  // per epilogue warp: 32 rows x 64 columns, bf16/fp16
    static constexpr int kSmem = kStages * kStageBytes + kEpiBytes + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr int kTmemCols = 2 * BN;
};

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &z, int &mt, int &nt)
{
    const int per_batch = tiles_m * tiles_n;
    z = t / per_batch;
    t -= z * per_batch;
    const int group = t / (kGroupM * tiles_n);
    const int first_m = group * kGroupM;
    const int gm = min(kGroupM, tiles_m - first_m);
    const int r = t - group * kGroupM * tiles_n;
    mt = first_m + r % gm;
    nt = r / gm;
}

// Segment of output column n (constant indices only: a dynamically indexed
// kernel parameter would be copied to local memory).
__device__ __forceinline__ int segment_of(const TcGemmParams &p, int n)
{
    return (p.nseg > 2 && n >= p.seg_n0[2]) ? 2 : ((p.nseg > 1 && n >= p.seg_n0[1]) ? 1 : 0);
}
__device__ __forceinline__ int segment_start(const TcGemmParams &p, int sg)
{
    return sg == 0 ? 0 : (sg == 1 ? p.seg_n0[1] : p.seg_n0[2]);
}

// RoPE of row m's columns [n0, n0 + NC) of its segment, in place (NC covers
// whole half-split groups: the chunk starts on a group boundary).  False,
// with the position flag raised, when the row's position is out of range.
template <int NC>
__device__ __forceinline__ bool apply_rope(const Epilogue &e, int m, int n0, float (&v)[64])
{
    if (e.rope_mode == kRopeNone) return true;
    const int pos = e.rope_pos ? e.rope_pos[m] : m;
    if (pos < 0 || pos >= e.max_seq) {
        if (n0 == 0 && e.status) atomicOr(e.status, kStatusPos);
        return false;
    }
    const int dim = e.rope_dim, half = dim / 2;
    const float2 *tab = e.rope_table + (int64_t)pos * half;
    if (e.rope_mode == kRopeInterleaved && dim == 64 && NC == 64 && n0 % 64 == 0) {
        // One whole group: its 32 (cos, sin) pairs in 16 16-byte loads (a
        // table row is 256 bytes, 16-byte aligned).
        const float4 *tab4 = reinterpret_cast<const float4 *>(tab);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 cs = tab4[i];
            float x0 = v[4 * i], x1 = v[4 * i + 1];
            v[4 * i] = x0 * cs.x - x1 * cs.y;
            v[4 * i + 1] = x0 * cs.y + x1 * cs.x;
            x0 = v[4 * i + 2];
            x1 = v[4 * i + 3];
            v[4 * i + 2] = x0 * cs.z - x1 * cs.w;
            v[4 * i + 3] = x0 * cs.w + x1 * cs.z;
        }
    } else if (e.rope_mode == kRopeInterleaved) {
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) {
            const float2 cs = tab[((n0 + 2 * i) % dim) >> 1];
            const float x0 = v[2 * i], x1 = v[2 * i + 1];
            v[2 * i] = x0 * cs.x - x1 * cs.y;
            v[2 * i + 1] = x0 * cs.y + x1 * cs.x;
        }
    } else if (dim == 64) {
        // Pairs (i, i + 32) of each 64-column group: compile-time indices
        // keep v in registers.
#pragma unroll
        for (int g = 0; g < NC; g += 64)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float2 cs = tab[i];
                const float x0 = v[g + i], x1 = v[g + i + 32];
                v[g + i] = x0 * cs.x - x1 * cs.y;
                v[g + i + 32] = x0 * cs.y + x1 * cs.x;
            }
    } else {
        // Narrower groups: runtime indices, on a local copy.
        float t[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) t[j] = v[j];
        for (int g = 0; g < NC; g += dim)
            for (int i = 0; i < half; ++i) {
                const float2 cs = tab[i];
                const float x0 = t[g + i], x1 = t[g + i + half];
                t[g + i] = x0 * cs.x - x1 * cs.y;
                t[g + i + half] = x0 * cs.y + x1 * cs.x;
            }
#pragma unroll
        for (int j = 0; j < NC; ++j) v[j] = t[j];
    }
    return true;
}

// The 16-bit words of NC output values: fp16 operands of the prefill
// attention saturate at 65504 and raise the range flag (rows of batch entry z
// that no query sees excepted), the rest is bfloat16.
template <int NC>
__device__ __forceinline__ void pack_out(const Epilogue &e, int z, int m, const float (&v)[64], uint32_t (&w)[32])
{
    if (e.out_f16) {
        bool over = false;
#pragma unroll
        for (int i = 0; i < NC; ++i) over |= ptx::beyond_f16(v[i]);
        if (over && e.range_start && m >= e.range_start[z] + e.range_len) over = false;
        if (over && e.status) atomicOr(e.status, kStatusF16Range);
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) w[i] = ptx::pack_f16_satfinite(v[2 * i], v[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) w[i] = ptx::pack_bf16(v[2 * i], v[2 * i + 1]);
    }
}

// Epilogue e applied to columns [n0, n0 + NC) of its segment, stored by this
// thread.  A row whose RoPE position is out of range is written as zeros
// (or, for a cache row, not written).
template <int NC>
__device__ __forceinline__ void store_chunk_seg(const TcGemmParams &p, const Epilogue &e, int z, int m, int n0,
                                                float (&v)[64])
{
    if (!apply_rope<NC>(e, m, n0, v)) {
        if (e.row_seq) return;
#pragma unroll
        for (int i = 0; i < NC; ++i) v[i] = 0.f;
    }
    uint16_t *dst;
    if (e.row_seq) {
        const int sq = e.row_seq[m], ps = e.row_pos[m];
        if (sq < 0 || sq >= e.max_batch || ps < 0 || ps >= e.max_seq) {
            if (n0 == 0 && e.status) atomicOr(e.status, (sq < 0 || sq >= e.max_batch) ? kStatusSeq : kStatusPos);
            return;
        }
        dst = (uint16_t *)e.out + ((int64_t)sq * e.seq_rows + ps) * e.ldc + n0;
    } else {
        dst = (uint16_t *)e.out + (int64_t)z * e.batch_stride + (int64_t)m * e.ldc + n0;
    }
    uint32_t w[32];
    pack_out<NC>(e, z, m, v, w);
#pragma unroll
    for (int i = 0; i < NC / 2; i += 4)
        *reinterpret_cast<uint4 *>(dst + 2 * i) = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
}

// Row m's 64 output columns [n0, n0 + 64) of its segment as the 32 words of
// a staged tensor store: zeros for rows past M (which the store clips) and
// for rows whose RoPE position is out of range.
__device__ __forceinline__ void stage_words_seg(const TcGemmParams &p, const Epilogue &e, int z, int m, int n0,
                                                float (&v)[64], uint32_t (&w)[32])
{
    if (m >= p.M || !apply_rope<64>(e, m, n0, v)) {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
        return;
    }
    pack_out<64>(e, z, m, v, w);
}

// Epilogue of one accumulator row chunk of NC columns starting at output
// column ng (of the concatenated product) of row m of batch entry z.
template <int NC>
__device__ __forceinline__ void store_chunk(const TcGemmParams &p, int z, int m, int ng, float (&v)[64])
{
    if (m >= p.M || ng >= p.N) return;
    const int sg = segment_of(p, ng);
    if (sg == 0) store_chunk_seg<NC>(p, p.epi[0], z, m, ng, v);
    else if (sg == 1) store_chunk_seg<NC>(p, p.epi[1], z, m, ng - p.seg_n0[1], v);
    else store_chunk_seg<NC>(p, p.epi[2], z, m, ng - p.seg_n0[2], v);
}

// Row tile mt of batch entry z lies wholly past the rows in use (see
// Epilogue::range_start): no role loads, multiplies or stores it.  Read after
// the wait for the previous kernel, which may write the limits.
__device__ __forceinline__ bool unit_skipped(const TcGemmParams &p, int z, int mt)
{
    const Epilogue &e = p.epi[0];
    return p.nseg == 1 && e.range_start && mt * kBM >= e.range_start[z] + e.range_len;
}

template <int BN, bool kBMN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                   const __grid_constant__ CUtensorMap tmC2, TcGemmParams p)
{
    using C = Cfg<BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * C::kABytes;
    uint8_t *sEpi = sB + S * C::kBBytes;  // epilogue staging, 4 KB per epilogue warp (1024-byte aligned)
    uint64_t *full = (uint64_t *)(sEpi + C::kEpiBytes);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_drain = acc_empty + 2;  // the MMA thread's issued MMAs completed (give-up path)
    uint32_t *tmem_slot = (uint32_t *)(mma_drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&acc_full[i], 1);
            ptx::mbar_init(&acc_empty[i], kEpiWarps);
        }
        ptx::mbar_init(mma_drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int num_tiles = p.tiles_m * p.tiles_n * p.batch;
    const int num_units = num_tiles * p.splits;
    const int nk = (p.K + kBK - 1) / kBK;
    bool ok = true;

    if (threadIdx.x == 0) ptx::pdl_trigger();
    if (warp == 0) {
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&tmA);
            ptx::prefetch_tmap(&tmB0);
            if (p.nseg > 1) ptx::prefetch_tmap(&tmB1);
            if (p.nseg > 2) ptx::prefetch_tmap(&tmB2);
            int stage = 0;
            uint32_t phase = 0;
            int pending[S];
#pragma unroll
            for (int i = 0; i < S; ++i) pending[i] = -1;
            // Weight (B) tile kb of a unit into a stage.  With a single row
            // tile every weight byte is read once: it is marked evict-first so
            // that the stream does not push reusable lines out of L2.
            const bool stream_b = p.tiles_m == 1 && p.batch == 1;
            const uint64_t evict_first = ptx::policy_evict_first();
            auto load_b = [&](int st, const CUtensorMap *tmB, int z, int brow, int kb) {
                uint8_t *dB = sB + st * C::kBBytes;
                if (!kBMN && stream_b) {
                    ptx::tma_load_2d_hint(dB, tmB, &full[st], kb * kBK, brow, evict_first);
                } else if (!kBMN) {
                    ptx::tma_load_2d(dB, tmB, &full[st], (int)(z * p.b_col_batch) + kb * kBK,
                                     (int)(z * p.b_row_batch) + brow);
                } else {
#pragma unroll
                    for (int a = 0; a < BN / 64; ++a)
                        ptx::tma_load_2d(dB + a * (kBK * 128), tmB, &full[st], (int)(z * p.b_col_batch) + brow + a * 64,
                                         (int)(z * p.b_row_batch) + kb * kBK);
                }
            };
            // The weights do not depend on earlier kernels: the first unit's
            // first stages of B go out before the wait for the previous
            // kernel, overlapping its tail.
            int pre = 0;
            // (Not when tiles may be skipped: whether this one is, is known
            // only after the wait.)
            if ((int)blockIdx.x < num_units && !(p.nseg == 1 && p.epi[0].range_start)) {
                int z, mt, nt;
                const int u = blockIdx.x;
                tile_coords(u % num_tiles, p.tiles_m, p.tiles_n, z, mt, nt);
                const int kb0 = (u / num_tiles) * p.kb_per_split, kb1 = min(nk, kb0 + p.kb_per_split);
                const int sg = segment_of(p, nt * BN);
                const CUtensorMap *tmB = sg == 0 ? &tmB0 : (sg == 1 ? &tmB1 : &tmB2);
                pre = max(0, min(S, kb1 - kb0));
                for (int i = 0; i < pre; ++i) {
                    ptx::mbar_expect_tx(&full[i], C::kStageBytes);
                    load_b(i, tmB, z, nt * BN - segment_start(p, sg), kb0 + i);
                }
            }
            ptx::pdl_wait();
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                int z, mt, nt;
                tile_coords(u % num_tiles, p.tiles_m, p.tiles_n, z, mt, nt);
                if (unit_skipped(p, z, mt)) continue;
                const int ks = u / num_tiles;
                const int kb0 = ks * p.kb_per_split, kb1 = min(nk, kb0 + p.kb_per_split);
                const int ax = (int)(z * p.a_col_batch), ay = (int)(z * p.a_row_batch) + mt * kBM;
                const int sg = segment_of(p, nt * BN);
                const CUtensorMap *tmB = sg == 0 ? &tmB0 : (sg == 1 ? &tmB1 : &tmB2);
                const int brow = nt * BN - segment_start(p, sg);  // first weight row of the tile in its segment
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (pre > 0) {
                        // Stage already armed and holding its weights.
                        --pre;
                    } else {
                        if (!ptx::mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_cycles)) {
                            ok = false;
                            break;
                        }
                        ptx::mbar_expect_tx(&full[stage], C::kStageBytes);
                        load_b(stage, tmB, z, brow, kb);
                    }
                    ptx::tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], ax + kb * kBK, ay);
                    pending[stage] = (int)phase;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) *abort_flag = 1;
            // Drain: every copy this CTA issued must land before it exits.
            volatile int never = 0;
            for (int i = 0; i < S; ++i)
                if (pending[i] >= 0) ptx::mbar_wait(&full[i], (uint32_t)pending[i], &never);
        }
    } else if (warp == 1) {
        ptx::pdl_wait();
        if (ptx::elect_one()) {
            constexpr uint32_t idesc = ptx::idesc_bf16(kBM, BN, false, kBMN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                {
                    int z, mt, nt;
                    tile_coords(u % num_tiles, p.tiles_m, p.tiles_n, z, mt, nt);
                    if (unit_skipped(p, z, mt)) continue;
                }
                const int ks = u / num_tiles;
                const int kb0 = ks * p.kb_per_split, kb1 = min(nk, kb0 + p.kb_per_split);
                if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag, p.wait_cycles)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_u32(sA + stage * C::kABytes);
                    const uint32_t b0 = ptx::smem_u32(sB + stage * C::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = ptx::sdesc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = kBMN ? ptx::sdesc_sw128(b0 + k * 2048, kBK * 128, 1024)
                                                 : ptx::sdesc_sw128(b0 + k * 32, 16, 1024);
                        ptx::mma_bf16(d, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                ptx::mma_commit(&acc_full[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            if (!ok) {
                *abort_flag = 1;
                // Giving up: the MMAs already issued still read shared memory
                // and write tensor memory; they complete before the CTA frees
                // either.
                ptx::mma_commit(mma_drain);
                volatile int never = 0;
                ptx::mbar_wait(mma_drain, 0, &never);
            }
        }
    } else {
        ptx::pdl_wait();
        const int quad = warp % 4;  // tensor-memory lane quadrant this warp may access
        // Warps w and w + 4 share a quadrant and split the tile's columns:
        // half eh takes [eh BN / 2, (eh + 1) BN / 2) (RoPE in the half-split
        // form needs whole 64-column groups: at BN = 64 half 0 takes them all).
        const int eh = (warp - 2) / 4;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            int z, mt, nt;
            tile_coords(u % num_tiles, p.tiles_m, p.tiles_n, z, mt, nt);
            if (unit_skipped(p, z, mt)) continue;
            const int ks = u / num_tiles;
            const int sg = segment_of(p, nt * BN);
            const bool half_rope = (sg == 0 ? p.epi[0].rope_mode : (sg == 1 ? p.epi[1].rope_mode : p.epi[2].rope_mode)) ==
                                   kRopeHalf;
            // (Warp-uniform outcome: the tensor-memory loads below are warp-wide.)
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.wait_cycles))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const int m = mt * kBM + quad * 32 + lane;
            const uint32_t tbase = tmem + acc * BN + ((uint32_t)(quad * 32) << 16);
            const int c_lo = eh * (BN / 2), c_hi = c_lo + BN / 2;
            if (p.partial) {
                // Split-K: raw fp32 partial sums; the reduce kernel applies the epilogue.
                for (int c = c_lo; c < c_hi; c += 32) {
                    uint32_t r0[32];
                    ptx::tmem_ld32(tbase + c, r0);
                    ptx::tmem_ld_wait();
                    const int n0 = nt * BN + c;
                    if (m < p.M && n0 < p.N) {
                        float *dst = p.partial + ((int64_t)ks * p.M + m) * p.N + n0;
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) =
                                make_float4(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1]),
                                            __uint_as_float(r0[i + 2]), __uint_as_float(r0[i + 3]));
                    }
                }
            } else if (p.tma_store) {
                // Whole 64-column chunks: converted, staged in this warp's
                // 32-row buffer in the 128-byte swizzle and written by one
                // tensor store, which clips rows past M and columns past the
                // segment.  At BN = 64 half 0 takes the tile.
                const int s_lo = BN >= 128 ? c_lo : (eh == 0 ? 0 : BN), s_hi = BN >= 128 ? c_hi : BN;
                uint8_t *buf = sEpi + (warp - 2) * 4096;
                for (int c = s_lo; c < s_hi; c += 64) {
                    uint32_t r0[32], r1[32];
                    ptx::tmem_ld32(tbase + c, r0);
                    ptx::tmem_ld32(tbase + c + 32, r1);
                    ptx::tmem_ld_wait();
                    float v[64];
#pragma unroll
                    for (int i = 0; i < 32; ++i) { v[i] = __uint_as_float(r0[i]); v[32 + i] = __uint_as_float(r1[i]); }
                    const int ng = nt * BN + c;
                    const int sgc = segment_of(p, ng);
                    const int n0 = ng - segment_start(p, sgc);
                    uint32_t w[32];
                    if (sgc == 0) stage_words_seg(p, p.epi[0], z, m, n0, v, w);
                    else if (sgc == 1) stage_words_seg(p, p.epi[1], z, m, n0, v, w);
                    else stage_words_seg(p, p.epi[2], z, m, n0, v, w);
                    // The previous store from this buffer has read it.
                    if (lane == 0) ptx::bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const CUtensorMap *tmC = sgc == 0 ? &tmC0 : (sgc == 1 ? &tmC1 : &tmC2);
                        ptx::tma_store_3d(tmC, buf, n0, mt * kBM + quad * 32, z);
                        ptx::bulk_commit_group();
                    }
                }
            } else if (half_rope) {
                const int h_lo = BN >= 128 ? c_lo : (eh == 0 ? 0 : BN), h_hi = BN >= 128 ? c_hi : BN;
                for (int c = h_lo; c < h_hi; c += 64) {
                    uint32_t r0[32], r1[32];
                    ptx::tmem_ld32(tbase + c, r0);
                    ptx::tmem_ld32(tbase + c + 32, r1);
                    ptx::tmem_ld_wait();
                    float v[64];
#pragma unroll
                    for (int i = 0; i < 32; ++i) { v[i] = __uint_as_float(r0[i]); v[32 + i] = __uint_as_float(r1[i]); }
                    store_chunk<64>(p, z, m, nt * BN + c, v);
                }
            } else {
                for (int c = c_lo; c < c_hi; c += 32) {
                    uint32_t r0[32];
                    ptx::tmem_ld32(tbase + c, r0);
                    ptx::tmem_ld_wait();
                    float v[64];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r0[i]);
                    store_chunk<32>(p, z, m, nt * BN + c, v);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (lane == 0) ptx::bulk_wait_group0();  // this warp's tensor stores are complete
        if (!ok) *abort_flag = 1;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, kStatusTimeout);
}

// Sum of the split-K partials of one NC-column chunk of one row, then the
// usual epilogue (RoPE, cache scatter, conversion).  With NC = 8 a warp
// reads 1 KB of each split's partials contiguously; the partial loads of all
// splits are issued before the sums (they are independent).
template <int NC>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(TcGemmParams p)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int chunks = p.N / NC;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)p.M * chunks) return;
    const int m = (int)(i / chunks), n0 = (int)(i % chunks) * NC;
    float v[64];
#pragma unroll
    for (int j = 0; j < NC; ++j) v[j] = 0.f;
    const int64_t split_stride = (int64_t)p.M * p.N / 4;
    const float4 *src = reinterpret_cast<const float4 *>(p.partial + (int64_t)m * p.N + n0);
    int ks = 0;
    if (NC == 8) {
        for (; ks + 4 <= p.splits; ks += 4) {
            float4 w[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                w[u][0] = __ldcs(src + (ks + u) * split_stride);
                w[u][1] = __ldcs(src + (ks + u) * split_stride + 1);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                v[0] += w[u][0].x; v[1] += w[u][0].y; v[2] += w[u][0].z; v[3] += w[u][0].w;
                v[4] += w[u][1].x; v[5] += w[u][1].y; v[6] += w[u][1].z; v[7] += w[u][1].w;
            }
        }
    }
    for (; ks < p.splits; ++ks) {
#pragma unroll
        for (int j = 0; j < NC / 4; ++j) {
            const float4 w = __ldcs(src + ks * split_stride + j);
            v[4 * j] += w.x;
            v[4 * j + 1] += w.y;
            v[4 * j + 2] += w.z;
            v[4 * j + 3] += w.w;
        }
    }
    store_chunk<NC>(p, 0, m, n0, v);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

}  // namespace

// 2-D 16-bit tensor map over a row-major view with a (box_cols x box_rows)
// box, zero fill out of bounds; 128-byte swizzle for 64-column boxes, 64-byte
// swizzle for 32-column boxes.
bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_cols * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Map for tensor stores of 16-bit elements laid out [batch][rows][cols] with
// the given row and batch strides (elements): 64-column x box_rows boxes in
// the 128-byte swizzle.  The store clips at every dimension's end, so a tile
// never writes past its own batch entry's rows.
bool make_tmap_store16(CUtensorMap *m, void *ptr, int64_t rows, int64_t cols, int64_t ld, int64_t batch,
                       int64_t batch_stride, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const int64_t bstride = batch > 1 ? batch_stride : rows * ld;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(bstride * 2)};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The column segments of a product (one, unless the call is grouped) and the
// total width.
static int segments_of(const GemmArgs &a, GemmSegment (&sg)[kMaxSeg], int &n_total)
{
    if (a.nseg <= 0) {
        sg[0].B = a.B;
        sg[0].epi = a.epi;
        sg[0].N = a.N;
        n_total = a.N;
        return 1;
    }
    n_total = 0;
    for (int i = 0; i < a.nseg && i < kMaxSeg; ++i) {
        sg[i] = a.seg[i];
        n_total += a.seg[i].N;
    }
    return a.nseg;
}

bool gemm_tc_supported(const GemmArgs &a)
{
    auto al = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    if (a.nseg < 0 || a.nseg > kMaxSeg || (a.nseg > 0 && (a.trans_b || a.batch != 1))) return false;
    GemmSegment sg[kMaxSeg];
    int n_total = 0;
    const int ns = segments_of(a, sg, n_total);
    if (!al(a.A.ptr) || (a.A.ld * 2) % 16) return false;
    if ((a.a_col_batch * 2) % 16 || (a.b_col_batch * 2) % 16) return false;
    for (int i = 0; i < ns; ++i) {
        const GemmSegment &g = sg[i];
        if (!al(g.B.ptr) || !al(g.epi.out) || (g.B.ld * 2) % 16 || (g.epi.ldc * 2) % 16) return false;
        if (g.N % (ns > 1 ? 64 : 32) || (g.epi.batch_stride * 2) % 16) return false;
        if (g.epi.rope_mode == kRopeHalf && (g.epi.rope_dim > 64 || 64 % g.epi.rope_dim || g.N % 64)) return false;
    }
    if (a.trans_b && n_total % 64) return false;
    return true;
}

// Tile width and K split: large GEMMs take the widest tile that still gives
// every SM a tile; skinny ones (few output tiles, e.g. one decode token per
// sequence) split K so that the work units fill whole waves of SMs.
GemmPlan gemm_tc_plan(const GemmArgs &a_in, int num_sms)
{
    GemmSegment sg[kMaxSeg];
    int n_total = 0;
    const int ns = segments_of(a_in, sg, n_total);
    GemmArgs a = a_in;
    a.N = n_total;
    a.epi = sg[0].epi;
    // Every segment boundary must fall on a tile boundary.
    auto fits = [&](int bn) {
        if (ns == 1) return a.N % bn == 0;
        for (int i = 0; i < ns; ++i)
            if (sg[i].N % bn) return false;
        return true;
    };
    auto tiles = [&](int bn) { return ((a.M + kBM - 1) / kBM) * ((a.N + bn - 1) / bn) * a.batch; };
    GemmPlan pl;
    pl.bn = 64;
    if (fits(256) && tiles(256) >= num_sms) pl.bn = 256;
    else if (fits(128) && tiles(128) >= num_sms) pl.bn = 128;
    pl.splits = 1;
    const int nk = (a.K + kBK - 1) / kBK;
    const bool skinny = a.M <= kBM;  // one row tile: the GEMM streams the weights once
    if ((skinny || tiles(64) < num_sms) && a.batch == 1 && a.epi.batch_stride == 0 && !a.trans_b) {
        // Estimated time ~ bytes moved (weights, plus the fp32 partials written
        // and read back) / fraction of the SMs kept busy over whole waves.
        const double wbytes = 2.0 * a.N * a.K + 2.0 * a.M * a.K;
        auto cost = [&](int units, int sp) {
            const int waves = (units + num_sms - 1) / num_sms;
            const double eff = (double)units / ((double)waves * num_sms);
            return (wbytes + (sp > 1 ? 8.0 * sp * a.M * a.N : 0.0)) / eff;
        };
        double best = cost(tiles(pl.bn), 1);
        for (int bn : {256, 128, 64}) {
            if (bn != 64 && !fits(bn)) continue;
            const int t = tiles(bn);
            for (int sp = 1; sp <= std::min(nk, 64); ++sp) {
                const int kbps = (nk + sp - 1) / sp;
                const int real = (nk + kbps - 1) / kbps;
                const double c = cost(t * real, real);
                if (c < 0.95 * best) {
                    best = c;
                    pl.bn = bn;
                    pl.splits = real;
                }
            }
        }
    }
    pl.kb_per_split = (nk + pl.splits - 1) / pl.splits;
    return pl;
}

size_t gemm_tc_workspace(const GemmArgs &a, int num_sms)
{
    GemmSegment sg[kMaxSeg];
    int n_total = 0;
    segments_of(a, sg, n_total);
    GemmPlan pl = gemm_tc_plan(a, num_sms);
    return pl.splits > 1 ? (size_t)pl.splits * a.M * n_total * sizeof(float) : 0;
}

template <int BN, bool kBMN>
static cudaError_t launch(const GemmArgs &a, const GemmPlan &pl, int num_sms, cudaStream_t s)
{
    using C = Cfg<BN>;
    GemmSegment sg[kMaxSeg];
    int n_total = 0;
    const int ns = segments_of(a, sg, n_total);
    CUtensorMap ta, tb[kMaxSeg];
    if (!make_tmap_bf16(&ta, a.A.ptr, a.A.rows, a.A.cols, a.A.ld, 64, kBM)) return cudaErrorInvalidValue;
    for (int i = 0; i < ns; ++i) {
        const Mat2D &B = sg[i].B;
        if (!make_tmap_bf16(&tb[i], B.ptr, B.rows, B.cols, B.ld, 64, kBMN ? kBK : BN)) return cudaErrorInvalidValue;
    }
    for (int i = ns; i < kMaxSeg; ++i) tb[i] = tb[0];
    TcGemmParams p;
    p.M = a.M; p.N = n_total; p.K = a.K; p.batch = a.batch;
    p.a_row_batch = a.a_row_batch; p.a_col_batch = a.a_col_batch;
    p.b_row_batch = a.b_row_batch; p.b_col_batch = a.b_col_batch;
    p.tiles_m = (a.M + kBM - 1) / kBM;
    p.tiles_n = (n_total + BN - 1) / BN;
    p.splits = pl.splits;
    p.kb_per_split = pl.kb_per_split;
    p.partial = pl.splits > 1 ? a.split_ws : nullptr;
    p.nseg = ns;
    p.seg_n0[0] = 0;
    bool half_rope = false;
    for (int i = 0; i < ns; ++i) {
        p.epi[i] = sg[i].epi;
        p.seg_n0[i + 1] = p.seg_n0[i] + sg[i].N;
        half_rope = half_rope || sg[i].epi.rope_mode == kRopeHalf;
    }
    for (int i = ns; i < kMaxSeg; ++i) p.epi[i] = sg[0].epi;
    p.status = sg[0].epi.status;
    p.wait_cycles = gemm_wait_cycles();
    // Staged tensor stores for plain row-major outputs: not for split-K
    // partials, nor for rows scattered to cache positions.
    CUtensorMap tc[kMaxSeg];
    bool tma = pl.splits == 1;
    for (int i = 0; i < ns && tma; ++i) {
        const Epilogue &e = sg[i].epi;
        tma = !e.row_seq && (a.batch == 1 || (e.batch_stride * 2) % 16 == 0) &&
              make_tmap_store16(&tc[i], e.out, a.M, sg[i].N, e.ldc, a.batch, e.batch_stride, 32);
    }
    p.tma_store = tma ? 1 : 0;
    if (!tma) tc[0] = ta;  // unused placeholders
    for (int i = tma ? ns : 1; i < kMaxSeg; ++i) tc[i] = tc[0];
    if (pl.splits > 1 && !a.split_ws) return cudaErrorInvalidValue;
    const int units = p.tiles_m * p.tiles_n * a.batch * p.splits;
    static std::atomic<int> smem_dev{-1};
    cudaError_t e = smem_limit_once(smem_dev, (const void *)gemm_tc_kernel<BN, kBMN>, C::kSmem);
    if (e != cudaSuccess) return e;
    e = launch_ex(gemm_tc_kernel<BN, kBMN>, dim3(std::min(units, num_sms)), dim3(kThreads), C::kSmem, s, 1, ta,
                  tb[0], tb[1], tb[2], tc[0], tc[1], tc[2], p);
    note_launch();
    if (e != cudaSuccess) return e;
    if (pl.splits > 1) {
        const int nc = half_rope ? 64 : 8;
        const int64_t threads = (int64_t)a.M * (n_total / nc);
        const unsigned blocks = (unsigned)((threads + 255) / 256);
        if (nc == 64) e = launch_ex(splitk_reduce_kernel<64>, dim3(blocks), dim3(256), 0, s, 1, p);
        else e = launch_ex(splitk_reduce_kernel<8>, dim3(blocks), dim3(256), 0, s, 1, p);
        note_launch();
    }
    return e;
}

long long ptx_default_wait_cycles() { return ptx::kWaitCycles; }

cudaError_t gemm_tc(const GemmArgs &a, int num_sms, cudaStream_t s)
{
    if (a.M == 0 || (a.nseg == 0 && a.N == 0) || a.batch == 0) return cudaSuccess;
    if (!gemm_tc_supported(a)) return cudaErrorInvalidValue;
    const GemmPlan pl = gemm_tc_plan(a, num_sms);
    if (a.trans_b) {
        if (pl.bn == 256) return launch<256, true>(a, pl, num_sms, s);
        if (pl.bn == 128) return launch<128, true>(a, pl, num_sms, s);
        return launch<64, true>(a, pl, num_sms, s);
    }
    if (pl.bn == 256) return launch<256, false>(a, pl, num_sms, s);
    if (pl.bn == 128) return launch<128, false>(a, pl, num_sms, s);
    return launch<64, false>(a, pl, num_sms, s);
}

}  // namespace mla

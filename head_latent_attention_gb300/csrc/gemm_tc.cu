// Projection GEMM on the 5th-generation tensor cores (tcgen05), bfloat16 in,
// fp32 accumulation in tensor memory, with the RoPE / cache-append epilogue.
//
// C[M, N] = A[M, K] B^T per batch entry.  Persistent kernel, one CTA per SM:
//   warp 0      TMA producer: 128x64 A tiles and BNx64 B tiles into a ring of
//               128-byte-swizzled shared-memory stages;
//   warp 1      MMA issuer: tcgen05.mma M=128, N=BN, K=16 into one of two
//               tensor-memory accumulators (so the epilogue of one tile
//               overlaps the main loop of the next);
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows (one row per
//               thread), RoPE on column pairs, bfloat16 conversion, and the
//               store to the output or to the (sequence, position) cache row.
// Every mbarrier wait is bounded: on timeout the CTA raises the status word's
// timeout bit, stops issuing, drains its own copies and frees tensor memory.
#include <cudaTypedefs.h>

#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kGroupM = 16;  // raster: 16 M-tiles share each sweep over N (L2 reuse)

struct TcGemmParams {
    int M, N, K, batch;
    int64_t a_row_batch, a_col_batch, b_row_batch, b_col_batch;
    int tiles_m, tiles_n;
    Epilogue epi;
    uint32_t *status;
};

template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
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

// Epilogue of one accumulator row chunk of NC columns (32 or 64) starting at
// output column n0 of row m of batch entry z.
template <int NC>
__device__ __forceinline__ void store_chunk(const TcGemmParams &p, int z, int m, int n0, float (&v)[64])
{
    const Epilogue &e = p.epi;
    if (m >= p.M || n0 >= p.N) return;
    if (e.rope_mode != kRopeNone) {
        const int pos = e.rope_pos ? e.rope_pos[m] : m;
        if (pos < 0 || pos >= e.max_seq) {
            if (n0 == 0 && e.status) atomicOr(e.status, kStatusPos);
            return;
        }
        const int dim = e.rope_dim, half = dim / 2;
        const float2 *tab = e.rope_table + (int64_t)pos * half;
        if (e.rope_mode == kRopeInterleaved) {
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) {
                const float2 cs = tab[((n0 + 2 * i) % dim) >> 1];
                const float x0 = v[2 * i], x1 = v[2 * i + 1];
                v[2 * i] = x0 * cs.x - x1 * cs.y;
                v[2 * i + 1] = x0 * cs.y + x1 * cs.x;
            }
        } else {
            // NC covers whole groups: the chunk starts on a group boundary.
            for (int g = 0; g < NC; g += dim)
                for (int i = 0; i < half; ++i) {
                    const float2 cs = tab[i];
                    const float x0 = v[g + i], x1 = v[g + i + half];
                    v[g + i] = x0 * cs.x - x1 * cs.y;
                    v[g + i + half] = x0 * cs.y + x1 * cs.x;
                }
        }
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
    if (e.out_f16) {
#pragma unroll
        for (int i = 0; i < NC; i += 8)
            *reinterpret_cast<uint4 *>(dst + i) =
                make_uint4(ptx::pack_f16(v[i], v[i + 1]), ptx::pack_f16(v[i + 2], v[i + 3]),
                           ptx::pack_f16(v[i + 4], v[i + 5]), ptx::pack_f16(v[i + 6], v[i + 7]));
    } else {
#pragma unroll
        for (int i = 0; i < NC; i += 8)
            *reinterpret_cast<uint4 *>(dst + i) =
                make_uint4(ptx::pack_bf16(v[i], v[i + 1]), ptx::pack_bf16(v[i + 2], v[i + 3]),
                           ptx::pack_bf16(v[i + 4], v[i + 5]), ptx::pack_bf16(v[i + 6], v[i + 7]));
    }
}

template <int BN, bool kBMN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   TcGemmParams p)
{
    using C = Cfg<BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * C::kABytes;
    uint64_t *full = (uint64_t *)(sB + S * C::kBBytes);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = (uint32_t *)(acc_empty + 2);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&acc_full[i], 1);
            ptx::mbar_init(&acc_empty[i], 4);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int num_tiles = p.tiles_m * p.tiles_n * p.batch;
    const int nk = (p.K + kBK - 1) / kBK;
    bool ok = true;

    if (warp == 0) {
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&tmA);
            ptx::prefetch_tmap(&tmB);
            int stage = 0;
            uint32_t phase = 0;
            int pending[S];
#pragma unroll
            for (int i = 0; i < S; ++i) pending[i] = -1;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int z, mt, nt;
                tile_coords(t, p.tiles_m, p.tiles_n, z, mt, nt);
                const int ax = (int)(z * p.a_col_batch), ay = (int)(z * p.a_row_batch) + mt * kBM;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                    ptx::mbar_expect_tx(&full[stage], C::kStageBytes);
                    ptx::tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], ax + kb * kBK, ay);
                    uint8_t *dB = sB + stage * C::kBBytes;
                    if (!kBMN) {
                        ptx::tma_load_2d(dB, &tmB, &full[stage], (int)(z * p.b_col_batch) + kb * kBK,
                                         (int)(z * p.b_row_batch) + nt * BN);
                    } else {
#pragma unroll
                        for (int a = 0; a < BN / 64; ++a)
                            ptx::tma_load_2d(dB + a * (kBK * 128), &tmB, &full[stage],
                                             (int)(z * p.b_col_batch) + nt * BN + a * 64,
                                             (int)(z * p.b_row_batch) + kb * kBK);
                    }
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
        if (ptx::elect_one()) {
            constexpr uint32_t idesc = ptx::idesc_bf16(kBM, BN, false, kBMN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_u32(sA + stage * C::kABytes);
                    const uint32_t b0 = ptx::smem_u32(sB + stage * C::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = ptx::sdesc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = kBMN ? ptx::sdesc_sw128(b0 + k * 2048, kBK * 128, 1024)
                                                 : ptx::sdesc_sw128(b0 + k * 32, 16, 1024);
                        ptx::mma_bf16(d, ad, bd, idesc, (kb | k) != 0);
                    }
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                ptx::mma_commit(&acc_full[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        const int quad = warp % 4;  // tensor-memory lane quadrant this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        const bool half_rope = p.epi.rope_mode == kRopeHalf;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            int z, mt, nt;
            tile_coords(t, p.tiles_m, p.tiles_n, z, mt, nt);
            if (!ptx::mbar_wait(&acc_full[acc], acc_phase, abort_flag)) { ok = false; break; }
            ptx::tc_fence_after();
            const int m = mt * kBM + quad * 32 + lane;
            const uint32_t tbase = tmem + acc * BN + ((uint32_t)(quad * 32) << 16);
            if (half_rope) {
                for (int c = 0; c < BN; c += 64) {
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
                for (int c = 0; c < BN; c += 32) {
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

bool gemm_tc_supported(const GemmArgs &a)
{
    auto al = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    if (!al(a.A.ptr) || !al(a.B.ptr) || !al(a.epi.out)) return false;
    if ((a.A.ld * 2) % 16 || (a.B.ld * 2) % 16 || (a.epi.ldc * 2) % 16) return false;
    if (a.N % 32 || (a.a_col_batch * 2) % 16 || (a.b_col_batch * 2) % 16 || (a.epi.batch_stride * 2) % 16)
        return false;
    if (a.epi.rope_mode == kRopeHalf && (a.epi.rope_dim > 64 || 64 % a.epi.rope_dim || a.N % 64)) return false;
    if (a.trans_b && a.N % 64) return false;
    return true;
}

template <int BN, bool kBMN>
static cudaError_t launch(const GemmArgs &a, int num_sms, cudaStream_t s)
{
    using C = Cfg<BN>;
    CUtensorMap ta, tb;
    if (!make_tmap_bf16(&ta, a.A.ptr, a.A.rows, a.A.cols, a.A.ld, 64, kBM)) return cudaErrorInvalidValue;
    if (!kBMN) {
        if (!make_tmap_bf16(&tb, a.B.ptr, a.B.rows, a.B.cols, a.B.ld, 64, BN)) return cudaErrorInvalidValue;
    } else {
        if (!make_tmap_bf16(&tb, a.B.ptr, a.B.rows, a.B.cols, a.B.ld, 64, kBK)) return cudaErrorInvalidValue;
    }
    TcGemmParams p;
    p.M = a.M; p.N = a.N; p.K = a.K; p.batch = a.batch;
    p.a_row_batch = a.a_row_batch; p.a_col_batch = a.a_col_batch;
    p.b_row_batch = a.b_row_batch; p.b_col_batch = a.b_col_batch;
    p.tiles_m = (a.M + kBM - 1) / kBM;
    p.tiles_n = (a.N + BN - 1) / BN;
    p.epi = a.epi;
    p.status = a.epi.status;
    const int tiles = p.tiles_m * p.tiles_n * a.batch;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, kBMN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    gemm_tc_kernel<BN, kBMN><<<std::min(tiles, num_sms), kThreads, C::kSmem, s>>>(ta, tb, p);
    note_launch();
    return cudaGetLastError();
}

cudaError_t gemm_tc(const GemmArgs &a, int num_sms, cudaStream_t s)
{
    if (a.M == 0 || a.N == 0 || a.batch == 0) return cudaSuccess;
    if (!gemm_tc_supported(a)) return cudaErrorInvalidValue;
    auto tiles = [&](int bn) { return ((a.M + kBM - 1) / kBM) * ((a.N + bn - 1) / bn) * a.batch; };
    int bn = 64;
    if (a.N % 256 == 0 && tiles(256) >= num_sms) bn = 256;
    else if (a.N % 128 == 0 && tiles(128) >= num_sms) bn = 128;
    if (a.trans_b) {
        if (bn == 256) return launch<256, true>(a, num_sms, s);
        if (bn == 128) return launch<128, true>(a, num_sms, s);
        return launch<64, true>(a, num_sms, s);
    }
    if (bn == 256) return launch<256, false>(a, num_sms, s);
    if (bn == 128) return launch<128, false>(a, num_sms, s);
    return launch<64, false>(a, num_sms, s);
}

}  // namespace mla

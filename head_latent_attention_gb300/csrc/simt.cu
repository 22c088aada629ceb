// CUDA-core kernels: projection GEMM with RoPE / cache-append epilogue,
// split-KV latent decode with a log-sum-exp combine, and causal flash-style
// prefill.  Used for the float32 dtype (no TF32: its 2^-11 unit roundoff is
// too coarse for float32 parity) and instantiated for bfloat16 as well.
#include <float.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kTile = 64;
constexpr int kTileK = 16;

// Rotation of element c of a rope group held in a shared-memory row: the
// pair partner is c ^ 1 (interleaved, deepseek-mla apply_rotary_emb) or
// c +- dim/2 (half-split, mla_attn _apply_rope).
__device__ __forceinline__ float rope_elem(const float *row, int c, int dim, int mode,
                                          const float2 *table, int pos)
{
    if (mode == kRopeInterleaved) {
        int i = (c % dim) >> 1;
        float2 cs = table[(int64_t)pos * (dim / 2) + i];
        float x0 = row[c & ~1], x1 = row[c | 1];
        return (c & 1) ? x0 * cs.y + x1 * cs.x : x0 * cs.x - x1 * cs.y;
    }
    int half = dim / 2;
    int i = c % half;
    float2 cs = table[(int64_t)pos * half + i];
    int base = c - (c % dim);
    float x0 = row[base + i], x1 = row[base + i + half];
    return (c % dim) < half ? x0 * cs.x - x1 * cs.y : x0 * cs.y + x1 * cs.x;
}

template <typename T, bool kTransB>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a)
{
    __shared__ float As[kTileK][kTile + 4];
    __shared__ float Bs[kTileK][kTile + 4];
    __shared__ float Cs[kTile][kTile + 1];
    const int z = blockIdx.z;
    const T *A = (const T *)a.A.ptr + (int64_t)z * (a.a_row_batch * a.A.ld + a.a_col_batch);
    const T *Bm = (const T *)a.B.ptr + (int64_t)z * (a.b_row_batch * a.B.ld + a.b_col_batch);
    const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < a.K; k0 += kTileK) {
        for (int i = tid; i < kTile * kTileK; i += 256) {
            int r = i / kTileK, c = i % kTileK;
            int m = m0 + r, k = k0 + c;
            As[c][r] = (m < a.M && k < a.K) ? to_f32(A[(int64_t)m * a.A.ld + k]) : 0.f;
            int n, kk;
            if (kTransB) { n = n0 + i % kTile; kk = k0 + i / kTile; }
            else { n = n0 + r; kk = k; }
            float bv = 0.f;
            if (n < a.N && kk < a.K)
                bv = kTransB ? to_f32(Bm[(int64_t)kk * a.B.ld + n]) : to_f32(Bm[(int64_t)n * a.B.ld + kk]);
            if (kTransB) Bs[i / kTile][i % kTile] = bv;
            else Bs[c][r] = bv;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kTileK; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { av[i] = As[kk][ty * 4 + i]; bv[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
    __syncthreads();
    const Epilogue &e = a.epi;
    for (int idx = tid; idx < kTile * kTile; idx += 256) {
        int r = idx / kTile, c = idx % kTile;
        int m = m0 + r, n = n0 + c;
        if (m >= a.M || n >= a.N) continue;
        float v = Cs[r][c];
        if (e.rope_mode != kRopeNone) {
            int pos = e.rope_pos ? e.rope_pos[m] : m;
            if (pos < 0 || pos >= e.max_seq) {
                if (c == 0 && e.status) atomicOr(e.status, kStatusPos);
                continue;
            }
            v = rope_elem(Cs[r], c, e.rope_dim, e.rope_mode, e.rope_table, pos);
        }
        T *dst;
        if (e.row_seq) {
            int sq = e.row_seq[m], p = e.row_pos[m];
            if (sq < 0 || sq >= e.max_batch || p < 0 || p >= e.max_seq) {
                if (c == 0 && e.status)
                    atomicOr(e.status, (sq < 0 || sq >= e.max_batch) ? kStatusSeq : kStatusPos);
                continue;
            }
            dst = (T *)e.out + ((int64_t)sq * e.seq_rows + p) * e.ldc + n;
        } else {
            dst = (T *)e.out + (int64_t)z * e.batch_stride + (int64_t)m * e.ldc + n;
        }
        *dst = from_f32<T>(v);
    }
}

// ---------------------------------------------------------------------------
// Split-KV latent decode.  Block = (split, sequence b, group of HG heads that
// share one latent block); keys [split*chunk, min(L_b, (split+1)*chunk)).
// Scores s_hj = q_abs,h . c_j + q_rope,h . k_R,j; the partial state of each
// (b, split, h) is (max m in log2 units, sum l of 2^(s*scale_log2 - m),
// O = sum 2^(...) c_j).
// ---------------------------------------------------------------------------
template <typename T, int HG>
__global__ void __launch_bounds__(256) decode_partial_kernel(DecodeArgs a)
{
    extern __shared__ float sm[];
    const int split = blockIdx.x, b = blockIdx.y, hg = blockIdx.z;
    const int h0 = hg * HG;
    const int dq = a.r_lat + a.d_rope;
    float *qs = sm;                    // [HG][dq]
    float *ss = qs + HG * dq;          // [HG][chunk]
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int L = a.seq_lens[b];
    float *ml = a.ml_part + (((int64_t)b * a.n_split + split) * a.H + h0) * 2;
    float *op = a.o_part + (((int64_t)b * a.n_split + split) * a.H + h0) * a.r_lat;
    if (L < 1 || L > a.max_seq) {
        if (tid == 0 && split == 0 && hg == 0) atomicOr(a.status, kStatusLen);
        if (tid < HG) { ml[tid * 2] = -INFINITY; ml[tid * 2 + 1] = 0.f; }
        return;
    }
    const int j0 = split * a.chunk, j1 = min(L, j0 + a.chunk);
    if (j0 >= j1) {
        if (tid < HG) { ml[tid * 2] = -INFINITY; ml[tid * 2 + 1] = 0.f; }
        return;
    }
    // Latent columns this head group reads.
    const int lat_col = (h0 / a.heads_per_block_lat) * a.r_lat;
    for (int i = tid; i < HG * dq; i += 256) {
        int h = i / dq, c = i % dq;
        float v;
        if (c < a.r_lat) v = to_f32(((const T *)a.q_abs)[((int64_t)b * a.H + h0 + h) * a.r_lat + c]);
        else v = to_f32(((const T *)a.q_rope)[((int64_t)b * a.H + h0 + h) * a.d_rope + (c - a.r_lat)]);
        qs[i] = v;
    }
    __syncthreads();
    const T *lat = (const T *)a.lat + (int64_t)b * a.max_seq * a.lat_stride + lat_col;
    const T *rope = a.rope ? (const T *)a.rope + (int64_t)b * a.max_seq * a.rope_stride : nullptr;
    for (int j = j0 + warp; j < j1; j += 8) {
        float part[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) part[h] = 0.f;
        for (int c = lane; c < dq; c += 32) {
            float kv = c < a.r_lat ? to_f32(lat[(int64_t)j * a.lat_stride + c])
                                   : to_f32(rope[(int64_t)j * a.rope_stride + (c - a.r_lat)]);
#pragma unroll
            for (int h = 0; h < HG; ++h) part[h] = fmaf(qs[h * dq + c], kv, part[h]);
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            float v = part[h];
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) ss[h * a.chunk + (j - j0)] = v * a.scale_log2;
        }
    }
    __syncthreads();
    // Per-head max and exponentials (warp h handles head h, h < HG <= 8).
    __shared__ float mh[8], lh[8];
    if (warp < HG) {
        float m = -INFINITY;
        for (int j = lane; j < j1 - j0; j += 32) m = fmaxf(m, ss[warp * a.chunk + j]);
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float l = 0.f;
        for (int j = lane; j < j1 - j0; j += 32) {
            float p = exp2f(ss[warp * a.chunk + j] - m);
            ss[warp * a.chunk + j] = p;
            l += p;
        }
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) { mh[warp] = m; lh[warp] = l; }
    }
    __syncthreads();
    if (tid < HG) { ml[tid * 2] = mh[tid]; ml[tid * 2 + 1] = lh[tid]; }
    for (int c = tid; c < a.r_lat; c += 256) {
        float acc[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) acc[h] = 0.f;
        for (int j = j0; j < j1; ++j) {
            float cv = to_f32(lat[(int64_t)j * a.lat_stride + c]);
#pragma unroll
            for (int h = 0; h < HG; ++h) acc[h] = fmaf(ss[h * a.chunk + (j - j0)], cv, acc[h]);
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) op[(int64_t)h * a.r_lat + c] = acc[h];
    }
}

// o_lat[b, h] = sum_s 2^(m_s - m*) O_s / sum_s 2^(m_s - m*) l_s.
template <typename T>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeArgs a)
{
    const int h = blockIdx.x, b = blockIdx.y;
    __shared__ float w[64];
    __shared__ float inv_den;
    if (threadIdx.x == 0) {
        float m = -INFINITY;
        for (int s = 0; s < a.n_split; ++s)
            m = fmaxf(m, a.ml_part[(((int64_t)b * a.n_split + s) * a.H + h) * 2]);
        float den = 0.f;
        for (int s = 0; s < a.n_split; ++s) {
            const float *ml = a.ml_part + (((int64_t)b * a.n_split + s) * a.H + h) * 2;
            float ws = (ml[1] > 0.f) ? exp2f(ml[0] - m) : 0.f;
            w[s] = ws;
            den += ws * ml[1];
        }
        inv_den = den > 0.f ? 1.f / den : 0.f;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < a.r_lat; c += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < a.n_split; ++s)
            if (w[s] != 0.f)
                acc += w[s] * a.o_part[(((int64_t)b * a.n_split + s) * a.H + h) * a.r_lat + c];
        ((T *)a.o_lat)[((int64_t)b * a.H + h) * a.r_lat + c] = from_f32<T>(acc * inv_den);
    }
}

// ---------------------------------------------------------------------------
// Causal flash-style prefill.  Block = (64-query tile, head h, sequence b).
// Query i sits at position start_pos[b] + i and sees keys 0..that position.
// ---------------------------------------------------------------------------
constexpr int kPQ = 64;   // queries per block
constexpr int kPK = 32;   // keys per step

template <typename T>
__global__ void __launch_bounds__(256) prefill_kernel(PrefillArgs a)
{
    extern __shared__ float sm[];
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int dq = a.d_qk_nope + a.d_rope, dv = a.d_v;
    float *Qs = sm;                    // [kPQ][dq]
    float *Ks = Qs + kPQ * dq;         // [kPK][dq]
    float *Vs = Ks + kPK * dq;         // [kPK][dv]
    float *Ps = Vs + kPK * dv;         // [kPQ][kPK + 1]
    const int tid = threadIdx.x;
    const int sp = a.start_pos[b];
    const int i0 = qt * kPQ;
    const int nq = min(kPQ, a.S - i0);
    for (int idx = tid; idx < kPQ * dq; idx += 256) {
        int r = idx / dq, c = idx % dq;
        float v = 0.f;
        if (r < nq) {
            int64_t t = (int64_t)b * a.S + i0 + r;
            v = c < a.d_qk_nope ? to_f32(((const T *)a.q_nope)[(t * a.H + h) * a.d_qk_nope + c])
                                : to_f32(((const T *)a.q_rope)[(t * a.H + h) * a.d_rope + c - a.d_qk_nope]);
        }
        Qs[idx] = v;
    }
    const int r = tid / 4, sub = tid % 4;   // row r, quarter of the keys / value columns
    const int my_pos = sp + i0 + r;
    const int cols = (dv + 3) / 4;          // value columns owned by this thread
    float o[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int last_key = sp + i0 + nq - 1;
    for (int k0 = 0; k0 <= last_key; k0 += kPK) {
        __syncthreads();
        for (int idx = tid; idx < kPK * dq; idx += 256) {
            int j = idx / dq, c = idx % dq, key = k0 + j;
            float v = 0.f;
            if (key <= last_key) {
                if (c < a.d_qk_nope)
                    v = to_f32(((const T *)a.k)[(((int64_t)b * a.kv_rows + key) * a.H + h) * a.d_qk_nope + c]);
                else
                    v = to_f32(((const T *)a.rope)[((int64_t)b * a.max_seq + key) * a.rope_stride + c - a.d_qk_nope]);
            }
            Ks[idx] = v;
        }
        for (int idx = tid; idx < kPK * dv; idx += 256) {
            int j = idx / dv, c = idx % dv, key = k0 + j;
            Vs[idx] = key <= last_key
                          ? to_f32(((const T *)a.v)[(((int64_t)b * a.kv_rows + key) * a.H + h) * dv + c])
                          : 0.f;
        }
        __syncthreads();
        float s[8];
        float tmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int j = sub * 8 + u, key = k0 + j;
            float acc = 0.f;
            for (int c = 0; c < dq; ++c) acc = fmaf(Qs[r * dq + c], Ks[j * dq + c], acc);
            s[u] = (r < nq && key <= my_pos) ? acc * a.scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, s[u]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        float m_new = fmaxf(m, tmax);
        float corr = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float p = (s[u] == -INFINITY) ? 0.f : exp2f(s[u] - m_new);
            Ps[r * (kPK + 1) + sub * 8 + u] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        l = l * corr + psum;
        m = m_new;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (i >= cols) break;
            int c = sub * cols + i;
            if (c >= dv) break;
            float acc = o[i] * corr;
            for (int j = 0; j < kPK; ++j) acc = fmaf(Ps[r * (kPK + 1) + j], Vs[j * dv + c], acc);
            o[i] = acc;
        }
    }
    if (r < nq) {
        int64_t t = (int64_t)b * a.S + i0 + r;
        float inv = l > 0.f ? 1.f / l : 0.f;
        for (int i = 0; i < cols; ++i) {
            int c = sub * cols + i;
            if (c < dv) ((T *)a.o)[(t * a.H + h) * dv + c] = from_f32<T>(o[i] * inv);
        }
    }
}

template <typename T>
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s)
{
    dim3 grid((a.N + kTile - 1) / kTile, (a.M + kTile - 1) / kTile, a.batch);
    if (a.trans_b) gemm_simt_kernel<T, true><<<grid, 256, 0, s>>>(a);
    else gemm_simt_kernel<T, false><<<grid, 256, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

template <typename T, int HG>
cudaError_t launch_decode_hg(const DecodeArgs &a, cudaStream_t s)
{
    size_t smem = sizeof(float) * (size_t)HG * (a.r_lat + a.d_rope + a.chunk);
    static std::atomic<int> smem_dev{-1};
    static int smem_set = 0;
    if ((int)smem > smem_set) smem_dev = -1;  // the chunk size can grow the request
    cudaError_t e = smem_limit_once(smem_dev, (const void *)decode_partial_kernel<T, HG>, (int)smem);
    if (e == cudaSuccess && (int)smem > smem_set) smem_set = (int)smem;
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_split, a.B, a.H / HG);
    profile_begin(MLA_PROFILE_DECODE_ATTENTION, s);
    decode_partial_kernel<T, HG><<<grid, 256, smem, s>>>(a);
    profile_end(MLA_PROFILE_DECODE_ATTENTION, s);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    decode_combine_kernel<T><<<dim3(a.H, a.B), 256, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s)
{
    int hpb = a.heads_per_block_lat;
    if (hpb % 8 == 0) return launch_decode_hg<T, 8>(a, s);
    if (hpb % 4 == 0) return launch_decode_hg<T, 4>(a, s);
    if (hpb % 2 == 0) return launch_decode_hg<T, 2>(a, s);
    return launch_decode_hg<T, 1>(a, s);
}

template <typename T>
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s)
{
    int dq = a.d_qk_nope + a.d_rope;
    size_t smem = sizeof(float) * ((size_t)kPQ * dq + (size_t)kPK * dq + (size_t)kPK * a.d_v +
                                   (size_t)kPQ * (kPK + 1));
    static std::atomic<int> smem_dev{-1};
    static int smem_set = 0;
    if ((int)smem > smem_set) smem_dev = -1;  // the head widths can grow the request
    cudaError_t e = smem_limit_once(smem_dev, (const void *)prefill_kernel<T>, (int)smem);
    if (e == cudaSuccess && (int)smem > smem_set) smem_set = (int)smem;
    if (e != cudaSuccess) return e;
    dim3 grid((a.S + kPQ - 1) / kPQ, a.H, a.B);
    profile_begin(MLA_PROFILE_PREFILL_ATTENTION, s);
    prefill_kernel<T><<<grid, 256, smem, s>>>(a);
    profile_end(MLA_PROFILE_PREFILL_ATTENTION, s);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_simt(int dtype, const GemmArgs &a, cudaStream_t s)
{
    if (a.M == 0 || a.N == 0 || a.batch == 0) return cudaSuccess;
    return dtype == MLA_DTYPE_F32 ? launch_gemm<float>(a, s) : launch_gemm<bf16>(a, s);
}

cudaError_t decode_simt(const DecodeArgs &a, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    return a.dtype == MLA_DTYPE_F32 ? launch_decode<float>(a, s) : launch_decode<bf16>(a, s);
}

cudaError_t prefill_simt(const PrefillArgs &a, cudaStream_t s)
{
    if (a.B == 0 || a.S == 0) return cudaSuccess;
    return a.dtype == MLA_DTYPE_F32 ? launch_prefill<float>(a, s) : launch_prefill<bf16>(a, s);
}

}  // namespace mla

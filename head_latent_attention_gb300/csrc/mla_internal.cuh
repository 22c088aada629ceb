// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "mla.h"

struct mla_handle {
    mla_config cfg;      // the layer this handle computes (a shard's own part for MLRA shards)
    int shard, n_shards; // MLRA sub-head tensor parallelism: this handle's part (0 of 1 otherwise)
    int device;
    int num_sms;
    int rope_dim;        // rotated width: d_rope (decoupled), d_nope (small), 0 (MLRA)
    float2 *rope_table;  // [max_seq, rope_dim / 2] (cos, sin) of pos * base^(-2i/rope_dim)
    uint32_t *status;    // device status word for calls without a workspace
    int decode_clusters; // co-resident 2-CTA clusters of the tensor-core decode (0: not used)
};

namespace mla {

// Launch bookkeeping and the optional timing hook (api.cu).
void note_launch(int n = 1);
// Give-up limit (SM clock cycles) of the projection GEMM's bounded waits:
// the default (about one second) unless mla_set_wait_limit changed it.
long long gemm_wait_cycles();
long long ptx_default_wait_cycles();  // ptx::kWaitCycles, for host code without ptx.cuh
void profile_begin(int which, cudaStream_t s);
void profile_end(int which, cudaStream_t s);

// Raise a kernel's dynamic shared-memory limit once per device (call site
// keeps `set_on_device`, initially -1): the attribute need not be set per
// launch, and setting it only once keeps launches cheap and capturable.
// Threads that race on the first launch both set the same attribute, which
// is harmless; the atomic keeps the cache itself well defined.
inline cudaError_t smem_limit_once(std::atomic<int> &set_on_device, const void *func, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (set_on_device.load(std::memory_order_relaxed) == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) set_on_device.store(dev, std::memory_order_relaxed);
    return e;
}

// Launch of a tensor-core-path kernel with programmatic stream serialisation
// (and, when cluster_x > 1, a cluster of cluster_x CTAs along x): the kernel
// may begin while its predecessor in the stream finishes, so every kernel
// launched this way calls ptx::pdl_wait() before touching memory that other
// kernels write.  Setting the environment variable MLA_PDL=0 before the first
// launch turns the attribute off (plain stream order).
bool pdl_enabled();
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             int cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Workspace status bits (mirrors the values documented in mla.h).
constexpr uint32_t kStatusPos = 1u;
constexpr uint32_t kStatusSeq = 2u;
constexpr uint32_t kStatusLen = 4u;
constexpr uint32_t kStatusTimeout = 8u;
constexpr uint32_t kStatusF16Range = 16u;  // an fp16 operand of prefill was saturated

// Workspace: the first 256 bytes hold the status word; call scratch follows.
constexpr size_t kWsHeader = 256;

enum RopeMode { kRopeNone = 0, kRopeInterleaved = 1, kRopeHalf = 2 };

// Element types the kernels are instantiated for.
using bf16 = __nv_bfloat16;

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// Output stage of a projection GEMM C[M, N] = A[M, K] B^T.
//  - Row destination: row m goes to out + m * ldc, or, when row_seq is set, to
//    cache row (row_seq[m], row_pos[m]) = out + (seq * seq_rows + pos) * ldc
//    (rows whose sequence or position is out of range are skipped and flagged).
//  - Optional RoPE on every column (groups of rope_dim columns; tiles never
//    straddle a group): the position of row m is rope_pos[m], or m when
//    rope_pos is null.
struct Epilogue {
    void *out = nullptr;
    int64_t ldc = 0;
    int64_t batch_stride = 0;  // elements between batch entries of out
    const int32_t *row_seq = nullptr;
    const int32_t *row_pos = nullptr;
    int64_t seq_rows = 0;
    int max_batch = 0;
    int max_seq = 0;
    int rope_mode = kRopeNone;
    int rope_dim = 0;
    const float2 *rope_table = nullptr;
    const int32_t *rope_pos = nullptr;
    uint32_t *status = nullptr;  // device status word (index flags, timeouts)
    bool out_f16 = false;        // tensor-core path: store fp16 instead of bfloat16
    // Rows in use: with range_start set, only rows m < range_start[z] +
    // range_len of batch entry z are needed (the cache rows a prefill's
    // queries can see; the rest of a sequence's rows may hold anything).  The
    // tensor-core GEMM skips whole row tiles past that limit (single-segment
    // products) and checks only rows below it against fp16's range.
    const int32_t *range_start = nullptr;
    int range_len = 0;
};

// Row-major 2-D view of a tensor: rows x cols elements, row stride ld.
struct Mat2D {
    const void *ptr = nullptr;
    int64_t rows = 0, cols = 0, ld = 0;
};

// C[M, N] = A[M, K] B^T per batch entry z.  Batch entry z reads A from the
// block at (z * a_row_batch, z * a_col_batch) of the A view and B from
// (z * b_row_batch, z * b_col_batch) of the B view.  B holds element (n, k)
// at (row n, col k) (K contiguous, "K-major") unless trans_b, in which case
// at (row k, col n) (N contiguous, "MN-major").
// One column segment of a grouped product: output columns [n0, n0 + N) of
// the concatenated result take their weights from B ([N, K] row-major) and
// their epilogue from epi.  Tensor-core path only; widths multiple of 64.
struct GemmSegment {
    Mat2D B;
    Epilogue epi;
    int N = 0;
};
constexpr int kMaxSeg = 3;

struct GemmArgs {
    Mat2D A;
    int64_t a_row_batch = 0, a_col_batch = 0;
    Mat2D B;
    int64_t b_row_batch = 0, b_col_batch = 0;
    bool trans_b = false;
    int M = 0, N = 0, K = 0, batch = 1;
    Epilogue epi;
    float *split_ws = nullptr;  // tensor-core split-K partials (gemm_tc_workspace bytes)
    // nseg > 0: one launch computes A [B_0 | B_1 | ...]^T over the segments
    // below (same A, K and split workspace; B, N and epi above are unused).
    // Decode-sized projections that share their input stream their weights
    // as one GEMM this way.
    int nseg = 0;
    GemmSegment seg[kMaxSeg];
};

struct GemmPlan {
    int bn, splits, kb_per_split;
};

// CUDA-core kernels (the float32 path).
cudaError_t gemm_simt(int dtype, const GemmArgs &a, cudaStream_t s);

// Tensor-core (tcgen05) projection GEMM for bfloat16.  Requirements checked by
// gemm_tc_supported(): 16-byte aligned views and row strides, N % 32 == 0,
// batch offsets on 16-byte boundaries, output rows 16-byte aligned.
bool gemm_tc_supported(const GemmArgs &a);
GemmPlan gemm_tc_plan(const GemmArgs &a, int num_sms);
size_t gemm_tc_workspace(const GemmArgs &a, int num_sms);  // split-K scratch bytes (0: none)
cudaError_t gemm_tc(const GemmArgs &a, int num_sms, cudaStream_t s);

struct DecodeArgs {
    int dtype;
    int B, H, r_lat, d_rope;   // r_lat: latent width one head attends over
    int heads_per_block_lat;   // heads sharing one latent block (H for MLA, H/L for MLRA)
    const void *q_abs;         // [B, H, r_lat]
    const void *q_rope;        // [B, H, d_rope] or null
    const void *lat;           // cache latent rows
    int64_t lat_stride;
    const void *rope;          // cache rope rows or null
    int64_t rope_stride;
    int max_seq;
    const int32_t *seq_lens;   // device [B]
    float scale_log2;          // softmax scale * log2(e)
    float *o_part;             // [B, n_split, H, r_lat]
    float *ml_part;            // [B, n_split, H, 2] (running max in log2 units, sum)
    int n_split, chunk;
    void *o_lat;               // [B, H, r_lat] (dtype)
    uint32_t *status;
};
cudaError_t decode_simt(const DecodeArgs &a, cudaStream_t s);

// Split-KV schedule shared by the decode kernels, in the workspace.  The
// concatenation of all sequences' keys is cut into n contiguous ranges, one
// per CTA or cluster; a range splits into one segment per sequence it
// touches, and the partial result of range c for sequence b goes to slot
// c + b (unique, since ranges and sequences both advance monotonically):
// the latent average over the segment's keys, normalised by its own row sum
// and rounded to bfloat16 like a whole sequence's result, with its reference
// max (log2 units) and row sum in fp32.
struct DecodeSched {
    int *prefix;       // [B + 1] prefix sums of the valid lengths (invalid ones count 0)
    int *chunk;        // [1] keys per range of the uniform split
    int *range_start;  // [n + 1] first key of each range; [n] = total keys
    int *range_b0;     // [n] first sequence of each range (B when empty)
    int *seq_fc;       // [B] first range covering each sequence (-1: empty or invalid)
    int *seq_lc;       // [B] last range covering each sequence
};
// Tensor-core split-KV decode (decode_tc.cu): DECOUPLED, bfloat16, H <= 128,
// r_kv == 512, d_rope == 64.
struct DecodeTcArgs {
    int B, H, r_kv, d_rope, max_batch, max_seq, n_clusters;
    const void *q_abs;        // [B, kQChunks, kQRows, 8] (head-interleaved 16-byte chunks, see kQChunks)
    const void *q_rope;       // [B, H, d_rope]
    const void *lat;          // cache latent rows
    int64_t lat_stride;
    const void *rope;         // cache rope rows
    int64_t rope_stride;
    const int32_t *seq_lens;  // device [B]
    DecodeSched sc;           // written by decode_schedule (n = n_clusters)
    float scale_log2;
    void *o_lat;              // [B, H, r_kv] bf16
    bf16 *o_part;             // [n_clusters + B, H, r_kv] normalised partial averages
    float *ml_part;           // [n_clusters + B, H, 2]
    uint32_t *status;
};
int decode_tc_max_clusters();

size_t decode_sched_bytes(int B, int n);
DecodeSched decode_sched_at(void *base, int B, int n);
// seg_cost == 0: uniform ranges of `chunk` keys.  seg_cost > 0: ranges of
// equal estimated cost, a sequence start counting as seg_cost extra keys
// (the per-segment overhead of the kernel), which also moves range starts
// that fall within seg_cost keys after a sequence start onto that start.
// decode_schedule runs right before the absorption kernel, which lets the
// split-KV kernel start only after its own wait for the scheduler (the decode
// kernels read the schedule before their own dependency wait; see
// decode_tc.cu), so callers launch it first.
void decode_schedule(const int32_t *seq_lens, int B, int max_seq, int n_ranges, int seg_cost, const DecodeSched &sc,
                     uint32_t *status, cudaStream_t s);
// Log-sum-exp merge of the partials of split sequences into o_lat.
void decode_combine(const DecodeSched &sc, int B, int H, int r_lat, const bf16 *o_part, const float *ml_part,
                    void *o_lat, cudaStream_t s);

// Absorbed decode queries (absorb_tc.cu): q_abs[b, h] = W_UK,h^T q_nope[b, h]
// with W_UK,h = rows [128 h, 128 h + 128) of W_UK viewed as [H * 128, r_lat].
// bfloat16, d_nope == 128, r_lat in {256, 512}.
// The absorbed decode query of the tensor-core MLA decode, head-interleaved:
// per sequence, kQChunks 16-byte chunks (8 latent columns each) of kQRows
// head rows, chunk c of head h at ((b * kQChunks + c) * kQRows + h) * 16
// bytes, so that a warp's load of one chunk for 32 heads is 512 contiguous
// bytes.  Rows of heads >= H are not written.
constexpr int kQChunks = 64;
constexpr int kQRows = 128;

struct AbsorbArgs {
    int B, H, r_lat, d_nope;
    const void *q_nope;  // [B, H * 128]
    const void *W_UK;
    void *q_abs;         // [B, H, r_lat], or the interleaved layout above (r_lat = 512)
    bool interleave;
    uint32_t *status;
};
bool absorb_supported(int r_lat, int d_nope);
cudaError_t absorb(const AbsorbArgs &a, cudaStream_t s);

// Merge of the split-KV partials fused with the value up-projection
// (finish_tc.cu): o[b, h] = W_UV,h o_lat[b, h] with o_lat merged on chip from
// the partials decode_tc / mlra_tc leave (same slot layout as decode_combine).
// bfloat16, d_v == 128, r_lat in {256, 512}; W_UV,h = rows [128 h, 128 h + 128)
// of W_UV viewed as [H * 128, r_lat].
struct FinishArgs {
    int B, H, r_lat, d_v;
    const int *seq_fc, *seq_lc;  // ranges covering each sequence (DecodeSched)
    const bf16 *o_part;  // [slots, H, r_lat] normalised partial averages
    const float *ml_part;  // [slots, H, 2] (max in log2 units, row sum)
    const void *o_lat;  // [B, H, r_lat] (single-range sequences)
    const void *W_UV;
    void *o;            // [B, H, d_v]
    uint32_t *status;
};
bool decode_finish_supported(int r_lat, int d_v);
cudaError_t decode_finish(const FinishArgs &a, cudaStream_t s);

// Tensor-core split-KV decode for MLRA (mlra_tc.cu): bfloat16, latent blocks
// of 256 columns, at most 16 heads per block, no rope.
struct MlraTcArgs {
    int B, H, L, r_kv, max_batch, max_seq, n_ctas;
    const void *q_abs;  // [B, H, 256] (head h reads block h / (H / L))
    const void *lat;    // [max_batch * max_seq, lat_stride]
    int64_t lat_stride;
    const int32_t *seq_lens;
    int *prefix, *chunk;  // workspace: [B + 1], [1]
    float scale_log2;
    void *o_lat;          // [B, H, 256]
    bf16 *o_part;         // [(n_ctas + B), H, 256] normalised partial averages
    float *ml_part;       // [(n_ctas + B), H, 2]
    uint32_t *status;
};
bool mlra_tc_supported(int H, int L, int r_kv, int d_rope);
int mlra_tc_ctas();
cudaError_t mlra_tc(const MlraTcArgs &a, cudaStream_t s);
bool decode_tc_supported(int H, int r_kv, int d_rope);
cudaError_t decode_tc(const DecodeTcArgs &a, cudaStream_t s);

// Tensor-core causal prefill (prefill_tc.cu): bfloat16, (d_nope, d_rope, d_v)
// in {(128, 64, 128), (64, 0, 64), (128, 0, 128)}.
struct PrefillTcArgs {
    int B, S, H, d_nope, d_rope, d_v, max_batch, max_seq;
    int64_t kv_rows;
    const void *q_nope, *q_rope;  // [B*S, H*d_nope], [B*S, H*d_rope]
    const void *k, *v;            // fp16 workspace [B*kv_rows, Hkv*d_nope], [B*kv_rows, Hkv*d_v]
    int kv_group = 1;             // query heads per key/value head (Hkv = H / kv_group)
    const void *rope;             // rope cache rows (decoupled, bfloat16)
    int64_t rope_stride;
    void *k_rope16;               // fp16 workspace copy of the rope keys [B*kv_rows, 64]
    const int32_t *start_pos;     // device [B]
    float scale_log2;
    void *o;                      // [B, S, H, d_v]
    uint32_t *status;
};
bool prefill_tc_supported(int d_nope, int d_rope, int d_v);
// start_pos[b] = seq_lens[b] - 1 for a decode step that runs the prefill
// kernels (small-model form); -1 (zero output) and a flag for bad lengths.
cudaError_t positions_from_lengths(const int32_t *seq_lens, int B, int max_seq, int32_t *start_pos,
                                   uint32_t *status, cudaStream_t s);
cudaError_t prefill_tc(const PrefillTcArgs &a, cudaStream_t s);

struct PrefillArgs {
    int dtype;
    int B, S, H, d_qk_nope, d_rope, d_v;
    const void *q_nope;        // [B, S, H, d_qk_nope]
    const void *q_rope;        // [B, S, H, d_rope] or null
    const void *k;             // [B, kv_rows, H, d_qk_nope]
    const void *v;             // [B, kv_rows, H, d_v]
    int64_t kv_rows;
    const void *rope;          // cache rope rows (decoupled) or null
    int64_t rope_stride;
    int max_seq;
    const int32_t *start_pos;  // device [B]
    float scale_log2;
    void *o;                   // [B, S, H, d_v]
};
cudaError_t prefill_simt(const PrefillArgs &a, cudaStream_t s);

}  // namespace mla

// Output projection for callers that cannot allocate device memory.
//
// mla_out_proj needs a caller-provided workspace when the token count is small
// (the decode step), because its tensor-core GEMM then splits the reduction
// dimension and keeps fp32 partial sums in scratch memory.  Some callers have
// no way to provide that memory: a plugin inside an inference runtime that has
// reserved all device memory for its own pool and hands its plugins no
// scratch, or code on a latency-critical path where cudaMalloc's implicit
// device synchronisation is not acceptable.  mla_out_proj_static computes the
// same projection with its scratch in a fixed buffer that belongs to the
// library itself, so it allocates nothing.
#include <atomic>

#include "mla_internal.cuh"

namespace {

// Split-K partial sums of one call.  Every GPU that loads the library holds
// this buffer until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device.  In host code the symbol
// names a host-side stand-in, not device memory, so the address is looked up
// with cudaGetSymbolAddress once per device (with that device current).
// Threads that make their first call on a device at the same time may both
// look it up; they store the same address, and the atomics keep the cache
// itself well defined.
constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices] = {};

cudaError_t static_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" mla_status mla_out_proj_static(mla_handle *h, const mla_weights *w, const void *o, int64_t T,
                                          void *y, void *stream)
{
    if (!h || !w || T < 0) return MLA_ERR_INVALID_ARG;
    if (T == 0) return MLA_OK;
    const mla_config &c = h->cfg;
    if (!o || !y || !w->W_O || T > INT32_MAX) return MLA_ERR_INVALID_ARG;
    if (c.dtype == MLA_DTYPE_BF16) {
        for (const void *p : {o, (const void *)y, w->W_O})
            if ((uintptr_t)p & 15u) return MLA_ERR_INVALID_ARG;
    }
    const int K = c.n_heads * c.d_v;
    mla::GemmArgs g;
    g.A = mla::Mat2D{o, T, K, K};
    g.B = mla::Mat2D{w->W_O, c.d_model, K, K};
    g.M = (int)T;
    g.N = c.d_model;
    g.K = K;
    g.epi.out = y;
    g.epi.ldc = c.d_model;
    g.epi.status = h->status;
    cudaStream_t s = (cudaStream_t)stream;
    if (c.dtype != MLA_DTYPE_BF16)
        return mla::gemm_simt(MLA_DTYPE_F32, g, s) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
    if (!mla::gemm_tc_supported(g)) return MLA_ERR_UNSUPPORTED;
    // The partial sums of this call must fit the fixed buffer.
    if (mla::gemm_tc_workspace(g, h->num_sms) > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (static_scratch(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
    // Every split writes its whole slice of the partial sums before the
    // reduction reads it, so nothing in the buffer needs clearing.
    g.split_ws = (float *)scratch;
    return mla::gemm_tc(g, h->num_sms, s) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

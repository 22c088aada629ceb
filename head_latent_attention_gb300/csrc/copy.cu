// Stream-ordered copy between any two device-accessible buffers, done by the
// SMs: device memory, or pinned host memory, which a kernel reaches over the
// host link through the same pointer under unified addressing.  Launched
// like the library's other kernels (programmatic dependent launch), it lets
// a step's input staging and result read-back chain with the kernels around
// them instead of waiting for a copy engine on each side.
#include <algorithm>

#include "mla_internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

// 16-byte vectors over the aligned body, bytes for the rest.  The first
// kernel of the next call may be scheduled at once; this one waits for the
// previous kernel (which may still read dst or write src) before touching
// memory.
__global__ void __launch_bounds__(256) copy_kernel(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src,
                                                   size_t bytes)
{
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nthr = (size_t)gridDim.x * blockDim.x;
    const bool vec = (((uintptr_t)dst | (uintptr_t)src) & 15u) == 0;
    const size_t nv = vec ? bytes / 16 : 0;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    for (size_t i = tid; i < nv; i += nthr) d4[i] = s4[i];
    for (size_t i = nv * 16 + tid; i < bytes; i += nthr) dst[i] = src[i];
}

// The pointer through which a kernel reaches p, or null when it cannot
// (pageable host memory that was not registered, or an unknown pointer).
void *device_view(void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // the failed query leaves an error status behind: clear it
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost)
        return a.devicePointer;
    return nullptr;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (bytes == 0) return MLA_OK;
    if (!dst || !src) return MLA_ERR_INVALID_ARG;
    uint8_t *d = (uint8_t *)device_view(dst);
    const uint8_t *s = (const uint8_t *)device_view(const_cast<void *>(src));
    if (!d || !s) return MLA_ERR_INVALID_ARG;
    if ((d < s + bytes) && (s < d + bytes)) return MLA_ERR_INVALID_ARG;  // overlapping ranges
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MLA_ERR_CUDA;
    const size_t work = (bytes + 15) / 16;
    const unsigned blocks = (unsigned)std::max<size_t>(1, std::min<size_t>((size_t)sms * 2, (work + 255) / 256));
    const cudaError_t e = launch_ex(copy_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, 1, d, s, bytes);
    note_launch();
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

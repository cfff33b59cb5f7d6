// noalloc.cu -- rra_sparse_encode_noalloc: the sparse encoder for callers
// that cannot allocate device memory.
//
// rra_sparse_encode needs scratch (one 32-bit count per 1024-element chunk,
// and one total per 4096 chunks) and takes it from a per-device workspace that
// grows with cudaMalloc.  Some callers cannot allow that: processes whose
// device memory is handed out by their own allocator or budgeted up front,
// latency-critical loops in which an allocation's implicit device
// synchronisation is not acceptable, and libraries that must not call into
// the CUDA allocator behind their host framework's back.  This entry point
// uses a fixed scratch array that lives in the library image instead: a
// file-scope __device__ array of kNoallocScratchWords words (about 1 MiB),
// present on every GPU that loads the library until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "rra.h"
#include "rra_device.cuh"
#include "rra_kernels.h"

namespace {

// one word per 1024-element chunk of the largest input, then one per 4096
// chunks
constexpr long long kNoallocChunks = (long long)RRA_NOALLOC_MAX_COUNT / 1024;
constexpr long long kNoallocScratchWords = kNoallocChunks + (kNoallocChunks + 4095) / 4096;

// The scratch itself.  In host code this name is only a host-side stand-in,
// not a device address: the address a kernel may use comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoallocScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device, on the first call with that device current.  The address
// stays valid for the life of the device's primary context; after a
// cudaDeviceReset the entry point must not be called again in this process.
cudaError_t scratch_for_current_device(uint32_t **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_ptr[dev] = static_cast<uint32_t *>(p);
    }
    *out = g_ptr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" rra_status rra_sparse_encode_noalloc(const void *x, size_t n, rra_dtype dtype,
                                                float threshold, uint32_t *hdr, void *vals,
                                                int32_t *idx, void *stream)
{
    if (!x || n == 0 || !hdr || !vals || !idx ||
        !(dtype == RRA_F32 || dtype == RRA_F16 || dtype == RRA_BF16) ||
        !(threshold >= 0.0f && threshold < 1.0f))
        return RRA_ERR_INVALID;
    if (n > (size_t)RRA_NOALLOC_MAX_COUNT ||
        rra::sparse_encode_scratch_words((long long)n) > kNoallocScratchWords)
        return RRA_ERR_INVALID; // beyond the fixed scratch: use rra_sparse_encode
    uint32_t *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess)
        return RRA_ERR_CUDA;
    // every count and segment word is written in a call before that call
    // reads it, so nothing needs clearing, before or between calls
    return rra::launch_sparse_encode(x, (long long)n, dtype, 1.0 - (double)threshold, hdr, vals,
                                     idx, scratch,
                                     reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RRA_OK
               : RRA_ERR_CUDA;
}

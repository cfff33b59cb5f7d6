// ring_sparse.cu -- instantiations of the fused ring kernel for the
// kCodecSparse wire format(s): every input dtype and slice width, the
// bulk-copy path with one or several ranks per warp, and the generic path;
// its own translation unit so that the library compiles in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_sparse(int codec, int in_t, bool fast, int groups, bool one)
{
    if (codec == kCodecSparse && groups == 1) {
        if (in_t == kF32) {
            if (!fast)
                return (const void *)ring_kernel<kCodecSparse, kF32, false, 1, false>;
            return one ? (const void *)ring_kernel<kCodecSparse, kF32, true, 1, true>
                       : (const void *)ring_kernel<kCodecSparse, kF32, true, 1, false>;
        }
        if (in_t == kF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecSparse, kF16, false, 1, false>;
            return one ? (const void *)ring_kernel<kCodecSparse, kF16, true, 1, true>
                       : (const void *)ring_kernel<kCodecSparse, kF16, true, 1, false>;
        }
        if (in_t == kBF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecSparse, kBF16, false, 1, false>;
            return one ? (const void *)ring_kernel<kCodecSparse, kBF16, true, 1, true>
                       : (const void *)ring_kernel<kCodecSparse, kBF16, true, 1, false>;
        }
    }
    return nullptr;
}

} // namespace rra

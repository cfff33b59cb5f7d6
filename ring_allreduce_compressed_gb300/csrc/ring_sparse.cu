// ring_sparse.cu -- instantiations of the fused ring kernel for the
// kCodecSparse wire format(s); compiled as its own translation unit so
// that the library builds in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_sparse(int codec, int in_t, bool fast)
{
    if (codec == kCodecSparse) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecSparse, kF32, true>
                        : (const void *)ring_kernel<kCodecSparse, kF32, false>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecSparse, kF16, true>
                        : (const void *)ring_kernel<kCodecSparse, kF16, false>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecSparse, kBF16, true>
                        : (const void *)ring_kernel<kCodecSparse, kBF16, false>;
    }
    return nullptr;
}

} // namespace rra

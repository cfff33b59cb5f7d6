// ring_sparse.cu -- instantiations of the fused ring kernel for the
// kCodecSparse wire format(s), every input dtype, the bulk-copy and the
// generic input path, and the supported slice widths; its own translation unit
// so that the library compiles in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_sparse(int codec, int in_t, bool fast, int groups)
{
    if (codec == kCodecSparse && groups == 1) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecSparse, kF32, true, 1>
                        : (const void *)ring_kernel<kCodecSparse, kF32, false, 1>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecSparse, kF16, true, 1>
                        : (const void *)ring_kernel<kCodecSparse, kF16, false, 1>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecSparse, kBF16, true, 1>
                        : (const void *)ring_kernel<kCodecSparse, kBF16, false, 1>;
    }
    return nullptr;
}

} // namespace rra

// ring_none.cu -- instantiations of the fused ring kernel for the
// kCodecNone wire format(s); compiled as its own translation unit so
// that the library builds in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_none(int codec, int in_t, bool fast)
{
    if (codec == kCodecNone) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecNone, kF32, true>
                        : (const void *)ring_kernel<kCodecNone, kF32, false>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecNone, kF16, true>
                        : (const void *)ring_kernel<kCodecNone, kF16, false>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecNone, kBF16, true>
                        : (const void *)ring_kernel<kCodecNone, kBF16, false>;
    }
    return nullptr;
}

} // namespace rra

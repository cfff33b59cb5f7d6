// ring_bfp.cu -- instantiations of the fused ring kernel for the
// kCodecBfp8, kCodecBfp4 wire format(s); compiled as its own translation unit so
// that the library builds in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_bfp(int codec, int in_t, bool fast)
{
    if (codec == kCodecBfp8) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF32, true>
                        : (const void *)ring_kernel<kCodecBfp8, kF32, false>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF16, true>
                        : (const void *)ring_kernel<kCodecBfp8, kF16, false>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kBF16, true>
                        : (const void *)ring_kernel<kCodecBfp8, kBF16, false>;
    }
    if (codec == kCodecBfp4) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF32, true>
                        : (const void *)ring_kernel<kCodecBfp4, kF32, false>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF16, true>
                        : (const void *)ring_kernel<kCodecBfp4, kF16, false>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kBF16, true>
                        : (const void *)ring_kernel<kCodecBfp4, kBF16, false>;
    }
    return nullptr;
}

} // namespace rra

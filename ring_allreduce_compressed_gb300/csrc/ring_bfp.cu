// ring_bfp.cu -- instantiations of the fused ring kernel for the
// kCodecBfp8, kCodecBfp4 wire format(s), every input dtype, the bulk-copy and the
// generic input path, and the supported slice widths; its own translation unit
// so that the library compiles in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_bfp(int codec, int in_t, bool fast, int groups)
{
    if (codec == kCodecBfp8 && groups == 1) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF32, true, 1>
                        : (const void *)ring_kernel<kCodecBfp8, kF32, false, 1>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF16, true, 1>
                        : (const void *)ring_kernel<kCodecBfp8, kF16, false, 1>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kBF16, true, 1>
                        : (const void *)ring_kernel<kCodecBfp8, kBF16, false, 1>;
    }
    if (codec == kCodecBfp8 && groups == 2) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF32, true, 2>
                        : (const void *)ring_kernel<kCodecBfp8, kF32, false, 2>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF16, true, 2>
                        : (const void *)ring_kernel<kCodecBfp8, kF16, false, 2>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kBF16, true, 2>
                        : (const void *)ring_kernel<kCodecBfp8, kBF16, false, 2>;
    }
    if (codec == kCodecBfp8 && groups == 4) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF32, true, 4>
                        : (const void *)ring_kernel<kCodecBfp8, kF32, false, 4>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kF16, true, 4>
                        : (const void *)ring_kernel<kCodecBfp8, kF16, false, 4>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp8, kBF16, true, 4>
                        : (const void *)ring_kernel<kCodecBfp8, kBF16, false, 4>;
    }
    if (codec == kCodecBfp4 && groups == 1) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF32, true, 1>
                        : (const void *)ring_kernel<kCodecBfp4, kF32, false, 1>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF16, true, 1>
                        : (const void *)ring_kernel<kCodecBfp4, kF16, false, 1>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kBF16, true, 1>
                        : (const void *)ring_kernel<kCodecBfp4, kBF16, false, 1>;
    }
    if (codec == kCodecBfp4 && groups == 2) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF32, true, 2>
                        : (const void *)ring_kernel<kCodecBfp4, kF32, false, 2>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF16, true, 2>
                        : (const void *)ring_kernel<kCodecBfp4, kF16, false, 2>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kBF16, true, 2>
                        : (const void *)ring_kernel<kCodecBfp4, kBF16, false, 2>;
    }
    if (codec == kCodecBfp4 && groups == 4) {
        if (in_t == kF32)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF32, true, 4>
                        : (const void *)ring_kernel<kCodecBfp4, kF32, false, 4>;
        if (in_t == kF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kF16, true, 4>
                        : (const void *)ring_kernel<kCodecBfp4, kF16, false, 4>;
        if (in_t == kBF16)
            return fast ? (const void *)ring_kernel<kCodecBfp4, kBF16, true, 4>
                        : (const void *)ring_kernel<kCodecBfp4, kBF16, false, 4>;
    }
    return nullptr;
}

} // namespace rra

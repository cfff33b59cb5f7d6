// ring_none.cu -- instantiations of the fused ring kernel for the
// kCodecNone wire format: every input dtype and slice width, the
// bulk-copy path with one or several ranks per warp, and the generic path;
// its own translation unit so that the library compiles in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_none(int codec, int in_t, bool fast, int groups, bool one)
{
    if (codec == kCodecNone && groups == 1) {
        if (in_t == kF32) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF32, false, 1, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF32, true, 1, true>
                       : (const void *)ring_kernel<kCodecNone, kF32, true, 1, false>;
        }
        if (in_t == kF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF16, false, 1, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF16, true, 1, true>
                       : (const void *)ring_kernel<kCodecNone, kF16, true, 1, false>;
        }
        if (in_t == kBF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kBF16, false, 1, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kBF16, true, 1, true>
                       : (const void *)ring_kernel<kCodecNone, kBF16, true, 1, false>;
        }
    }
    if (codec == kCodecNone && groups == 2) {
        if (in_t == kF32) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF32, false, 2, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF32, true, 2, true>
                       : (const void *)ring_kernel<kCodecNone, kF32, true, 2, false>;
        }
        if (in_t == kF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF16, false, 2, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF16, true, 2, true>
                       : (const void *)ring_kernel<kCodecNone, kF16, true, 2, false>;
        }
        if (in_t == kBF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kBF16, false, 2, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kBF16, true, 2, true>
                       : (const void *)ring_kernel<kCodecNone, kBF16, true, 2, false>;
        }
    }
    if (codec == kCodecNone && groups == 4) {
        if (in_t == kF32) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF32, false, 4, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF32, true, 4, true>
                       : (const void *)ring_kernel<kCodecNone, kF32, true, 4, false>;
        }
        if (in_t == kF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF16, false, 4, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF16, true, 4, true>
                       : (const void *)ring_kernel<kCodecNone, kF16, true, 4, false>;
        }
        if (in_t == kBF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kBF16, false, 4, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kBF16, true, 4, true>
                       : (const void *)ring_kernel<kCodecNone, kBF16, true, 4, false>;
        }
    }
    if (codec == kCodecNone && groups == 8) {
        if (in_t == kF32) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF32, false, 8, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF32, true, 8, true>
                       : (const void *)ring_kernel<kCodecNone, kF32, true, 8, false>;
        }
        if (in_t == kF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kF16, false, 8, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kF16, true, 8, true>
                       : (const void *)ring_kernel<kCodecNone, kF16, true, 8, false>;
        }
        if (in_t == kBF16) {
            if (!fast)
                return (const void *)ring_kernel<kCodecNone, kBF16, false, 8, false>;
            return one ? (const void *)ring_kernel<kCodecNone, kBF16, true, 8, true>
                       : (const void *)ring_kernel<kCodecNone, kBF16, true, 8, false>;
        }
    }
    return nullptr;
}

} // namespace rra

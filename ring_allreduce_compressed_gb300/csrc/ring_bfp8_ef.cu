// ring_bfp8_ef.cu -- instantiations of the fused ring kernel for the block-FP8
// wire format with error feedback: every input kind and slice width, the
// staged path in each rank-to-warp mapping, and the generic path; its own
// translation unit so that the library compiles in parallel.
#include "ring_kernel.cuh"

namespace rra {

const void *ring_fn_bfp8_ef(int in_t, bool fast, int groups, int mode)
{
    switch (groups) {
    case 1: return ring_variant<kCodecBfp8, 1, true>(in_t, fast, mode);
    case 2: return ring_variant<kCodecBfp8, 2, true>(in_t, fast, mode);
    case 4: return ring_variant<kCodecBfp8, 4, true>(in_t, fast, mode);
    case 8: return ring_variant<kCodecBfp8, 8, true>(in_t, fast, mode);
    default: return nullptr;
    }
}

} // namespace rra

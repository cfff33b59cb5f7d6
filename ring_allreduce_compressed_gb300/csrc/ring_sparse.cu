// ring_sparse.cu -- instantiations of the fused ring kernel for the sparse values + indices
// wire format: every input dtype and slice width, the staged path in each
// rank-to-warp mapping, and the generic path; its own translation unit so
// that the library compiles in parallel.
#include "ring_kernel.cuh"
#include "wire_sparse.cuh"

namespace rra {

const void *ring_fn_sparse(int in_t, bool fast, int groups, int mode)
{
    switch (groups) {
    case 1: return ring_variant<kCodecSparse, 1>(in_t, fast, mode);
    case 2: return ring_variant<kCodecSparse, 2>(in_t, fast, mode);
    case 4: return ring_variant<kCodecSparse, 4>(in_t, fast, mode);
    default: return nullptr;
    }
}

} // namespace rra

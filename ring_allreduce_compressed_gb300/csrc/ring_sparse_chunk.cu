// ring_sparse_chunk.cu -- the per-chunk sparse ring ("CCCL通信压缩库" §2.1:
// the sparsity of the tensor about to be sent decides between the dense
// tensor and its nonzero values + indices): the count pass that gives the
// nonzero count of every (hop, chunk) message before the ring starts, and
// the instantiations of the fused ring kernel for the per-chunk format.
//
// Why a count pass.  A rank's message for chunk c at hop h is its partial
// P_h = x_{c+1} + ... + x_{c+h} (fp32, added in ring order), and its format
// depends on the nonzero count of all of P_h.  The ring streams every chunk
// slice by slice, so the first slice of P_h is sent long before the last one
// exists.  The receiver adds the whole restored message whatever its format
// (decompress, then reduce, §2.2), so P_h does not depend on the formats of
// earlier hops, and one pass over the inputs -- each thread adding the ranks'
// elements of one position in ring order -- gives every count.
#include "ring_kernel.cuh"
#include "wire_sparse.cuh"

namespace rra {

namespace {

constexpr int kCountThreads = 256;
constexpr int kCountWarps = kCountThreads / 32;

// Nonzero counts of every message (see SpCountArgs).  Block b works on chunk
// c = b / bpc; a warp takes 256 consecutive elements of the chunk at a time,
// 8 per lane, and for each hop h adds rank (c + h) mod N's elements to its
// running fp32 partial and counts the elements whose bits are not +0.0.
template <int IN_KIND, bool VEC>
__global__ void __launch_bounds__(kCountThreads)
    sparse_chunk_count_kernel(const __grid_constant__ SpCountArgs a)
{
    constexpr bool PREV = IN_KIND == kF32Diff;
    constexpr int LT = PREV ? kF32 : IN_KIND;
    constexpr int es = dtype_size(LT);
    __shared__ unsigned long long s_cnt[kCountWarps][kMaxRanks];
    __shared__ bool s_last;
    const int N = a.N;
    const int c = blockIdx.x / a.bpc, sub = blockIdx.x % a.bpc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nh = a.h_hi - a.h_lo + 1;
    for (int i = threadIdx.x; i < kCountWarps * kMaxRanks; i += blockDim.x)
        (&s_cnt[0][0])[i] = 0ull;
    __syncthreads();

    const long long lo = min((long long)c * a.n, a.T);
    const long long len = min(lo + a.n, a.T) - lo;
    const long long wstride = (long long)a.bpc * kCountWarps * kTile;
    for (long long w0 = ((long long)sub * kCountWarps + warp) * kTile; w0 < len; w0 += wstride) {
        const long long e = w0 + 8 * lane; // chunk-relative first element of this lane
        const int valid = (int)min(max(len - e, 0LL), 8LL);
        const long long off = lo + e;
        float p[8];
#pragma unroll 4
        for (int h = a.h_lo; h <= a.h_hi; ++h) {
            int r = c + h;
            r -= r >= N ? N : 0;
            r -= r >= N ? N : 0;
            float x[8];
            const char *src = reinterpret_cast<const char *>(a.in[r]) + off * es;
            if (VEC && valid == 8)
                load8_vec<LT>(src, x);
            else
                load8_scalar<LT>(src, valid, x);
            if constexpr (PREV) {
                float q[8];
                if (VEC && valid == 8)
                    load8_vec<kF32>(a.prev[r] + off, q);
                else
                    load8_scalar<kF32>(a.prev[r] + off, valid, q);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    x[i] = __fsub_rn(x[i], q[i]);
            }
            if (h == a.h_lo) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    p[i] = x[i];
            } else {
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const float2 s2 =
                        __fadd2_rn(make_float2(x[i], x[i + 1]), make_float2(p[i], p[i + 1]));
                    p[i] = s2.x;
                    p[i + 1] = s2.y;
                }
            }
            // positions past the chunk's end hold +0.0 on both sides
            unsigned nz = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                nz += __float_as_uint(p[i]) != 0u ? 1u : 0u;
            const unsigned wc = __reduce_add_sync(kFull, nz);
            if (lane == 0)
                s_cnt[warp][h - a.h_lo] += wc;
        }
    }
    __syncthreads();
    if (threadIdx.x < nh) {
        unsigned long long t = 0;
#pragma unroll
        for (int w = 0; w < kCountWarps; ++w)
            t += s_cnt[w][threadIdx.x];
        if (t)
            atomicAdd(a.acc + (size_t)(a.h_lo + threadIdx.x - 1) * N + c, t);
    }
    // the last block to finish publishes the totals and clears the
    // accumulator and the ticket for the next call
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int i = threadIdx.x; i < N * N; i += blockDim.x)
            a.out[i] = atomicExch(a.acc + i, 0ull);
        __syncthreads();
        if (threadIdx.x == 0)
            *a.ticket = 0u;
    }
}

template <int IN_KIND> const void *count_fn(bool vec)
{
    return vec ? (const void *)sparse_chunk_count_kernel<IN_KIND, true>
               : (const void *)sparse_chunk_count_kernel<IN_KIND, false>;
}

} // namespace

cudaError_t launch_sparse_chunk_count(const SpCountArgs &a, int in_kind, bool vec,
                                      cudaStream_t st)
{
    const void *fn = nullptr;
    switch (in_kind) {
    case kF32: fn = count_fn<kF32>(vec); break;
    case kF16: fn = count_fn<kF16>(vec); break;
    case kBF16: fn = count_fn<kBF16>(vec); break;
    case kF32Diff: fn = count_fn<kF32Diff>(vec); break;
    default: return cudaErrorInvalidValue;
    }
    void *args[] = {const_cast<SpCountArgs *>(&a)};
    return cudaLaunchKernel(fn, dim3(a.N * a.bpc), dim3(kCountThreads), args, 0, st);
}

const void *ring_fn_sparse_chunk(int in_t, bool fast, int groups, int mode)
{
    switch (groups) {
    case 1: return ring_variant<kCodecSparseChunk, 1>(in_t, fast, mode);
    case 2: return ring_variant<kCodecSparseChunk, 2>(in_t, fast, mode);
    case 4: return ring_variant<kCodecSparseChunk, 4>(in_t, fast, mode);
    default: return nullptr;
    }
}

} // namespace rra

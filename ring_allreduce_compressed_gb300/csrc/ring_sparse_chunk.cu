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
#include <algorithm>

#include "ring_kernel.cuh"
#include "wire_sparse.cuh"

namespace rra {

namespace {

constexpr int kCountThreads = 256;
constexpr int kCountWarps = kCountThreads / 32;

// Nonzero counts of every message (see SpCountArgs).  Block b works on chunk
// c = b / bpc; a warp takes 256 consecutive elements of the chunk at a time,
// 8 per lane, and for each hop h adds rank (c + h) mod N's elements to its
// running fp32 partial and counts the elements whose bits are not +0.0
// (per lane in registers with at most 16 hops, else per warp and position).
// The raw 16-byte words of a batch of hops (8 words per lane: 8 hops of
// 16-bit data, 4 of fp32, 2 of fp32 with a prev stream) are loaded before
// any is used, so every lane keeps up to 8 loads in flight (and three
// blocks fit an SM).
// NH16: at most 16 hops (N <= 16); each lane then keeps its counts of every
// hop in registers and reduces them over the warp once, at the end.
template <int IN_KIND, bool VEC, bool NH16>
__global__ void __launch_bounds__(kCountThreads, 3)
    sparse_chunk_count_kernel(const __grid_constant__ SpCountArgs a)
{
    constexpr bool PREV = IN_KIND == kF32Diff;
    constexpr int LT = PREV ? kF32 : IN_KIND;
    constexpr int es = dtype_size(LT);
    constexpr int kWords = (es == 4 ? 2 : 1) * (PREV ? 2 : 1); // 16-byte words per hop
    constexpr int kBatch = 8 / kWords;                          // hops per batch
    using E = typename Elem<LT>::type;
    __shared__ unsigned long long s_cnt[kCountWarps][kMaxRanks];
    __shared__ bool s_last;
    const int N = a.N;
    const int c = blockIdx.x / a.bpc, sub = blockIdx.x % a.bpc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nh = a.h_hi - a.h_lo + 1;
    for (int i = threadIdx.x; i < kCountWarps * kMaxRanks; i += blockDim.x)
        (&s_cnt[0][0])[i] = 0ull;
    __syncthreads();

    // the raw words of 8 elements of rank r at element offset off
    auto fetch = [&](int r, long long off, uint4 (&w)[kWords]) {
        const uint4 *src =
            reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(a.in[r]) + off * es);
#pragma unroll
        for (int k = 0; k < (es == 4 ? 2 : 1); ++k)
            w[k] = __ldg(src + k);
        if constexpr (PREV) {
            const uint4 *ps = reinterpret_cast<const uint4 *>(a.prev[r] + off);
            w[2] = __ldg(ps);
            w[3] = __ldg(ps + 1);
        }
    };
    // the 8 fp32 input values (cur - prev with a prev stream) of raw words
    auto widen = [&](const uint4 (&w)[kWords], float (&x)[8]) {
        if constexpr (es == 4) {
            const float *f = reinterpret_cast<const float *>(&w[0]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = f[i];
        } else {
            const E *e = reinterpret_cast<const E *>(&w[0]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = to_f32(e[i]);
        }
        if constexpr (PREV) {
            const float *q = reinterpret_cast<const float *>(&w[2]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = __fsub_rn(x[i], q[i]);
        }
    };
    // the same from bounds-checked element loads (ragged end, unaligned)
    auto load_scalar = [&](int r, long long off, int valid, float (&x)[8]) {
        load8_scalar<LT>(reinterpret_cast<const char *>(a.in[r]) + off * es, valid, x);
        if constexpr (PREV) {
            float q[8];
            load8_scalar<kF32>(a.prev[r] + off, valid, q);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = __fsub_rn(x[i], q[i]);
        }
    };
    auto rank_of = [&](int h) {
        int r = c + h;
        r -= r >= N ? N : 0;
        r -= r >= N ? N : 0;
        return r;
    };

    const long long lo = min((long long)c * a.n, a.T);
    const long long len = min(lo + a.n, a.T) - lo;
    const long long wstride = (long long)a.bpc * kCountWarps * kTile;
    if constexpr (NH16) {
        uint32_t cnt[16];
#pragma unroll
        for (int hh = 0; hh < 16; ++hh)
            cnt[hh] = 0u;
        for (long long w0 = ((long long)sub * kCountWarps + warp) * kTile; w0 < len; w0 += wstride) {
            const long long e = w0 + 8 * lane;
            const int valid = (int)min(max(len - e, 0LL), 8LL);
            const long long off = lo + e;
            const bool vec = VEC && valid == 8;
            float p[8];
#pragma unroll
            for (int b = 0; b < 16 / kBatch; ++b) {
                uint4 w[kBatch][kWords];
                if (vec) {
#pragma unroll
                    for (int j = 0; j < kBatch; ++j)
                        if (b * kBatch + j < nh)
                            fetch(rank_of(a.h_lo + b * kBatch + j), off, w[j]);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int hh = b * kBatch + j;
                    if (hh < nh) {
                        float x[8];
                        if (vec)
                            widen(w[j], x);
                        else
                            load_scalar(rank_of(a.h_lo + hh), off, valid, x);
                        if (hh == 0) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                p[i] = x[i];
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {
                                const float2 s2 = __fadd2_rn(make_float2(x[i], x[i + 1]),
                                                             make_float2(p[i], p[i + 1]));
                                p[i] = s2.x;
                                p[i + 1] = s2.y;
                            }
                        }
                        // positions past the chunk's end hold +0.0 on both sides
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            cnt[hh] += __float_as_uint(p[i]) != 0u ? 1u : 0u;
                    }
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < 16; ++hh) {
            const unsigned wc = __reduce_add_sync(kFull, cnt[hh]);
            if (lane == 0 && hh < nh)
                s_cnt[warp][hh] += wc;
        }
    } else
    for (long long w0 = ((long long)sub * kCountWarps + warp) * kTile; w0 < len; w0 += wstride) {
        const long long e = w0 + 8 * lane; // chunk-relative first element of this lane
        const int valid = (int)min(max(len - e, 0LL), 8LL);
        const long long off = lo + e;
        const bool vec = VEC && valid == 8;
        float p[8];
        for (int h0 = a.h_lo; h0 <= a.h_hi; h0 += kBatch) {
            uint4 w[kBatch][kWords];
            if (vec) {
#pragma unroll
                for (int j = 0; j < kBatch; ++j)
                    if (h0 + j <= a.h_hi)
                        fetch(rank_of(h0 + j), off, w[j]);
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int h = h0 + j;
                if (h > a.h_hi)
                    break;
                float x[8];
                if (vec)
                    widen(w[j], x);
                else
                    load_scalar(rank_of(h), off, valid, x);
                if (h == a.h_lo) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        p[i] = x[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const float2 s2 = __fadd2_rn(make_float2(x[i], x[i + 1]),
                                                     make_float2(p[i], p[i + 1]));
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

template <int IN_KIND> const void *count_fn(bool vec, bool nh16)
{
    if (nh16)
        return vec ? (const void *)sparse_chunk_count_kernel<IN_KIND, true, true>
                   : (const void *)sparse_chunk_count_kernel<IN_KIND, false, true>;
    return vec ? (const void *)sparse_chunk_count_kernel<IN_KIND, true, false>
               : (const void *)sparse_chunk_count_kernel<IN_KIND, false, false>;
}

} // namespace

// One wave of resident blocks, split evenly over the chunks (at least one
// block per chunk, at most one per 2048 elements of a chunk).
cudaError_t launch_sparse_chunk_count(const SpCountArgs &args, int in_kind, bool vec,
                                      cudaStream_t st)
{
    const void *fn = nullptr;
    const bool nh16 = args.h_hi - args.h_lo + 1 <= 16;
    switch (in_kind) {
    case kF32: fn = count_fn<kF32>(vec, nh16); break;
    case kF16: fn = count_fn<kF16>(vec, nh16); break;
    case kBF16: fn = count_fn<kBF16>(vec, nh16); break;
    case kF32Diff: fn = count_fn<kF32Diff>(vec, nh16); break;
    default: return cudaErrorInvalidValue;
    }
    // resident blocks per SM of each variant, asked once
    static int occ_cache[16] = {};
    int &occ = occ_cache[in_kind * 4 + (vec ? 2 : 0) + (nh16 ? 1 : 0)];
    if (occ < 1 &&
        (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kCountThreads, 0) != cudaSuccess ||
         occ < 1))
        occ = 1;
    SpCountArgs a = args;
    const long long per_chunk = (a.n + kCountWarps * kTile - 1) / (kCountWarps * kTile);
    a.bpc = (int)std::max(1LL, std::min(per_chunk, (long long)num_sms() * occ / a.N));
    void *p[] = {&a};
    return cudaLaunchKernel(fn, dim3(a.N * a.bpc), dim3(kCountThreads), p, 0, st);
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

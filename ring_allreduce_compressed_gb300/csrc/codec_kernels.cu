// codec_kernels.cu -- standalone streaming codec kernels for sm_103a
// ("CCCL通信压缩库" §2.1: block floating point with one shared exponent per
// 128-element block and 8- or 4-bit mantissas; sparse values + indices when
// the sparsity exceeds a threshold; difference against the previous round).
// All of them are HBM-bound streams: 128-bit loads and stores where the
// buffers allow, grid-stride loops over warp-sized tiles.
#include "bfp_group.cuh"
#include "rra_device.cuh"
#include "rra_kernels.h"
#include <algorithm>
#include <map>
#include <mutex>

namespace rra {

int num_sms()
{
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0)
            sms = 1;
    }
    return sms;
}

namespace {

constexpr int kThreads = 256;

inline int grid_for(long long work_items, int per_block)
{
    long long g = (work_items + per_block - 1) / per_block;
    long long cap = (long long)num_sms() * 16;
    if (g > cap)
        g = cap;
    return (int)(g < 1 ? 1 : g);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- BFP encode
// One warp per 256-element tile (two 128-element blocks, one per half-warp).
template <int IN_T, int BITS>
__global__ void __launch_bounds__(kThreads) bfp_encode_kernel(const void *__restrict__ x, long long n,
                                                              int8_t *__restrict__ exps,
                                                              uint8_t *__restrict__ mants, int vec)
{
    constexpr int es = dtype_size(IN_T);
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (kThreads / 32);
    const long long tiles = (n + kTile - 1) / kTile;
    for (long long t = blockIdx.x * (long long)(kThreads / 32) + (threadIdx.x >> 5); t < tiles;
         t += warps) {
        const long long e0 = t * kTile + 8 * lane;
        const int vl = (int)max(0LL, min(8LL, n - e0));
        float v[8];
        const char *src = reinterpret_cast<const char *>(x) + e0 * es;
        if (vec && vl == 8)
            load8_vec<IN_T>(src, v);
        else
            load8_scalar<IN_T>(src, vl, v);
        // the ring's encoder (half-warp maximum by warp reductions, codes
        // from one fma each) gives offset codes m + 2^(bits-1); flipping the
        // top bit of every code gives the two's complement this API stores
        int e;
        uint32_t w[2];
        BfpGroup<BITS>::encode(v, e, w);
        const long long blk = (t * kTile + 128 * (lane >> 4)) / kBlock;
        if ((lane & 15) == 0 && blk * kBlock < n)
            exps[blk] = (int8_t)e;
        if constexpr (BITS == 8) {
            const uint2 c2 = make_uint2(w[0] ^ 0x80808080u, w[1] ^ 0x80808080u);
            if (vec && vl == 8) {
                *reinterpret_cast<uint2 *>(mants + e0) = c2;
            } else {
                for (int i = 0; i < vl; ++i)
                    mants[e0 + i] = (uint8_t)(((i < 4 ? c2.x : c2.y) >> (8 * (i & 3))) & 0xffu);
            }
        } else {
            const uint32_t u = w[0] ^ 0x88888888u;
            if (vec && vl == 8) {
                *reinterpret_cast<uint32_t *>(mants + e0 / 2) = u;
            } else {
                const int nb = (vl + 1) / 2; // an odd tail keeps its high nibble 0
                for (int b = 0; b < nb; ++b)
                    mants[e0 / 2 + b] = (uint8_t)((u >> (8 * b)) & (2 * b + 1 < vl ? 0xffu : 0x0fu));
            }
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) bfp_decode_kernel(const int8_t *__restrict__ exps,
                                                              const uint8_t *__restrict__ mants,
                                                              long long n, float *__restrict__ out,
                                                              int accumulate, int vec)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (kThreads / 32);
    const long long tiles = (n + kTile - 1) / kTile;
    // two's complement codes -> the offset codes m + 2^(bits-1) the ring's
    // decoder reads (flip the top bit of every code)
    constexpr uint32_t kFlip = BITS == 8 ? 0x80808080u : 0x88888888u;
    for (long long t = blockIdx.x * (long long)(kThreads / 32) + (threadIdx.x >> 5); t < tiles;
         t += warps) {
        const long long e0 = t * kTile + 8 * lane;
        const int vl = (int)max(0LL, min(8LL, n - e0));
        if (vl == 0)
            continue;
        const int e = __ldg(exps + e0 / kBlock);
        uint32_t w[2] = {0u, 0u};
        if constexpr (BITS == 8) {
            if (vec && vl == 8) {
                const uint2 u = __ldg(reinterpret_cast<const uint2 *>(mants + e0));
                w[0] = u.x;
                w[1] = u.y;
            } else {
                for (int i = 0; i < vl; ++i)
                    w[i >> 2] |= (uint32_t)mants[e0 + i] << (8 * (i & 3));
            }
        } else {
            if (vec && vl == 8) {
                w[0] = __ldg(reinterpret_cast<const uint32_t *>(mants + e0 / 2));
            } else {
                for (int b = 0; b < (vl + 1) / 2; ++b)
                    w[0] |= (uint32_t)mants[e0 / 2 + b] << (8 * b);
            }
        }
        // positions past n decode code 0 (flipped to the offset code of 0)
        w[0] ^= kFlip;
        w[1] ^= kFlip;
        // every m * 2^(e-q) is an exact float (|m| < 2^7, e - q >= -132), so
        // the fused decode-and-add rounds once, like decoding then adding
        float v[8];
        if (accumulate) {
            float o[8];
            if (vec && vl == 8)
                load8_vec<kF32>(out + e0, o);
            else
                load8_scalar<kF32>(out + e0, vl, o);
            BfpGroup<BITS>::decode_add(w, e, o, v);
        } else {
            BfpGroup<BITS>::decode(w, e, v);
        }
        store8(out + e0, kF32, v, vl, vec != 0);
    }
}

// ---------------------------------------------------------------- sparse encode
// Tile of 4096 elements per block: 256 threads x 16 elements (two groups of
// 8 consecutive elements per thread).  Pass 1 counts the tile's nonzeros;
// pass 2 (one block) turns the counts into exclusive offsets, decides the
// format and writes the header; pass 3 writes the values and indices: a
// thread's slot comes from a warp ballot/popc prefix and a block prefix sum
// over the warps; the tile's compacted run is staged in shared memory and
// leaves in consecutive stores at the tile's offset.
constexpr int kSpTile = 4096;

// Nonzero mask of the 8 elements at e0 (bit i: element e0+i is not +0.0),
// from the elements' own bits, which are also returned (a 16-bit element
// zero-extended): an fp16 or bf16 element widens to +0.0 exactly when its 16
// bits are zero, so no conversion is needed.
template <int IN_T>
__device__ __forceinline__ uint32_t nz_mask8_bits(const void *x, long long n, long long e0,
                                                  int vec, uint32_t w[8])
{
    const int vl = (int)max(0LL, min(8LL, n - e0));
    if constexpr (IN_T == kF32) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(x) + e0;
        if (vec && vl == 8) {
            const uint4 a = reinterpret_cast<const uint4 *>(p)[0];
            const uint4 b = reinterpret_cast<const uint4 *>(p)[1];
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = i < vl ? p[i] : 0u;
        }
    } else {
        const uint16_t *p = reinterpret_cast<const uint16_t *>(x) + e0;
        if (vec && vl == 8) {
            const uint4 a = *reinterpret_cast<const uint4 *>(p);
            const uint32_t h[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[2 * i] = h[i] & 0xffffu;
                w[2 * i + 1] = h[i] >> 16;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = i < vl ? (uint32_t)p[i] : 0u;
        }
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m |= (w[i] != 0u ? 1u : 0u) << i;
    return m;
}

template <int IN_T>
__global__ void __launch_bounds__(kThreads) sparse_count_kernel(const void *__restrict__ x,
                                                                long long n, uint32_t *counts,
                                                                int vec)
{
    __shared__ uint32_t wsum[kThreads / 32];
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
        uint32_t c = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[8];
            const long long e0 = t * kSpTile + (long long)h * 2048 + 8 * threadIdx.x;
            c += __popc(nz_mask8_bits<IN_T>(x, n, e0, vec, w));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            c += __shfl_xor_sync(kFull, c, o);
        if ((threadIdx.x & 31) == 0)
            wsum[threadIdx.x >> 5] = c;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t s = 0;
            for (int w = 0; w < kThreads / 32; ++w)
                s += wsum[w];
            counts[t] = s;
        }
        __syncthreads();
    }
}

// Exclusive prefix of the tile counts, in place, in segments of kSegTiles
// tiles: block s scans segment s (every thread four consecutive counts, one
// 16-byte load; warp shuffles; one shared-memory pass over the warp totals)
// and writes the segment's total to seg[s].  A tile's offset in the output is
// then its in-segment prefix plus the totals of the segments before it.
constexpr int kSegTiles = 4096;
constexpr int kScanThreads = kSegTiles / 4;

__global__ void __launch_bounds__(kScanThreads) sparse_segscan_kernel(uint32_t *counts,
                                                                      long long tiles,
                                                                      uint32_t *seg)
{
    __shared__ uint32_t wsum[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long t0 = (long long)blockIdx.x * kSegTiles + 4LL * threadIdx.x;
    uint32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        v[j] = t0 + j < tiles ? counts[t0 + j] : 0u;
    const uint32_t s = v[0] + v[1] + v[2] + v[3];
    uint32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, w, o);
            if (lane >= o)
                w += t;
        }
        wsum[lane] = w; // inclusive totals of warps 0..lane
    }
    __syncthreads();
    uint32_t run = (warp > 0 ? wsum[warp - 1] : 0u) + incl - s;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (t0 + j < tiles) {
            counts[t0 + j] = run;
            run += v[j];
        }
    if (threadIdx.x == 0)
        seg[blockIdx.x] = wsum[kScanThreads / 32 - 1];
}

// Exclusive prefix of a thread's count c (0..8) over the lanes of its warp,
// and the warp's total, from four ballots of the count's bits.
__device__ __forceinline__ uint32_t warp_prefix8(uint32_t c, int lane, uint32_t &total)
{
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t before = 0;
    total = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t m = __ballot_sync(kFull, (c >> b) & 1u);
        before += (uint32_t)__popc(m & lt) << b;
        total += (uint32_t)__popc(m) << b;
    }
    return before;
}

// Emit pass: every tile's nonzero values and indices at its offset (the
// tile's in-segment prefix plus the totals of the segments before it), or,
// for a dense message, a bit copy of x.  The format is decided from the
// total of all segments, which every block adds up for itself; block 0
// writes the header.  Inside a tile the compacted run is staged in shared
// memory (positions from warp ballots and a block prefix over the warp
// totals) and leaves in consecutive, coalesced stores, two elements per
// thread and store.  A 16-bit value and its index in the tile share one
// staged word.  The next tile's input is loaded before the current tile's
// run is written, so its latency overlaps the stores.
template <int IN_T>
__global__ void __launch_bounds__(kThreads, 6) sparse_emit_kernel(const void *__restrict__ x, long long n,
                                                               const uint32_t *__restrict__ offsets,
                                                               const uint32_t *__restrict__ seg,
                                                               long long nseg, double lim,
                                                               uint32_t *__restrict__ hdr,
                                                               void *__restrict__ vals,
                                                               int32_t *__restrict__ idx, int vec,
                                                               int pairs)
{
    using E = typename Elem<IN_T>::type;
    constexpr int es = dtype_size(IN_T);
    constexpr bool W16 = es == 2;
    constexpr int kWarps = kThreads / 32;
    __shared__ uint32_t wsum[2 * kWarps];  // warp totals, then their exclusive prefixes
    __shared__ uint32_t swd[kSpTile];      // 16-bit: value | index << 16; fp32: value bits
    __shared__ uint16_t sidx[W16 ? 1 : kSpTile]; // fp32: the index in the tile
    __shared__ unsigned long long s_total;
    __shared__ uint32_t s_local;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    if (warp == 0) { // the total of all segments
        unsigned long long t = 0;
        for (long long i = lane; i < nseg; i += 32)
            t += seg[i];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            t += __shfl_xor_sync(kFull, t, o);
        if (lane == 0)
            s_total = t;
    }
    __syncthreads();
    const unsigned long long total = s_total;
    const bool sparse = (double)total < lim;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        hdr[0] = sparse ? 1u : 0u;
        hdr[1] = (uint32_t)total;
    }
    if (!sparse) { // dense message: vals = x, bit for bit
        const long long groups = (n + 7) / 8;
        for (long long gi = blockIdx.x * (long long)kThreads + threadIdx.x; gi < groups;
             gi += (long long)gridDim.x * kThreads) {
            const long long e0 = gi * 8;
            const int vl = (int)min(8LL, n - e0);
            const char *src = reinterpret_cast<const char *>(x) + e0 * es;
            char *dst = reinterpret_cast<char *>(vals) + e0 * es;
            if (vec && vl == 8) {
#pragma unroll
                for (int b = 0; b < es / 2; ++b)
                    reinterpret_cast<uint4 *>(dst)[b] = reinterpret_cast<const uint4 *>(src)[b];
            } else {
                for (int i = 0; i < vl; ++i)
                    reinterpret_cast<E *>(dst)[i] = reinterpret_cast<const E *>(src)[i];
            }
        }
        return;
    }
    uint32_t bits[2][8], msk[2];
    uint32_t off_next = 0; // the next tile's offset within its segment
    auto load_tile = [&](long long t) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long e0 = t * kSpTile + (long long)h * 2048 + 8 * threadIdx.x;
            msk[h] = nz_mask8_bits<IN_T>(x, n, e0, vec, bits[h]);
        }
        off_next = offsets[t];
    };
    long long t = blockIdx.x;
    if (t < tiles)
        load_tile(t);
    for (; t < tiles; t += gridDim.x) {
        // positions in the tile's compacted run: half 0 (every thread) before
        // half 1, a thread's 8 elements in order within each half
        uint32_t before[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t wt;
            before[h] = warp_prefix8(__popc(msk[h]), lane, wt);
            if (lane == 0)
                wsum[h * kWarps + warp] = wt;
        }
        __syncthreads();
        if (warp == 0) { // exclusive prefix over (half, warp), and the tile's total
            const uint32_t v = lane < 2 * kWarps ? wsum[lane] : 0u;
            uint32_t incl = v;
#pragma unroll
            for (int o = 1; o < 2 * kWarps; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o)
                    incl += y;
            }
            if (lane < 2 * kWarps)
                wsum[lane] = incl - v;
            if (lane == 2 * kWarps - 1)
                s_local = incl;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t q = wsum[h * kWarps + warp] + before[h];
            const uint32_t e0 = h * 2048 + 8 * threadIdx.x; // within the tile
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((msk[h] >> i) & 1u) {
                    if constexpr (W16) {
                        swd[q] = bits[h][i] | ((e0 + i) << 16); // value bits | index
                    } else {
                        swd[q] = bits[h][i];
                        sidx[q] = (uint16_t)(e0 + i);
                    }
                    ++q;
                }
        }
        const uint32_t local = s_local;
        __syncthreads();
        uint32_t base = off_next;
        const uint32_t tseg = (uint32_t)(t / kSegTiles);
        for (uint32_t s2 = 0; s2 < tseg; ++s2)
            base += seg[s2];
        // the next tile's input, in flight while this tile's run is written
        const long long tn = t + gridDim.x;
        if (tn < tiles)
            load_tile(tn);
        const int32_t t0 = (int32_t)(t * kSpTile);
        int32_t *ip = idx + base;
        if constexpr (W16) {
            uint16_t *vp = reinterpret_cast<uint16_t *>(vals) + base;
            if (pairs && (base & 1u) == 0u) { // pairs: a 4-byte value and an 8-byte index store
                for (uint32_t k = 2 * threadIdx.x; k < local; k += 2 * kThreads) {
                    const uint32_t a = swd[k];
                    if (k + 1 < local) {
                        const uint32_t b = swd[k + 1];
                        *reinterpret_cast<uint32_t *>(vp + k) = (a & 0xffffu) | (b << 16);
                        *reinterpret_cast<int2 *>(ip + k) =
                            make_int2(t0 + (int32_t)(a >> 16), t0 + (int32_t)(b >> 16));
                    } else {
                        vp[k] = (uint16_t)a;
                        ip[k] = t0 + (int32_t)(a >> 16);
                    }
                }
            } else {
                for (uint32_t k = threadIdx.x; k < local; k += kThreads) {
                    const uint32_t a = swd[k];
                    vp[k] = (uint16_t)a;
                    ip[k] = t0 + (int32_t)(a >> 16);
                }
            }
        } else {
            uint32_t *vp = reinterpret_cast<uint32_t *>(vals) + base;
            for (uint32_t k = threadIdx.x; k < local; k += kThreads) {
                vp[k] = swd[k];
                ip[k] = t0 + (int32_t)sidx[k];
            }
        }
        __syncthreads(); // the staging arrays are reused by the next tile
    }
}

// ---------------------------------------------------------------- sparse decode
// Dense message: a streaming copy (or add) of the values into acc.
template <int IN_T>
__global__ void __launch_bounds__(kThreads) sparse_dense_kernel(const uint32_t *__restrict__ hdr,
                                                                const void *__restrict__ vals,
                                                                long long n, float *__restrict__ acc,
                                                                int accumulate, int vec)
{
    constexpr int es = dtype_size(IN_T);
    const bool sparse = hdr[0] != 0u;
    if (sparse) // sparse_fill_kernel or sparse_scatter_kernel restores it
        return;
    const long long groups = (n + 7) / 8;
    for (long long gi = blockIdx.x * (long long)kThreads + threadIdx.x; gi < groups;
         gi += (long long)gridDim.x * kThreads) {
        const long long e0 = gi * 8;
        const int vl = (int)min(8LL, n - e0);
        float v[8];
        const char *src = reinterpret_cast<const char *>(vals) + e0 * es;
        if (vec && vl == 8)
            load8_vec<IN_T>(src, v);
        else
            load8_scalar<IN_T>(src, vl, v);
        if (accumulate) {
            float o[8];
            if (vec && vl == 8)
                load8_vec<kF32>(acc + e0, o);
            else
                load8_scalar<kF32>(acc + e0, vl, o);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __fadd_rn(o[i], v[i]);
        }
        store8(acc + e0, kF32, v, vl, vec != 0);
    }
}

// Sparse message, accumulate == 0: one pass over acc in 4096-element tiles.
// First the position in the (ascending) index list where each tile starts,
// one binary search per tile; then every tile is built in shared memory
// (+0.0, then its values, read with consecutive threads) and written once.
// An index outside its tile (out of order, or outside [0, n)) is never
// written.
__global__ void __launch_bounds__(kThreads) sparse_tile_starts_kernel(
    const uint32_t *__restrict__ hdr, const int32_t *__restrict__ idx, long long n,
    uint32_t *__restrict__ start, int accumulate)
{
    if (hdr[0] == 0u || accumulate)
        return;
    const long long nnz = min((long long)hdr[1], n); // a header never lists more than n
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    for (long long t = blockIdx.x * (long long)kThreads + threadIdx.x; t <= tiles;
         t += (long long)gridDim.x * kThreads) {
        long long lo = 0, hi = nnz;
        if (t == tiles) {
            lo = nnz;
        } else {
            const long long target = t * kSpTile;
            while (lo < hi) {
                const long long mid = (lo + hi) >> 1;
                if ((long long)idx[mid] < target)
                    lo = mid + 1;
                else
                    hi = mid;
            }
        }
        start[t] = (uint32_t)lo;
    }
}

template <int IN_T>
__global__ void __launch_bounds__(kThreads) sparse_fill_kernel(const uint32_t *__restrict__ hdr,
                                                               const void *__restrict__ vals,
                                                               const int32_t *__restrict__ idx,
                                                               const uint32_t *__restrict__ start,
                                                               long long n, float *acc,
                                                               int accumulate, int vec)
{
    using E = typename Elem<IN_T>::type;
    __shared__ __align__(16) float tile[kSpTile];
    if (hdr[0] == 0u || accumulate)
        return;
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
        const long long t0 = t * kSpTile, t1 = min(n, t0 + kSpTile);
        for (int i = threadIdx.x; i < kSpTile; i += kThreads)
            tile[i] = 0.0f;
        __syncthreads();
        const long long kb = start[t], ke = start[t + 1];
#pragma unroll 4
        for (long long k = kb + threadIdx.x; k < ke; k += kThreads) {
            const long long i = idx[k];
            if (i >= t0 && i < t1)
                tile[i - t0] = to_f32(reinterpret_cast<const E *>(vals)[k]);
        }
        __syncthreads();
        const int len = (int)(t1 - t0);
        if (vec && len == kSpTile) {
            float4 *dst = reinterpret_cast<float4 *>(acc + t0);
            for (int j = threadIdx.x; j < kSpTile / 4; j += kThreads)
                dst[j] = reinterpret_cast<const float4 *>(tile)[j];
        } else {
            for (int j = threadIdx.x; j < len; j += kThreads)
                acc[t0 + j] = tile[j];
        }
        __syncthreads(); // the tile is rebuilt for the next position
    }
}

// Sparse message, accumulate != 0: acc[i] += v at the listed positions.
template <int IN_T>
__global__ void __launch_bounds__(kThreads) sparse_scatter_kernel(const uint32_t *__restrict__ hdr,
                                                                  const void *__restrict__ vals,
                                                                  const int32_t *__restrict__ idx,
                                                                  long long n, float *acc,
                                                                  int accumulate)
{
    using E = typename Elem<IN_T>::type;
    if (hdr[0] == 0u || !accumulate)
        return;
    const long long nnz = min((long long)hdr[1], n); // a header never lists more than n
    for (long long k = blockIdx.x * (long long)kThreads + threadIdx.x; k < nnz;
         k += (long long)gridDim.x * kThreads) {
        const long long i = idx[k];
        if (i < 0 || i >= n)
            continue; // malformed index: skip rather than write out of bounds
        const float v = to_f32(reinterpret_cast<const E *>(vals)[k]);
        acc[i] = accumulate ? __fadd_rn(acc[i], v) : v;
    }
}

// ---------------------------------------------------------------- diff
__global__ void __launch_bounds__(kThreads) diff_kernel(const float *cur, const float *prev,
                                                        float *diff, long long n, int vec)
{
    const long long groups = (n + 7) / 8;
    for (long long gi = blockIdx.x * (long long)kThreads + threadIdx.x; gi < groups;
         gi += (long long)gridDim.x * kThreads) {
        const long long e0 = gi * 8;
        const int vl = (int)min(8LL, n - e0);
        float a[8], b[8];
        if (vec && vl == 8) {
            load8_vec<kF32>(cur + e0, a);
            load8_vec<kF32>(prev + e0, b);
        } else {
            load8_scalar<kF32>(cur + e0, vl, a);
            load8_scalar<kF32>(prev + e0, vl, b);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = __fsub_rn(a[i], b[i]);
        store8(diff + e0, kF32, a, vl, vec != 0);
    }
}

// ---------------------------------------------------------------- codec statistics
// One warp per 128-element BFP block (4 elements a lane).  Blocks are cut
// from the start of each ring chunk of every rank's buffer, as the ring's
// first hop encodes them.  A nonzero element (fp32 bits not +0.0) is flushed
// by a BFP code of q = bits - 2 fraction bits when it rounds to code 0, that
// is when |x| <= 2^(e - q - 1) for the block exponent e.
// Grid: blockIdx.y = r * N + c (rank r, chunk c); the blocks along x stride
// over the chunk's 128-element blocks, a warp at a time, so no index needs a
// division.

// 2^k as an fp32 value for k in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2_exact(int k)
{
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// 4 elements of dtype IN_T at p widened to fp32; the first `valid` are read
// (vec: all 4 present and p aligned to 4 elements)
template <int IN_T>
__device__ __forceinline__ void load4(const void *p, int valid, bool vec, float v[4])
{
    using E = typename Elem<IN_T>::type;
    if (vec && valid == 4) {
        if constexpr (IN_T == kF32) {
            const float4 x = __ldg(reinterpret_cast<const float4 *>(p));
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        } else {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
            const E *e = reinterpret_cast<const E *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = to_f32(e[i]);
        }
        return;
    }
    const E *e = reinterpret_cast<const E *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = i < valid ? to_f32(e[i]) : 0.0f;
}

template <int IN_T>
__global__ void __launch_bounds__(kThreads) codec_stats_kernel(const __grid_constant__ StatsArgs a,
                                                               int vec)
{
    constexpr int es = dtype_size(IN_T);
    const int lane = threadIdx.x & 31;
    const int r = (int)(blockIdx.y / (unsigned)a.N), c = (int)(blockIdx.y % (unsigned)a.N);
    const long long lo = min(a.T, (long long)c * a.n), hi = min(a.T, lo + a.n);
    const char *base = reinterpret_cast<const char *>(a.in[r]);
    uint32_t cnt_nz = 0, cnt_f4 = 0, cnt_f8 = 0;
    const long long step = (long long)gridDim.x * (kThreads / 32) * kBlock;
    for (long long e0 = lo + ((long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kBlock;
         e0 < hi; e0 += step) {
        const int len = (int)min((long long)kBlock, hi - e0);
        const int valid = min(max(len - 4 * lane, 0), 4);
        float v[4];
        load4<IN_T>(base + (e0 + 4 * lane) * es, valid, vec != 0, v);
        unsigned mx = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            mx = max(mx, __float_as_uint(v[i]) & 0x7fffffffu);
        mx = __reduce_max_sync(kFull, mx);
        const int e = max((int)(mx >> 23), 1) - 127;
        const float t4 = pow2_exact(e - 3), t8 = pow2_exact(e - 7);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // absent positions read +0.0: never counted
            const bool nz = __float_as_uint(v[i]) != 0u;
            const float m = fabsf(v[i]);
            cnt_nz += nz ? 1u : 0u;
            cnt_f4 += nz && m <= t4 ? 1u : 0u;
            cnt_f8 += nz && m <= t8 ? 1u : 0u;
        }
    }
    cnt_nz = __reduce_add_sync(kFull, cnt_nz);
    cnt_f4 = __reduce_add_sync(kFull, cnt_f4);
    cnt_f8 = __reduce_add_sync(kFull, cnt_f8);
    if (lane == 0) {
        if (cnt_nz)
            atomicAdd(a.stats + 1, (unsigned long long)cnt_nz);
        if (cnt_f4)
            atomicAdd(a.stats + 2, (unsigned long long)cnt_f4);
        if (cnt_f8)
            atomicAdd(a.stats + 3, (unsigned long long)cnt_f8);
    }
    // the element count: one thread per (rank, chunk)
    if (blockIdx.x == 0 && threadIdx.x == 0 && hi > lo)
        atomicAdd(a.stats + 0, (unsigned long long)(hi - lo));
}

} // namespace

// ---------------------------------------------------------------- launchers

cudaError_t launch_codec_stats(const StatsArgs &a, int dtype, cudaStream_t st)
{
    // y: (rank, chunk); x: enough blocks of 8 warps for about 16 blocks per SM
    const long long nb = (a.n + kBlock - 1) / kBlock;
    const long long per_chunk = (nb + kThreads / 32 - 1) / (kThreads / 32);
    const long long want = std::max(1LL, (long long)num_sms() * 16 / ((long long)a.N * a.N));
    const dim3 grid((unsigned)std::max(1LL, std::min(per_chunk, want)), (unsigned)(a.N * a.N));
    const int es = dtype == kF32 ? 4 : 2;
    int vec = (a.n * es) % 16 == 0 ? 1 : 0; // 4-element runs aligned in every chunk
    for (int r = 0; r < a.N; ++r)
        vec = vec && aligned16(a.in[r]);
    if (dtype == kF32)
        codec_stats_kernel<kF32><<<grid, kThreads, 0, st>>>(a, vec);
    else if (dtype == kF16)
        codec_stats_kernel<kF16><<<grid, kThreads, 0, st>>>(a, vec);
    else
        codec_stats_kernel<kBF16><<<grid, kThreads, 0, st>>>(a, vec);
    return cudaGetLastError();
}

cudaError_t launch_bfp_encode(const void *x, long long n, int dtype, int bits, int8_t *exps,
                              uint8_t *mants, cudaStream_t st)
{
    const int es = dtype_size(dtype);
    const int vec = aligned16(x) && ((reinterpret_cast<uintptr_t>(mants) & 7u) == 0) ? 1 : 0;
    (void)es;
    const int grid = grid_for((n + kTile - 1) / kTile, kThreads / 32);
#define RRA_ENC(T, B) bfp_encode_kernel<T, B><<<grid, kThreads, 0, st>>>(x, n, exps, mants, vec)
    if (bits == 8) {
        if (dtype == kF32) RRA_ENC(kF32, 8);
        else if (dtype == kF16) RRA_ENC(kF16, 8);
        else RRA_ENC(kBF16, 8);
    } else {
        if (dtype == kF32) RRA_ENC(kF32, 4);
        else if (dtype == kF16) RRA_ENC(kF16, 4);
        else RRA_ENC(kBF16, 4);
    }
#undef RRA_ENC
    return cudaGetLastError();
}

cudaError_t launch_bfp_decode(const int8_t *exps, const uint8_t *mants, long long n, int bits,
                              float *out, int accumulate, cudaStream_t st)
{
    const int vec = aligned16(out) && ((reinterpret_cast<uintptr_t>(mants) & 7u) == 0) ? 1 : 0;
    const int grid = grid_for((n + kTile - 1) / kTile, kThreads / 32);
    if (bits == 8)
        bfp_decode_kernel<8><<<grid, kThreads, 0, st>>>(exps, mants, n, out, accumulate, vec);
    else
        bfp_decode_kernel<4><<<grid, kThreads, 0, st>>>(exps, mants, n, out, accumulate, vec);
    return cudaGetLastError();
}

// Scratch: one count (then offset) per 4096-element tile, then one total per
// segment of 4096 tiles.
long long sparse_encode_scratch_words(long long n)
{
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    return tiles + (tiles + kSegTiles - 1) / kSegTiles;
}

cudaError_t launch_sparse_encode(const void *x, long long n, int dtype, double one_minus_thr,
                                 uint32_t *hdr, void *vals, int32_t *idx, uint32_t *scratch,
                                 cudaStream_t st)
{
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    const long long nseg = (tiles + kSegTiles - 1) / kSegTiles;
    uint32_t *seg = scratch + tiles;
    const double lim = one_minus_thr * (double)n; // sparse iff nnz < lim
    const int vec = aligned16(x) && aligned16(vals) ? 1 : 0;
    const int grid = grid_for(tiles, 1);
    const int egrid = grid;
    // pairs of 16-bit values and of indices leave in one store each
    const int pairs = (reinterpret_cast<uintptr_t>(vals) & 3u) == 0 &&
                      (reinterpret_cast<uintptr_t>(idx) & 7u) == 0;
#define RRA_SP(T)                                                                              \
    do {                                                                                       \
        sparse_count_kernel<T><<<grid, kThreads, 0, st>>>(x, n, scratch, vec);                 \
        sparse_segscan_kernel<<<(unsigned)nseg, kScanThreads, 0, st>>>(scratch, tiles, seg);   \
        sparse_emit_kernel<T><<<egrid, kThreads, 0, st>>>(x, n, scratch, seg, nseg, lim, hdr,  \
                                                          vals, idx, vec, pairs);              \
    } while (0)
    if (dtype == kF32) RRA_SP(kF32);
    else if (dtype == kF16) RRA_SP(kF16);
    else RRA_SP(kBF16);
#undef RRA_SP
    return cudaGetLastError();
}

// Scratch of the decoder, one per (device, stream): where each tile's values
// start.  Grown on demand; decodes on different streams never share one, and
// the lock is held until the launches are queued, so no growth by another
// thread frees a buffer under a launch.
std::mutex g_dec_mu;
std::map<std::pair<int, cudaStream_t>, std::pair<uint32_t *, long long>> g_dec_ws;

cudaError_t launch_sparse_decode(const uint32_t *hdr, const void *vals, const int32_t *idx,
                                 long long n, int dtype, float *acc, int accumulate,
                                 cudaStream_t st)
{
    const long long words = (n + kSpTile - 1) / kSpTile + 1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_dec_mu);
    auto &ws = g_dec_ws[{dev, st}];
    if (ws.second < words) {
        if (ws.first) {
            cudaDeviceSynchronize(); // a decode in flight may still read it
            cudaFree(ws.first);
            ws.first = nullptr;
            ws.second = 0;
        }
        const long long want = std::max(words, 1LL << 12);
        e = cudaMalloc(&ws.first, (size_t)want * sizeof(uint32_t));
        if (e != cudaSuccess) {
            ws.first = nullptr;
            return e;
        }
        ws.second = want;
    }
    uint32_t *const scratch = ws.first;
    const int vec = aligned16(vals) && aligned16(acc) ? 1 : 0;
    const int g1 = grid_for((n + 7) / 8, kThreads);
    const int g2 = num_sms() * 4;
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    const int gs = (int)std::min<long long>((tiles + 1 + kThreads - 1) / kThreads, 65535);
    const int gf = (int)std::min<long long>(tiles, (long long)num_sms() * 8);
#define RRA_SD(T)                                                                                  \
    do {                                                                                           \
        sparse_dense_kernel<T><<<g1, kThreads, 0, st>>>(hdr, vals, n, acc, accumulate, vec);       \
        sparse_tile_starts_kernel<<<gs, kThreads, 0, st>>>(hdr, idx, n, scratch, accumulate);      \
        sparse_fill_kernel<T><<<gf, kThreads, 0, st>>>(hdr, vals, idx, scratch, n, acc,            \
                                                       accumulate, vec);                           \
        sparse_scatter_kernel<T><<<g2, kThreads, 0, st>>>(hdr, vals, idx, n, acc, accumulate);     \
    } while (0)
    if (dtype == kF32) RRA_SD(kF32);
    else if (dtype == kF16) RRA_SD(kF16);
    else RRA_SD(kBF16);
#undef RRA_SD
    return cudaGetLastError();
}

cudaError_t launch_diff_encode(const float *cur, const float *prev, float *diff, long long n,
                               cudaStream_t st)
{
    const int vec = aligned16(cur) && aligned16(prev) && aligned16(diff) ? 1 : 0;
    diff_kernel<<<grid_for((n + 7) / 8, kThreads), kThreads, 0, st>>>(cur, prev, diff, n, vec);
    return cudaGetLastError();
}

} // namespace rra

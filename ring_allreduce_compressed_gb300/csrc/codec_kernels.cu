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

// Decode helpers of the standalone BFP decoder: two's complement codes
// unpacked to integers, each scaled by 2^(e-q) (exact: |m| < 2^7 and
// e - q >= -132, so every product is a representable float).  (A variant
// that converts to the ring's offset codes and decodes with its fma path
// measured 30 % slower on this write-mostly stream.)
__device__ __forceinline__ float pow2i(int k)
{
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}
template <int BITS> __device__ __forceinline__ float bfp_value(int m, int e)
{
    return __fmul_rn(__int2float_rn(m), pow2i(e - (BITS - 2)));
}
// 8-bit codes: byte i = element i; 4-bit: nibble i = element i (2j low, 2j+1 high)
__device__ __forceinline__ void unpack8(uint2 u, int m[8])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = (int)(int8_t)((u.x >> (8 * i)) & 0xff);
        m[i + 4] = (int)(int8_t)((u.y >> (8 * i)) & 0xff);
    }
}
__device__ __forceinline__ void unpack4(uint32_t u, int m[8])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int nib = (u >> (4 * i)) & 0xf;
        m[i] = nib >= 8 ? nib - 16 : nib;
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
    for (long long t = blockIdx.x * (long long)(kThreads / 32) + (threadIdx.x >> 5); t < tiles;
         t += warps) {
        const long long e0 = t * kTile + 8 * lane;
        const int vl = (int)max(0LL, min(8LL, n - e0));
        if (vl == 0)
            continue;
        const int e = exps[e0 / kBlock];
        int m[8];
        if constexpr (BITS == 8) {
            if (vec && vl == 8) {
                unpack8(*reinterpret_cast<const uint2 *>(mants + e0), m);
            } else {
                for (int i = 0; i < 8; ++i)
                    m[i] = i < vl ? (int)(int8_t)mants[e0 + i] : 0;
            }
        } else {
            uint32_t u = 0;
            if (vec && vl == 8) {
                u = *reinterpret_cast<const uint32_t *>(mants + e0 / 2);
            } else {
                for (int b = 0; b < (vl + 1) / 2; ++b)
                    u |= (uint32_t)mants[e0 / 2 + b] << (8 * b);
            }
            unpack4(u, m);
        }
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = bfp_value<BITS>(m[i], e);
        if (accumulate) {
            float o[8];
            if (vec && vl == 8)
                load8_vec<kF32>(out + e0, o);
            else
                load8_scalar<kF32>(out + e0, vl, o);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __fadd_rn(o[i], v[i]);
        }
        store8(out + e0, kF32, v, vl, vec != 0);
    }
}

// ---------------------------------------------------------------- sparse encode
// Three passes over chunks of 1024 elements ([cccl] §2.1's values +
// indices), each chunk handled by one warp, no block-wide step anywhere:
//   count  the nonzeros of every chunk;
//   scan   their exclusive prefix (segments of 4096 chunks, then the
//          segments' own prefix, whose total decides the format and goes
//          into the header);
//   emit   every chunk's nonzero values and indices at its offset, or, for
//          a dense message, a bit copy of x.
// Lane L holds the chunk's 16-byte words L, 32 + L, 64 + L, ... (8 16-bit
// or 4 fp32 elements each).  The chunk's run (word by word, lanes and
// elements in order: ascending indices) is staged in the warp's own part of
// shared memory -- a 16-bit value and its index in the chunk share one word
// -- and leaves in 16-byte index stores and 8-byte (16-bit values) or
// 16-byte (fp32) value stores aligned to the output.
constexpr int kSpChunk = 1024;  // elements per chunk
constexpr int kSegChunks = 4096; // chunks per scan segment
constexpr int kScanThreads = kSegChunks / 4;

template <int IN_T> struct SpChunk {
    static constexpr int es = dtype_size(IN_T);
    static constexpr int epw = 16 / es;             // elements per 16-byte word
    static constexpr int words = kSpChunk / epw / 32; // 16-byte words per lane (4 or 8)
};

// Bit 15 set iff the low 16 bits of w are nonzero, bit 31 iff the high 16
// bits are; no other bit set.  (w & 0x7fff) + 0x7fff carries into bit 15
// exactly when the low 15 bits are not all zero, and cannot carry further.
__device__ __forceinline__ uint32_t nz16(uint32_t w)
{
    return (((w & 0x7fff7fffu) + 0x7fff7fffu) | w) & 0x80008000u;
}

__device__ __forceinline__ uint32_t u4_at(const uint4 &q, int k)
{
    return k == 0 ? q.x : k == 1 ? q.y : k == 2 ? q.z : q.w;
}

// Nonzero mask of one 16-byte word of dtype IN_T (bit i: element i).  An
// element is zero iff its bits are all zero (+0.0 in every dtype).
template <int IN_T> __device__ __forceinline__ uint32_t word_mask(const uint4 &q)
{
    if constexpr (dtype_size(IN_T) == 2) {
        // the top bits of bytes 1 and 3 of nz16 flag the two elements of a
        // 32-bit word; gather them into the top bits of four bytes and
        // collect those (the four products land on distinct bits)
        const uint32_t u0 = __byte_perm(nz16(q.x), nz16(q.y), 0x7531);
        const uint32_t u1 = __byte_perm(nz16(q.z), nz16(q.w), 0x7531);
        return ((u0 * 0x00204081u) >> 28) | (((u1 * 0x00204081u) >> 28) << 4);
    } else {
        return (q.x != 0u ? 1u : 0u) | (q.y != 0u ? 2u : 0u) | (q.z != 0u ? 4u : 0u) |
               (q.w != 0u ? 8u : 0u);
    }
}

// Number of nonzero elements of one 16-byte word of dtype IN_T.
template <int IN_T> __device__ __forceinline__ uint32_t word_count(const uint4 &q)
{
    if constexpr (dtype_size(IN_T) == 2)
        return (uint32_t)__popc(nz16(q.x) | (nz16(q.y) >> 1) | (nz16(q.z) >> 2) |
                                (nz16(q.w) >> 3));
    else
        return (q.x != 0u ? 1u : 0u) + (q.y != 0u ? 1u : 0u) + (q.z != 0u ? 1u : 0u) +
               (q.w != 0u ? 1u : 0u);
}

// The count pass reads x once more than the output needs.  It keeps its
// last 64 MB of x (half the 129 MB L2) with the evict-last priority, and the
// emit pass, which takes the chunks from the last one down, reads them from
// L2 first; every other read of x is a streaming (evict-first) load.
constexpr long long kKeepBytes = 64ll << 20;

// One 16-byte global load with the L2 evict-last policy.
__device__ __forceinline__ uint4 ld_keep(const uint4 *p)
{
    uint64_t pol;
    uint4 r;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// This lane's words of chunk c (zero past n): one 16-byte load each when the
// chunk is whole and x aligned (kept in L2 with keep set), else element
// loads.
template <int IN_T>
__device__ __forceinline__ void load_chunk(const void *x, long long n, long long c, int lane,
                                           int vec, uint4 (&q)[SpChunk<IN_T>::words],
                                           bool keep = false)
{
    constexpr int es = SpChunk<IN_T>::es, EPW = SpChunk<IN_T>::epw, W = SpChunk<IN_T>::words;
    const long long base = c * kSpChunk;
    if (vec && base + kSpChunk <= n) {
        const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(x) +
                                                           base * es);
        if (keep) {
#pragma unroll
            for (int j = 0; j < W; ++j)
                q[j] = ld_keep(src + 32 * j + lane);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j)
                q[j] = __ldcs(src + 32 * j + lane);
        }
    } else {
#pragma unroll
        for (int j = 0; j < W; ++j) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            const long long e0 = base + (long long)(32 * j + lane) * EPW;
            for (int i = 0; i < EPW; ++i)
                if (e0 + i < n) {
                    if constexpr (es == 2)
                        w[i >> 1] |= (uint32_t)reinterpret_cast<const uint16_t *>(x)[e0 + i]
                                     << (16 * (i & 1));
                    else
                        w[i] = reinterpret_cast<const uint32_t *>(x)[e0 + i];
                }
            q[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Pass 1: counts[c] = nonzeros of chunk c.  Warps stride over the chunks;
// the next chunk's words are loaded before this one is counted.  The chunks
// of the last kKeepBytes of x stay in L2 for the emit pass.
template <int IN_T>
__global__ void __launch_bounds__(kThreads) sparse_count_kernel(const void *__restrict__ x,
                                                                long long n, long long chunks,
                                                                uint32_t *__restrict__ counts,
                                                                int vec)
{
    constexpr int W = SpChunk<IN_T>::words;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (kThreads / 32);
    long long c = blockIdx.x * (long long)(kThreads / 32) + (threadIdx.x >> 5);
    const long long keep_from = chunks - kKeepBytes / (kSpChunk * SpChunk<IN_T>::es);
    uint4 q[W];
    if (c < chunks)
        load_chunk<IN_T>(x, n, c, lane, vec, q, c >= keep_from);
    for (; c < chunks; c += warps) {
        uint32_t k = 0;
#pragma unroll
        for (int j = 0; j < W; ++j)
            k += word_count<IN_T>(q[j]);
        if (c + warps < chunks)
            load_chunk<IN_T>(x, n, c + warps, lane, vec, q, c + warps >= keep_from);
        k = __reduce_add_sync(kFull, k);
        if (lane == 0)
            counts[c] = k;
    }
}

// Pass 2a: exclusive prefix of the chunk counts, in place, in segments of
// kSegChunks chunks: block s scans segment s (every thread four consecutive
// counts; warp shuffles; one shared-memory pass over the warp totals) and
// writes the segment's total to seg[s].
// Pass 2b (one block): the segments' exclusive prefix, in place, and the
// header: the total nnz and the format (sparse iff nnz < lim).
// Inclusive scan of v over a block of kScanThreads threads; *all: the total.
__device__ __forceinline__ uint32_t scan_block(uint32_t v, uint32_t *wsum, uint32_t *all)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) {
        const uint32_t y = wsum[w];
        before += w < warp ? y : 0u;
        tot += y;
    }
    __syncthreads(); // (wsum is reused by the next scan)
    *all = tot;
    return before + incl;
}

__global__ void __launch_bounds__(kScanThreads) sparse_segscan_kernel(uint32_t *counts,
                                                                      long long chunks,
                                                                      uint32_t *seg)
{
    __shared__ uint32_t wsum[kScanThreads / 32];
    const long long t0 = (long long)blockIdx.x * kSegChunks + 4LL * threadIdx.x;
    uint32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        v[j] = t0 + j < chunks ? counts[t0 + j] : 0u;
    const uint32_t s = v[0] + v[1] + v[2] + v[3];
    uint32_t total;
    uint32_t run = scan_block(s, wsum, &total) - s;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (t0 + j < chunks) {
            counts[t0 + j] = run;
            run += v[j];
        }
    if (threadIdx.x == 0)
        seg[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) sparse_segbase_kernel(uint32_t *seg, long long nseg,
                                                                      double lim, uint32_t *hdr)
{
    __shared__ uint32_t wsum[kScanThreads / 32];
    uint32_t carry = 0;
    for (long long b0 = 0; b0 < nseg; b0 += kScanThreads) {
        const long long i = b0 + threadIdx.x;
        const uint32_t y = i < nseg ? seg[i] : 0u;
        uint32_t all;
        const uint32_t incl = scan_block(y, wsum, &all);
        if (i < nseg)
            seg[i] = carry + incl - y;
        carry += all;
    }
    if (threadIdx.x == 0) {
        hdr[0] = (double)carry < lim ? 1u : 0u;
        hdr[1] = carry;
    }
}

// Pass 3: every chunk's run at its offset (counts[c] + seg[c / kSegChunks]),
// or, when the header says dense, vals = x bit for bit.  The next chunk's
// words are loaded once this chunk is staged, so that their latency
// overlaps the stores.
template <int IN_T>
__global__ void __launch_bounds__(kThreads, 4) sparse_emit_kernel(
    const void *__restrict__ x, long long n, long long chunks, const uint32_t *__restrict__ offs,
    const uint32_t *__restrict__ segbase, const uint32_t *__restrict__ hdr, void *__restrict__ vals,
    int32_t *__restrict__ idx, int vec, int quads)
{
    using E = typename Elem<IN_T>::type;
    constexpr int es = SpChunk<IN_T>::es, EPW = SpChunk<IN_T>::epw, W = SpChunk<IN_T>::words;
    constexpr bool W16 = es == 2;
    constexpr int kWarps = kThreads / 32;
    // the staged run, 3 slots of room in front: slot k of the run sits at
    // position k + (ob & 3), so that a 4-aligned output group is one
    // 16-byte shared-memory word
    constexpr int kStage = kSpChunk + 4;
    __shared__ __align__(16) uint32_t swd[kWarps][kStage]; // 16-bit: value | index << 16; fp32: value
    __shared__ __align__(8) uint16_t sidx[W16 ? 1 : kWarps][W16 ? 4 : kStage]; // fp32: index in the chunk
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (hdr[0] == 0u) { // dense message: vals = x, bit for bit
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
                    reinterpret_cast<uint4 *>(dst)[b] = __ldcs(reinterpret_cast<const uint4 *>(src) + b);
            } else {
                for (int i = 0; i < vl; ++i)
                    reinterpret_cast<E *>(dst)[i] = reinterpret_cast<const E *>(src)[i];
            }
        }
        return;
    }
    uint32_t *wsd = swd[warp];
    uint16_t *wsi = sidx[W16 ? 0 : warp];
    const long long warps = (long long)gridDim.x * kWarps;
    // chunks are taken from the last one down: the count pass kept its last
    // kKeepBytes of x in L2, and these loads (evict-first) are their last use
    long long i = blockIdx.x * (long long)kWarps + warp;
    uint4 q[W];
    if (i < chunks)
        load_chunk<IN_T>(x, n, chunks - 1 - i, lane, vec, q);
    for (; i < chunks; i += warps) {
        const long long c = chunks - 1 - i;
        const uint32_t ob = offs[c] + segbase[c / kSegChunks]; // the run's first output position
        const uint32_t sh = ob & 3u;
        // this lane's masks (word j at bits j*EPW..) and slots
        uint32_t msk = 0, cw[W];
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const uint32_t m = word_mask<IN_T>(q[j]);
            msk |= m << (j * EPW);
            cw[j] = (uint32_t)__popc(m);
        }
        uint32_t slot[W];
        uint32_t run = sh; // the staging positions of the words before word j
#pragma unroll
        for (int j = 0; j < W; j += 2) {
            const uint32_t c2 = cw[j] | (cw[j + 1] << 16);
            uint32_t i2 = c2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, i2, o);
                if (lane >= o)
                    i2 += y;
            }
            const uint32_t t2 = __shfl_sync(kFull, i2, 31), e2 = i2 - c2;
            slot[j] = run + (e2 & 0xffffu);
            run += t2 & 0xffffu;
            slot[j + 1] = run + (e2 >> 16);
            run += t2 >> 16;
        }
        const uint32_t len = run - sh; // the chunk's nonzeros
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const uint32_t ib = (uint32_t)((32 * j + lane) * EPW);
#pragma unroll
            for (int i = 0; i < EPW; ++i)
                if ((msk >> (j * EPW + i)) & 1u) {
                    if constexpr (W16) {
                        const uint32_t v = (u4_at(q[j], i >> 1) >> (16 * (i & 1))) & 0xffffu;
                        wsd[slot[j]] = v | ((ib + i) << 16);
                    } else {
                        wsd[slot[j]] = u4_at(q[j], i);
                        wsi[slot[j]] = (uint16_t)(ib + i);
                    }
                    ++slot[j];
                }
        }
        __syncwarp();
        if (i + warps < chunks)
            load_chunk<IN_T>(x, n, chunks - 1 - (i + warps), lane, vec, q);
        // the run in 4-aligned groups; group g covers output positions
        // (ob & ~3) + 4g .., staged at positions 4g ..
        const int32_t t0 = (int32_t)(c * kSpChunk);
        const uint32_t ngr = (sh + len + 3u) >> 2;
        const long long obase = (long long)(ob - sh);
        for (uint32_t g = lane; g < ngr; g += 32) {
            const int k0 = (int)(4u * g) - (int)sh; // run position of the group's first slot
            const uint4 s4 = reinterpret_cast<const uint4 *>(wsd)[g];
            const uint32_t w4[4] = {s4.x, s4.y, s4.z, s4.w};
            int32_t i4[4];
            if constexpr (W16) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    i4[u] = t0 + (int32_t)(w4[u] >> 16);
            } else {
                const uint2 x2 = reinterpret_cast<const uint2 *>(wsi)[g];
                i4[0] = t0 + (int32_t)(x2.x & 0xffffu);
                i4[1] = t0 + (int32_t)(x2.x >> 16);
                i4[2] = t0 + (int32_t)(x2.y & 0xffffu);
                i4[3] = t0 + (int32_t)(x2.y >> 16);
            }
            const long long o = obase + 4LL * g;
            if (quads && k0 >= 0 && k0 + 4 <= (int)len) {
                *reinterpret_cast<int4 *>(idx + o) = make_int4(i4[0], i4[1], i4[2], i4[3]);
                if constexpr (W16)
                    *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(vals) + o) =
                        make_uint2(__byte_perm(w4[0], w4[1], 0x5410), __byte_perm(w4[2], w4[3], 0x5410));
                else
                    *reinterpret_cast<uint4 *>(reinterpret_cast<uint32_t *>(vals) + o) =
                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k0 + u;
                    if (k >= 0 && k < (int)len) {
                        idx[o + u] = i4[u];
                        if constexpr (W16)
                            reinterpret_cast<uint16_t *>(vals)[o + u] = (uint16_t)w4[u];
                        else
                            reinterpret_cast<uint32_t *>(vals)[o + u] = w4[u];
                    }
                }
            }
        }
        __syncwarp(); // (the staging area is reused by the next chunk)
    }
}

// ---------------------------------------------------------------- sparse decode
constexpr int kSpTile = 4096; // elements per decoder tile
// Dense message: a streaming copy (or add) of the values into acc, the
// whole grid striding over groups of 8 elements.
template <int IN_T>
__device__ __forceinline__ void dense_restore(const void *vals, long long n, float *acc,
                                              int accumulate, int vec)
{
    constexpr int es = dtype_size(IN_T);
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

// The decode is two kernels, one pass over acc in 4096-element tiles.  This
// one: a dense message is copied (or added) by the whole grid; for a sparse
// one, the position in the (ascending) index list where each tile starts,
// one binary search per tile and thread.  Then sparse_fill_kernel builds
// every tile of a sparse message in shared memory (+0.0, or acc's values
// when accumulating, then the listed values set or added, read with
// consecutive threads) and writes it once.  An index outside its tile (out
// of order, or outside [0, n)) is never used.
template <int IN_T>
__global__ void __launch_bounds__(kThreads) sparse_prep_kernel(const uint32_t *__restrict__ hdr,
                                                               const void *__restrict__ vals,
                                                               const int32_t *__restrict__ idx,
                                                               long long n, float *__restrict__ acc,
                                                               uint32_t *__restrict__ start,
                                                               int accumulate, int vec)
{
    if (hdr[0] == 0u) {
        dense_restore<IN_T>(vals, n, acc, accumulate, vec);
        return;
    }
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

// Pairs of a tile each thread holds in registers (the rest, if a tile lists
// more than kThreads * kFillPairs values, are read in a second loop).
constexpr int kFillPairs = 8;

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
    if (hdr[0] == 0u)
        return;
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    // The tile's listed (index, value) pairs k = kb + tid + kThreads*j are read
    // into registers one tile ahead: the next tile's loads are in flight
    // while this tile is written out.  Between tiles the buffer holds the
    // next tile's base: +0.0 (each thread zeroes the words it has just
    // written out) or, accumulating, acc's values (each thread loads the
    // words of the next tile that it will write out itself).
    int32_t pi[kFillPairs];
    float pv[kFillPairs];
    long long kb = 0, ke = 0;
    auto fetch = [&](long long t) {
        kb = start[t];
        ke = start[t + 1];
#pragma unroll
        for (int j = 0; j < kFillPairs; ++j) {
            const long long k = kb + threadIdx.x + (long long)kThreads * j;
            pi[j] = k < ke ? idx[k] : -1;
            pv[j] = k < ke ? to_f32(reinterpret_cast<const E *>(vals)[k]) : 0.0f;
        }
    };
    // this thread's words of tile t's base: acc's values accumulating, else +0.0
    auto load_base = [&](long long t) {
        const long long t0 = t * kSpTile;
        const int len = (int)(min(n, t0 + kSpTile) - t0);
        if (!accumulate) {
            for (int i = threadIdx.x; i < kSpTile; i += kThreads)
                tile[i] = 0.0f;
        } else if (vec && len == kSpTile) {
            const float4 *src = reinterpret_cast<const float4 *>(acc + t0);
            for (int j = threadIdx.x; j < kSpTile / 4; j += kThreads)
                reinterpret_cast<float4 *>(tile)[j] = src[j];
        } else {
            for (int j = threadIdx.x; j < len; j += kThreads)
                tile[j] = acc[t0 + j];
        }
    };
    long long t = blockIdx.x;
    if (t < tiles) {
        fetch(t);
        load_base(t);
    }
    __syncthreads();
    for (; t < tiles; t += gridDim.x) {
        const long long t0 = t * kSpTile, t1 = min(n, t0 + kSpTile);
        // set or add the pairs (an index outside the tile is never used);
        // the indices of one message are distinct, so no two threads touch
        // one word
#pragma unroll
        for (int j = 0; j < kFillPairs; ++j)
            if (pi[j] >= t0 && pi[j] < t1)
                tile[pi[j] - t0] = accumulate ? __fadd_rn(tile[pi[j] - t0], pv[j]) : pv[j];
        for (long long k = kb + threadIdx.x + (long long)kThreads * kFillPairs; k < ke;
             k += kThreads) {
            const long long i = idx[k];
            if (i >= t0 && i < t1) {
                const float v = to_f32(reinterpret_cast<const E *>(vals)[k]);
                tile[i - t0] = accumulate ? __fadd_rn(tile[i - t0], v) : v;
            }
        }
        __syncthreads();
        const long long tn = t + gridDim.x;
        if (tn < tiles)
            fetch(tn);
        const int len = (int)(t1 - t0);
        const long long tn0 = tn * kSpTile;
        const bool next_full = tn < tiles && tn0 + kSpTile <= n;
        if (vec && len == kSpTile && (!accumulate || tn >= tiles || next_full)) {
            // every thread moves the same float4 words out and in
            float4 *dst = reinterpret_cast<float4 *>(acc + t0);
            for (int j = threadIdx.x; j < kSpTile / 4; j += kThreads) {
                dst[j] = reinterpret_cast<const float4 *>(tile)[j];
                reinterpret_cast<float4 *>(tile)[j] =
                    !accumulate ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                    : tn < tiles ? reinterpret_cast<const float4 *>(acc + tn0)[j]
                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        } else {
            for (int j = threadIdx.x; j < len; j += kThreads)
                acc[t0 + j] = tile[j];
            if (tn < tiles) {
                __syncthreads(); // the element loop above maps threads differently
                load_base(tn);
            }
        }
        __syncthreads(); // the tile holds the next base before the next scatter
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
// One warp per 256-element tile: two 128-element BFP blocks, one per
// half-warp, 8 elements a lane.  Blocks are cut from the start of each ring
// chunk of every rank's buffer, as the ring's first hop encodes them.  A
// nonzero element (fp32 bits not +0.0) is flushed by a BFP code of q =
// bits - 2 fraction bits when it rounds to code 0, that is when
// |x| <= 2^(e - q - 1) for the block exponent e.
// Grid: blockIdx.y = r * N + c (rank r, chunk c); the blocks along x stride
// over the chunk's tiles, a warp at a time, so no index needs a division.

// 2^k as an fp32 value for k in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2_exact(int k)
{
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

template <int IN_T>
__global__ void __launch_bounds__(kThreads) codec_stats_kernel(const __grid_constant__ StatsArgs a,
                                                               int vec)
{
    constexpr int es = dtype_size(IN_T);
    const int lane = threadIdx.x & 31;
    const int r = (int)(blockIdx.y / (unsigned)a.N), c = (int)(blockIdx.y % (unsigned)a.N);
    const long long lo = min(a.T, (long long)c * a.n), hi = min(a.T, lo + a.n);
    const long long len = hi - lo;
    const char *base = reinterpret_cast<const char *>(a.in[r]) + lo * es;
    uint32_t cnt_nz = 0, cnt_f4 = 0, cnt_f8 = 0;
    // kStatsU tiles per warp and iteration, all loaded before any is
    // counted, so that every lane keeps kStatsU loads in flight
    constexpr int kStatsU = 2;
    const long long step = (long long)gridDim.x * (kThreads / 32) * kTile;
    for (long long w0 = ((long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kTile;
         w0 < len; w0 += kStatsU * step) {
        float v[kStatsU][8];
#pragma unroll
        for (int u = 0; u < kStatsU; ++u) {
            const long long e = w0 + u * step + 8 * lane; // chunk-relative
            const int valid = (int)min(max(len - e, 0LL), 8LL);
            if (vec && valid == 8)
                load8_vec<IN_T>(base + e * es, v[u]);
            else
                load8_scalar<IN_T>(base + e * es, valid, v[u]); // +0.0 past the end
        }
#pragma unroll
        for (int u = 0; u < kStatsU; ++u) {
            if (w0 + u * step >= len) // (warp-uniform)
                break;
            // the half-warp's block maximum: non-negative floats order like
            // their bit patterns
            unsigned mx = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mx = max(mx, __float_as_uint(v[u][i]) & 0x7fffffffu);
            const unsigned m_lo = __reduce_max_sync(kFull, lane < 16 ? mx : 0u);
            const unsigned m_hi = __reduce_max_sync(kFull, lane < 16 ? 0u : mx);
            const int e = max((int)((lane < 16 ? m_lo : m_hi) >> 23), 1) - 127;
            // |x| <= 2^k as bit patterns (both non-negative)
            const unsigned t4 = __float_as_uint(pow2_exact(e - 3));
            const unsigned t8 = __float_as_uint(pow2_exact(e - 7));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // absent positions read +0.0: never counted
                const unsigned b = __float_as_uint(v[u][i]);
                const unsigned m = b & 0x7fffffffu;
                const bool nz = b != 0u;
                cnt_nz += nz ? 1u : 0u;
                cnt_f4 += nz && m <= t4 ? 1u : 0u;
                cnt_f8 += nz && m <= t8 ? 1u : 0u;
            }
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
    const long long nt = (a.n + kTile - 1) / kTile; // 256-element tiles per chunk
    const long long per_chunk = (nt + kThreads / 32 - 1) / (kThreads / 32);
    const long long want = std::max(1LL, (long long)num_sms() * 16 / ((long long)a.N * a.N));
    const dim3 grid((unsigned)std::max(1LL, std::min(per_chunk, want)), (unsigned)(a.N * a.N));
    const int es = dtype == kF32 ? 4 : 2;
    int vec = (a.n * es) % 16 == 0 ? 1 : 0; // 8-element runs aligned in every chunk
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

// Scratch: one count (then offset) per 1024-element chunk, then one total
// (then base) per segment of 4096 chunks.  Every word is written by a call
// before that call reads it: nothing needs clearing, before or between calls.
long long sparse_encode_scratch_words(long long n)
{
    const long long chunks = (n + kSpChunk - 1) / kSpChunk;
    return chunks + (chunks + kSegChunks - 1) / kSegChunks;
}

// Resident blocks per SM of a kernel, asked once per kernel.
template <typename K> int blocks_per_sm(K kernel)
{
    static int occ = 0;
    if (occ < 1 &&
        (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess ||
         occ < 1))
        occ = 1;
    return occ;
}

cudaError_t launch_sparse_encode(const void *x, long long n, int dtype, double one_minus_thr,
                                 uint32_t *hdr, void *vals, int32_t *idx, uint32_t *scratch,
                                 cudaStream_t st)
{
    const long long chunks = (n + kSpChunk - 1) / kSpChunk;
    const long long nseg = (chunks + kSegChunks - 1) / kSegChunks;
    uint32_t *counts = scratch;
    uint32_t *seg = counts + chunks;
    const double lim = one_minus_thr * (double)n; // sparse iff nnz < lim
    const int vec = aligned16(x) && aligned16(vals) ? 1 : 0;
    const int es = dtype == kF32 ? 4 : 2;
    // 4-element groups of the run leave in one index and one value store
    const int quads = (reinterpret_cast<uintptr_t>(idx) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(vals) & (uintptr_t)(4 * es - 1)) == 0;
    const long long wblocks = (chunks + kThreads / 32 - 1) / (kThreads / 32); // a warp per chunk
#define RRA_SP(T)                                                                              \
    do {                                                                                       \
        const int cg = (int)std::max(1LL, std::min(wblocks, (long long)num_sms() *             \
                                                     blocks_per_sm(sparse_count_kernel<T>)));  \
        const int eg = (int)std::max(1LL, std::min(wblocks, (long long)num_sms() *             \
                                                     blocks_per_sm(sparse_emit_kernel<T>)));   \
        sparse_count_kernel<T><<<cg, kThreads, 0, st>>>(x, n, chunks, counts, vec);            \
        sparse_segscan_kernel<<<(unsigned)nseg, kScanThreads, 0, st>>>(counts, chunks, seg);   \
        sparse_segbase_kernel<<<1, kScanThreads, 0, st>>>(seg, nseg, lim, hdr);                \
        sparse_emit_kernel<T><<<eg, kThreads, 0, st>>>(x, n, chunks, counts, seg, hdr, vals,   \
                                                       idx, vec, quads);                       \
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
    // the dense stream's grid; its threads also cover the tiles + 1 starts
    const long long tiles = (n + kSpTile - 1) / kSpTile;
    const int g1 = grid_for((n + 7) / 8, kThreads);
    const int gf = (int)std::min<long long>(tiles, (long long)num_sms() * 8);
    // the format is in the device header: for a dense message the first
    // kernel does all the work and the fill returns at once
#define RRA_SD(T)                                                                                  \
    do {                                                                                           \
        sparse_prep_kernel<T><<<g1, kThreads, 0, st>>>(hdr, vals, idx, n, acc, scratch,            \
                                                       accumulate ? 1 : 0, vec);                   \
        sparse_fill_kernel<T><<<gf, kThreads, 0, st>>>(hdr, vals, idx, scratch, n, acc,            \
                                                       accumulate ? 1 : 0, vec);                   \
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

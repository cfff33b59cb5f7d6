// ring_kernel.cuh -- the fused two-pass ring for N simulated ranks on one
// sm_103a GPU ("从零实现集合通信", "两趟实现 ring allreduce"; "CCCL通信压缩库"
// §2.1-§2.2).
//
// Mapping.  One thread block runs the whole ring for one slice position t
// (TW = 256*G consecutive elements of every chunk) at a time; a persistent
// block loops over slice positions.  Simulated rank r is warp r mod W (a warp
// plays ceil(N/W) ranks).  Lane L of a warp holds G groups of 8 elements:
// group gi covers elements [256*gi + 8L, 256*gi + 8L + 8) of the slice, so a
// 128-element BFP block is one half-warp of one group.
//
// The ring edge r -> r+1 is a FIFO of K receive slots in shared memory owned
// by rank r+1, with a "full" and an "empty" mbarrier per slot: the sender
// waits for "empty", writes the encoded message, arrives on "full"; the
// receiver waits for "full", copies the message to registers, arrives on
// "empty" (before it sends, so even K = 1 cannot deadlock).  Every wait is
// bounded (time limit + a device status word): a rank that never publishes
// ends the launch with a latched error instead of a hang.
//
// Step g of one slice position (g = 1..2N-1 for the allreduce) for rank r
// always concerns chunk c = (r - g) mod N:
//   g = 1          reduce-scatter step 1: encode own x_r[c], send to r+1.
//   g = 2..N-1     reduce-scatter step g: receive the partial of chunk c, add
//                  own fp32 x_r[c] (ring order), encode, send.
//   g = N          owner: c = r; S_r = x_r[r] + received; allreduce: encode
//                  S_r once, output its decoded value and send the codes
//                  (allgather step 1); reduce-scatter: output S_r.
//   g = N+1..2N-2  allgather step g-N+1: receive codes of chunk c, output
//                  their decoded value, forward the same codes.
//   g = 2N-1       receive the last chunk (c = r+1), output, no send.
// Input slices are staged into shared memory with one-dimensional bulk async
// copies (cp.async.bulk + mbarrier transaction counts), D loads ahead per
// rank, on the fast path (16-byte aligned buffers and chunk sizes); the
// generic path loads elements directly with bounds checks.  Every index in
// the step loop advances incrementally: no division in the hot loop.
#pragma once

#include "rra_device.cuh"
#include "rra_kernels.h"

namespace rra {

// ---------------------------------------------------------------- BFP arithmetic
// Encode: the code m = clamp(rne(v * 2^k), +-M) with k = q - e is read from
// the bits of t = fma(v, 2^k, 1.5*2^23).  The exact v*2^k lies in
// (-2^(q+1), 2^(q+1)), so the exact sum lies in [2^23, 2^24) where the float
// grid spacing is 1: the fma's single rounding is round-to-nearest-even of
// v*2^k (the constant is even), and t's low byte is m in two's complement.
// Decode: the code byte xor 0x80 (nibble xor 0x8), placed under the upper
// bytes of 1.5*2^23 by a byte permute, is the float 1.5*2^23 + m + 2^(bits-1);
// subtracting that offset gives m exactly, m * 2^(e-q) is exact, and
// fma(m, 2^(e-q), x) is the correctly rounded x + decode(m).  No integer <->
// float conversion instruction is used.
constexpr float kMagic = 12582912.0f; // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;

template <int BITS> struct BfpGroup {
    static constexpr int q = BITS - 2;
    static constexpr int M = (1 << (BITS - 1)) - 1;

    // Codes of one lane's 8 values; e is the half-warp block exponent.
    // w[0..1] = 8 bytes (BITS 8) or w[0] = 8 nibbles (BITS 4).
    __device__ __forceinline__ static void encode(const float v[8], int &e, uint32_t w[2])
    {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        e = bfp_exponent(amax);
        int k = q - e;
        float x[8];
        float ax = amax;
        if (k > 127) { // blocks below 2^(q-127): pre-scale by an exact 2^64
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = __fmul_rn(v[i], 1.8446744073709552e19f);
            ax = __fmul_rn(amax, 1.8446744073709552e19f);
            k -= 64;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = v[i];
        }
        const float s = pow2i(k);
        float t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            t[i] = __fmaf_rn(x[i], s, kMagic);
        if (__fmul_rn(ax, s) >= (float)M + 0.5f) { // some value rounds past the clamp
#pragma unroll
            for (int i = 0; i < 8; ++i)
                t[i] = fminf(fmaxf(t[i], kMagic - (float)M), kMagic + (float)M);
        }
        uint32_t u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            u[i] = __float_as_uint(t[i]);
        const uint32_t b0 = __byte_perm(__byte_perm(u[0], u[1], 0x0040),
                                        __byte_perm(u[2], u[3], 0x0040), 0x5410);
        const uint32_t b1 = __byte_perm(__byte_perm(u[4], u[5], 0x0040),
                                        __byte_perm(u[6], u[7], 0x0040), 0x5410);
        if constexpr (BITS == 8) {
            w[0] = b0;
            w[1] = b1;
        } else {
            // bytes hold m & 0xff; pairs of low nibbles into one byte each
            uint32_t c0 = b0 & 0x0f0f0f0fu, c1 = b1 & 0x0f0f0f0fu;
            c0 |= c0 >> 4; // byte 0: n0 | n1 << 4, byte 2: n2 | n3 << 4
            c1 |= c1 >> 4;
            w[0] = __byte_perm(c0, c1, 0x6420);
            w[1] = 0;
        }
    }

    // m_i as exact floats.
    __device__ __forceinline__ static void codes(const uint32_t w[2], float mf[8])
    {
        constexpr float off = kMagic + (float)(1 << (BITS - 1));
        if constexpr (BITS == 8) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t x = w[h] ^ 0x80808080u;
                mf[4 * h + 0] = __uint_as_float(__byte_perm(x, kMagicBits, 0x7640)) - off;
                mf[4 * h + 1] = __uint_as_float(__byte_perm(x, kMagicBits, 0x7641)) - off;
                mf[4 * h + 2] = __uint_as_float(__byte_perm(x, kMagicBits, 0x7642)) - off;
                mf[4 * h + 3] = __uint_as_float(__byte_perm(x, kMagicBits, 0x7643)) - off;
            }
        } else {
            const uint32_t x = w[0] ^ 0x88888888u;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mf[i] = __uint_as_float(((x >> (4 * i)) & 0xfu) | kMagicBits) - off;
        }
    }

    // Decoded values m_i * 2^(e-q) (exact).
    __device__ __forceinline__ static void decode(const uint32_t w[2], int e, float out[8])
    {
        float mf[8];
        codes(w, mf);
        const float s = pow2i(e - q);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            out[i] = __fmul_rn(mf[i], s);
    }

    // acc_i = x_i + m_i * 2^(e-q) with one rounding (the product is exact).
    __device__ __forceinline__ static void decode_add(const uint32_t w[2], int e, const float x[8],
                                                      float acc[8])
    {
        float mf[8];
        codes(w, mf);
        const float s = pow2i(e - q);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = __fmaf_rn(mf[i], s, x[i]);
    }
};

// ---------------------------------------------------------------- wire formats
// A Wire holds one lane's share of a message in registers.
// All value arrays are updated in place (one array of 8G floats per lane
// keeps the register footprint small).
//  encode_store<DEC>: encode the lane's fp32 values v into a slot; with DEC,
//                     v is replaced by what a receiver decodes; returns the
//                     wire bytes.
//  load / store:      slot <-> registers (allgather forwarding); load returns
//                     the wire bytes.
//  decode_add:        v = v + decoded message (positions a sparse message
//                     does not carry keep v).
//  values:            v = decoded values (0 where a sparse message carries none).

template <int CODEC, int G> struct Wire;

template <int G> struct Wire<kCodecNone, G> {
    static constexpr int kSlot = kTile * 4 * G;
    float f[8 * G];
    template <bool DEC>
    __device__ __forceinline__ uint32_t encode_store(float (&v)[8 * G], int V, int lane,
                                                     unsigned char *slot, double, unsigned char *)
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float4 *p = reinterpret_cast<float4 *>(slot + gi * kTile * 4) + 2 * lane;
            p[0] = make_float4(v[8 * gi + 0], v[8 * gi + 1], v[8 * gi + 2], v[8 * gi + 3]);
            p[1] = make_float4(v[8 * gi + 4], v[8 * gi + 5], v[8 * gi + 6], v[8 * gi + 7]);
        }
        return 4u * (uint32_t)V;
    }
    __device__ __forceinline__ uint32_t load(const unsigned char *slot, int lane, int V)
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            const float4 *p = reinterpret_cast<const float4 *>(slot + gi * kTile * 4) + 2 * lane;
            const float4 a = p[0], b = p[1];
            f[8 * gi + 0] = a.x; f[8 * gi + 1] = a.y; f[8 * gi + 2] = a.z; f[8 * gi + 3] = a.w;
            f[8 * gi + 4] = b.x; f[8 * gi + 5] = b.y; f[8 * gi + 6] = b.z; f[8 * gi + 7] = b.w;
        }
        return 4u * (uint32_t)V;
    }
    __device__ __forceinline__ void store(unsigned char *slot, int lane) const
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float4 *p = reinterpret_cast<float4 *>(slot + gi * kTile * 4) + 2 * lane;
            p[0] = make_float4(f[8 * gi + 0], f[8 * gi + 1], f[8 * gi + 2], f[8 * gi + 3]);
            p[1] = make_float4(f[8 * gi + 4], f[8 * gi + 5], f[8 * gi + 6], f[8 * gi + 7]);
        }
    }
    __device__ __forceinline__ void decode_add(float (&v)[8 * G], int, unsigned char *) const
    {
#pragma unroll
        for (int i = 0; i < 8 * G; ++i)
            v[i] = __fadd_rn(v[i], f[i]);
    }
    __device__ __forceinline__ void values(float (&v)[8 * G], int, unsigned char *) const
    {
#pragma unroll
        for (int i = 0; i < 8 * G; ++i)
            v[i] = f[i];
    }
};

// Block floating point.  Slot: 16 bytes of exponents (2G used; byte b is the
// exponent of the slice's block b), then the mantissas in element order
// (group gi at 16 + gi * 256*BITS/8; lane L at 8L bytes (8-bit) or 4L bytes
// (4-bit) within the group).
template <int BITS, int G> struct WireBfp {
    static constexpr int kMB = kTile * BITS / 8;
    static constexpr int kSlot = 16 + kMB * G;
    uint32_t w[G][2];
    int e[G];
    template <bool DEC>
    __device__ __forceinline__ uint32_t encode_store(float (&v)[8 * G], int V, int lane,
                                                     unsigned char *slot, double, unsigned char *)
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            BfpGroup<BITS>::encode(v + 8 * gi, e[gi], w[gi]);
            if (DEC)
                BfpGroup<BITS>::decode(w[gi], e[gi], v + 8 * gi);
        }
        store(slot, lane);
        return bfp_msg_bytes(V, BITS);
    }
    __device__ __forceinline__ uint32_t load(const unsigned char *slot, int lane, int V)
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            e[gi] = (int)(int8_t)slot[2 * gi + (lane >> 4)];
            if constexpr (BITS == 8) {
                const uint2 u = reinterpret_cast<const uint2 *>(slot + 16 + gi * kMB)[lane];
                w[gi][0] = u.x;
                w[gi][1] = u.y;
            } else {
                w[gi][0] = reinterpret_cast<const uint32_t *>(slot + 16 + gi * kMB)[lane];
                w[gi][1] = 0;
            }
        }
        return bfp_msg_bytes(V, BITS);
    }
    __device__ __forceinline__ void store(unsigned char *slot, int lane) const
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            if ((lane & 15) == 0)
                slot[2 * gi + (lane >> 4)] = (unsigned char)(int8_t)e[gi];
            if constexpr (BITS == 8)
                reinterpret_cast<uint2 *>(slot + 16 + gi * kMB)[lane] =
                    make_uint2(w[gi][0], w[gi][1]);
            else
                reinterpret_cast<uint32_t *>(slot + 16 + gi * kMB)[lane] = w[gi][0];
        }
    }
    __device__ __forceinline__ void decode_add(float (&v)[8 * G], int, unsigned char *) const
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
            BfpGroup<BITS>::decode_add(w[gi], e[gi], v + 8 * gi, v + 8 * gi);
    }
    __device__ __forceinline__ void values(float (&v)[8 * G], int, unsigned char *) const
    {
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
            BfpGroup<BITS>::decode(w[gi], e[gi], v + 8 * gi);
    }
};
template <int G> struct Wire<kCodecBfp8, G> : WireBfp<8, G> {};
template <int G> struct Wire<kCodecBfp4, G> : WireBfp<4, G> {};

// Sparse values + indices (one 256-element slice per message, G = 1).
// Slot: {uint32 fmt, uint32 nnz} padded to 16 bytes, fp32 values[256],
// int32 indices[256] (slice-relative, ascending).  Dense fallback: fmt 0,
// values[0..len) in place.  Compaction: per-lane nonzero masks and a warp
// inclusive scan of their popcounts give every lane's first output position.
template <> struct Wire<kCodecSparse, 1> {
    static constexpr int kSlot = 16 + kTile * 8;
    uint32_t fmt, nnz;
    float f[8];
    int ix[8];
    __device__ __forceinline__ static float *vals(unsigned char *s)
    {
        return reinterpret_cast<float *>(s + 16);
    }
    __device__ __forceinline__ static int *idxs(unsigned char *s)
    {
        return reinterpret_cast<int *>(s + 16 + kTile * 4);
    }
    __device__ __forceinline__ uint32_t bytes(int V) const
    {
        return V == 0 ? 0u : 8u + (fmt ? 8u * nnz : 4u * (uint32_t)V);
    }
    template <bool DEC>
    __device__ __forceinline__ uint32_t encode_store(float (&acc)[8], int V, int lane,
                                                     unsigned char *slot, double one_minus_thr,
                                                     unsigned char *)
    {
        // the receiver restores every value exactly (absent ones are +0.0),
        // so the decoded values are acc itself
        uint32_t nzm = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (8 * lane + i < V && __float_as_uint(acc[i]) != 0u)
                nzm |= 1u << i;
        }
        const int cnt = __popc(nzm);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += t;
        }
        const int total = __shfl_sync(kFull, incl, 31);
        fmt = (double)total < one_minus_thr * (double)V ? 1u : 0u;
        nnz = (uint32_t)total;
        if (lane == 0)
            *reinterpret_cast<uint2 *>(slot) = make_uint2(fmt, nnz);
        if (fmt) {
            int pos = incl - cnt;
            float *v = vals(slot);
            int *x = idxs(slot);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((nzm >> i) & 1u) {
                    v[pos] = acc[i];
                    x[pos] = 8 * lane + i;
                    ++pos;
                }
        } else {
            float4 *p = reinterpret_cast<float4 *>(vals(slot)) + 2 * lane;
            p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        return bytes(V);
    }
    __device__ __forceinline__ uint32_t load(const unsigned char *slot, int lane, int V)
    {
        const uint2 h = *reinterpret_cast<const uint2 *>(slot);
        fmt = h.x;
        nnz = h.y;
        unsigned char *s = const_cast<unsigned char *>(slot);
        if (!fmt) {
            const float4 *p = reinterpret_cast<const float4 *>(vals(s)) + 2 * lane;
            const float4 a = p[0], b = p[1];
            f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
            f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = lane + 32 * i;
                if (k < (int)nnz) {
                    f[i] = vals(s)[k];
                    ix[i] = idxs(s)[k];
                }
            }
        }
        return bytes(V);
    }
    __device__ __forceinline__ void store(unsigned char *slot, int lane) const
    {
        if (lane == 0)
            *reinterpret_cast<uint2 *>(slot) = make_uint2(fmt, nnz);
        if (!fmt) {
            float4 *p = reinterpret_cast<float4 *>(vals(slot)) + 2 * lane;
            p[0] = make_float4(f[0], f[1], f[2], f[3]);
            p[1] = make_float4(f[4], f[5], f[6], f[7]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = lane + 32 * i;
                if (k < (int)nnz) {
                    vals(slot)[k] = f[i];
                    idxs(slot)[k] = ix[i];
                }
            }
        }
    }
    // Sparse messages: scatter the pairs into the warp's scratch (values +
    // presence bytes), then read this lane's 8 positions.
    __device__ __forceinline__ uint32_t gather(int lane, unsigned char *scratch, float v[8]) const
    {
        if (!fmt) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = f[i];
            return 0xffu;
        }
        float *sval = reinterpret_cast<float *>(scratch);
        unsigned char *spres = scratch + kTile * 4;
        *reinterpret_cast<uint2 *>(spres + 8 * lane) = make_uint2(0u, 0u);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = lane + 32 * i;
            if (k < (int)nnz) {
                sval[ix[i]] = f[i];
                spres[ix[i]] = 1;
            }
        }
        __syncwarp();
        uint32_t pres = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (spres[8 * lane + i]) {
                pres |= 1u << i;
                v[i] = sval[8 * lane + i];
            } else {
                v[i] = 0.0f;
            }
        }
        __syncwarp();
        return pres;
    }
    __device__ __forceinline__ void decode_add(float (&x)[8], int lane,
                                               unsigned char *scratch) const
    {
        float v[8];
        const uint32_t pres = gather(lane, scratch, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            x[i] = ((pres >> i) & 1u) ? __fadd_rn(x[i], v[i]) : x[i];
    }
    __device__ __forceinline__ void values(float (&v)[8], int lane, unsigned char *scratch) const
    {
        gather(lane, scratch, v);
    }
};

// ---------------------------------------------------------------- helpers

// Bounded wait used only to drain this warp's own bulk copies before exit:
// it ignores the status word (copies in flight must land before the block's
// shared memory is released) and gives up only at the time limit.
__device__ __forceinline__ void drain_phase(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns)
            break;
}

// A (slot, phase) position in a FIFO of depth n, advanced without division.
struct Fifo {
    int slot, phase;
    __device__ __forceinline__ void advance(int n)
    {
        if (++slot == n) {
            slot = 0;
            phase ^= 1;
        }
    }
};

// ---------------------------------------------------------------- kernel

template <int CODEC, int IN_T, bool FAST, int G>
__global__ void __launch_bounds__(kMaxWarps * 32, 2) ring_kernel(const __grid_constant__ RingArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    using Msg = Wire<CODEC, G>;
    constexpr int es = dtype_size(IN_T);
    constexpr int TW = kTile * G; // elements per rank per step
    const int N = a.N;
    const int W = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int K = a.K, D = a.D;
    const Layout Lo =
        make_layout(N, K, D, a.slot_bytes, a.stage_bytes, W, FAST, CODEC == kCodecSparse);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lo.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + Lo.empty);
    uint64_t *sbar = reinterpret_cast<uint64_t *>(smem + Lo.stage_bar);
    unsigned long long *rsent = reinterpret_cast<unsigned long long *>(smem + Lo.rank_state);
    unsigned long long *rrecv = rsent + N;
    unsigned char *slots = smem + Lo.slots;
    unsigned char *stages = smem + Lo.stages;
    unsigned char *scratch = smem + Lo.scratch + warp * (kTile * 4 + kTile);

    for (int i = threadIdx.x; i < N * K; i += blockDim.x) {
        mbar_init(full + i, 1);
        mbar_init(empty + i, 1);
    }
    if constexpr (FAST)
        for (int i = threadIdx.x; i < N * D; i += blockDim.x)
            mbar_init(sbar + i, 1);
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        rsent[i] = 0;
        rrecv[i] = 0;
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < 2 * N; i += blockDim.x)
            a.zero[i] = 0ull;
    mbar_fence_init();
    __syncthreads();

    const bool allred = a.mode == kModeAllreduce;
    const int Gs = allred ? 2 * N - 1 : N; // steps per slice position
    const int M = allred ? 2 * N - 2 : N - 1;
    const long long n = a.n, T = a.T;
    const int out_es = dtype_size(a.out_t);
    // shortest chunk: every slice position below it is full in every chunk
    const long long min_len = T - (long long)(N - 1) * n;

    auto slice_len = [&](int c, long long t0) -> int {
        if (t0 + TW <= min_len)
            return TW;
        long long lo = (long long)c * n, hi = lo + n;
        lo = lo < T ? lo : T;
        hi = hi < T ? hi : T;
        const long long v = hi - lo - t0;
        return (int)(v < 0 ? 0 : (v > TW ? TW : v));
    };

    // ---- staged input loads.  All ranks consume loads in the same order
    // (slice iteration, step 1..N), so one cursor gives the next load to
    // issue for every rank; "issued" and "consumed" count loads per rank.
    long long cur_item = blockIdx.x; // slice position of the next load to issue
    int cur_g = 1;                   // its step
    long long issued = 0, consumed = 0;
    auto issue_one = [&](int r, int d) { // lane 0: load (cur_item, cur_g) of rank r into stage d
        int c = r - cur_g;
        c += c < 0 ? N : 0;
        const long long t0 = cur_item * TW;
        const uint32_t bytes = (uint32_t)slice_len(c, t0) * es;
        uint64_t *bar = sbar + r * D + d;
        unsigned char *dst = stages + (size_t)(r * D + d) * a.stage_bytes;
        if (bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        const long long eo = (long long)c * n + t0;
        const char *src = reinterpret_cast<const char *>(a.in[r]) + eo * es;
        if (a.has_prev) {
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_g2s(dst, src, bytes, bar);
            bulk_g2s(dst + TW * 4, a.prev[r] + eo, bytes, bar);
        } else {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(dst, src, bytes, bar);
        }
    };
    auto cursor_next = [&]() {
        if (++cur_g > N) {
            cur_g = 1;
            cur_item += gridDim.x;
        }
    };
    if constexpr (FAST) {
        while (issued < D && cur_item < a.tiles) {
            if (lane == 0)
                for (int r = warp; r < N; r += W)
                    issue_one(r, (int)issued);
            ++issued;
            cursor_next();
        }
        __syncwarp();
    }

    Fifo rcv{0, 0}, snd{0, 0}, stg{0, 0};
    bool ok = true;
    long long j = 0;
    for (long long item = blockIdx.x; ok && item < a.tiles; item += gridDim.x, ++j) {
        const long long t0 = item * TW;
        for (int g = 1; ok && g <= Gs; ++g) {
            const bool do_recv = g >= 2;
            const bool do_send = g <= M;
            const bool rs_part = g <= N;
            for (int r = warp; r < N; r += W) {
                int c = r - g;
                c += c < 0 ? N : 0;
                c += c < 0 ? N : 0;
                const int V = slice_len(c, t0);
                const long long ebase = (long long)c * n + t0 + 8 * lane;

                // ---- own input (reduce-scatter steps and the owner step)
                float v[8 * G];
                if (rs_part) {
                    if constexpr (FAST) {
                        ok = wait_phase(sbar + r * D + stg.slot, (uint32_t)stg.phase,
                                        a.timeout_ns, a.status);
                        if (!ok)
                            break;
                        const unsigned char *sp =
                            stages + (size_t)(r * D + stg.slot) * a.stage_bytes;
#pragma unroll
                        for (int gi = 0; gi < G; ++gi)
                            load8_vec<IN_T>(sp + (gi * kTile + 8 * lane) * es, v + 8 * gi);
                        if (a.has_prev) {
#pragma unroll
                            for (int gi = 0; gi < G; ++gi) {
                                float p[8];
                                load8_vec<kF32>(sp + TW * 4 + (gi * kTile + 8 * lane) * 4, p);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    v[8 * gi + i] = __fsub_rn(v[8 * gi + i], p[i]);
                            }
                        }
                        if (V < TW) {
#pragma unroll
                            for (int gi = 0; gi < G; ++gi)
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    if (gi * kTile + 8 * lane + i >= V)
                                        v[8 * gi + i] = 0.0f;
                        }
                    } else {
#pragma unroll
                        for (int gi = 0; gi < G; ++gi) {
                            const int vl = min(max(V - gi * kTile - 8 * lane, 0), 8);
                            const long long eo = ebase + gi * kTile;
                            load8_scalar<IN_T>(reinterpret_cast<const char *>(a.in[r]) + eo * es,
                                               vl, v + 8 * gi);
                            if (a.has_prev) {
                                float p[8];
                                load8_scalar<kF32>(a.prev[r] + eo, vl, p);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    v[8 * gi + i] = __fsub_rn(v[8 * gi + i], p[i]);
                            }
                        }
                    }
                }

                // ---- receive from rank r-1 (steps 2..Gs)
                Msg w;
                uint32_t rb = 0;
                if (do_recv) {
                    ok = wait_phase(full + r * K + rcv.slot, (uint32_t)rcv.phase, a.timeout_ns,
                                    a.status);
                    if (!ok)
                        break;
                    rb = w.load(slots + (size_t)(r * K + rcv.slot) * a.slot_bytes, lane, V);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(empty + r * K + rcv.slot);
                        rrecv[r] += rb;
                    }
                }

                // ---- reserve the slot of rank r+1
                const int dst = r + 1 == N ? 0 : r + 1;
                unsigned char *dslot = nullptr;
                if (do_send) {
                    ok = wait_phase(empty + dst * K + snd.slot, (uint32_t)(snd.phase ^ 1),
                                    a.timeout_ns, a.status);
                    if (!ok)
                        break;
                    dslot = slots + (size_t)(dst * K + snd.slot) * a.slot_bytes;
                }

                // ---- compute (in place in v)
                bool do_out = false;
                uint32_t sb = 0;
                if (rs_part) {
                    if (do_recv)
                        w.decode_add(v, lane, scratch);
                    Msg ws;
                    if (g < N) {
                        sb = ws.template encode_store<false>(v, V, lane, dslot, a.one_minus_thr,
                                                             scratch);
                    } else {
                        do_out = true;
                        if (allred) {
                            // N = 1 has no allgather step: encode into the rank's
                            // own (otherwise unused) mailbox slot for its output
                            unsigned char *es_slot =
                                dslot ? dslot : slots + (size_t)(r * K) * a.slot_bytes;
                            sb = ws.template encode_store<true>(v, V, lane, es_slot,
                                                                a.one_minus_thr, scratch);
                            if (!dslot)
                                sb = 0;
                        }
                    }
                } else {
                    w.values(v, lane, scratch);
                    do_out = true;
                    if (do_send) { // allgather: forward the received codes unchanged
                        w.store(dslot, lane);
                        sb = rb;
                    }
                }
                if (do_send) {
                    __syncwarp();
                    if (lane == 0) {
                        if (!(r == a.withhold_rank && g == a.withhold_step && j == 0))
                            mbar_arrive(full + dst * K + snd.slot);
                        rsent[r] += sb;
                    }
                }

                // ---- output epilogue: average, previous-round base, cast
                if (do_out) {
#pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
                        const int vl = min(max(V - gi * kTile - 8 * lane, 0), 8);
                        const long long eo = ebase + gi * kTile;
                        float wv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            wv[i] = a.average ? __fdiv_rn(v[8 * gi + i], (float)N)
                                              : v[8 * gi + i];
                        if (a.base) {
                            float bb[8];
                            if (a.vec_base && vl == 8)
                                load8_vec<kF32>(a.base + eo, bb);
                            else
                                load8_scalar<kF32>(a.base + eo, vl, bb);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                wv[i] = __fadd_rn(bb[i], wv[i]);
                        }
                        store8(reinterpret_cast<char *>(a.out[r]) + eo * out_es, a.out_t, wv,
                               vl, a.vec_out != 0);
                    }
                }
            }
            if (!ok)
                break;
            // ---- refill the consumed stage and advance the shared counters
            if (FAST && rs_part) {
                __syncwarp();
                if (issued == consumed + D && cur_item < a.tiles) {
                    if (lane == 0)
                        for (int r = warp; r < N; r += W)
                            issue_one(r, stg.slot);
                    ++issued;
                    cursor_next();
                }
                ++consumed;
                stg.advance(D);
            }
            if (do_recv)
                rcv.advance(K);
            if (do_send)
                snd.advance(K);
        }
    }

    // ---- drain this warp's staged copies that are still in flight
    if constexpr (FAST) {
        __syncwarp();
        for (int r = warp; r < N; r += W)
            for (long long L = consumed; L < issued; ++L)
                drain_phase(sbar + r * D + (int)(L % D), (uint32_t)((L / D) & 1), a.timeout_ns);
    }
    // ---- per-rank byte counters
    if (lane == 0)
        for (int r = warp; r < N; r += W) {
            if (rsent[r])
                atomicAdd(a.sent + r, rsent[r]);
            if (rrecv[r])
                atomicAdd(a.recv + r, rrecv[r]);
        }
}

} // namespace rra

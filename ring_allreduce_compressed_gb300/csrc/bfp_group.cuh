// bfp_group.cuh -- block floating point arithmetic on one warp's 256
// elements (two 128-element blocks, one per half-warp; 8 elements a lane),
// shared by the fused ring and the standalone BFP codec kernels ("CCCL通信
// 压缩库" §2.1: one shared exponent per block, a fixed-width signed mantissa
// per element).
#pragma once

#include "rra_device.cuh"

namespace rra {

// ---------------------------------------------------------------- BFP arithmetic
// Encode: the code m = clamp(rne(v * 2^k), +-M) with k = q - e is read from
// the bits of t = fma(v, 2^k, 1.5*2^23 + 2^(bits-1)).  The exact v*2^k lies
// in (-2^(q+1), 2^(q+1)), so the exact sum lies in [2^23, 2^24) where the
// float grid spacing is 1: the fma's single rounding is round-to-nearest-even
// of v*2^k (the constant is an even integer), and t's low byte (nibble) is the
// offset code m + 2^(bits-1), always in [1, 2^bits - 1].  Inside the ring a
// message carries these offset codes (the standalone codec entry points write
// two's complement, as their interface states).
// Decode: the offset code placed under the upper bytes of 1.5*2^23 by a byte
// permute is the float F = 1.5*2^23 + m + 2^(bits-1).  fma(F, 2^-q,
// -(1.5*2^23 + 2^(bits-1)) * 2^-q) = m * 2^-q exactly (every term is a
// power-of-two multiple of an exact float and the result is representable),
// and fma(m * 2^-q, 2^e, x) is the correctly rounded x + m * 2^(e-q): the
// product is exact.  2^e is a normal float for every block exponent e in
// [-126, 127], so no case split is needed.  No integer <-> float conversion
// instruction is used.
constexpr float kMagic = 12582912.0f; // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;

template <int BITS> struct BfpGroup {
    static constexpr int q = BITS - 2;
    static constexpr int M = (1 << (BITS - 1)) - 1;
    static constexpr float kEnc = kMagic + (float)(1 << (BITS - 1)); // code offset folded in
    static constexpr float kInvQ = 1.0f / (float)(1 << q);           // 2^-q

    // 2^e for a block exponent e in [-126, 127] (always a normal float).
    __device__ __forceinline__ static float scale(int e) { return __int_as_float((e + 127) << 23); }

    // Offset codes of one lane's 8 values; e is the half-warp block exponent.
    // w[0..1] = 8 bytes (BITS 8) or w[0] = 8 nibbles (BITS 4).
    __device__ __forceinline__ static void encode(const float v[8], int &e, uint32_t w[2])
    {
        float lmax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            lmax = fmaxf(lmax, fabsf(v[i]));
        // half-warp maximum: non-negative floats order like their bit patterns,
        // so two warp-wide unsigned max reductions (one per half) give it
        const unsigned lane = threadIdx.x & 31u;
        const unsigned bits = __float_as_uint(lmax);
        const unsigned lo = __reduce_max_sync(kFull, lane < 16 ? bits : 0u);
        const unsigned hi = __reduce_max_sync(kFull, lane < 16 ? 0u : bits);
        const unsigned ab = lane < 16 ? lo : hi;
        // biased exponent of the maximum; zero and subnormal maxima count as
        // biased 1, i.e. e = -126
        const int E = max((int)(ab >> 23), 1);
        e = E - 127;
        // 2^k with k = q - e = q + 127 - E: a normal float unless E < q, a
        // block below 2^(q-126) that is first scaled up by an exact 2^64
        float x[8];
        float ax = __uint_as_float(ab);
        int sb = q + 254 - E; // biased exponent of 2^k
        if (E < q) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = __fmul_rn(v[i], 1.8446744073709552e19f);
            ax = __fmul_rn(ax, 1.8446744073709552e19f);
            sb -= 64;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = v[i];
        }
        const float s = __int_as_float(sb << 23);
        float t[8];
        const float2 s2 = make_float2(s, s), c2 = make_float2(kEnc, kEnc);
#pragma unroll
        for (int i = 0; i < 8; i += 2) { // paired fp32 fma: two IEEE fmas per instruction
            const float2 r = __ffma2_rn(make_float2(x[i], x[i + 1]), s2, c2);
            t[i] = r.x;
            t[i + 1] = r.y;
        }
        if (__fmul_rn(ax, s) >= (float)M + 0.5f) { // some value rounds past the clamp
#pragma unroll
            for (int i = 0; i < 8; ++i)
                t[i] = fminf(fmaxf(t[i], kEnc - (float)M), kEnc + (float)M);
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
            // every byte holds an offset code below 16: pairs of them into one
            // byte each (byte 0: n0 | n1 << 4, byte 2: n2 | n3 << 4)
            const uint32_t c0 = b0 | (b0 >> 4), c1 = b1 | (b1 >> 4);
            w[0] = __byte_perm(c0, c1, 0x6420);
            w[1] = 0;
        }
    }

    // m_i * 2^-q as exact floats, in pairs (element 2j in .x, 2j+1 in .y).
    __device__ __forceinline__ static void codes(const uint32_t w[2], float2 mf[4])
    {
        constexpr float off = -(kMagic + (float)(1 << (BITS - 1))) * kInvQ;
        const float2 iq2 = make_float2(kInvQ, kInvQ), off2 = make_float2(off, off);
        if constexpr (BITS == 8) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t x = w[h];
                mf[2 * h + 0] = __ffma2_rn(
                    make_float2(__uint_as_float(__byte_perm(x, kMagicBits, 0x7640)),
                                __uint_as_float(__byte_perm(x, kMagicBits, 0x7641))),
                    iq2, off2);
                mf[2 * h + 1] = __ffma2_rn(
                    make_float2(__uint_as_float(__byte_perm(x, kMagicBits, 0x7642)),
                                __uint_as_float(__byte_perm(x, kMagicBits, 0x7643))),
                    iq2, off2);
            }
        } else {
            const uint32_t x = w[0];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mf[j] = __ffma2_rn(
                    make_float2(__uint_as_float(((x >> (8 * j)) & 0xfu) | kMagicBits),
                                __uint_as_float(((x >> (8 * j + 4)) & 0xfu) | kMagicBits)),
                    iq2, off2);
        }
    }

    // Decoded values m_i * 2^(e-q) (exact).
    __device__ __forceinline__ static void decode(const uint32_t w[2], int e, float out[8])
    {
        float2 mf[4];
        codes(w, mf);
        const float s = scale(e);
        const float2 s2 = make_float2(s, s);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 r = __fmul2_rn(mf[j], s2);
            out[2 * j] = r.x;
            out[2 * j + 1] = r.y;
        }
    }

    // acc_i = x_i + m_i * 2^(e-q) with one rounding (the product is exact).
    __device__ __forceinline__ static void decode_add(const uint32_t w[2], int e, const float x[8],
                                                      float acc[8])
    {
        float2 mf[4];
        codes(w, mf);
        const float s = scale(e);
        const float2 s2 = make_float2(s, s);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 r = __ffma2_rn(mf[j], s2, make_float2(x[2 * j], x[2 * j + 1]));
            acc[2 * j] = r.x;
            acc[2 * j + 1] = r.y;
        }
    }
};

} // namespace rra

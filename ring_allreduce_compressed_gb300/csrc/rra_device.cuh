// rra_device.cuh -- device building blocks shared by the sm_103a kernels:
// PTX wrappers (mbarrier, bulk async copy, global timer), bounded waits,
// the per-warp tile layout, dtype conversions and the block-floating-point
// arithmetic.
//
// Tile layout used everywhere: a warp handles a slice of 256 elements; lane L
// holds elements [8L, 8L+8).  A 128-element BFP block is therefore one
// half-warp (lanes 0-15 and 16-31).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rra {

constexpr int kTile = 256;       // elements per warp slice (= RRA_RING_SLICE)
constexpr int kEpl = 8;          // elements per lane
constexpr int kBlock = 128;      // BFP block (= RRA_BFP_BLOCK)
constexpr unsigned kFull = 0xffffffffu;

enum Dtype { kF32 = 0, kF16 = 1, kBF16 = 2 };
// Ring kernel input kind: fp32 inputs cur together with a second fp32 stream
// prev, sent as the difference cur - prev.
constexpr int kF32Diff = 3;
enum Status : unsigned { kStOk = 0, kStTimeout = 4 };

__host__ __device__ constexpr int dtype_size(int t) { return t == kF32 || t == kF32Diff ? 4 : 2; }

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once (release at CTA scope: prior shared-memory writes of this
// thread, and those ordered before it by a warp barrier, become visible to a
// thread that observes the phase flip with an acquire wait).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t tx)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(tx)
                 : "memory");
}

// One test of an mbarrier phase (acquire on success); it may block for a
// short, hardware-chosen time before returning false.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// One-dimensional bulk copy global -> this CTA's shared memory, completing
// "bytes" transaction bytes on the mbarrier.  dst and src 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Warp-uniform bounded wait for the phase of parity "parity" of an mbarrier.
// Every lane waits (each gets acquire ordering).  The common case -- the
// neighbour publishes within microseconds -- touches nothing but the
// mbarrier: the clock is read every 256 polls, and the device status word
// (an error latched by another warp) only once the wait has lasted more than
// kPollAfterNs, so no global-memory round trip sits on the critical path.
// Gives up at the time limit (latching kStTimeout) or when another warp has
// latched an error.  Returns true iff every lane saw the phase complete.
constexpr uint64_t kPollAfterNs = 20000;

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                           unsigned *status)
{
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = global_ns();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait(bar, parity)) {
                ok = true;
                break;
            }
            if ((it & 255u) == 0u) {
                const uint64_t dt = global_ns() - t0;
                if (dt > kPollAfterNs && *reinterpret_cast<volatile unsigned *>(status) != 0u)
                    break;
                if (dt > limit_ns) {
                    atomicCAS(status, 0u, (unsigned)kStTimeout);
                    break;
                }
            }
        }
    }
    return __all_sync(kFull, ok);
}

// ---------------------------------------------------------------- mailbox helpers

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

// Rare path of a wait (the phase was not complete at the first test): kept
// out of line so that the common path stays a few instructions.
static __device__ __noinline__ bool wait_slow(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                              unsigned *status)
{
    return wait_phase(bar, parity, limit_ns, status);
}

// Warp-uniform: true once every lane has observed the phase (acquire).
__device__ __forceinline__ bool wait_ready(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                           unsigned *status)
{
    if (__all_sync(kFull, mbar_try_wait(bar, parity)))
        return true;
    return wait_slow(bar, parity, limit_ns, status);
}

// ---------------------------------------------------------------- dtypes

template <int T> struct Elem;
template <> struct Elem<kF32> {
    using type = float;
};
template <> struct Elem<kF16> {
    using type = __half;
};
template <> struct Elem<kBF16> {
    using type = __nv_bfloat16;
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 8 consecutive elements of dtype IN_T at p (16-byte aligned for 16-bit
// types, 32-byte for fp32) widened to fp32.
template <int IN_T> __device__ __forceinline__ void load8_vec(const void *p, float v[8])
{
    if constexpr (IN_T == kF32) {
        const float4 a = reinterpret_cast<const float4 *>(p)[0];
        const float4 b = reinterpret_cast<const float4 *>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        using E = typename Elem<IN_T>::type;
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const E *e = reinterpret_cast<const E *>(&u);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = to_f32(e[i]);
    }
}

// Bounds-checked element loads (any alignment); absent elements read as 0.
template <int IN_T>
__device__ __forceinline__ void load8_scalar(const void *base, int valid, float v[8])
{
    using E = typename Elem<IN_T>::type;
    const E *p = reinterpret_cast<const E *>(base);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = i < valid ? to_f32(p[i]) : 0.0f;
}

__device__ __forceinline__ uint16_t f32_to_16(float v, int t)
{
    if (t == kF16)
        return __half_as_ushort(__float2half_rn(v));
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// 8 fp32 values as 4 packed pairs of 16-bit out_t (round to nearest even).
template <int OUT_T> __device__ __forceinline__ void pack16x8(const float v[8], uint32_t h[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (OUT_T == kF16) {
            const __half2 p = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            h[i] = *reinterpret_cast<const uint32_t *>(&p);
        } else {
            const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            h[i] = *reinterpret_cast<const uint32_t *>(&p);
        }
    }
}

// Store 8 fp32 values as out_t (round to nearest even); vectorised when the
// destination is 16-byte aligned and all 8 are present.  Each output type
// has its own straight-line path, so a runtime out_t costs one branch.
__device__ __forceinline__ void store8(void *base, int out_t, const float v[8], int valid,
                                       bool vec)
{
    if (out_t == kF32) {
        float *p = reinterpret_cast<float *>(base);
        if (vec && valid >= 8) {
            reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < valid)
                    p[i] = v[i];
        }
        return;
    }
    uint32_t h[4];
    if (out_t == kF16)
        pack16x8<kF16>(v, h);
    else
        pack16x8<kBF16>(v, h);
    uint16_t *p = reinterpret_cast<uint16_t *>(base);
    if (vec && valid >= 8) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid)
                p[i] = (uint16_t)(h[i / 2] >> (16 * (i % 2)));
    }
}

// Full, aligned group of 8: a 16-byte (or two) vector store of out_t.
__device__ __forceinline__ void store8_full(void *p, int out_t, const float v[8])
{
    if (out_t == kF32) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
        return;
    }
    uint32_t h[4];
    if (out_t == kF16)
        pack16x8<kF16>(v, h);
    else
        pack16x8<kBF16>(v, h);
    *reinterpret_cast<uint4 *>(p) = make_uint4(h[0], h[1], h[2], h[3]);
}

// ---------------------------------------------------------------- BFP

// Wire bytes of one BFP message covering len elements.
__host__ __device__ __forceinline__ uint32_t bfp_msg_bytes(int len, int bits)
{
    return (uint32_t)((len + kBlock - 1) / kBlock + (bits == 8 ? len : (len + 1) / 2));
}

} // namespace rra

// ring_kernel.cuh -- the fused two-pass ring for N simulated ranks on one
// sm_103a GPU ("从零实现集合通信", "两趟实现 ring allreduce"; "CCCL通信压缩库"
// §2.1-§2.2).
//
// Mapping.  One thread block runs the whole ring for one 256-element slice
// position t of every chunk at a time (a persistent block loops over slice
// positions).  Simulated rank r is warp r mod W (a warp plays ceil(N/W)
// ranks).  The ring edge r -> r+1 is a FIFO of K receive slots in shared
// memory owned by rank r+1, with a "full" and an "empty" mbarrier per slot:
// the sender waits for "empty", writes the encoded message, arrives on
// "full"; the receiver waits for "full", copies the message out, arrives on
// "empty".  Every wait is bounded (time limit + a device status word), so a
// rank that never publishes ends the launch with a latched error instead of
// a hang.
//
// Step g of one slice position (g = 1..2N-1 for the allreduce) for rank r
// always concerns chunk c = (r - g) mod N:
//   g = 1          reduce-scatter step 1: encode own x_r[c], send to r+1.
//   g = 2..N-1     reduce-scatter step g: receive partial of chunk c, add own
//                  fp32 x_r[c] (ring order), encode, send.
//   g = N          owner: c = r; S_r = x_r[r] + received; allreduce: encode
//                  S_r once, output its decoded value and send the codes
//                  (allgather step 1); reduce-scatter: output S_r.
//   g = N+1..2N-2  allgather step g-N+1: receive codes of chunk c, output
//                  their decoded value, forward the same codes.
//   g = 2N-1       receive the last chunk (c = r+1), output, no send.
// Input slices are staged into shared memory with one-dimensional bulk
// async copies (cp.async.bulk + mbarrier transaction counts), D loads ahead
// per rank, on the fast path (16-byte aligned buffers and chunk sizes); the
// generic path loads elements directly with bounds checks.
#pragma once

#include "rra_device.cuh"
#include "rra_kernels.h"

namespace rra {

__device__ __forceinline__ int mod_n(int a, int n)
{
    int m = a % n;
    return m < 0 ? m + n : m;
}

// ---------------------------------------------------------------- wire formats
// Each Wire<> holds one lane's share of a message in registers.
//  encode_store: encode the lane's fp32 values into a slot; dec receives what
//                a receiver decodes (the owner outputs it); returns wire bytes.
//  load / store: copy a message slot <-> registers (allgather forwarding).
//  decode:       the lane's 8 values and a presence mask (sparse slices
//                carry only some positions).

template <int CODEC> struct Wire;

template <> struct Wire<kCodecNone> {
    static constexpr int kSlot = kTile * 4;
    float f[8];
    __device__ __forceinline__ uint32_t encode_store(const float acc[8], int V, int lane,
                                                     unsigned char *slot, double, float dec[8])
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            f[i] = acc[i];
            dec[i] = acc[i];
        }
        store(slot, lane);
        return 4u * (uint32_t)V;
    }
    __device__ __forceinline__ uint32_t load(const unsigned char *slot, int lane, int V)
    {
        const float4 *p = reinterpret_cast<const float4 *>(slot) + 2 * lane;
        const float4 a = p[0], b = p[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        return 4u * (uint32_t)V;
    }
    __device__ __forceinline__ void store(unsigned char *slot, int lane) const
    {
        float4 *p = reinterpret_cast<float4 *>(slot) + 2 * lane;
        p[0] = make_float4(f[0], f[1], f[2], f[3]);
        p[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __device__ __forceinline__ uint32_t decode(int, unsigned char *, float v[8]) const
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = f[i];
        return 0xffu;
    }
};

// Block floating point.  Slot: 16 bytes of exponents (2 used), then the
// mantissas (8 bytes per lane at 8 bits, 4 bytes per lane at 4 bits).
template <int BITS> struct WireBfp {
    static constexpr int kSlot = 16 + kTile * BITS / 8;
    uint32_t c0, c1;
    int e;
    __device__ __forceinline__ uint32_t encode_store(const float acc[8], int V, int lane,
                                                     unsigned char *slot, double, float dec[8])
    {
        e = bfp_exponent(halfwarp_absmax(acc));
        int m[8];
        bfp_codes<BITS>(acc, e, m);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dec[i] = bfp_value<BITS>(m[i], e);
        if constexpr (BITS == 8) {
            const uint2 u = pack8(m);
            c0 = u.x;
            c1 = u.y;
        } else {
            c0 = pack4(m);
            c1 = 0;
        }
        store(slot, lane);
        return bfp_msg_bytes(V, BITS);
    }
    __device__ __forceinline__ uint32_t load(const unsigned char *slot, int lane, int V)
    {
        e = (int)(int8_t)slot[lane >> 4];
        if constexpr (BITS == 8) {
            const uint2 u = reinterpret_cast<const uint2 *>(slot + 16)[lane];
            c0 = u.x;
            c1 = u.y;
        } else {
            c0 = reinterpret_cast<const uint32_t *>(slot + 16)[lane];
            c1 = 0;
        }
        return bfp_msg_bytes(V, BITS);
    }
    __device__ __forceinline__ void store(unsigned char *slot, int lane) const
    {
        if ((lane & 15) == 0)
            slot[lane >> 4] = (unsigned char)(int8_t)e;
        if constexpr (BITS == 8)
            reinterpret_cast<uint2 *>(slot + 16)[lane] = make_uint2(c0, c1);
        else
            reinterpret_cast<uint32_t *>(slot + 16)[lane] = c0;
    }
    __device__ __forceinline__ uint32_t decode(int, unsigned char *, float v[8]) const
    {
        int m[8];
        if constexpr (BITS == 8)
            unpack8(make_uint2(c0, c1), m);
        else
            unpack4(c0, m);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = bfp_value<BITS>(m[i], e);
        return 0xffu;
    }
};
template <> struct Wire<kCodecBfp8> : WireBfp<8> {};
template <> struct Wire<kCodecBfp4> : WireBfp<4> {};

// Sparse values + indices.  Slot: {uint32 fmt, uint32 nnz} padded to 16
// bytes, fp32 values[256], int32 indices[256] (slice-relative, ascending).
// Dense fallback: fmt 0, values[0..len) in place.  Compaction: per-lane
// nonzero masks, a warp inclusive scan of their popcounts gives every
// lane's first output position.
template <> struct Wire<kCodecSparse> {
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
    __device__ __forceinline__ uint32_t encode_store(const float acc[8], int V, int lane,
                                                     unsigned char *slot, double one_minus_thr,
                                                     float dec[8])
    {
        uint32_t nzm = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            dec[i] = acc[i];
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
    // Dense: all positions.  Sparse: scatter the pairs into the warp's
    // scratch (values + presence bytes), then read this lane's 8 positions.
    __device__ __forceinline__ uint32_t decode(int lane, unsigned char *scratch, float v[8]) const
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
};

// ---------------------------------------------------------------- kernel

// Bounded wait used only to drain this warp's own bulk copies before exit:
// it ignores the status word (copies in flight must land before the block's
// shared memory can be released) and gives up only at the time limit.
__device__ __forceinline__ void drain_phase(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns)
            break;
}

template <int CODEC, int IN_T, bool FAST>
__global__ void __launch_bounds__(kMaxWarps * 32) ring_kernel(const __grid_constant__ RingArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    using W_t = Wire<CODEC>;
    constexpr int es = dtype_size(IN_T);
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
    long long *next_issue = reinterpret_cast<long long *>(smem + Lo.rank_state);
    long long *consumed = next_issue + N;
    unsigned long long *rsent = reinterpret_cast<unsigned long long *>(consumed + N);
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
        next_issue[i] = 0;
        consumed[i] = 0;
        rsent[i] = 0;
        rrecv[i] = 0;
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < 2 * N; i += blockDim.x)
            a.zero[i] = 0ull;
    mbar_fence_init();
    __syncthreads();

    const bool allred = a.mode == kModeAllreduce;
    const int G = allred ? 2 * N - 1 : N; // steps per slice position
    const int M = allred ? 2 * N - 2 : N - 1; // messages per ring edge per slice position
    const int P = N;                          // staged input loads per rank per slice position
    const long long n = a.n, T = a.T;
    const int out_es = dtype_size(a.out_t);

    auto chunk_len = [&](int c) -> long long {
        long long lo = (long long)c * n, hi = lo + n;
        lo = lo < T ? lo : T;
        hi = hi < T ? hi : T;
        return hi - lo;
    };

    // Lane 0 of the owning warp: enqueue staged load number L of rank r
    // (slice iteration L / P, step L % P + 1).  Returns false if that slice
    // position does not exist.
    auto issue = [&](int r, long long L) -> bool {
        const long long jj = L / P;
        const int gg = (int)(L % P) + 1;
        const long long item = blockIdx.x + jj * gridDim.x;
        if (item >= a.tiles)
            return false;
        const int c = mod_n(r - gg, N);
        const long long t0 = item * kTile;
        long long V = chunk_len(c) - t0;
        V = V < 0 ? 0 : (V > kTile ? kTile : V);
        const int d = (int)(L % D);
        uint64_t *bar = sbar + r * D + d;
        unsigned char *dst = stages + (size_t)(r * D + d) * a.stage_bytes;
        const uint32_t bytes = (uint32_t)(V * es);
        if (bytes == 0) {
            mbar_arrive(bar);
            return true;
        }
        const long long eo = (long long)c * n + t0;
        const char *src = reinterpret_cast<const char *>(a.in[r]) + eo * es;
        if (a.has_prev) {
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_g2s(dst, src, bytes, bar);
            bulk_g2s(dst + kTile * 4, a.prev[r] + eo, bytes, bar);
        } else {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(dst, src, bytes, bar);
        }
        return true;
    };

    if constexpr (FAST) {
        if (lane == 0)
            for (int r = warp; r < N; r += W) {
                long long L = 0;
                while (L < D && issue(r, L))
                    ++L;
                next_issue[r] = L;
            }
        __syncwarp();
    }

    bool ok = true;
    long long j = 0;
    for (long long item = blockIdx.x; ok && item < a.tiles; item += gridDim.x, ++j) {
        const long long t0 = item * kTile;
        for (int g = 1; ok && g <= G; ++g) {
            for (int r = warp; r < N; r += W) {
                const int c = mod_n(r - g, N);
                long long Vl = chunk_len(c) - t0;
                const int V = (int)(Vl < 0 ? 0 : (Vl > kTile ? kTile : Vl));
                const int vl = min(max(V - 8 * lane, 0), 8);
                const long long eoff = (long long)c * n + t0 + 8 * lane;

                // ---- own input (reduce-scatter steps and the owner step)
                float x[8];
                if (g <= N) {
                    if constexpr (FAST) {
                        const long long L = j * P + (g - 1);
                        const int d = (int)(L % D);
                        ok = wait_phase(sbar + r * D + d, (uint32_t)((L / D) & 1), a.timeout_ns,
                                        a.status);
                        if (!ok)
                            break;
                        const unsigned char *sp = stages + (size_t)(r * D + d) * a.stage_bytes;
                        load8_vec<IN_T>(sp + 8 * lane * es, x);
                        if (a.has_prev) {
                            float p[8];
                            load8_vec<kF32>(sp + kTile * 4 + 8 * lane * 4, p);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                x[i] = __fsub_rn(x[i], p[i]);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (i >= vl)
                                x[i] = 0.0f;
                        __syncwarp();
                        if (lane == 0) {
                            consumed[r] = L + 1;
                            if (next_issue[r] == L + D && issue(r, L + D))
                                next_issue[r] = L + D + 1;
                        }
                    } else {
                        load8_scalar<IN_T>(reinterpret_cast<const char *>(a.in[r]) + eoff * es,
                                           vl, x);
                        if (a.has_prev) {
                            float p[8];
                            load8_scalar<kF32>(a.prev[r] + eoff, vl, p);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                x[i] = __fsub_rn(x[i], p[i]);
                        }
                    }
                }

                // ---- receive from rank r-1 (steps 2..G)
                W_t w;
                uint32_t rb = 0;
                if (g >= 2) {
                    const long long m = j * M + (g - 2);
                    const int s = (int)(m % K);
                    ok = wait_phase(full + r * K + s, (uint32_t)((m / K) & 1), a.timeout_ns,
                                    a.status);
                    if (!ok)
                        break;
                    rb = w.load(slots + (size_t)(r * K + s) * a.slot_bytes, lane, V);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(empty + r * K + s);
                        rrecv[r] += rb;
                    }
                }

                // ---- compute this step's outgoing message and/or output
                float outv[8];
                bool do_out = false;
                bool do_send = g <= M;
                W_t ws;
                unsigned char *dslot = nullptr;
                int dst = r + 1 == N ? 0 : r + 1;
                long long ms = j * M + (g - 1);
                int ss = (int)(ms % K);
                if (do_send) {
                    ok = wait_phase(empty + dst * K + ss, (uint32_t)(((ms / K) & 1) ^ 1),
                                    a.timeout_ns, a.status);
                    if (!ok)
                        break;
                    dslot = slots + (size_t)(dst * K + ss) * a.slot_bytes;
                }
                uint32_t sb = 0;
                if (g <= N) {
                    float acc[8];
                    if (g >= 2) {
                        float dv[8];
                        const uint32_t pres = w.decode(lane, scratch, dv);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc[i] = ((pres >> i) & 1u) ? __fadd_rn(x[i], dv[i]) : x[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc[i] = x[i];
                    }
                    if (g < N) {
                        float dec[8];
                        sb = ws.encode_store(acc, V, lane, dslot, a.one_minus_thr, dec);
                    } else {
                        do_out = true;
                        if (allred) {
                            // N = 1 has no allgather step: encode into the rank's
                            // own (otherwise unused) mailbox slot for its output
                            unsigned char *es_slot =
                                dslot ? dslot : slots + (size_t)(r * K) * a.slot_bytes;
                            sb = ws.encode_store(acc, V, lane, es_slot, a.one_minus_thr, outv);
                            if (!dslot)
                                sb = 0;
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                outv[i] = acc[i];
                        }
                    }
                } else {
                    float dv[8];
                    const uint32_t pres = w.decode(lane, scratch, dv);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        outv[i] = ((pres >> i) & 1u) ? dv[i] : 0.0f;
                    do_out = true;
                    if (do_send) {
                        // allgather: forward the received codes unchanged
                        w.store(dslot, lane);
                        sb = rb;
                    }
                }
                if (do_send) {
                    __syncwarp();
                    if (lane == 0) {
                        const bool withheld =
                            r == a.withhold_rank && g == a.withhold_step && j == 0;
                        if (!withheld)
                            mbar_arrive(full + dst * K + ss);
                        rsent[r] += sb;
                    }
                }

                // ---- output epilogue: average, previous-round base, cast
                if (do_out) {
                    float wv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        wv[i] = a.average ? __fdiv_rn(outv[i], (float)N) : outv[i];
                    if (a.base) {
                        float bb[8];
                        if (a.vec_base && vl == 8)
                            load8_vec<kF32>(a.base + eoff, bb);
                        else
                            load8_scalar<kF32>(a.base + eoff, vl, bb);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            wv[i] = __fadd_rn(bb[i], wv[i]);
                    }
                    store8(reinterpret_cast<char *>(a.out[r]) + eoff * out_es, a.out_t, wv, vl,
                           a.vec_out != 0);
                }
            }
        }
    }

    // ---- drain this warp's staged copies that are still in flight
    if constexpr (FAST) {
        __syncwarp();
        for (int r = warp; r < N; r += W) {
            const long long from = consumed[r], to = next_issue[r];
            for (long long L = from; L < to; ++L)
                drain_phase(sbar + r * D + (int)(L % D), (uint32_t)((L / D) & 1), a.timeout_ns);
        }
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

// coll_kernels.cu -- ring allgather, binomial broadcast and tree allreduce for
// N simulated ranks on one sm_103a GPU ("从零实现集合通信": per-rank byte/step
// table -- allgather T(N-1)/N in N-1 steps, broadcast T over a log2(N) tree,
// tree allreduce T log2 N in 2 log2 N steps; "练习": the tree variant).
//
// Same machinery as the fused ring (ring_kernel.cuh).  A block runs the
// collective for one slice position (TW = 256*G elements) at a time and
// strides over slice positions; simulated rank r is warp r mod W.  Every edge
// of the communication graph is a FIFO of K slots in shared memory owned by
// its receiver, with a "full" and an "empty" mbarrier per slot and bounded
// waits.  Data a rank reads from its own buffer is staged with bulk async
// copies on the fast path (16-byte aligned buffers and slice boundaries).
//
//  allgather   ring edges r -> r+1; step g = 1..N, chunk (r - g + 1) mod N:
//              g = 1 sends the rank's own chunk, g >= 2 stores the received
//              chunk into the rank's buffer and forwards it while g < N.
//  broadcast   binomial tree from the root: relative rank q = (r - root) mod N
//              receives at level floor(log2 q) from q - 2^level and forwards
//              at every later level k with q + 2^k < N, from its receive slot.
//  tree        fp32.  Each rank accumulates in its staged slice: at reduce
//              level k, r with r mod 2^(k+1) = 2^k sends to r - 2^k, which
//              adds (receiver's partial + sender's partial, round to nearest
//              even); then the binomial broadcast of rank 0's sum.
// Each tree/broadcast edge carries one message per slice position, so one
// FIFO position per block serves all of them; ring edges carry N-1 messages
// per slice position, one per step.  Within a level, a warp does all of its
// ranks' sends before any of their receives, so a warp that plays both ends
// of an edge (N > 16) never waits on itself.
//  broadcast   (BFP) the same tree carrying the root's block-floating-point
//              codes, each edge copied by its receiver: the root encodes
//              each slice once into its own slot and stores the decoded
//              values; every other rank copies its parent's codes into its
//              own slot (if it has children) and stores the decoded values;
//              a slot is freed when all of its rank's children have copied
//              it (an mbarrier counting the children).
#include "ring_kernel.cuh" // BfpGroup: the BFP arithmetic of the ring
#include "rra_device.cuh"
#include "rra_kernels.h"

namespace rra {

namespace {

// One lane's 8 consecutive elements of ES bytes each (16 or 32 bytes).
template <int ES> struct Vec8 {
    uint4 u[ES / 2];
    __device__ __forceinline__ void load(const void *p)
    {
#pragma unroll
        for (int i = 0; i < ES / 2; ++i)
            u[i] = reinterpret_cast<const uint4 *>(p)[i];
    }
    __device__ __forceinline__ void store(void *p) const
    {
#pragma unroll
        for (int i = 0; i < ES / 2; ++i)
            reinterpret_cast<uint4 *>(p)[i] = u[i];
    }
    // the first `valid` elements at p (any alignment); the rest read as zero
    __device__ __forceinline__ void load_elems(const void *p, int valid)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if constexpr (ES == 4)
                reinterpret_cast<uint32_t *>(u)[i] =
                    i < valid ? reinterpret_cast<const uint32_t *>(p)[i] : 0u;
            else
                reinterpret_cast<uint16_t *>(u)[i] =
                    i < valid ? reinterpret_cast<const uint16_t *>(p)[i] : (uint16_t)0;
        }
    }
    __device__ __forceinline__ void store_elems(void *p, int valid) const
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid) {
                if constexpr (ES == 4)
                    reinterpret_cast<uint32_t *>(p)[i] = reinterpret_cast<const uint32_t *>(u)[i];
                else
                    reinterpret_cast<uint16_t *>(p)[i] = reinterpret_cast<const uint16_t *>(u)[i];
            }
    }
};

// Shared-memory carve-up of a collective kernel (host and device agree via
// coll_layout in rra_kernels.h).
struct CollSmem {
    uint64_t *full, *empty, *sbar;
    unsigned long long *rsent, *rrecv;
    unsigned char *slots, *stages;
};

__device__ __forceinline__ CollSmem coll_carve(unsigned char *smem, const CopyArgs &a, int edges,
                                               int stagers, bool fast)
{
    const CollLayout L =
        coll_layout(a.N, edges, a.K, stagers, a.D, a.slot_bytes, a.stage_bytes, fast);
    CollSmem s;
    s.full = reinterpret_cast<uint64_t *>(smem + L.full);
    s.empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    s.sbar = reinterpret_cast<uint64_t *>(smem + L.stage_bar);
    s.rsent = reinterpret_cast<unsigned long long *>(smem + L.counters);
    s.rrecv = s.rsent + a.N;
    s.slots = smem + L.slots;
    s.stages = smem + L.stages;
    return s;
}

// empty_count(edge): arrivals that free a slot of that edge (1 by default)
template <class EmptyCount>
__device__ __forceinline__ void coll_init(const CollSmem &s, const CopyArgs &a, int edges,
                                          int stagers, bool fast, EmptyCount empty_count)
{
    for (int i = threadIdx.x; i < edges * a.K; i += blockDim.x) {
        mbar_init(s.full + i, 1);
        mbar_init(s.empty + i, (uint32_t)empty_count(i / a.K));
    }
    if (fast)
        for (int i = threadIdx.x; i < stagers * a.D; i += blockDim.x)
            mbar_init(s.sbar + i, 1);
    for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
        s.rsent[i] = 0;
        s.rrecv[i] = 0;
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < 2 * a.N; i += blockDim.x)
            a.zero[i] = 0ull;
    mbar_fence_init();
    __syncthreads();
}

__device__ __forceinline__ void coll_init(const CollSmem &s, const CopyArgs &a, int edges,
                                          int stagers, bool fast)
{
    coll_init(s, a, edges, stagers, fast, [](int) { return 1; });
}

// Per-rank byte counters: in registers when every warp plays one rank, in
// shared memory otherwise; added to the device counters once per block.
template <bool ONE> struct Bytes {
    unsigned long long sent = 0, recv = 0;
    __device__ __forceinline__ void add_sent(const CollSmem &s, int r, unsigned long long b)
    {
        if (ONE)
            sent += b;
        else
            s.rsent[r] += b;
    }
    __device__ __forceinline__ void add_recv(const CollSmem &s, int r, unsigned long long b)
    {
        if (ONE)
            recv += b;
        else
            s.rrecv[r] += b;
    }
    __device__ __forceinline__ void flush(const CollSmem &s, const CopyArgs &a, int warp, int W)
    {
        if ((threadIdx.x & 31) != 0)
            return;
        if (ONE) {
            if (warp < a.N) {
                if (sent)
                    atomicAdd(a.sent + warp, sent);
                if (recv)
                    atomicAdd(a.recv + warp, recv);
            }
        } else {
            for (int r = warp; r < a.N; r += W) {
                if (s.rsent[r])
                    atomicAdd(a.sent + r, s.rsent[r]);
                if (s.rrecv[r])
                    atomicAdd(a.recv + r, s.rrecv[r]);
            }
        }
    }
};

__device__ __forceinline__ int clamp_len(long long v, int w)
{
    return (int)(v < 0 ? 0 : (v > w ? w : v));
}

} // namespace

// ---------------------------------------------------------------- allgather
template <int ES, bool FAST, int G, bool ONE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) allgather_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int TW = kTile * G;
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.K, D = a.D;
    const CollSmem s = coll_carve(smem, a, N, N, FAST);
    coll_init(s, a, N, N, FAST);
    const long long n = a.n, T = a.T;
    const int rstride = ONE ? N : W;
    const int tiles = (int)a.tiles;
    const long long min_len = T - (long long)(N - 1) * n; // shortest chunk
    auto slice_len = [&](int c, long long t0) -> int {
        if (t0 + TW <= min_len)
            return TW;
        long long lo = (long long)c * n, hi = lo + n;
        lo = lo < T ? lo : T;
        hi = hi < T ? hi : T;
        return clamp_len(hi - lo - t0, TW);
    };
    // staged loads: each rank's own chunk, one slice per slice position
    int cur_item = blockIdx.x, inflight = 0;
    auto issue = [&](int r, int d) { // lane 0
        const long long t0 = (long long)cur_item * TW;
        const uint32_t bytes = (uint32_t)slice_len(r, t0) * ES;
        uint64_t *bar = s.sbar + r * D + d;
        if (bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(s.stages + (size_t)(r * D + d) * a.stage_bytes,
                 reinterpret_cast<const char *>(a.buf[r]) + ((long long)r * n + t0) * ES, bytes,
                 bar);
    };
    if constexpr (FAST) {
        while (inflight < D && cur_item < tiles) {
            if (lane == 0)
                for (int r = warp; r < N; r += rstride)
                    issue(r, inflight);
            ++inflight;
            cur_item += gridDim.x;
        }
        __syncwarp();
    }
    Bytes<ONE> by;
    Fifo rcv{0, 0}, snd{0, 0}, stg{0, 0};
    bool ok = true;
    for (int item = blockIdx.x; ok && item < tiles; item += gridDim.x) {
        const long long t0 = (long long)item * TW;
        const bool first = item == (int)blockIdx.x;
        for (int g = 1; ok && g <= N; ++g) {
            const bool fwd = g < N;
            for (int r = warp; r < N; r += rstride) {
                int c = r - g + 1;
                c += c < 0 ? N : 0;
                const int V = slice_len(c, t0);
                const int dst = r + 1 == N ? 0 : r + 1;
                const unsigned char *src;
                if (g == 1) {
                    if (FAST) {
                        if (!(ok = wait_ready(s.sbar + r * D + stg.slot, (uint32_t)stg.phase,
                                              a.timeout_ns, a.status)))
                            break;
                        src = s.stages + (size_t)(r * D + stg.slot) * a.stage_bytes;
                    } else {
                        src = reinterpret_cast<const unsigned char *>(a.buf[r]) +
                              ((long long)r * n + t0) * ES;
                    }
                } else {
                    if (!(ok = wait_ready(s.full + r * K + rcv.slot, (uint32_t)rcv.phase,
                                          a.timeout_ns, a.status)))
                        break;
                    src = s.slots + (size_t)(r * K + rcv.slot) * a.slot_bytes;
                }
                if (fwd && !(ok = wait_ready(s.empty + dst * K + snd.slot,
                                             (uint32_t)(snd.phase ^ 1), a.timeout_ns, a.status)))
                    break;
                unsigned char *dslot = s.slots + (size_t)(dst * K + snd.slot) * a.slot_bytes;
                char *mine = reinterpret_cast<char *>(a.buf[r]) + ((long long)c * n + t0) * ES;
                const bool global_src = !FAST && g == 1;
#pragma unroll 1
                for (int gi = 0; gi < G; ++gi) {
                    const int e = gi * kTile + 8 * lane;
                    const int vl = min(max(V - e, 0), 8);
                    if (gi * kTile >= V)
                        break;
                    Vec8<ES> v;
                    if (global_src)
                        v.load_elems(src + (size_t)e * ES, vl);
                    else
                        v.load(src + (size_t)e * ES);
                    if (g >= 2) {
                        if (FAST && vl == 8)
                            v.store(mine + (size_t)e * ES);
                        else
                            v.store_elems(mine + (size_t)e * ES, vl);
                    }
                    if (fwd)
                        v.store(dslot + (size_t)e * ES);
                }
                __syncwarp();
                if (lane == 0) {
                    if (g >= 2) {
                        mbar_arrive(s.empty + r * K + rcv.slot);
                        by.add_recv(s, r, (unsigned long long)V * ES);
                    }
                    if (fwd) {
                        if (!(first && r == a.withhold_rank && g == a.withhold_step))
                            mbar_arrive(s.full + dst * K + snd.slot);
                        by.add_sent(s, r, (unsigned long long)V * ES);
                    }
                }
            }
            if (!ok)
                break;
            if (FAST && g == 1) { // the own-chunk stage is consumed: refill it
                __syncwarp();
                if (inflight == D && cur_item < tiles) {
                    if (lane == 0)
                        for (int r = warp; r < N; r += rstride)
                            issue(r, stg.slot);
                    cur_item += gridDim.x;
                } else {
                    --inflight;
                }
                stg.advance(D);
            }
            if (g >= 2)
                rcv.advance(K);
            if (fwd)
                snd.advance(K);
        }
    }
    if constexpr (FAST) {
        __syncwarp();
        for (int r = warp; r < N; r += W) {
            Fifo d = stg;
            for (int L = 0; L < inflight; ++L) {
                drain_phase(s.sbar + r * D + d.slot, (uint32_t)d.phase, a.timeout_ns);
                d.advance(D);
            }
        }
    }
    by.flush(s, a, warp, W);
}

// ---------------------------------------------------------------- broadcast
// Pull model: every edge of the binomial tree is copied by its receiver.  A
// rank with children holds the slice in its own slot: the root copies it
// there from its stage (or its buffer on the generic path), every other such
// rank from its parent's slot; every non-root rank stores it into its
// buffer.  A slot is freed once all of its rank's children have copied it
// (its "empty" mbarrier counts them).  A warp plays its ranks in increasing
// relative rank, so a parent it plays always publishes before a child it
// plays waits for it.
template <int ES, bool FAST, int G, bool ONE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) broadcast_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int TW = kTile * G;
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.K, D = a.D;
    const int root = a.root;
    int L = 0;
    while ((1 << L) < N)
        ++L;
    // relative rank q: parent q - 2^floor(log2 q); children q + 2^k for every
    // k with 2^k > q and q + 2^k < N
    auto children = [&](int q) -> int {
        int c = 0;
        for (int k = q > 0 ? 32 - __clz(q) : 0; k < L; ++k)
            c += q + (1 << k) < N ? 1 : 0;
        return c;
    };
    auto rel = [&](int r) -> int {
        const int q = r - root;
        return q < 0 ? q + N : q;
    };
    // slot FIFO of rank r, freed by its children; one stager (the root)
    const CollSmem s = coll_carve(smem, a, N, 1, FAST);
    coll_init(s, a, N, 1, FAST, [&](int r) { return max(children(rel(r)), 1); });
    const long long T = a.T;
    const int tiles = (int)a.tiles;
    const bool root_warp = root % W == warp;
    int cur_item = blockIdx.x, inflight = 0;
    auto issue = [&](int d) { // lane 0 of the root's warp
        const long long t0 = (long long)cur_item * TW;
        const uint32_t bytes = (uint32_t)clamp_len(T - t0, TW) * ES;
        uint64_t *bar = s.sbar + d;
        if (bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(s.stages + (size_t)d * a.stage_bytes,
                 reinterpret_cast<const char *>(a.buf[root]) + t0 * ES, bytes, bar);
    };
    if constexpr (FAST) {
        while (inflight < D && cur_item < tiles) {
            if (lane == 0 && root_warp)
                issue(inflight);
            ++inflight;
            cur_item += gridDim.x;
        }
        __syncwarp();
    }
    // the level at which relative rank q's withheld publish is checked: a
    // rank publishes once for all its children, so the fault-injection step
    // (a 1-based level) withholds it when q has a child at that level
    const int wlevel = a.withhold_step - 1;
    Bytes<ONE> by;
    Fifo e{0, 0}, stg{0, 0};
    bool ok = true;
    for (int item = blockIdx.x; ok && item < tiles; item += gridDim.x) {
        const long long t0 = (long long)item * TW;
        const bool first = item == (int)blockIdx.x;
        const int V = clamp_len(T - t0, TW);
        const unsigned long long mb = (unsigned long long)V * ES;
        for (int q = ONE ? rel(warp) : 0; ok && q < N; q += ONE ? N : 1) {
            int r = q + root;
            r -= r >= N ? N : 0;
            if (!ONE && r % W != warp)
                continue;
            const int nch = children(q);
            unsigned char *own = s.slots + (size_t)(r * K + e.slot) * a.slot_bytes;
            char *mine = reinterpret_cast<char *>(a.buf[r]) + t0 * ES;
            // a rank with children first waits until they have all copied the
            // message that last used this slot
            if (nch > 0 && !(ok = wait_ready(s.empty + r * K + e.slot, (uint32_t)(e.phase ^ 1),
                                             a.timeout_ns, a.status)))
                break;
            int p = 0; // absolute rank of the parent
            if (q == 0) {
                if (FAST && !(ok = wait_ready(s.sbar + stg.slot, (uint32_t)stg.phase,
                                              a.timeout_ns, a.status)))
                    break;
                if (nch > 0) {
                    const unsigned char *src =
                        FAST ? s.stages + (size_t)stg.slot * a.stage_bytes
                             : reinterpret_cast<const unsigned char *>(a.buf[root]) + t0 * ES;
#pragma unroll 1
                    for (int gi = 0; gi < G; ++gi) {
                        if (gi * kTile >= V)
                            break;
                        const int el = gi * kTile + 8 * lane;
                        Vec8<ES> v;
                        if (FAST)
                            v.load(src + (size_t)el * ES);
                        else
                            v.load_elems(src + (size_t)el * ES, min(max(V - el, 0), 8));
                        v.store(own + (size_t)el * ES);
                    }
                }
            } else {
                p = q - (1 << (31 - __clz(q))) + root;
                p -= p >= N ? N : 0;
                if (!(ok = wait_ready(s.full + p * K + e.slot, (uint32_t)e.phase, a.timeout_ns,
                                      a.status)))
                    break;
                const unsigned char *pslot = s.slots + (size_t)(p * K + e.slot) * a.slot_bytes;
#pragma unroll 1
                for (int gi = 0; gi < G; ++gi) { // copy the parent's slice
                    if (gi * kTile >= V)
                        break;
                    const int el = gi * kTile + 8 * lane;
                    const int vl = min(max(V - el, 0), 8);
                    Vec8<ES> v;
                    v.load(pslot + (size_t)el * ES);
                    if (nch > 0)
                        v.store(own + (size_t)el * ES);
                    if (FAST && vl == 8)
                        v.store(mine + (size_t)el * ES);
                    else
                        v.store_elems(mine + (size_t)el * ES, vl);
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (q > 0) {
                    mbar_arrive(s.empty + p * K + e.slot); // done with the parent's slot
                    by.add_recv(s, r, mb);
                }
                if (nch > 0) {
                    const bool withheld = first && r == a.withhold_rank && wlevel >= 0 &&
                                          wlevel < L && q < (1 << wlevel) &&
                                          q + (1 << wlevel) < N;
                    if (!withheld)
                        mbar_arrive(s.full + r * K + e.slot);
                    by.add_sent(s, r, mb * (unsigned long long)nch);
                }
            }
        }
        if (!ok)
            break;
        if (FAST) { // the root's stage is consumed: refill it
            __syncwarp();
            if (inflight == D && cur_item < tiles) {
                if (lane == 0 && root_warp)
                    issue(stg.slot);
                cur_item += gridDim.x;
            } else {
                --inflight;
            }
            stg.advance(D);
        }
        e.advance(K);
    }
    if constexpr (FAST) {
        __syncwarp();
        if (root_warp) {
            Fifo d = stg;
            for (int i = 0; i < inflight; ++i) {
                drain_phase(s.sbar + d.slot, (uint32_t)d.phase, a.timeout_ns);
                d.advance(D);
            }
        }
    }
    by.flush(s, a, warp, W);
}

// ---------------------------------------------------------------- BFP broadcast
// Message of one slice in a slot: 16 exponent bytes (byte b: block b), then
// the codes of group gi at 16 + gi * 256*BITS/8, lane L at 8L (BITS 8) or 4L
// (BITS 4) bytes within the group -- the layout of the ring's BFP messages.
template <int BITS> struct BfpSlot {
    static constexpr int kMB = kTile * BITS / 8;
    __device__ __forceinline__ static void put(unsigned char *slot, int gi, int lane, int e,
                                               const uint32_t w[2])
    {
        if ((lane & 15) == 0)
            slot[2 * gi + (lane >> 4)] = (unsigned char)(int8_t)e;
        if constexpr (BITS == 8)
            reinterpret_cast<uint2 *>(slot + 16 + gi * kMB)[lane] = make_uint2(w[0], w[1]);
        else
            reinterpret_cast<uint32_t *>(slot + 16 + gi * kMB)[lane] = w[0];
    }
    __device__ __forceinline__ static void get(const unsigned char *slot, int gi, int lane, int &e,
                                               uint32_t w[2])
    {
        e = (int)(int8_t)slot[2 * gi + (lane >> 4)];
        if constexpr (BITS == 8) {
            const uint2 u = reinterpret_cast<const uint2 *>(slot + 16 + gi * kMB)[lane];
            w[0] = u.x;
            w[1] = u.y;
        } else {
            w[0] = reinterpret_cast<const uint32_t *>(slot + 16 + gi * kMB)[lane];
            w[1] = 0;
        }
    }
};

// 8 elements of dtype dt at p widened to fp32; the first `valid` are read,
// the rest are +0.0 (vec: 16-byte aligned, all 8 present)
__device__ __forceinline__ void load8_dt(const void *p, int dt, int valid, bool vec, float v[8])
{
    if (dt == kF32) {
        if (vec && valid == 8)
            load8_vec<kF32>(p, v);
        else
            load8_scalar<kF32>(p, valid, v);
    } else if (dt == kF16) {
        if (vec && valid == 8)
            load8_vec<kF16>(p, v);
        else
            load8_scalar<kF16>(p, valid, v);
    } else {
        if (vec && valid == 8)
            load8_vec<kBF16>(p, v);
        else
            load8_scalar<kBF16>(p, valid, v);
    }
}

template <int BITS, bool FAST, int G, bool ONE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    broadcast_bfp_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    using BG = BfpGroup<BITS>;
    using SL = BfpSlot<BITS>;
    constexpr int TW = kTile * G;
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.K, D = a.D, dt = a.dt, es = a.es;
    const int root = a.root;
    int L = 0;
    while ((1 << L) < N)
        ++L;
    // relative rank q: parent q - 2^floor(log2 q); children q + 2^k for every
    // k with 2^k > q and q + 2^k < N
    auto children = [&](int q) -> int {
        int c = 0;
        for (int k = q > 0 ? 32 - __clz(q) : 0; k < L; ++k)
            c += q + (1 << k) < N ? 1 : 0;
        return c;
    };
    auto rel = [&](int r) -> int {
        const int q = r - root;
        return q < 0 ? q + N : q;
    };
    // a rank's slot is freed once every child has copied the message out
    const CollSmem s = coll_carve(smem, a, N, 1, FAST);
    coll_init(s, a, N, 1, FAST, [&](int r) { return max(children(rel(r)), 1); });
    const long long T = a.T;
    const int tiles = (int)a.tiles;
    const bool root_warp = root % W == warp;
    int cur_item = blockIdx.x, inflight = 0;
    auto issue = [&](int d) { // lane 0 of the root's warp
        const long long t0 = (long long)cur_item * TW;
        const uint32_t bytes = (uint32_t)clamp_len(T - t0, TW) * es;
        uint64_t *bar = s.sbar + d;
        if (bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(s.stages + (size_t)d * a.stage_bytes,
                 reinterpret_cast<const char *>(a.buf[root]) + t0 * es, bytes, bar);
    };
    if constexpr (FAST) {
        while (inflight < D && cur_item < tiles) {
            if (lane == 0 && root_warp)
                issue(inflight);
            ++inflight;
            cur_item += gridDim.x;
        }
        __syncwarp();
    }
    Bytes<ONE> by;
    Fifo e{0, 0}, stg{0, 0};
    bool ok = true;
    for (int item = blockIdx.x; ok && item < tiles; item += gridDim.x) {
        const long long t0 = (long long)item * TW;
        const bool first = item == (int)blockIdx.x;
        const int V = clamp_len(T - t0, TW);
        const unsigned long long mb = bfp_msg_bytes(V, BITS);
        // a warp plays its ranks in increasing relative rank, so a parent it
        // plays always publishes before a child it plays waits for it
        for (int q = ONE ? rel(warp) : 0; ok && q < N; q += ONE ? N : 1) {
            int r = q + root;
            r -= r >= N ? N : 0;
            if (!ONE && r % W != warp)
                continue;
            const int nch = children(q);
            unsigned char *own = s.slots + (size_t)(r * K + e.slot) * a.slot_bytes;
            char *mine = reinterpret_cast<char *>(a.buf[r]) + t0 * es;
            // a rank with children first waits until they have all copied the
            // message that last used this slot
            if (nch > 0 && !(ok = wait_ready(s.empty + r * K + e.slot, (uint32_t)(e.phase ^ 1),
                                             a.timeout_ns, a.status)))
                break;
            int p = 0; // absolute rank of the parent
            if (q == 0) {
                if (FAST && !(ok = wait_ready(s.sbar + stg.slot, (uint32_t)stg.phase,
                                              a.timeout_ns, a.status)))
                    break;
                const unsigned char *src =
                    FAST ? s.stages + (size_t)stg.slot * a.stage_bytes
                         : reinterpret_cast<const unsigned char *>(a.buf[root]) + t0 * es;
#pragma unroll 1
                for (int gi = 0; gi < G; ++gi) { // encode once, keep the decoded values
                    if (gi * kTile >= V)
                        break;
                    const int el = gi * kTile + 8 * lane;
                    const int vl = min(max(V - el, 0), 8);
                    float v[8];
                    load8_dt(src + (size_t)el * es, dt, vl, FAST, v); // +0.0 past the end
                    int ex;
                    uint32_t w[2];
                    BG::encode(v, ex, w);
                    SL::put(own, gi, lane, ex, w);
                    BG::decode(w, ex, v);
                    store8(mine + (size_t)el * es, dt, v, vl, FAST);
                }
            } else {
                p = q - (1 << (31 - __clz(q))) + root;
                p -= p >= N ? N : 0;
                if (!(ok = wait_ready(s.full + p * K + e.slot, (uint32_t)e.phase, a.timeout_ns,
                                      a.status)))
                    break;
                const unsigned char *pslot = s.slots + (size_t)(p * K + e.slot) * a.slot_bytes;
#pragma unroll 1
                for (int gi = 0; gi < G; ++gi) { // copy the parent's codes, store decoded
                    if (gi * kTile >= V)
                        break;
                    const int el = gi * kTile + 8 * lane;
                    int ex;
                    uint32_t w[2];
                    SL::get(pslot, gi, lane, ex, w);
                    if (nch > 0)
                        SL::put(own, gi, lane, ex, w);
                    float v[8];
                    BG::decode(w, ex, v);
                    store8(mine + (size_t)el * es, dt, v, min(max(V - el, 0), 8), FAST);
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (q > 0) {
                    mbar_arrive(s.empty + p * K + e.slot); // done with the parent's slot
                    by.add_recv(s, r, mb);
                }
                if (nch > 0) {
                    // fault injection: a withheld rank never publishes its message
                    if (!(first && r == a.withhold_rank && a.withhold_step >= 1))
                        mbar_arrive(s.full + r * K + e.slot);
                    by.add_sent(s, r, mb * (unsigned long long)nch);
                }
            }
        }
        if (!ok)
            break;
        if (FAST) { // the root's stage is consumed: refill it
            __syncwarp();
            if (inflight == D && cur_item < tiles) {
                if (lane == 0 && root_warp)
                    issue(stg.slot);
                cur_item += gridDim.x;
            } else {
                --inflight;
            }
            stg.advance(D);
        }
        e.advance(K);
    }
    if constexpr (FAST) {
        __syncwarp();
        if (root_warp) {
            Fifo d = stg;
            for (int i = 0; i < inflight; ++i) {
                drain_phase(s.sbar + d.slot, (uint32_t)d.phase, a.timeout_ns);
                d.advance(D);
            }
        }
    }
    by.flush(s, a, warp, W);
}

// ---------------------------------------------------------------- tree allreduce
// Pull model on the ranks' own stages (no slots): every rank stages its slice
// (its fp32 partial) and accumulates in it.
//  reduce     at level k, rank r with r mod 2^(k+1) = 0 and r + 2^k < N waits
//             until rank r + 2^k's partial is final and adds it, from that
//             rank's stage, into its own (receiver's partial + sender's,
//             round to nearest even: the binomial order).  A rank's partial
//             is final once it has received at every level below its own
//             sending level (the lowest set bit of r); it then publishes it
//             ("reduce-full").
//  broadcast  rank 0's stage holds the sum.  Every other rank waits for its
//             parent's "broadcast-full" (parent: r with its highest set bit
//             cleared), copies the parent's stage into its own (if it has
//             children) and into its buffer, then publishes.
// A stage is refilled once every rank that reads it -- the reduce parent and
// the broadcast children -- has arrived on its "empty" barrier.  Barriers per
// (rank, stage): full[r] reduce-full, full[N + r] broadcast-full, empty[r].
// A warp walks its ranks downwards in the reduce (children first) and
// upwards in the broadcast (parents first), so it never waits on a rank it
// plays later.
template <bool FAST, int G, bool ONE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) tree_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int TW = kTile * G;
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D; // stages per rank; the barrier FIFOs have D positions (a.K == D)
    int L = 0;
    while ((1 << L) < N)
        ++L;
    auto bc_children = [&](int r) -> int { // children in the broadcast from rank 0
        int c = 0;
        for (int k = r > 0 ? 32 - __clz(r) : 0; k < L; ++k)
            c += r + (1 << k) < N ? 1 : 0;
        return c;
    };
    // readers of rank r's stage: its reduce parent, its broadcast children
    auto readers = [&](int r) -> int { return (r > 0 ? 1 : 0) + bc_children(r); };
    const CollSmem s = coll_carve(smem, a, 2 * N, N, true);
    coll_init(s, a, 2 * N, N, FAST,
              [&](int edge) { return edge < N ? max(readers(edge), 1) : 1; });
    const long long T = a.T;
    const int rstride = ONE ? N : W;
    const int tiles = (int)a.tiles;
    int cur_item = blockIdx.x, inflight = 0;
    auto stage_of = [&](int r, int d) -> float * {
        return reinterpret_cast<float *>(s.stages + (size_t)(r * D + d) * a.stage_bytes);
    };
    auto issue = [&](int r, int d) { // lane 0
        const long long t0 = (long long)cur_item * TW;
        const uint32_t bytes = (uint32_t)clamp_len(T - t0, TW) * 4;
        uint64_t *bar = s.sbar + r * D + d;
        if (bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(stage_of(r, d), reinterpret_cast<const float *>(a.buf[r]) + t0, bytes, bar);
    };
    if constexpr (FAST) {
        while (inflight < D && cur_item < tiles) {
            if (lane == 0)
                for (int r = warp; r < N; r += rstride)
                    issue(r, inflight);
            ++inflight;
            cur_item += gridDim.x;
        }
        __syncwarp();
    }
    // the last rank this warp plays (the reduce walks them downwards)
    const int r_last = warp + ((N - 1 - warp) / rstride) * rstride;
    Bytes<ONE> by;
    Fifo stg{0, 0};
    bool ok = true;
    for (int item = blockIdx.x; ok && item < tiles; item += gridDim.x) {
        const long long t0 = (long long)item * TW;
        const bool first = item == (int)blockIdx.x;
        const int V = clamp_len(T - t0, TW);
        const int ng = (V + kTile - 1) / kTile;
        const unsigned long long mb = 4ull * (unsigned long long)V;
        const int d = stg.slot;
        const uint32_t ph = (uint32_t)stg.phase;
        // ---- binomial reduce to rank 0, children before parents
        for (int r = r_last; ok && r >= warp; r -= rstride) {
            float *acc = stage_of(r, d);
            if (FAST) {
                if (!(ok = wait_ready(s.sbar + r * D + d, ph, a.timeout_ns, a.status)))
                    break;
            } else {
                // the one stage's last readers must be done before it is refilled
                if (!first && !(ok = wait_ready(s.empty + r * D + d, ph ^ 1u, a.timeout_ns,
                                                a.status)))
                    break;
                const float *src = reinterpret_cast<const float *>(a.buf[r]) + t0;
#pragma unroll 1
                for (int gi = 0; gi < ng; ++gi) {
                    const int el = gi * kTile + 8 * lane;
                    float x[8];
                    load8_scalar<kF32>(src + el, min(max(V - el, 0), 8), x);
                    reinterpret_cast<float4 *>(acc + el)[0] = make_float4(x[0], x[1], x[2], x[3]);
                    reinterpret_cast<float4 *>(acc + el)[1] = make_float4(x[4], x[5], x[6], x[7]);
                }
                __syncwarp();
            }
            const int klast = r == 0 ? L : __ffs(r) - 1; // r receives at levels below this
            for (int k = 0; k < klast; ++k) {
                const int child = r + (1 << k);
                if (child >= N)
                    break;
                if (!(ok = wait_ready(s.full + child * D + d, ph, a.timeout_ns, a.status)))
                    break;
                const float *msg = stage_of(child, d);
#pragma unroll 1
                for (int gi = 0; gi < ng; ++gi) {
                    const int el = gi * kTile + 8 * lane;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float4 m = reinterpret_cast<const float4 *>(msg + el)[h];
                        float4 x = reinterpret_cast<float4 *>(acc + el)[h];
                        const float2 lo = __fadd2_rn(make_float2(x.x, x.y), make_float2(m.x, m.y));
                        const float2 hi = __fadd2_rn(make_float2(x.z, x.w), make_float2(m.z, m.w));
                        reinterpret_cast<float4 *>(acc + el)[h] = make_float4(lo.x, lo.y, hi.x, hi.y);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s.empty + child * D + d); // done reading the child's stage
                    by.add_recv(s, r, mb);
                }
            }
            if (!ok)
                break;
            if (r > 0 && lane == 0) { // the partial is final: publish it
                if (!(first && r == a.withhold_rank && a.withhold_step == klast + 1))
                    mbar_arrive(s.full + r * D + d);
                by.add_sent(s, r, mb);
            }
        }
        if (!ok)
            break;
        // ---- binomial broadcast of rank 0's sum, parents before children
        for (int r = warp; ok && r < N; r += rstride) {
            float *acc = stage_of(r, d);
            float *out = reinterpret_cast<float *>(a.buf[r]) + t0;
            const int nch = bc_children(r);
            if (r > 0) {
                const int p = r - (1 << (31 - __clz(r)));
                if (!(ok = wait_ready(s.full + (N + p) * D + d, ph, a.timeout_ns, a.status)))
                    break;
                const float *src = stage_of(p, d);
#pragma unroll 1
                for (int gi = 0; gi < ng; ++gi) {
                    const int el = gi * kTile + 8 * lane;
                    float x[8];
                    load8_vec<kF32>(src + el, x);
                    if (nch > 0) {
                        reinterpret_cast<float4 *>(acc + el)[0] = make_float4(x[0], x[1], x[2], x[3]);
                        reinterpret_cast<float4 *>(acc + el)[1] = make_float4(x[4], x[5], x[6], x[7]);
                    }
                    store8(out + el, kF32, x, min(max(V - el, 0), 8), FAST);
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s.empty + p * D + d); // done reading the parent's stage
                    by.add_recv(s, r, mb);
                }
            } else {
#pragma unroll 1
                for (int gi = 0; gi < ng; ++gi) {
                    const int el = gi * kTile + 8 * lane;
                    float x[8];
                    load8_vec<kF32>(acc + el, x);
                    store8(out + el, kF32, x, min(max(V - el, 0), 8), FAST);
                }
                __syncwarp();
            }
            if (lane == 0) {
                if (nch > 0) {
                    // fault injection: the broadcast levels are steps L+1..2L;
                    // a rank publishes once, withheld when it has a child at
                    // the withheld level
                    const int wl = a.withhold_step - L - 1;
                    const bool withheld = first && r == a.withhold_rank && wl >= 0 && wl < L &&
                                          r < (1 << wl) && r + (1 << wl) < N;
                    if (!withheld)
                        mbar_arrive(s.full + (N + r) * D + d);
                    by.add_sent(s, r, mb * (unsigned long long)nch);
                }
                if (readers(r) == 0) // N = 1: nobody else frees the stage
                    mbar_arrive(s.empty + r * D + d);
            }
        }
        if (!ok)
            break;
        if (FAST) {
            // refill this item's stages once their readers are done with them
            __syncwarp();
            if (inflight == D && cur_item < tiles) {
                for (int r = warp; ok && r < N; r += rstride)
                    ok = wait_ready(s.empty + r * D + d, ph, a.timeout_ns, a.status);
                if (!ok)
                    break;
                if (lane == 0)
                    for (int r = warp; r < N; r += rstride)
                        issue(r, d);
                cur_item += gridDim.x;
            } else {
                --inflight;
            }
        }
        stg.advance(D);
    }
    if constexpr (FAST) {
        __syncwarp();
        for (int r = warp; r < N; r += W) {
            Fifo dd = stg;
            for (int i = 0; i < inflight; ++i) {
                drain_phase(s.sbar + r * D + dd.slot, (uint32_t)dd.phase, a.timeout_ns);
                dd.advance(D);
            }
        }
    }
    by.flush(s, a, warp, W);
}

// ---------------------------------------------------------------- launchers

namespace {

template <int ES, int G> const void *ag_fn(bool fast, bool one)
{
    if (fast)
        return one ? (const void *)allgather_kernel<ES, true, G, true>
                   : (const void *)allgather_kernel<ES, true, G, false>;
    return one ? (const void *)allgather_kernel<ES, false, G, true>
               : (const void *)allgather_kernel<ES, false, G, false>;
}
template <int ES, int G> const void *bc_fn(bool fast, bool one)
{
    if (fast)
        return one ? (const void *)broadcast_kernel<ES, true, G, true>
                   : (const void *)broadcast_kernel<ES, true, G, false>;
    return one ? (const void *)broadcast_kernel<ES, false, G, true>
               : (const void *)broadcast_kernel<ES, false, G, false>;
}
template <int G> const void *tr_fn(bool fast, bool one)
{
    if (fast)
        return one ? (const void *)tree_kernel<true, G, true> : (const void *)tree_kernel<true, G, false>;
    return one ? (const void *)tree_kernel<false, G, true> : (const void *)tree_kernel<false, G, false>;
}

template <int ES> const void *coll_fn_es(int which, int groups, bool fast, bool one)
{
    switch (which * 10 + groups) {
    case 1: return ag_fn<ES, 1>(fast, one);
    case 2: return ag_fn<ES, 2>(fast, one);
    case 4: return ag_fn<ES, 4>(fast, one);
    case 11: return bc_fn<ES, 1>(fast, one);
    case 12: return bc_fn<ES, 2>(fast, one);
    case 14: return bc_fn<ES, 4>(fast, one);
    default: return nullptr;
    }
}

} // namespace

template <int BITS, int G> const void *bb_fn(bool fast, bool one)
{
    if (fast)
        return one ? (const void *)broadcast_bfp_kernel<BITS, true, G, true>
                   : (const void *)broadcast_bfp_kernel<BITS, true, G, false>;
    return one ? (const void *)broadcast_bfp_kernel<BITS, false, G, true>
               : (const void *)broadcast_bfp_kernel<BITS, false, G, false>;
}

const void *bcast_bfp_fn(int bits, int groups, bool fast, bool one)
{
    switch (bits * 10 + groups) {
    case 81: return bb_fn<8, 1>(fast, one);
    case 82: return bb_fn<8, 2>(fast, one);
    case 84: return bb_fn<8, 4>(fast, one);
    case 41: return bb_fn<4, 1>(fast, one);
    case 42: return bb_fn<4, 2>(fast, one);
    case 44: return bb_fn<4, 4>(fast, one);
    default: return nullptr;
    }
}

const void *coll_fn(int which, int es, int groups, bool fast, bool one)
{
    if (which == 2) {
        switch (groups) {
        case 1: return tr_fn<1>(fast, one);
        case 2: return tr_fn<2>(fast, one);
        case 4: return tr_fn<4>(fast, one);
        default: return nullptr;
        }
    }
    return es == 4 ? coll_fn_es<4>(which, groups, fast, one) : coll_fn_es<2>(which, groups, fast, one);
}

} // namespace rra

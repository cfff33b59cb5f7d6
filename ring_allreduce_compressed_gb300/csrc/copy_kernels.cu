// copy_kernels.cu -- allgather (ring), binomial broadcast and tree allreduce
// for N simulated ranks on one sm_103a GPU ("从零实现集合通信": per-rank
// byte/step table -- allgather T(N-1)/N in N-1 steps, broadcast T over a
// log2(N) tree, tree allreduce T log2 N in 2 log2 N steps; "练习": the tree
// variant).
//
// Same machinery as the fused ring: a block handles one 256-element slice
// position at a time, simulated rank r is warp r mod W, messages travel
// through per-rank shared-memory mailboxes guarded by full/empty mbarriers
// with bounded waits, and on the fast path the data a rank reads from its own
// buffer is staged with bulk async copies.  Allgather and broadcast copy
// element bits unchanged (2- or 4-byte elements); the tree adds in fp32 with
// round to nearest even in the binomial order.
#include "rra_device.cuh"
#include "rra_kernels.h"

namespace rra {

namespace {

__device__ __forceinline__ int modn(int a, int n)
{
    int m = a % n;
    return m < 0 ? m + n : m;
}

__device__ __forceinline__ long long clampv(long long v)
{
    return v < 0 ? 0 : (v > kTile ? kTile : v);
}

// One lane's 8 raw elements (ES bytes each), in memory order.
template <int ES> struct Raw8 {
    uint4 u[ES / 2]; // 16 bytes per 8 two-byte elements, 32 per 8 four-byte ones
    __device__ __forceinline__ void load_vec(const void *p)
    {
#pragma unroll
        for (int i = 0; i < ES / 2; ++i)
            u[i] = reinterpret_cast<const uint4 *>(p)[i];
    }
    __device__ __forceinline__ void store_vec(void *p) const
    {
#pragma unroll
        for (int i = 0; i < ES / 2; ++i)
            reinterpret_cast<uint4 *>(p)[i] = u[i];
    }
    __device__ __forceinline__ void load_elems(const void *p, int valid)
    {
        unsigned char *d = reinterpret_cast<unsigned char *>(u);
        const unsigned char *s = reinterpret_cast<const unsigned char *>(p);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < valid) {
                if constexpr (ES == 4)
                    reinterpret_cast<uint32_t *>(d)[i] = reinterpret_cast<const uint32_t *>(s)[i];
                else
                    reinterpret_cast<uint16_t *>(d)[i] = reinterpret_cast<const uint16_t *>(s)[i];
            } else {
                if constexpr (ES == 4)
                    reinterpret_cast<uint32_t *>(d)[i] = 0u;
                else
                    reinterpret_cast<uint16_t *>(d)[i] = 0u;
            }
        }
    }
    __device__ __forceinline__ void store_elems(void *p, int valid) const
    {
        const unsigned char *s = reinterpret_cast<const unsigned char *>(u);
        unsigned char *d = reinterpret_cast<unsigned char *>(p);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid) {
                if constexpr (ES == 4)
                    reinterpret_cast<uint32_t *>(d)[i] = reinterpret_cast<const uint32_t *>(s)[i];
                else
                    reinterpret_cast<uint16_t *>(d)[i] = reinterpret_cast<const uint16_t *>(s)[i];
            }
    }
};

__device__ __forceinline__ void drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns)
            break;
}

struct Smem {
    uint64_t *full, *empty, *sbar;
    long long *next_issue, *consumed;
    unsigned long long *rsent, *rrecv;
    unsigned char *slots, *stages, *extra;
};

__device__ __forceinline__ Smem carve(unsigned char *smem, const CopyArgs &a, int W, bool fast)
{
    const Layout Lo = make_layout(a.N, a.K, a.D, a.slot_bytes, a.stage_bytes, W, fast, false);
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(smem + Lo.full);
    s.empty = reinterpret_cast<uint64_t *>(smem + Lo.empty);
    s.sbar = reinterpret_cast<uint64_t *>(smem + Lo.stage_bar);
    s.next_issue = reinterpret_cast<long long *>(smem + Lo.rank_state);
    s.consumed = s.next_issue + a.N;
    s.rsent = reinterpret_cast<unsigned long long *>(s.consumed + a.N);
    s.rrecv = s.rsent + a.N;
    s.slots = smem + Lo.slots;
    s.stages = smem + Lo.stages;
    s.extra = smem + Lo.total; // tree: per-rank fp32 accumulators follow the layout
    return s;
}

__device__ __forceinline__ void init_smem(const Smem &s, const CopyArgs &a, bool fast)
{
    for (int i = threadIdx.x; i < a.N * a.K; i += blockDim.x) {
        mbar_init(s.full + i, 1);
        mbar_init(s.empty + i, 1);
    }
    if (fast)
        for (int i = threadIdx.x; i < a.N * a.D; i += blockDim.x)
            mbar_init(s.sbar + i, 1);
    for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
        s.next_issue[i] = 0;
        s.consumed[i] = 0;
        s.rsent[i] = 0;
        s.rrecv[i] = 0;
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < 2 * a.N; i += blockDim.x)
            a.zero[i] = 0ull;
    mbar_fence_init();
    __syncthreads();
}

// Staged load number L (one per slice position) of rank r: bytes [src, +bytes)
// into stage L % D.  Lane 0 only.
__device__ __forceinline__ void stage_issue(const Smem &s, const CopyArgs &a, int r, long long L,
                                            const void *src, uint32_t bytes)
{
    const int d = (int)(L % a.D);
    uint64_t *bar = s.sbar + r * a.D + d;
    if (bytes == 0) {
        mbar_arrive(bar);
        return;
    }
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(s.stages + (size_t)(r * a.D + d) * a.stage_bytes, src, bytes, bar);
}

__device__ __forceinline__ void finish(const Smem &s, const CopyArgs &a, int W, int warp,
                                       int lane, bool fast)
{
    if (fast) {
        __syncwarp();
        for (int r = warp; r < a.N; r += W)
            for (long long L = s.consumed[r]; L < s.next_issue[r]; ++L)
                drain(s.sbar + r * a.D + (int)(L % a.D), (uint32_t)((L / a.D) & 1), a.timeout_ns);
    }
    if (lane == 0)
        for (int r = warp; r < a.N; r += W) {
            if (s.rsent[r])
                atomicAdd(a.sent + r, s.rsent[r]);
            if (s.rrecv[r])
                atomicAdd(a.recv + r, s.rrecv[r]);
        }
}

// Wait for mailbox message number m of rank q (slot m % K).
__device__ __forceinline__ bool mb_wait_full(const Smem &s, const CopyArgs &a, int q,
                                             long long m)
{
    return wait_phase(s.full + q * a.K + (int)(m % a.K), (uint32_t)((m / a.K) & 1), a.timeout_ns,
                      a.status);
}
__device__ __forceinline__ bool mb_wait_empty(const Smem &s, const CopyArgs &a, int q,
                                              long long m)
{
    return wait_phase(s.empty + q * a.K + (int)(m % a.K), (uint32_t)(((m / a.K) & 1) ^ 1),
                      a.timeout_ns, a.status);
}
__device__ __forceinline__ unsigned char *mb_slot(const Smem &s, const CopyArgs &a, int q,
                                                  long long m)
{
    return s.slots + (size_t)(q * a.K + (int)(m % a.K)) * a.slot_bytes;
}

} // namespace

// ---------------------------------------------------------------- allgather
// In place: chunk r of buf[r] is rank r's contribution.  Step g = 1..N for
// rank r concerns chunk c = (r - g + 1) mod N: g = 1 reads its own chunk and
// sends it; g >= 2 receives chunk c, stores it into buf[r] and (g <= N-1)
// forwards it unchanged.
template <int ES, bool FAST>
__global__ void __launch_bounds__(kMaxWarps * 32) allgather_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Smem s = carve(smem, a, W, FAST);
    init_smem(s, a, FAST);
    const long long n = a.n, T = a.T;
    auto chunk_len = [&](int c) -> long long {
        long long lo = (long long)c * n, hi = lo + n;
        lo = lo < T ? lo : T;
        hi = hi < T ? hi : T;
        return hi - lo;
    };
    auto issue = [&](int r, long long L) -> bool {
        const long long item = blockIdx.x + L * gridDim.x;
        if (item >= a.tiles)
            return false;
        const long long t0 = item * kTile;
        const uint32_t bytes = (uint32_t)(clampv(chunk_len(r) - t0) * ES);
        stage_issue(s, a, r, L,
                    reinterpret_cast<const char *>(a.buf[r]) + ((long long)r * n + t0) * ES,
                    bytes);
        return true;
    };
    if (FAST) {
        if (lane == 0)
            for (int r = warp; r < N; r += W) {
                long long L = 0;
                while (L < a.D && issue(r, L))
                    ++L;
                s.next_issue[r] = L;
            }
        __syncwarp();
    }
    const int M = N - 1;
    bool ok = true;
    long long j = 0;
    for (long long item = blockIdx.x; ok && item < a.tiles; item += gridDim.x, ++j) {
        const long long t0 = item * kTile;
        for (int g = 1; ok && g <= N; ++g) {
            for (int r = warp; r < N; r += W) {
                const int c = modn(r - g + 1, N);
                const int V = (int)clampv(chunk_len(c) - t0);
                const int vl = min(max(V - 8 * lane, 0), 8);
                char *mine = reinterpret_cast<char *>(a.buf[r]) + ((long long)c * n + t0 + 8 * lane) * ES;
                Raw8<ES> v;
                if (g == 1) {
                    if constexpr (FAST) {
                        const int d = (int)(j % a.D);
                        ok = wait_phase(s.sbar + r * a.D + d, (uint32_t)((j / a.D) & 1),
                                        a.timeout_ns, a.status);
                        if (!ok)
                            break;
                        v.load_vec(s.stages + (size_t)(r * a.D + d) * a.stage_bytes + 8 * lane * ES);
                        __syncwarp();
                        if (lane == 0) {
                            s.consumed[r] = j + 1;
                            if (s.next_issue[r] == j + a.D && issue(r, j + a.D))
                                s.next_issue[r] = j + a.D + 1;
                        }
                    } else {
                        v.load_elems(mine, vl);
                    }
                } else {
                    const long long m = j * M + (g - 2);
                    ok = mb_wait_full(s, a, r, m);
                    if (!ok)
                        break;
                    v.load_vec(mb_slot(s, a, r, m) + 8 * lane * ES);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(s.empty + r * a.K + (int)(m % a.K));
                        s.rrecv[r] += (unsigned long long)V * ES;
                    }
                    if (FAST && vl == 8)
                        v.store_vec(mine);
                    else
                        v.store_elems(mine, vl);
                }
                if (g <= M) {
                    const int dst = r + 1 == N ? 0 : r + 1;
                    const long long m = j * M + (g - 1);
                    ok = mb_wait_empty(s, a, dst, m);
                    if (!ok)
                        break;
                    v.store_vec(mb_slot(s, a, dst, m) + 8 * lane * ES);
                    __syncwarp();
                    if (lane == 0) {
                        if (!(r == a.withhold_rank && g == a.withhold_step && j == 0))
                            mbar_arrive(s.full + dst * a.K + (int)(m % a.K));
                        s.rsent[r] += (unsigned long long)V * ES;
                    }
                }
            }
        }
    }
    finish(s, a, W, warp, lane, FAST);
}

// ---------------------------------------------------------------- broadcast
// Binomial tree from a.root over the whole buffer.  Relative rank q =
// (r - root) mod N receives its copy at level floor(log2 q) from q - 2^level
// (one mailbox message per slice position) and forwards it at every later
// level k with q + 2^k < N.  The root copies its own slice into its own
// (otherwise unused) mailbox slot so that every sender reads from its slot;
// a receiver keeps its slot until its last forward.
template <int ES, bool FAST>
__global__ void __launch_bounds__(kMaxWarps * 32) broadcast_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Smem s = carve(smem, a, W, FAST);
    init_smem(s, a, FAST);
    const long long T = a.T;
    int L = 0;
    while ((1 << L) < N)
        ++L;
    const int root = a.root;
    auto issue = [&](long long Li) -> bool {
        const long long item = blockIdx.x + Li * gridDim.x;
        if (item >= a.tiles)
            return false;
        const long long t0 = item * kTile;
        stage_issue(s, a, root, Li, reinterpret_cast<const char *>(a.buf[root]) + t0 * ES,
                    (uint32_t)(clampv(T - t0) * ES));
        return true;
    };
    if (FAST) {
        if (lane == 0 && root % W == warp) {
            long long Li = 0;
            while (Li < a.D && issue(Li))
                ++Li;
            s.next_issue[root] = Li;
        }
        __syncwarp();
    }
    // last level at which relative rank q forwards (-1: none)
    auto last_send = [&](int q) -> int {
        int k0 = 0;
        if (q > 0) {
            int fl = 31 - __clz(q);
            k0 = fl + 1;
        }
        int last = -1;
        for (int k = k0; k < L; ++k)
            if (q + (1 << k) < N)
                last = k;
        return last;
    };
    bool ok = true;
    long long j = 0;
    for (long long item = blockIdx.x; ok && item < a.tiles; item += gridDim.x, ++j) {
        const long long t0 = item * kTile;
        const int V = (int)clampv(T - t0);
        const int vl = min(max(V - 8 * lane, 0), 8);
        const long long eo = t0 + 8 * lane;
        // the root puts its slice into its own slot
        if (root % W == warp) {
            Raw8<ES> v;
            if constexpr (FAST) {
                const int d = (int)(j % a.D);
                ok = wait_phase(s.sbar + root * a.D + d, (uint32_t)((j / a.D) & 1), a.timeout_ns,
                                a.status);
                if (ok) {
                    v.load_vec(s.stages + (size_t)(root * a.D + d) * a.stage_bytes + 8 * lane * ES);
                    __syncwarp();
                    if (lane == 0) {
                        s.consumed[root] = j + 1;
                        if (s.next_issue[root] == j + a.D && issue(j + a.D))
                            s.next_issue[root] = j + a.D + 1;
                    }
                }
            } else {
                v.load_elems(reinterpret_cast<const char *>(a.buf[root]) + eo * ES, vl);
            }
            if (ok)
                v.store_vec(mb_slot(s, a, root, j) + 8 * lane * ES);
            __syncwarp();
        }
        for (int k = 0; ok && k < L; ++k) {
            // senders at level k: relative q < 2^k with q + 2^k < N
            for (int r = warp; ok && r < N; r += W) {
                const int q = modn(r - root, N);
                if (!(q < (1 << k) && q + (1 << k) < N))
                    continue;
                const int child = (q + (1 << k) + root) % N;
                ok = mb_wait_empty(s, a, child, j);
                if (!ok)
                    break;
                Raw8<ES> v;
                v.load_vec(mb_slot(s, a, r, j) + 8 * lane * ES);
                v.store_vec(mb_slot(s, a, child, j) + 8 * lane * ES);
                __syncwarp();
                if (lane == 0) {
                    if (!(r == a.withhold_rank && k + 1 == a.withhold_step && j == 0))
                        mbar_arrive(s.full + child * a.K + (int)(j % a.K));
                    s.rsent[r] += (unsigned long long)V * ES;
                }
                if (q > 0 && k == last_send(q) && lane == 0)
                    mbar_arrive(s.empty + r * a.K + (int)(j % a.K));
            }
            // receivers at level k: relative q in [2^k, 2^(k+1))
            for (int r = warp; ok && r < N; r += W) {
                const int q = modn(r - root, N);
                if (!(q >= (1 << k) && q < (2 << k)))
                    continue;
                ok = mb_wait_full(s, a, r, j);
                if (!ok)
                    break;
                Raw8<ES> v;
                v.load_vec(mb_slot(s, a, r, j) + 8 * lane * ES);
                char *mine = reinterpret_cast<char *>(a.buf[r]) + eo * ES;
                if (FAST && vl == 8)
                    v.store_vec(mine);
                else
                    v.store_elems(mine, vl);
                __syncwarp();
                if (lane == 0) {
                    s.rrecv[r] += (unsigned long long)V * ES;
                    if (last_send(q) < 0)
                        mbar_arrive(s.empty + r * a.K + (int)(j % a.K));
                }
            }
        }
        __syncwarp();
    }
    finish(s, a, W, warp, lane, FAST);
}

// ---------------------------------------------------------------- tree allreduce
// fp32, in place.  Per slice position every rank copies its slice into its
// fp32 accumulator in shared memory; reduce level k: rank r with
// r mod 2^(k+1) = 2^k sends its accumulator to r - 2^k, which adds it
// (receiver's partial + sender's partial); then the binomial broadcast of
// rank 0's accumulator.  Rank q's mailbox gets nred(q) reduce messages
// (levels 0..nred(q)-1) and, for q > 0, one broadcast message per position.
template <bool FAST>
__global__ void __launch_bounds__(kMaxWarps * 32) tree_kernel(const __grid_constant__ CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int N = a.N, W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Smem s = carve(smem, a, W, FAST);
    init_smem(s, a, FAST);
    float *accs = reinterpret_cast<float *>(s.extra); // [N][256]
    const long long T = a.T;
    int L = 0;
    while ((1 << L) < N)
        ++L;
    auto nred = [&](int q) -> int {
        int c = 0;
        for (int k = 0; k < L; ++k)
            if ((q & ((2 << k) - 1)) == 0 && q + (1 << k) < N)
                ++c;
        return c;
    };
    auto msgs = [&](int q) -> int { return nred(q) + (q != 0 ? 1 : 0); };
    auto issue = [&](int r, long long Li) -> bool {
        const long long item = blockIdx.x + Li * gridDim.x;
        if (item >= a.tiles)
            return false;
        const long long t0 = item * kTile;
        stage_issue(s, a, r, Li, reinterpret_cast<const float *>(a.buf[r]) + t0,
                    (uint32_t)(clampv(T - t0) * 4));
        return true;
    };
    if (FAST) {
        if (lane == 0)
            for (int r = warp; r < N; r += W) {
                long long Li = 0;
                while (Li < a.D && issue(r, Li))
                    ++Li;
                s.next_issue[r] = Li;
            }
        __syncwarp();
    }
    bool ok = true;
    long long j = 0;
    for (long long item = blockIdx.x; ok && item < a.tiles; item += gridDim.x, ++j) {
        const long long t0 = item * kTile;
        const int V = (int)clampv(T - t0);
        const int vl = min(max(V - 8 * lane, 0), 8);
        const long long eo = t0 + 8 * lane;
        // load every rank's slice into its accumulator
        for (int r = warp; ok && r < N; r += W) {
            float x[8];
            if constexpr (FAST) {
                const int d = (int)(j % a.D);
                ok = wait_phase(s.sbar + r * a.D + d, (uint32_t)((j / a.D) & 1), a.timeout_ns,
                                a.status);
                if (!ok)
                    break;
                load8_vec<kF32>(s.stages + (size_t)(r * a.D + d) * a.stage_bytes + 32 * lane, x);
                __syncwarp();
                if (lane == 0) {
                    s.consumed[r] = j + 1;
                    if (s.next_issue[r] == j + a.D && issue(r, j + a.D))
                        s.next_issue[r] = j + a.D + 1;
                }
            } else {
                load8_scalar<kF32>(reinterpret_cast<const float *>(a.buf[r]) + eo, vl, x);
            }
            float4 *p = reinterpret_cast<float4 *>(accs + r * kTile) + 2 * lane;
            p[0] = make_float4(x[0], x[1], x[2], x[3]);
            p[1] = make_float4(x[4], x[5], x[6], x[7]);
        }
        const unsigned long long mb = 4ull * (unsigned long long)V;
        // ---- binomial reduce to rank 0
        for (int k = 0; ok && k < L; ++k) {
            for (int r = warp; ok && r < N; r += W) { // senders first
                if ((r & ((2 << k) - 1)) != (1 << k))
                    continue;
                const int p = r - (1 << k);
                const long long m = j * msgs(p) + k;
                ok = mb_wait_empty(s, a, p, m);
                if (!ok)
                    break;
                const float4 *src = reinterpret_cast<const float4 *>(accs + r * kTile) + 2 * lane;
                float4 *dst = reinterpret_cast<float4 *>(mb_slot(s, a, p, m)) + 2 * lane;
                dst[0] = src[0];
                dst[1] = src[1];
                __syncwarp();
                if (lane == 0) {
                    if (!(r == a.withhold_rank && k + 1 == a.withhold_step && j == 0))
                        mbar_arrive(s.full + p * a.K + (int)(m % a.K));
                    s.rsent[r] += mb;
                }
            }
            for (int r = warp; ok && r < N; r += W) { // then receivers
                if ((r & ((2 << k) - 1)) != 0 || r + (1 << k) >= N)
                    continue;
                const long long m = j * msgs(r) + k;
                ok = mb_wait_full(s, a, r, m);
                if (!ok)
                    break;
                const float4 *src = reinterpret_cast<const float4 *>(mb_slot(s, a, r, m)) + 2 * lane;
                float4 *acc = reinterpret_cast<float4 *>(accs + r * kTile) + 2 * lane;
                const float4 m0 = src[0], m1 = src[1];
                float4 a0 = acc[0], a1 = acc[1];
                a0.x = __fadd_rn(a0.x, m0.x); a0.y = __fadd_rn(a0.y, m0.y);
                a0.z = __fadd_rn(a0.z, m0.z); a0.w = __fadd_rn(a0.w, m0.w);
                a1.x = __fadd_rn(a1.x, m1.x); a1.y = __fadd_rn(a1.y, m1.y);
                a1.z = __fadd_rn(a1.z, m1.z); a1.w = __fadd_rn(a1.w, m1.w);
                acc[0] = a0;
                acc[1] = a1;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s.empty + r * a.K + (int)(m % a.K));
                    s.rrecv[r] += mb;
                }
            }
        }
        // ---- rank 0 writes the result, then the binomial broadcast
        if (ok && warp == 0) {
            float x[8];
            load8_vec<kF32>(accs + 8 * lane, x);
            store8(reinterpret_cast<float *>(a.buf[0]) + eo, kF32, x, vl, FAST);
        }
        for (int k = 0; ok && k < L; ++k) {
            for (int r = warp; ok && r < N; r += W) { // senders: q < 2^k
                if (!(r < (1 << k) && r + (1 << k) < N))
                    continue;
                const int child = r + (1 << k);
                const long long m = j * msgs(child) + nred(child);
                ok = mb_wait_empty(s, a, child, m);
                if (!ok)
                    break;
                const float4 *src = reinterpret_cast<const float4 *>(accs + r * kTile) + 2 * lane;
                float4 *dst = reinterpret_cast<float4 *>(mb_slot(s, a, child, m)) + 2 * lane;
                dst[0] = src[0];
                dst[1] = src[1];
                __syncwarp();
                if (lane == 0) {
                    if (!(r == a.withhold_rank && L + k + 1 == a.withhold_step && j == 0))
                        mbar_arrive(s.full + child * a.K + (int)(m % a.K));
                    s.rsent[r] += mb;
                }
            }
            for (int r = warp; ok && r < N; r += W) { // receivers: q in [2^k, 2^(k+1))
                if (!(r >= (1 << k) && r < (2 << k)))
                    continue;
                const long long m = j * msgs(r) + nred(r);
                ok = mb_wait_full(s, a, r, m);
                if (!ok)
                    break;
                float x[8];
                load8_vec<kF32>(mb_slot(s, a, r, m) + 32 * lane, x);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s.empty + r * a.K + (int)(m % a.K));
                    s.rrecv[r] += mb;
                }
                float4 *acc = reinterpret_cast<float4 *>(accs + r * kTile) + 2 * lane;
                acc[0] = make_float4(x[0], x[1], x[2], x[3]);
                acc[1] = make_float4(x[4], x[5], x[6], x[7]);
                store8(reinterpret_cast<float *>(a.buf[r]) + eo, kF32, x, vl, FAST);
            }
        }
        __syncwarp();
    }
    finish(s, a, W, warp, lane, FAST);
}

// ---------------------------------------------------------------- launchers

static const void *copy_fn(int which, int es, bool fast)
{
    if (which == 0) {
        if (es == 4)
            return fast ? (const void *)allgather_kernel<4, true> : (const void *)allgather_kernel<4, false>;
        return fast ? (const void *)allgather_kernel<2, true> : (const void *)allgather_kernel<2, false>;
    }
    if (which == 1) {
        if (es == 4)
            return fast ? (const void *)broadcast_kernel<4, true> : (const void *)broadcast_kernel<4, false>;
        return fast ? (const void *)broadcast_kernel<2, true> : (const void *)broadcast_kernel<2, false>;
    }
    return fast ? (const void *)tree_kernel<true> : (const void *)tree_kernel<false>;
}

static cudaError_t launch_copy(int which, bool fast, const CopyArgs &a, int grid, int warps,
                               int smem, cudaStream_t st)
{
    const void *fn = copy_fn(which, a.es, fast);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    void *args[] = {const_cast<CopyArgs *>(&a)};
    return cudaLaunchKernel(fn, dim3(grid), dim3(warps * 32), args, (size_t)smem, st);
}

cudaError_t launch_allgather(bool fast, const CopyArgs &a, int grid, int warps, int smem,
                             cudaStream_t st)
{
    return launch_copy(0, fast, a, grid, warps, smem, st);
}
cudaError_t launch_broadcast(bool fast, const CopyArgs &a, int grid, int warps, int smem,
                             cudaStream_t st)
{
    return launch_copy(1, fast, a, grid, warps, smem, st);
}
cudaError_t launch_tree(bool fast, const CopyArgs &a, int grid, int warps, int smem,
                        cudaStream_t st)
{
    return launch_copy(2, fast, a, grid, warps, smem, st);
}

cudaError_t copy_kernel_attrs(int which, bool fast, int smem, int warps, int *blocks_per_sm)
{
    // element size does not change resource use materially; query the 4-byte variant
    const void *fn = copy_fn(which, 4, fast);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, warps * 32,
                                                         (size_t)smem);
}

} // namespace rra

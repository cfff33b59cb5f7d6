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
// The allgather alone (compressed allgather) skips steps 1..N-1: at g = N the
// owner encodes its own input chunk r, outputs its decoded value and sends
// the codes, and steps N+1..2N-1 run as above.
// Input slices are staged into shared memory with one-dimensional bulk async
// copies (cp.async.bulk + mbarrier transaction counts), D loads ahead per
// rank, on the fast path (16-byte aligned buffers and chunk sizes); the
// generic path loads elements directly with bounds checks.  Every index in
// the step loop advances incrementally: no division in the hot loop.
#pragma once

#include "bfp_group.cuh"
#include "rra_device.cuh"
#include "rra_kernels.h"

namespace rra {

// ---------------------------------------------------------------- wire formats
// What a step tells the wire codec about the message it moves (per-chunk
// sparse codec; the other codecs ignore it): fk = 2 * ((h-1)*N + c) + f,
// the message of chunk c at hop h and its format f (1 sparse, 0 dense,
// decided for the whole chunk before the ring starts), and base, the
// chunk-relative index of the slice's first element.
struct Msg {
    int fk;
    int base;
    __device__ __forceinline__ int sparse() const { return fk & 1; }
    __device__ __forceinline__ int key() const { return fk >> 1; }
};
// A message known to be dense: a codec with both forms overloads its
// operations on this type with dense-only code, so that steps whose
// messages are all dense carry no sparse instructions.  The other codecs
// take it as a Msg.
struct DenseMsg : Msg {
    __device__ __forceinline__ explicit DenseMsg(const Msg &m) : Msg(m) {}
};

// A message covers one slice of TW = 256*G elements.  The kernel streams it
// group by group (8 elements per lane, 256 per warp): a WireCodec's per-group
// operations move one group between registers and a slot, so only 8 values
// per lane are live at a time however large the slice is.
//  Reg                   one lane's share of one group of a message.
//  load / store          group gi: slot <-> Reg (allgather forwarding).
//                        Every operation also takes the step's Msg.
//  encode<DEC>           encode the lane's 8 fp32 values of group gi into the
//                        slot; with DEC, v becomes what a receiver decodes.
//                        Returns the group's wire bytes where they depend on
//                        the data (kVarBytes), else 0.
//  decode_add            v = v + decoded group (positions a sparse message
//                        does not carry keep v).
//  values                v = decoded group (0 where a sparse message has none).
//  bytes(V, slot)        wire bytes of a message of V elements.
//  kVarBytes             the wire bytes depend on the data; the kernel then
//                        sums group_bytes(m, V, gi) of the groups it loads and
//                        the returns of encode rather than re-reading headers.

template <int CODEC> struct WireCodec;

// Lossless: fp32, group gi at byte 1024*gi, lane L at 32L within the group.
template <> struct WireCodec<kCodecNone> {
    static constexpr bool kVarBytes = false;
    static constexpr int slot_bytes(int G) { return kTile * 4 * G; }
    struct Reg {
        float f[8];
    };
    __device__ __forceinline__ static void load(const unsigned char *slot, int gi, int lane,
                                                unsigned char *, const RingArgs &, Reg &m,
                                                const Msg &)
    {
        const float4 *p = reinterpret_cast<const float4 *>(slot + gi * kTile * 4) + 2 * lane;
        const float4 a = p[0], b = p[1];
        m.f[0] = a.x; m.f[1] = a.y; m.f[2] = a.z; m.f[3] = a.w;
        m.f[4] = b.x; m.f[5] = b.y; m.f[6] = b.z; m.f[7] = b.w;
    }
    __device__ __forceinline__ static void store(unsigned char *slot, int gi, int lane,
                                                 const Reg &m, const RingArgs &, const Msg &)
    {
        float4 *p = reinterpret_cast<float4 *>(slot + gi * kTile * 4) + 2 * lane;
        p[0] = make_float4(m.f[0], m.f[1], m.f[2], m.f[3]);
        p[1] = make_float4(m.f[4], m.f[5], m.f[6], m.f[7]);
    }
    template <bool DEC>
    __device__ __forceinline__ static uint32_t encode(float (&v)[8], unsigned char *slot, int gi,
                                                      int lane, int, const RingArgs &,
                                                      unsigned char *, const Msg &)
    {
        float4 *p = reinterpret_cast<float4 *>(slot + gi * kTile * 4) + 2 * lane;
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
        return 0u;
    }
    __device__ __forceinline__ static void decode_add(const Reg &m, float (&v)[8], int,
                                                      unsigned char *)
    {
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const float2 r =
                __fadd2_rn(make_float2(v[i], v[i + 1]), make_float2(m.f[i], m.f[i + 1]));
            v[i] = r.x;
            v[i + 1] = r.y;
        }
    }
    __device__ __forceinline__ static void values(const Reg &m, float (&v)[8], int,
                                                  unsigned char *)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = m.f[i];
    }
    __device__ __forceinline__ static uint32_t bytes(int V, const unsigned char *,
                                                     const RingArgs &, const Msg &)
    {
        return 4u * (uint32_t)V;
    }
};

// Block floating point: 16 header bytes of exponents (byte b is the exponent
// of the slice's 128-element block b), then the mantissas in element order
// (group gi at 16 + gi * 256*BITS/8; lane L at 8L bytes (8-bit) or 4L bytes
// (4-bit) within the group).
template <int BITS> struct CodecBfp {
    static constexpr bool kVarBytes = false;
    static constexpr int kMB = kTile * BITS / 8;
    static constexpr int slot_bytes(int G) { return 16 + kMB * G; }
    struct Reg {
        uint32_t w[2];
        int e;
    };
    __device__ __forceinline__ static void load(const unsigned char *slot, int gi, int lane,
                                                unsigned char *, const RingArgs &, Reg &m,
                                                const Msg &)
    {
        m.e = (int)(int8_t)slot[2 * gi + (lane >> 4)];
        if constexpr (BITS == 8) {
            const uint2 u = reinterpret_cast<const uint2 *>(slot + 16 + gi * kMB)[lane];
            m.w[0] = u.x;
            m.w[1] = u.y;
        } else {
            m.w[0] = reinterpret_cast<const uint32_t *>(slot + 16 + gi * kMB)[lane];
            m.w[1] = 0;
        }
    }
    __device__ __forceinline__ static void store(unsigned char *slot, int gi, int lane,
                                                 const Reg &m, const RingArgs &, const Msg &)
    {
        if ((lane & 15) == 0)
            slot[2 * gi + (lane >> 4)] = (unsigned char)(int8_t)m.e;
        if constexpr (BITS == 8)
            reinterpret_cast<uint2 *>(slot + 16 + gi * kMB)[lane] = make_uint2(m.w[0], m.w[1]);
        else
            reinterpret_cast<uint32_t *>(slot + 16 + gi * kMB)[lane] = m.w[0];
    }
    // encode group gi into the slot and return its codes
    __device__ __forceinline__ static void encode_reg(const float (&v)[8], unsigned char *slot,
                                                      int gi, int lane, Reg &m)
    {
        BfpGroup<BITS>::encode(v, m.e, m.w);
        if ((lane & 15) == 0)
            slot[2 * gi + (lane >> 4)] = (unsigned char)(int8_t)m.e;
        if constexpr (BITS == 8)
            reinterpret_cast<uint2 *>(slot + 16 + gi * kMB)[lane] = make_uint2(m.w[0], m.w[1]);
        else
            reinterpret_cast<uint32_t *>(slot + 16 + gi * kMB)[lane] = m.w[0];
    }
    template <bool DEC>
    __device__ __forceinline__ static uint32_t encode(float (&v)[8], unsigned char *slot, int gi,
                                                      int lane, int, const RingArgs &,
                                                      unsigned char *, const Msg &)
    {
        Reg m;
        encode_reg(v, slot, gi, lane, m);
        if (DEC)
            BfpGroup<BITS>::decode(m.w, m.e, v);
        return 0u;
    }
    __device__ __forceinline__ static void decode_add(const Reg &m, float (&v)[8], int,
                                                      unsigned char *)
    {
        BfpGroup<BITS>::decode_add(m.w, m.e, v, v);
    }
    __device__ __forceinline__ static void values(const Reg &m, float (&v)[8], int,
                                                  unsigned char *)
    {
        BfpGroup<BITS>::decode(m.w, m.e, v);
    }
    __device__ __forceinline__ static uint32_t bytes(int V, const unsigned char *,
                                                     const RingArgs &, const Msg &)
    {
        return bfp_msg_bytes(V, BITS);
    }
};
template <> struct WireCodec<kCodecBfp8> : CodecBfp<8> {};

// fp16 outputs straight from BFP8 offset codes.  A byte permute places an
// offset code b = m + 128 under the high byte 0x64 of an fp16 word: the half
// H = 1024 + b.  With s = 2^(e-q) and c = -1152 * s both fp16 numbers,
// fma(H, s, c) = (H - 1152) * s = m * 2^(e-q) exactly before its one
// rounding, so the result is the exact decoded value rounded once to fp16 --
// the same bits as rounding the fp32 decode to fp16.  s is an fp16 number for
// e - q in [-24, 15] and c for e - q in [-31, 5]; elsewhere the fp32 decode
// is used.  The table entry of block exponent e (index e + 128) holds the
// half2 words (s, s) and (c, c), or zero outside that range.
__device__ __forceinline__ uint2 bfp8_f16_entry(int e)
{
    const int k = e - BfpGroup<8>::q;
    if (k < -24 || k > 5)
        return make_uint2(0u, 0u);
    const uint32_t s = k >= -14 ? (uint32_t)(k + 15) << 10 : 1u << (k + 24);
    const uint32_t c = 0x8000u | ((uint32_t)(k + 25) << 10) | 0x80u; // -1.125 * 2^(k+10)
    return make_uint2(s | s << 16, c | c << 16);
}

// h[j] = fp16 pair (element 2j, 2j+1) of one lane's 8 codes; sc from the table.
__device__ __forceinline__ void bfp8_decode_f16(const uint32_t w[2], uint2 sc, uint32_t h[4])
{
    const __half2 s2 = *reinterpret_cast<const __half2 *>(&sc.x);
    const __half2 c2 = *reinterpret_cast<const __half2 *>(&sc.y);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t hw = __byte_perm(w[j >> 1], 0x64646464u, (j & 1) ? 0x4342 : 0x4140);
        const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&hw), s2, c2);
        h[j] = *reinterpret_cast<const uint32_t *>(&r);
    }
}
template <> struct WireCodec<kCodecBfp4> : CodecBfp<4> {};

// ---------------------------------------------------------------- kernel

// MODE kRanksShared: a warp may play several ranks (N > warps per block).
// MODE kRankPerWarp8 / kRankPerWarp16: every warp plays exactly one rank, so
// rank indices, addresses and byte counts stay in registers across the
// loops (each rank loop runs exactly once: the host launches W = N warps);
// blocks of at most 8 warps get up to 80 registers a thread (three blocks per
// SM), blocks of up to 16 warps 64 (two blocks per SM).
// EF: error feedback -- every value a rank encodes takes its residual first,
// and the residual keeps what the encoding lost (BFP instantiations only).
template <int CODEC, int IN_T, bool FAST, int G, int MODE, bool EF>
__global__ void __launch_bounds__(MODE == kRankPerWarp8 ? 8 * 32 : kMaxWarps * 32,
                                  MODE == kRankPerWarp8 ? 3 : 2)
    ring_kernel(const __grid_constant__ RingArgs a)
{
    constexpr bool ONE = MODE != kRanksShared;
    // kF32Diff: fp32 inputs cur with a second stream prev, encoded as cur - prev
    constexpr bool PREV = IN_T == kF32Diff;
    constexpr int LT = PREV ? kF32 : IN_T; // element type of the input buffers
    extern __shared__ __align__(128) unsigned char smem[];
    using C = WireCodec<CODEC>;
    using Reg = typename C::Reg;
    constexpr int es = dtype_size(LT);
    constexpr int TW = kTile * G; // elements per rank per step
    // The reduce-scatter group loop of the lossy codecs is unrolled (measured
    // faster: more independent work between the warp reductions), and so are
    // the BFP8 allgather loop that writes fp16 straight from the codes and the
    // allgather loop of the sparse codec (slices of at most 4 groups); the
    // other loops stay rolled to keep the code within the instruction cache.
    constexpr int kUnrollRS = CODEC != kCodecNone ? G : 1;
    constexpr int kUnrollAG = CODEC == kCodecSparse ? G : 1;
    const int N = a.N;
    const int W = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int K = a.K, D = a.D;
    // BFP8 allgather steps write fp16 outputs straight from the codes
    constexpr bool kDirect16 = CODEC == kCodecBfp8;
    const Layout Lo = make_layout(N, K, D, a.slot_bytes, a.stage_bytes, W, FAST,
                                  CODEC == kCodecSparse ? 1 : CODEC == kCodecSparseChunk ? 2 : 0,
                                  kDirect16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lo.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + Lo.empty);
    uint64_t *sbar = reinterpret_cast<uint64_t *>(smem + Lo.stage_bar);
    unsigned long long *rsent = reinterpret_cast<unsigned long long *>(smem + Lo.rank_state);
    unsigned long long *rrecv = rsent + N;
    unsigned char *slots = smem + Lo.slots;
    unsigned char *stages = smem + Lo.stages;
    unsigned char *scratch = smem + Lo.scratch + warp * (kTile * 4);
    unsigned char *fmt_s = smem + Lo.fmt; // per-chunk sparse: format of message (hop, chunk)

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
    const uint2 *lut = reinterpret_cast<const uint2 *>(smem + Lo.lut);
    if constexpr (kDirect16)
        for (int i = threadIdx.x; i < 256; i += blockDim.x)
            reinterpret_cast<uint2 *>(smem + Lo.lut)[i] = bfp8_f16_entry(i - 128);
    if constexpr (CODEC == kCodecSparseChunk) {
        // the format of every message of the call, from the count pass: the
        // message of chunk c at hop h is sparse iff nnz < (1 - threshold) * len
        for (int i = threadIdx.x; i < a.N * a.N; i += blockDim.x) {
            const long long c = i % a.N;
            const long long lo = min(c * a.n, a.T), hi = min(lo + a.n, a.T);
            fmt_s[i] = (double)a.sp_nnz[i] < a.one_minus_thr * (double)(hi - lo) ? 1 : 0;
        }
    }
    mbar_fence_init();
    __syncthreads();

    const bool allred = a.mode == kModeAllreduce;
    const bool agonly = a.mode == kModeAllgather; // the allgather pass alone
    const bool gather = allred || agonly;         // an allgather pass follows the owner
    const long long n = a.n, T = a.T;
    const int rstride = ONE ? N : W; // rank loop stride: one iteration when ONE
    unsigned long long my_sent = 0, my_recv = 0; // ONE: this warp's rank's bytes
    // shortest chunk: every slice position below it is full in every chunk
    const long long min_len = T - (long long)(N - 1) * n;

    // elements of chunk c in the slice at t0 (`full`: known full in every chunk)
    auto slice_len = [&](int c, long long t0, bool full = false) -> int {
        if (full || t0 + TW <= min_len)
            return TW;
        long long lo = (long long)c * n, hi = lo + n;
        lo = lo < T ? lo : T;
        hi = hi < T ? hi : T;
        const long long v = hi - lo - t0;
        return (int)(v < 0 ? 0 : (v > TW ? TW : v));
    };

    // ---- staged input loads.  All ranks consume loads in the same order
    // (slice iteration, step 1..N), so one cursor gives the next load to
    // issue for every rank; "inflight" counts loads issued and not consumed.
    int cur_item = blockIdx.x; // slice position of the next load to issue
    int cur_g = agonly ? N : 1; // its step (the allgather alone loads at the owner step only)
    // that slice position is full in every chunk
    bool cur_full = (long long)cur_item * TW + TW <= min_len;
    int inflight = 0;          // loads issued and not yet consumed, per rank
    const int tiles = (int)a.tiles;
    auto issue_one = [&](int r, int d) { // lane 0: load (cur_item, cur_g) of rank r into stage d
        int c = r - cur_g;
        c += c < 0 ? N : 0;
        const long long t0 = (long long)cur_item * TW;
        const uint32_t bytes = cur_full ? (uint32_t)(TW * es) : (uint32_t)slice_len(c, t0) * es;
        uint64_t *bar = sbar + r * D + d;
        unsigned char *dst = stages + (size_t)(r * D + d) * a.stage_bytes;
        if (!cur_full && bytes < (uint32_t)(TW * es)) {
            // a short slice: zero the rest of the stage (both streams), so
            // that the consumer reads +0.0 past the end without a test per
            // group; these stores precede the arrive that publishes the stage
            for (uint32_t o = bytes; o < (uint32_t)(TW * es); o += 4) {
                *reinterpret_cast<uint32_t *>(dst + o) = 0u;
                if constexpr (PREV)
                    *reinterpret_cast<uint32_t *>(dst + TW * 4 + o) = 0u;
            }
        }
        if (!cur_full && bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        const long long eo = (long long)c * n + t0;
        const char *src = reinterpret_cast<const char *>(a.in[r]) + eo * es;
        if constexpr (PREV) {
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
            cur_g = agonly ? N : 1;
            cur_item += gridDim.x;
            cur_full = (long long)cur_item * TW + TW <= min_len;
        }
    };
    if constexpr (FAST) {
        while (inflight < D && cur_item < tiles) {
            if (lane == 0)
                for (int r = warp; r < N; r += rstride)
                    issue_one(r, inflight);
            ++inflight;
            cursor_next();
        }
        __syncwarp();
    }

    Fifo rcv{0, 0}, snd{0, 0}, stg{0, 0};
    bool ok = true;
    long long t0 = 0;
    const bool first_item_withhold = a.withhold_rank >= 0;
    int withhold_g = 0; // step whose send is withheld in this slice (0: none)

    // run f(x, y) with the step's received and sent message; when both are
    // dense, as DenseMsg (the per-chunk sparse codec's dense-only code)
    auto with_msgs = [&](const Msg &x, const Msg &y, auto &&f) {
        if constexpr (CODEC == kCodecSparseChunk) {
            if (!x.sparse() && !y.sparse()) {
                f(DenseMsg(x), DenseMsg(y));
                return;
            }
        }
        f(x, y);
    };
    // the message of chunk c at hop h (h = N: the owner's) in the slice at t0
    auto msg_of = [&](int h, int c) -> Msg {
        if constexpr (CODEC == kCodecSparseChunk) {
            const int i = (h - 1) * N + c;
            return Msg{2 * i + fmt_s[i], (int)t0};
        } else {
            return Msg{0, 0};
        }
    };

    // group gi of rank r's own input for chunk c (staged on the fast path)
    auto input_group = [&](int r, int c, int V, int gi, const unsigned char *sp,
                           float (&v)[8]) {
        if constexpr (FAST) {
            // the stage is zero past the slice's end (see issue_one)
            load8_vec<LT>(sp + (gi * kTile + 8 * lane) * es, v);
            if constexpr (PREV) {
                float p[8];
                load8_vec<kF32>(sp + TW * 4 + (gi * kTile + 8 * lane) * 4, p);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = __fsub_rn(v[i], p[i]);
            }
        } else {
            const int vl = min(max(V - gi * kTile - 8 * lane, 0), 8);
            const long long eo = (long long)c * n + t0 + gi * kTile + 8 * lane;
            load8_scalar<LT>(reinterpret_cast<const char *>(a.in[r]) + eo * es, vl, v);
            if constexpr (PREV) {
                float p[8];
                load8_scalar<kF32>(a.prev[r] + eo, vl, p);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = __fsub_rn(v[i], p[i]);
            }
        }
    };
    // output epilogue of group gi: average, previous-round base, cast
    const float inv_n = ((N & (N - 1)) == 0) ? 1.0f / (float)N : 0.0f; // exact for powers of two
    const int out_t = a.out_t;
    const int osz = dtype_size(out_t);
    const bool plain_out = !a.average && !a.base && a.vec_out;
    const bool direct16 = kDirect16 && plain_out && out_t == kF16;
    auto output_group = [&](int r, int c, int V, int gi, float (&v)[8]) {
        const long long e0 = (long long)c * n + t0 + gi * kTile + 8 * lane;
        if (plain_out && V == TW) { // full slice, no epilogue arithmetic: vector store
            store8_full(reinterpret_cast<char *>(a.out[r]) + e0 * osz, out_t, v);
            return;
        }
        const int vl = V == TW ? 8 : min(max(V - gi * kTile - 8 * lane, 0), 8);
        if (a.average) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = inv_n != 0.0f ? __fmul_rn(v[i], inv_n) : __fdiv_rn(v[i], (float)N);
        }
        if (a.base) {
            float bb[8];
            if (a.vec_base && vl == 8)
                load8_vec<kF32>(a.base + e0, bb);
            else
                load8_scalar<kF32>(a.base + e0, vl, bb);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __fadd_rn(bb[i], v[i]);
        }
        store8(reinterpret_cast<char *>(a.out[r]) + e0 * osz, out_t, v, vl, a.vec_out != 0);
    };
    // error feedback of group gi: encode u = v + e into the slot, store
    // e = u - decoded and leave the decoded values in v
    auto encode_ef = [&](int r, int c, int V, int gi, float (&v)[8], unsigned char *dslot) {
        const long long e0 = (long long)c * n + t0 + gi * kTile + 8 * lane;
        const int vl = min(max(V - gi * kTile - 8 * lane, 0), 8);
        float *ep = a.resid[r] + e0;
        float e[8];
        if (a.vec_resid && vl == 8)
            load8_vec<kF32>(ep, e);
        else
            load8_scalar<kF32>(ep, vl, e);
        float u[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const float2 s2 = __fadd2_rn(make_float2(v[i], v[i + 1]), make_float2(e[i], e[i + 1]));
            u[i] = s2.x;
            u[i + 1] = s2.y;
            v[i] = s2.x;
            v[i + 1] = s2.y;
        }
        C::template encode<true>(v, dslot, gi, lane, V, a, scratch, Msg{0, 0});
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const float2 d2 = __fadd2_rn(make_float2(u[i], u[i + 1]), make_float2(-v[i], -v[i + 1]));
            e[i] = d2.x;
            e[i + 1] = d2.y;
        }
        store8(ep, kF32, e, vl, a.vec_resid != 0);
    };
    // One-group messages fit in registers: copy the message out and free its
    // slot before waiting for the next rank's slot, so even one slot per
    // edge cannot stall the ring.  Wider messages are streamed group by group
    // and their slot is freed at the end of the step (two slots per edge).
    constexpr bool kEarly = G == 1;
    auto release_early = [&](int r, const unsigned char *rslot, uint32_t rb, Reg &m,
                             const Msg &mg) {
        C::load(rslot, 0, lane, scratch, a, m, mg);
        if (ONE)
            my_recv += rb;
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(empty + r * K + rcv.slot);
            if (!ONE)
                rrecv[r] += rb;
        }
    };
    // Common case of a step's waits: every barrier it needs has already
    // completed, seen with one test each and one warp vote.  Otherwise the
    // step waits for them one by one (bounded).  A completed phase stays
    // complete until this rank acts on that barrier again, so the tests are
    // exact.  One-group messages free their receive slot before the send
    // wait, so they always take the one-by-one order.
    auto all_ready = [&](bool stage, bool recv, bool send, int r, int dst) -> bool {
        if constexpr (kEarly)
            return false;
        bool t = true;
        if (FAST && stage)
            t = mbar_try_wait(sbar + r * D + stg.slot, (uint32_t)stg.phase);
        if (recv)
            t &= mbar_try_wait(full + r * K + rcv.slot, (uint32_t)rcv.phase);
        if (send)
            t &= mbar_try_wait(empty + dst * K + snd.slot, (uint32_t)(snd.phase ^ 1));
        return __all_sync(kFull, t);
    };
    // after a step that consumed a staged load: refill that stage (the warp
    // barrier of the step's finish_step orders every lane's reads of the
    // stage before lane 0 issues the copy that overwrites it)
    auto stage_step = [&]() {
        if constexpr (FAST) {
            if (inflight == D && cur_item < tiles) { // refill the stage just consumed
                if (lane == 0)
                    for (int r = warp; r < N; r += rstride)
                        issue_one(r, stg.slot);
                cursor_next();
            } else {
                --inflight;
            }
            stg.advance(D);
        }
    };
    // publish: free the receive slot (if any), mark the sent message full
    auto finish_step = [&](int r, int g, bool recv, bool send, uint32_t rb, uint32_t sb) {
        if (ONE) {
            my_recv += recv ? rb : 0u;
            my_sent += send ? sb : 0u;
        }
        __syncwarp();
        if (lane == 0) {
            if (recv) {
                mbar_arrive(empty + r * K + rcv.slot);
                if (!ONE)
                    rrecv[r] += rb;
            }
            if (send) {
                const int dst = r + 1 == N ? 0 : r + 1;
                if (!((ONE || r == a.withhold_rank) && g == withhold_g))
                    mbar_arrive(full + dst * K + snd.slot);
                if (!ONE)
                    rsent[r] += sb;
            }
        }
    };

    for (int item = blockIdx.x; ok && item < tiles; item += gridDim.x) {
        t0 = (long long)item * TW;
        const bool item_full = t0 + TW <= min_len;
        // the fault-injection test withholds one send in each block's first slice
        withhold_g = first_item_withhold && item == (int)blockIdx.x &&
                             (!ONE || warp == a.withhold_rank)
                         ? a.withhold_step
                         : 0;

        // ---- reduce-scatter steps g = 1..N-1: send chunk (r-g) mod N
        for (int g = 1; ok && !agonly && g < N; ++g) {
            for (int r = warp; ONE || r < N; r += rstride) {
                int c = r - g;
                c += c < 0 ? N : 0;
                const int V = slice_len(c, t0, item_full);
                const int dst = r + 1 == N ? 0 : r + 1;
                const bool pre = all_ready(true, g >= 2, true, r, dst);
                if (!pre && FAST &&
                    !wait_ready(sbar + r * D + stg.slot, (uint32_t)stg.phase, a.timeout_ns,
                                a.status)) {
                    ok = false;
                    break;
                }
                if (!pre && g >= 2 &&
                    !wait_ready(full + r * K + rcv.slot, (uint32_t)rcv.phase, a.timeout_ns,
                                a.status)) {
                    ok = false;
                    break;
                }
                const unsigned char *sp = stages + (size_t)(r * D + stg.slot) * a.stage_bytes;
                const unsigned char *rslot = slots + (size_t)(r * K + rcv.slot) * a.slot_bytes;
                const Msg rmsg = g >= 2 ? msg_of(g - 1, c) : Msg{0, 0};
                const Msg smsg = msg_of(g, c);
                // wire bytes received and sent (data-dependent sizes are
                // summed group by group below)
                uint32_t rb = 0, sb = 0;
                Reg m0;
                if (g >= 2 && (kEarly || !C::kVarBytes))
                    with_msgs(rmsg, smsg, [&](const auto &rm, const auto &) {
                        rb = C::bytes(V, rslot, a, rm);
                        if (kEarly)
                            release_early(r, rslot, rb, m0, rm);
                    });
                if (!pre && !wait_ready(empty + dst * K + snd.slot, (uint32_t)(snd.phase ^ 1),
                                        a.timeout_ns, a.status)) {
                    ok = false;
                    break;
                }
                unsigned char *dslot = slots + (size_t)(dst * K + snd.slot) * a.slot_bytes;
                with_msgs(rmsg, smsg, [&](const auto &rm, const auto &sm) {
#pragma unroll kUnrollRS
                    for (int gi = 0; gi < G; ++gi) {
                        float v[8];
                        input_group(r, c, V, gi, sp, v);
                        if (g >= 2) {
                            Reg m;
                            if (kEarly) {
                                m = m0;
                            } else {
                                C::load(rslot, gi, lane, scratch, a, m, rm);
                                if constexpr (C::kVarBytes)
                                    rb += C::group_bytes(m, V, gi, rm);
                            }
                            C::decode_add(m, v, lane, scratch);
                        }
                        if constexpr (EF)
                            encode_ef(r, c, V, gi, v, dslot);
                        else
                            sb += C::template encode<false>(v, dslot, gi, lane, V, a, scratch, sm);
                    }
                    if constexpr (!C::kVarBytes)
                        sb = C::bytes(V, dslot, a, sm);
                });
                finish_step(r, g, g >= 2 && !kEarly, true, rb, sb);
                if (ONE)
                    break;
            }
            if (!ok)
                break;
            stage_step();
            if (g >= 2)
                rcv.advance(K);
            snd.advance(K);
        }
        if (!ok)
            break;

        // ---- owner step g = N: chunk r; allreduce encodes the full sum once
        for (int r = warp; ONE || r < N; r += rstride) {
            const int V = slice_len(r, t0, item_full);
            const int dst = r + 1 == N ? 0 : r + 1;
            const bool recv = N > 1 && !agonly, send = gather && N > 1;
            const bool pre = all_ready(true, recv, send, r, dst);
            if (!pre && FAST &&
                !wait_ready(sbar + r * D + stg.slot, (uint32_t)stg.phase, a.timeout_ns,
                            a.status)) {
                ok = false;
                break;
            }
            if (!pre && recv &&
                !wait_ready(full + r * K + rcv.slot, (uint32_t)rcv.phase, a.timeout_ns,
                            a.status)) {
                ok = false;
                break;
            }
            const unsigned char *sp = stages + (size_t)(r * D + stg.slot) * a.stage_bytes;
            const unsigned char *rslot = slots + (size_t)(r * K + rcv.slot) * a.slot_bytes;
            const Msg rmsg = recv ? msg_of(N - 1, r) : Msg{0, 0};
            const Msg smsg = msg_of(N, r);
            uint32_t rb = 0, sb = 0;
            Reg m0;
            if (recv && (kEarly || !C::kVarBytes))
                with_msgs(rmsg, smsg, [&](const auto &rm, const auto &) {
                    rb = C::bytes(V, rslot, a, rm);
                    if (kEarly)
                        release_early(r, rslot, rb, m0, rm);
                });
            if (!pre && send &&
                !wait_ready(empty + dst * K + snd.slot, (uint32_t)(snd.phase ^ 1), a.timeout_ns,
                            a.status)) {
                ok = false;
                break;
            }
            // N = 1 has no allgather step: encode into the rank's own (unused) slot
            unsigned char *dslot = send ? slots + (size_t)(dst * K + snd.slot) * a.slot_bytes
                                        : slots + (size_t)(r * K) * a.slot_bytes;
            bool done = false;
            if constexpr (kDirect16 && !EF) {
                // a full slice of plain fp16 outputs: encode the sum, send the
                // codes and write fp16 straight from them (a rolled loop: the
                // unrolled one measured slower, its code too large for the
                // instruction cache next to the unrolled loops)
                if (direct16 && send && recv && V == TW) {
                    uint4 *op = reinterpret_cast<uint4 *>(
                                    reinterpret_cast<__half *>(a.out[r]) + (long long)r * n + t0) +
                                lane;
#pragma unroll 1
                    for (int gi = 0; gi < G; ++gi) {
                        float v[8];
                        input_group(r, r, V, gi, sp, v);
                        Reg m;
                        if (kEarly)
                            m = m0;
                        else
                            C::load(rslot, gi, lane, scratch, a, m, rmsg);
                        C::decode_add(m, v, lane, scratch);
                        Reg w;
                        C::encode_reg(v, dslot, gi, lane, w);
                        uint32_t h[4];
                        const uint2 sc = lut[w.e + 128];
                        if (sc.x != 0u) {
                            bfp8_decode_f16(w.w, sc, h);
                        } else {
                            C::values(w, v, lane, scratch);
                            pack16x8<kF16>(v, h);
                        }
                        op[gi * (kTile / 8)] = make_uint4(h[0], h[1], h[2], h[3]);
                    }
                    done = true;
                }
            }
            if (!done)
                with_msgs(rmsg, smsg, [&](const auto &rm, const auto &sm) {
#pragma unroll 1
                    for (int gi = 0; gi < G; ++gi) {
                        float v[8];
                        input_group(r, r, V, gi, sp, v);
                        if (recv) {
                            Reg m;
                            if (kEarly) {
                                m = m0;
                            } else {
                                C::load(rslot, gi, lane, scratch, a, m, rm);
                                if constexpr (C::kVarBytes)
                                    rb += C::group_bytes(m, V, gi, rm);
                            }
                            C::decode_add(m, v, lane, scratch);
                        }
                        if (gather) {
                            if constexpr (EF)
                                encode_ef(r, r, V, gi, v, dslot);
                            else
                                sb += C::template encode<true>(v, dslot, gi, lane, V, a, scratch,
                                                               sm);
                        }
                        output_group(r, r, V, gi, v);
                    }
                });
            if constexpr (!C::kVarBytes)
                sb = C::bytes(V, dslot, a, smsg);
            finish_step(r, N, recv && !kEarly, send, rb, send ? sb : 0u);
            if (ONE)
                break;
        }
        if (!ok)
            break;
        stage_step();
        if (N > 1 && !agonly)
            rcv.advance(K);
        if (gather && N > 1)
            snd.advance(K);

        // ---- allgather steps g = N+1..2N-1: output chunk (r-g) mod N, forward its codes
        if (gather) {
            for (int g = N + 1; ok && g <= 2 * N - 1; ++g) {
                const bool fwd = g < 2 * N - 1;
                for (int r = warp; ONE || r < N; r += rstride) {
                    int c = r - g;
                    c += c < 0 ? N : 0;
                    c += c < 0 ? N : 0;
                    const int V = slice_len(c, t0, item_full);
                    const int dst = r + 1 == N ? 0 : r + 1;
                    const bool pre = all_ready(false, true, fwd, r, dst);
                    if (!pre && !wait_ready(full + r * K + rcv.slot, (uint32_t)rcv.phase,
                                            a.timeout_ns, a.status)) {
                        ok = false;
                        break;
                    }
                    const unsigned char *rslot =
                        slots + (size_t)(r * K + rcv.slot) * a.slot_bytes;
                    const Msg amsg = msg_of(N, c); // the owner's message, forwarded unchanged
                    uint32_t rb = 0;
                    Reg m0;
                    if (kEarly || !C::kVarBytes)
                        with_msgs(amsg, amsg, [&](const auto &am, const auto &) {
                            rb = C::bytes(V, rslot, a, am);
                            if (kEarly)
                                release_early(r, rslot, rb, m0, am);
                        });
                    if (!pre && fwd &&
                        !wait_ready(empty + dst * K + snd.slot, (uint32_t)(snd.phase ^ 1),
                                    a.timeout_ns, a.status)) {
                        ok = false;
                        break;
                    }
                    unsigned char *dslot = slots + (size_t)(dst * K + snd.slot) * a.slot_bytes;
                    bool done = false;
                    if constexpr (kDirect16) {
                        // a full slice of plain fp16 outputs: codes straight to fp16
                        if (direct16 && V == TW) {
                            uint4 *op = reinterpret_cast<uint4 *>(
                                            reinterpret_cast<__half *>(a.out[r]) +
                                            (long long)c * n + t0) +
                                        lane;
#pragma unroll
                            for (int gi = 0; gi < G; ++gi) {
                                Reg m;
                                if (kEarly)
                                    m = m0;
                                else
                                    C::load(rslot, gi, lane, scratch, a, m, amsg);
                                if (fwd)
                                    C::store(dslot, gi, lane, m, a, amsg);
                                uint32_t h[4];
                                const uint2 sc = lut[m.e + 128]; // m.e is a signed byte
                                if (sc.x != 0u) {
                                    bfp8_decode_f16(m.w, sc, h);
                                } else {
                                    float v[8];
                                    C::values(m, v, lane, scratch);
                                    pack16x8<kF16>(v, h);
                                }
                                op[gi * (kTile / 8)] = make_uint4(h[0], h[1], h[2], h[3]);
                            }
                            done = true;
                        }
                    }
                    if (!done)
                        with_msgs(amsg, amsg, [&](const auto &am, const auto &) {
#pragma unroll kUnrollAG
                            for (int gi = 0; gi < G; ++gi) {
                                Reg m;
                                if (kEarly) {
                                    m = m0;
                                } else {
                                    C::load(rslot, gi, lane, scratch, a, m, am);
                                    if constexpr (C::kVarBytes)
                                        rb += C::group_bytes(m, V, gi, am);
                                }
                                if (fwd)
                                    C::store(dslot, gi, lane, m, a, am);
                                float v[8];
                                C::values(m, v, lane, scratch);
                                output_group(r, c, V, gi, v);
                            }
                        });
                    __syncwarp();
                    finish_step(r, g, !kEarly, fwd, rb, rb);
                    if (ONE)
                        break;
                }
                if (!ok)
                    break;
                rcv.advance(K);
                if (fwd)
                    snd.advance(K);
            }
        }
    }

    // ---- drain this warp's staged copies that are still in flight
    if constexpr (FAST) {
        __syncwarp();
        // the loads in flight occupy the stages from stg on, in order
        for (int r = warp; r < N; r += W) {
            Fifo d = stg;
            for (int L = 0; L < inflight; ++L) {
                drain_phase(sbar + r * D + d.slot, (uint32_t)d.phase, a.timeout_ns);
                d.advance(D);
            }
        }
    }
    // ---- per-rank byte counters
    if (lane == 0) {
        if (ONE) {
            if (warp < N) {
                if (my_sent)
                    atomicAdd(a.sent + warp, my_sent);
                if (my_recv)
                    atomicAdd(a.recv + warp, my_recv);
            }
        } else {
            for (int r = warp; r < N; r += W) {
                if (rsent[r])
                    atomicAdd(a.sent + r, rsent[r]);
                if (rrecv[r])
                    atomicAdd(a.recv + r, rrecv[r]);
            }
        }
    }
}

// Kernel for one (codec, input dtype, slice width): the generic path, or the
// staged path in the given MODE.
template <int CODEC, int IN_T, int G, bool EF> const void *ring_variant(bool fast, int mode)
{
    if (!fast)
        return (const void *)ring_kernel<CODEC, IN_T, false, G, kRanksShared, EF>;
    switch (mode) {
    case kRankPerWarp8: return (const void *)ring_kernel<CODEC, IN_T, true, G, kRankPerWarp8, EF>;
    case kRankPerWarp16: return (const void *)ring_kernel<CODEC, IN_T, true, G, kRankPerWarp16, EF>;
    default: return (const void *)ring_kernel<CODEC, IN_T, true, G, kRanksShared, EF>;
    }
}
template <int CODEC, int G, bool EF = false> const void *ring_variant(int in_t, bool fast, int mode)
{
    switch (in_t) {
    case kF32: return ring_variant<CODEC, kF32, G, EF>(fast, mode);
    case kF16: return ring_variant<CODEC, kF16, G, EF>(fast, mode);
    case kBF16: return ring_variant<CODEC, kBF16, G, EF>(fast, mode);
    case kF32Diff: return ring_variant<CODEC, kF32Diff, G, EF>(fast, mode);
    default: return nullptr;
    }
}

} // namespace rra

// rra_kernels.h -- launch interface between the C ABI (rra_host.cu) and the
// kernel translation units.  Host-side only types; no torch, no CUDA types
// beyond cudaStream_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rra {

constexpr int kMaxRanks = 64;
constexpr int kMaxWarps = 16; // warps per block; ranks per warp = ceil(N / warps)

// kCodecSparse: one sparse/dense message per 256-element slice;
// kCodecSparseChunk: one message per ring chunk and hop, its format chosen
// from the chunk's nonzero count (the count pass below).
enum Codec { kCodecNone = 0, kCodecBfp8 = 1, kCodecBfp4 = 2, kCodecSparse = 3, kCodecSparseChunk = 4 };
enum Mode { kModeAllreduce = 0, kModeReduceScatter = 1, kModeAllgather = 2 };

// Launch shape of a ring kernel: blocks per SM, mailbox slots per edge,
// staging depth, 256-element groups per slice.  Zero fields: automatic.
struct Tune {
    int blocks = 0, K = 0, D = 0, G = 0;
    bool any() const { return blocks || K || D || G; }
};
// How simulated ranks map onto the warps of a ring kernel block.
enum RankMap { kRanksShared = 0, kRankPerWarp8 = 1, kRankPerWarp16 = 2 };

// Arguments of the fused ring kernel (reduce-scatter pass, owner finalise,
// allgather pass).  Passed by value as a __grid_constant__ parameter.
struct RingArgs {
    int N;          // simulated ranks
    int mode;       // kModeAllreduce / kModeReduceScatter / kModeAllgather
    int in_t;       // dtype of the inputs
    int out_t;      // dtype of the outputs
    int K;          // mailbox depth (messages in flight per ring edge)
    int D;          // input staging depth per rank (fast path)
    int slot_bytes; // bytes of one mailbox slot
    int stage_bytes;
    int average;       // divide the reduced value by N
    int has_prev;      // difference encoding: inputs are cur, prev[] given
    int withhold_rank; // fault injection (-1: off)
    int withhold_step;
    int vec_out;       // outputs allow 16-byte vector stores
    int vec_base;      // diff_base allows 16-byte vector loads
    int vec_resid;     // error-feedback residuals allow 16-byte vector access
    long long T;       // elements per rank
    long long n;       // chunk length ceil(T/N)
    long long tiles;   // slices per chunk ceil(n / 256)
    double one_minus_thr; // sparse: a message is sparse iff nnz < one_minus_thr * len
    int sp_full_lim;      // per-slice sparse: a full 256-element slice is sparse iff nnz < sp_full_lim
    int sp_icap;          // per-slice sparse: most (value, index) pairs of a sparse group = lim - 1
    int sp_sub;           // per-slice sparse: bytes of one group's sub-message in a slot
    const unsigned long long *sp_nnz; // per-chunk sparse: nnz[(h-1)*N + c] of the message of
                                      // chunk c at hop h (h = N: the owner's), from the count pass
    unsigned char *sp_spill; // per-chunk sparse: the pairs of a group beyond the slot's 128,
                             // (slot_bytes - 32) bytes per (block, slot)
    int slots_off;           // byte offset of the mailbox slots in the block's shared memory
    unsigned long long timeout_ns;
    unsigned long long *sent; // [N] device counters of this call
    unsigned long long *recv; // [N]
    unsigned long long *zero; // [2N] counters of the next call: block 0 clears them
    unsigned *status;         // device status word
    const float *base;        // diff_base or nullptr
    const void *in[kMaxRanks];
    const float *prev[kMaxRanks];
    float *resid[kMaxRanks]; // error-feedback residuals (kernels instantiated with EF)
    void *out[kMaxRanks];
};

// Arguments of the copy collectives (allgather, broadcast) and the tree.
struct CopyArgs {
    int N;
    int es;    // element size in bytes (2 or 4)
    int root;  // broadcast root
    int K;
    int D;
    int slot_bytes;
    int stage_bytes;
    int withhold_rank;
    int withhold_step;
    int bits;        // BFP broadcast: code width (8 or 4); 0 for plain copies
    int dt;          // BFP broadcast: element dtype (kF32 / kF16 / kBF16)
    long long T;
    long long n;     // allgather chunk length
    long long tiles; // slices per launch item range
    unsigned long long timeout_ns;
    unsigned long long *sent;
    unsigned long long *recv;
    unsigned long long *zero;
    unsigned *status;
    void *buf[kMaxRanks];
};

// Per-chunk sparse codec: nonzero count of every message of one call.
// Hop h = 1..N-1 carries the reduce-scatter partial x_{c+1} + ... + x_{c+h}
// of chunk c (fp32, ring order), hop N the owner's full sum, or, for the
// allgather alone, chunk c of buffer c.  Counts are summed into acc by
// atomics; the last block to finish moves them to out and clears acc and
// the ticket for the next call.
struct SpCountArgs {
    int N;
    int h_lo, h_hi;  // hops counted: allreduce 1..N, reduce-scatter 1..N-1, allgather N..N
    int bpc;         // blocks per chunk (set by the launcher)
    long long T, n;
    unsigned long long *acc; // [N * N], zero on entry
    unsigned long long *out; // [N * N]
    unsigned *ticket;        // zero on entry
    const void *in[kMaxRanks];
    const float *prev[kMaxRanks];
};
cudaError_t launch_sparse_chunk_count(const SpCountArgs &a, int in_kind, bool vec,
                                      cudaStream_t st);

// Shared-memory layout of the ring / copy kernels (host and device agree).
struct Layout {
    int full, empty, stage_bar, rank_state, slots, stages, scratch, lut, fmt, total;
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int N, int K, int D, int slot_bytes,
                                              int stage_bytes, int warps, bool fast,
                                              int sparse, bool lut)
{
    Layout L;
    int off = 0;
    L.full = off;
    off += N * K * 8;
    L.empty = off;
    off += N * K * 8;
    L.stage_bar = off;
    off += fast ? N * D * 8 : 0;
    L.rank_state = off; // per rank: next staged load to issue, loads consumed, sent, recv
    off += N * 32;
    off = align_up(off, 128);
    L.slots = off;
    off += N * K * slot_bytes;
    off = align_up(off, 128);
    L.stages = off;
    off += fast ? N * D * stage_bytes : 0;
    off = align_up(off, 16);
    L.scratch = off;
    off += sparse ? warps * 256 * 4 : 0; // per warp: one restored 256-element group
    off = align_up(off, 16);
    L.lut = off; // BFP8: 256 entries of 8 bytes (the fp16 output table)
    off += lut ? 256 * 8 : 0;
    off = align_up(off, 16);
    L.fmt = off; // per-chunk sparse: format byte of every (hop, chunk) message
    off += sparse == 2 ? N * N : 0;
    L.total = align_up(off, 128);
    return L;
}

// Shared-memory layout of the allgather / broadcast / tree kernels: `edges`
// slot FIFOs of K slots (full and empty barrier each), D stages for each of
// `stagers` ranks, per-rank byte counters.
struct CollLayout {
    int full, empty, stage_bar, counters, slots, stages, total;
};

__host__ __device__ inline CollLayout coll_layout(int N, int edges, int K, int stagers, int D,
                                                  int slot_bytes, int stage_bytes, bool stage)
{
    CollLayout L;
    int off = 0;
    L.full = off;
    off += edges * K * 8;
    L.empty = off;
    off += edges * K * 8;
    L.stage_bar = off;
    off += stagers * D * 8;
    L.counters = off;
    off += N * 16;
    off = align_up(off, 128);
    L.slots = off;
    off += edges * K * slot_bytes;
    off = align_up(off, 128);
    L.stages = off;
    off += stage ? stagers * D * stage_bytes : 0;
    L.total = align_up(off, 128);
    return L;
}

// Kernel entry points (one per translation unit family).  Each returns the
// launch's cudaError_t.
cudaError_t launch_ring(const void *fn, const RingArgs &a, int grid, int warps, int smem,
                        cudaStream_t st);

// Allgather (which 0), broadcast (1) or tree allreduce (2) kernel for
// element size es, slice width 256 * groups, staged or generic path, one rank
// per warp or several; nullptr if not instantiated.
const void *coll_fn(int which, int es, int groups, bool fast, bool one);
// BFP-compressed broadcast (bits 8 or 4); the element dtype is a kernel argument
const void *bcast_bfp_fn(int bits, int groups, bool fast, bool one);
cudaError_t launch_coll(const void *fn, const CopyArgs &a, int grid, int warps, int smem,
                        cudaStream_t st);

// Standalone codec kernels.
cudaError_t launch_bfp_encode(const void *x, long long n, int dtype, int bits, int8_t *exps,
                              uint8_t *mants, cudaStream_t st);
cudaError_t launch_bfp_decode(const int8_t *exps, const uint8_t *mants, long long n, int bits,
                              float *out, int accumulate, cudaStream_t st);
// The standalone sparse encoder.  scratch: sparse_encode_scratch_words(n)
// 32-bit words, needing no clearing (a call writes every word it reads).
cudaError_t launch_sparse_encode(const void *x, long long n, int dtype, double one_minus_thr,
                                 uint32_t *hdr, void *vals, int32_t *idx, uint32_t *scratch,
                                 cudaStream_t st);
long long sparse_encode_scratch_words(long long n);
cudaError_t launch_sparse_decode(const uint32_t *hdr, const void *vals, const int32_t *idx,
                                 long long n, int dtype, float *acc, int accumulate,
                                 cudaStream_t st);
cudaError_t launch_diff_encode(const float *cur, const float *prev, float *diff, long long n,
                               cudaStream_t st);

// Codec statistics over the N input buffers: stats[0..3] = elements, nonzero,
// flushed by BFP4, flushed by BFP8 (added to; the caller clears them).
struct StatsArgs {
    int N;
    long long T, n;
    unsigned long long *stats;
    const void *in[kMaxRanks];
};
cudaError_t launch_codec_stats(const StatsArgs &a, int dtype, cudaStream_t st);

int num_sms();

} // namespace rra

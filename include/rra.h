/*
 * rra.h -- C ABI of a GB300 (sm_103a) library for the chunked ring
 * allreduce coupled with gradient-compression codecs.
 *
 * N ranks are simulated as N buffers in the memory of ONE GPU.  A "send" is a
 * device-side write of the (encoded) message into the receiving rank's
 * receive slot; the receiving rank decodes it from there and accumulates in
 * fp32.  All functions take plain pointers and sizes; the caller keeps
 * ownership of every buffer it passes.
 *
 * Sources (cited by page title and section):
 *  [ring]  "从零实现集合通信" (collective ops from scratch), section
 *          "两趟实现 ring allreduce": tensor cut into N equal chunks, rank r
 *          owns chunk r; reduce-scatter pass of N-1 steps (at step s rank r
 *          sends chunk (r-s) mod N to rank r+1 and accumulates the chunk it
 *          receives), then an allgather pass of N-1 steps; the per-rank byte
 *          and step table (ring 2T(N-1)/N, tree T log2 N, broadcast T over a
 *          log2(N) tree, allgather and reduce_scatter T(N-1)/N each);
 *          section "练习" (tree variant chosen by message size, byte counter,
 *          receive timeout instead of hanging).
 *  [cccl]  "CCCL通信压缩库：突破LLM训练通信墙的工程实践": §2.1 sparse
 *          values+indices when sparsity exceeds a threshold (e.g. 50%),
 *          block floating point (one shared exponent per block of e.g. 128
 *          elements, 8- or 4-bit mantissas), difference against the previous
 *          round; §2.2 chunked compress -> send -> decompress -> reduce
 *          pipeline; §3.3 compression types and sparsity_threshold 0.5.
 *
 * Conventions shared by every entry point:
 *  - Device pointers are plain CUDA device addresses of the device that was
 *    current when the communicator was created (or, for the codec
 *    functions, the current device).  Arrays of N pointers ("in", "out",
 *    "buf", "diff_prev") are HOST arrays; they are read during the call and
 *    may be reused or freed as soon as it returns.
 *  - Elements are counted, not bytes.  "count" (T) is the number of
 *    elements of every rank's buffer.
 *  - Chunking: n = ceil(T/N); chunk c covers elements
 *    [c*n, min(T, (c+1)*n)); trailing chunks may be short or empty.
 *  - All work is enqueued asynchronously on "stream" (a cudaStream_t; NULL
 *    is the legacy default stream).  Argument errors are detected on the host
 *    before anything is enqueued and returned as RRA_ERR_INVALID /
 *    RRA_ERR_UNSUPPORTED; a failed launch returns RRA_ERR_CUDA.  Errors the
 *    device detects while running (a wait that ran out of time) are latched
 *    in the communicator and reported by rra_comm_status().
 *  - Inputs must be finite: NaN or infinity in an input is outside the
 *    contract (results unspecified, no fault).
 *  - Nothing on these paths allocates memory except rra_comm_create, and
 *    rra_sparse_encode / rra_sparse_decode when a stream's scratch is
 *    smaller than the call needs (its first call, or a larger n; see there).
 */
#ifndef RRA_H
#define RRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest number of simulated ranks one communicator supports. */
#define RRA_MAX_RANKS 64
/* Elements per block-floating-point block ([cccl] §2.1: "e.g. 128"). */
#define RRA_BFP_BLOCK 128
/* Elements per ring message slice: the ring streams each chunk through the
 * receive slots in slices of a multiple of this many elements.  With
 * RRA_SPARSE_PER_SLICE, every slice of this many elements is one sparse
 * codec message with its own header and its own sparse/dense choice
 * ([cccl] §2.2: the tensor is cut into small chunks that are compressed and
 * sent one after the other). */
#define RRA_RING_SLICE 256

/* Granularity of the sparse codec's sparse/dense decision
 * (rra_codec.sparse_granularity). */
#define RRA_SPARSE_PER_CHUNK 0 /* one message per ring chunk and hop (default) */
#define RRA_SPARSE_PER_SLICE 1 /* one message per RRA_RING_SLICE elements     */

typedef enum {
    RRA_OK = 0,
    RRA_ERR_INVALID = 1,     /* a NULL pointer, a size out of range, a bad enum */
    RRA_ERR_UNSUPPORTED = 2, /* valid arguments, combination not provided   */
    RRA_ERR_CUDA = 3,        /* a CUDA call or launch failed                */
    RRA_ERR_TIMEOUT = 4,     /* a device-side wait ran past its time limit   */
    RRA_ERR_NOMEM = 5        /* device memory allocation failed              */
} rra_status;

typedef enum { RRA_F32 = 0, RRA_F16 = 1, RRA_BF16 = 2 } rra_dtype;

typedef enum {
    RRA_CODEC_NONE = 0,   /* lossless: fp32 on the wire                      */
    RRA_CODEC_BFP = 1,    /* block floating point, 8- or 4-bit mantissas     */
    RRA_CODEC_SPARSE = 2  /* values + int32 indices, or dense fallback       */
} rra_codec_kind;

/*
 * Codec of one reducing call ([cccl] §3.2/§3.3 configuration fields).
 *  kind                what goes on the wire (above).
 *  bits                8 or 4 (RRA_CODEC_BFP only).
 *  sparsity_threshold  RRA_CODEC_SPARSE: a message is sent sparse iff its
 *                      sparsity (zeros / length) is strictly greater, i.e.
 *                      nnz < (1 - threshold) * length; must lie in [0, 1).
 *  diff_prev           NULL, or a host array of N device pointers to fp32
 *                      buffers of T elements: the previous round's values.
 *                      The ring then runs on cur - prev ([cccl] §2.1
 *                      difference encoding); requires in_t == RRA_F32.
 *  diff_base           NULL, or a device pointer to T fp32 values (the
 *                      previous round's result R_prev, shared by all ranks)
 *                      added back in the output epilogue.
 *  average             nonzero: the reduced value is divided by N (IEEE
 *                      division, round to nearest even) before diff_base is
 *                      added: out = diff_base + v / N.
 *  residual            NULL, or a host array of N device pointers to fp32
 *                      buffers of T elements: per-rank error-feedback
 *                      residuals, read and updated in place ([cccl] §5,
 *                      future directions: the precision a compression loses
 *                      is carried into the next round).  Every value rank r
 *                      encodes -- its reduce-scatter messages and, as owner,
 *                      its chunk's sum -- is encoded as u = v + e_r, and
 *                      e_r = u - decode(codes) is stored back; each element
 *                      is updated once per call.  RRA_CODEC_BFP only (the
 *                      other codecs lose nothing); start from zeros.  The
 *                      buffers must not overlap each other or any input,
 *                      output, diff_prev or diff_base buffer.
 *  sparse_granularity  RRA_CODEC_SPARSE: RRA_SPARSE_PER_CHUNK (0, default):
 *                      at every hop the sender's message for a chunk is one
 *                      message, sparse or dense by the nonzero count of the
 *                      whole chunk's partial ([cccl] §2.1: the sparsity of
 *                      the tensor about to be sent decides).  Before the ring
 *                      starts, a count pass over the inputs (one read of
 *                      every input) gives the count of every (chunk, hop)
 *                      message: each hop's partial is the ring-order sum of
 *                      the inputs of the ranks it has passed.  Chunks of more
 *                      than 2^31 - 1 elements are RRA_ERR_UNSUPPORTED (int32
 *                      indices).  RRA_SPARSE_PER_SLICE (1): one message per
 *                      RRA_RING_SLICE elements, each decided on its own.
 * A NULL rra_codec* means {RRA_CODEC_NONE, 0, 0, NULL, NULL, 0, NULL, 0}.
 */
typedef struct {
    rra_codec_kind kind;
    int bits;
    float sparsity_threshold;
    const float *const *diff_prev;
    const float *diff_base;
    int average;
    float *const *residual;
    int sparse_granularity;
} rra_codec;

/* Opaque communicator: owns the device-side byte counters, the status word
 * and the launch configuration of the N simulated ranks. */
typedef struct rra_comm rra_comm;

/*
 * Create a communicator for nranks simulated ranks on the current device.
 *  nranks     1..RRA_MAX_RANKS.
 *  max_count  largest "count" any later call may pass (>= 1).
 *  max_dtype  widest element type later calls may pass (informational; the
 *             library keeps no per-size buffers: receive slots live in
 *             on-chip shared memory of each launched block).
 *  out        receives the handle.
 * Allocates device memory for its counters and status (a few hundred
 * bytes) and for the sparse codec's message counts (16 * nranks^2 + 8 bytes).
 * Threads: one communicator serves one host thread at a time (its launch
 * caches, counter sets and last-call record have no lock); separate
 * communicators may be driven from separate threads.  Calls on one
 * communicator must also run in order on the GPU: each launch clears the
 * byte counters of the next call, so two calls on different streams need
 * an ordering between them (an event, or one stream) to count correctly.
 * rra_get_bytes and rra_comm_status wait on the stream of the last call.
 * Errors: RRA_ERR_INVALID (bad nranks, max_count 0, NULL out, bad dtype),
 * RRA_ERR_NOMEM, RRA_ERR_CUDA.
 */
rra_status rra_comm_create(int nranks, size_t max_count, rra_dtype max_dtype, rra_comm **out);

/* Destroy a communicator (synchronises the device first).  NULL is a no-op. */
rra_status rra_comm_destroy(rra_comm *comm);

/*
 * Two-pass ring allreduce ([ring] "两趟实现 ring allreduce"; [cccl] §2.1-2.2).
 *  in[r]     device pointer to rank r's T input elements of type in_t
 *            (with codec->diff_prev: the current round's fp32 values).
 *  out[r]    device pointer to rank r's T output elements of type out_t.
 *            out[r] may equal in[r] (in place); output buffers of different
 *            ranks must not overlap, and none may overlap diff_base.
 *  codec     NULL or a codec (above).
 * Schedule (steps s = 1..N-1 in each pass): reduce-scatter step s, rank r
 * sends chunk (r-s) mod N to rank r+1, which adds its own fp32 copy of that
 * chunk to the decoded message; after N-1 steps rank r owns the full sum S_r
 * of chunk r.  Lossless: S_r is sent as fp32.  With a codec, every hop
 * re-encodes the sender's fp32 partial, the owner encodes S_r once, the
 * allgather pass (step s: rank r sends chunk (r-s+1) mod N) forwards those
 * codes unchanged, and every rank, the owner included, outputs their decoded
 * value, so all N outputs are bit-identical.  Lossless sums follow the ring
 * order ((x_{c+1} + x_{c+2}) + ...) + x_c exactly (fp32, round to nearest
 * even, no FMA).  Output: cast to out_t with round to nearest even, after the
 * optional average and diff_base epilogue.
 * Wire formats of one message of len elements (NONE and BFP: a chunk's
 * message is the concatenation of its slices' messages, so these sizes add
 * up over any cut into slices of multiples of 128 elements):
 *  NONE   fp32[len]                                       4 len bytes
 *  BFP    int8 exps[ceil(len/128)] + mantissas            ceil(len/128) + len (8-bit)
 *                                                         or + ceil(len/2) (4-bit)
 *  SPARSE {uint32 fmt, uint32 nnz} + fp32 vals[nnz] + int32 idx[nnz]
 *         (relative to the message start, ascending) = 8 + 8 nnz bytes, or
 *         dense {fmt = 0, nnz} + fp32[len] = 8 + 4 len bytes; one message
 *         per chunk and hop (len = the chunk's length; an empty chunk sends
 *         nothing), or per RRA_RING_SLICE elements (sparse_granularity).
 * A sparse receiver restores the message -- the listed values at their
 * indices, +0.0 elsewhere -- and adds the whole restored chunk ([cccl] §2.2:
 * receive, decompress, then reduce), so the sparse ring's result equals the
 * lossless ring's bit for bit.
 * Errors: RRA_ERR_INVALID (NULL pointers, count 0 or > max_count, bad enums,
 * bits not 8/4, threshold outside [0,1), a bad sparse_granularity,
 * diff_prev with in_t != F32, out overlapping diff_base),
 * RRA_ERR_UNSUPPORTED (see sparse_granularity), RRA_ERR_CUDA.
 */
rra_status rra_ring_allreduce(rra_comm *comm, const void *const *in, void *const *out,
                              size_t count, rra_dtype in_t, rra_dtype out_t,
                              const rra_codec *codec, void *stream);

/*
 * Reduce-scatter: the first pass of the ring alone ([ring] table:
 * T(N-1)/N bytes per rank, N-1 steps).  Only chunk r of out[r] is written
 * (at its offset r*n); the rest of out[r] is left untouched.  The owner's
 * value is its fp32 sum S_r (not re-encoded), then the same epilogue and
 * cast as the allreduce.  Same arguments and errors as rra_ring_allreduce.
 */
rra_status rra_reduce_scatter(rra_comm *comm, const void *const *in, void *const *out,
                              size_t count, rra_dtype in_t, rra_dtype out_t,
                              const rra_codec *codec, void *stream);

/*
 * Allgather, in place ([ring] table: T(N-1)/N bytes per rank, N-1 steps):
 * on entry chunk r of buf[r] holds rank r's contribution; on return every
 * buf[r] holds all N chunks.  Elements are copied bit for bit, uncompressed
 * ([cccl] §2.1: allgather and broadcast stay conservative).
 * Errors: RRA_ERR_INVALID, RRA_ERR_CUDA.
 */
rra_status rra_allgather(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                         void *stream);

/*
 * Compressed allgather, in place ([cccl] §2.1, the operator-aware layer:
 * allgather and broadcast take lossless compression or a higher-precision
 * lossy one; §3.3: low-precision compression for all_gather once all_reduce
 * runs compressed).  On entry chunk r of buf[r] (dtype f32, f16 or bf16) is
 * rank r's contribution.  Its owner encodes it once -- BFP (codec->bits 8
 * or 4, lossy) or sparse values + indices (codec->sparsity_threshold and
 * sparse_granularity: one message per chunk, decided by the nonzero count
 * of chunk r of buf[r], which a count pass reads first, or one per slice;
 * lossless) -- the codes travel the ring of the allgather pass unchanged
 * (N-1 steps), and every rank, the owner included, stores the decoded chunk
 * in dtype (round to nearest even), so all buffers end identical.  Sparse
 * codes restore every element bit for bit.  Byte counters: the messages
 * each rank forwards (all chunks but chunk r+1) and receives.
 * codec NULL or RRA_CODEC_NONE: rra_allgather (a plain copy).
 * Errors: RRA_ERR_INVALID (as rra_allgather; diff_prev, diff_base, average
 * or residual set; a bad codec), RRA_ERR_CUDA.
 */
rra_status rra_allgather_codec(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                               const rra_codec *codec, void *stream);

/*
 * Broadcast from rank "root" over a binomial tree of depth ceil(log2 N)
 * ([ring] table: T bytes per receiving rank, log2(N) tree).  At level
 * k = 0..ceil(log2 N)-1 every relative rank q < 2^k with q + 2^k < N sends
 * its whole buffer to q + 2^k (relative rank q = (r - root) mod N).  Each
 * edge is copied by its receiver, from the parent's copy of the slice.  In
 * place, bit-exact copies.  Errors: RRA_ERR_INVALID (root outside 0..N-1,
 * ...), RRA_ERR_CUDA.
 */
rra_status rra_broadcast(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                         int root, void *stream);

/*
 * Compressed broadcast over the same binomial tree ([cccl] §2.1, the
 * operator-aware layer: broadcast takes a higher-precision lossy
 * compression; §3.3: low-precision compression for broadcast once
 * all_reduce runs compressed).  The root encodes its buffer once as block
 * floating point (codec->bits 8 or 4; 128-element blocks from the buffer
 * start), every tree edge carries those codes unchanged, and every rank,
 * the root included, stores the decoded buffer in dtype (round to nearest
 * even), so all buffers end identical.  Byte counters: the message
 * (ceil(count/128) exponent bytes + the codes) once per tree edge.
 * codec NULL or RRA_CODEC_NONE: rra_broadcast (a plain copy).
 * Errors: RRA_ERR_INVALID (as rra_broadcast; diff_prev, diff_base, average or
 * residual set; bits other than 8 or 4), RRA_ERR_UNSUPPORTED (the sparse
 * codec), RRA_ERR_CUDA.
 */
rra_status rra_broadcast_codec(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                               int root, const rra_codec *codec, void *stream);

/*
 * Tree allreduce ([ring] table: T log2 N bytes, 2 log2 N steps; "练习":
 * the tree variant for small messages).  Binomial reduce to rank 0 (at level
 * k every rank r with r mod 2^(k+1) = 0 and r + 2^k < N adds rank r+2^k's
 * fp32 partial to its own), then the binomial broadcast above from rank 0.
 * In place; dtype must be RRA_F32 (RRA_ERR_UNSUPPORTED otherwise).
 */
rra_status rra_tree_allreduce(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                              void *stream);

/*
 * Block-floating-point encode of x[0..n) ([cccl] §2.1, §3.3).  For each
 * 128-element block (the last one may be short): e = floor(log2 max|x|)
 * taken from the fp32 exponent bits (-126 for a zero or subnormal maximum),
 * q = bits-2, m_i = clamp(rne(x_i * 2^(q-e)), -(2^(bits-1)-1), 2^(bits-1)-1).
 *  x      device, n elements of dtype (widened to fp32 exactly).
 *  exps   device, ceil(n/128) int8 exponents.
 *  mants  device, n bytes (bits 8: int8 codes) or ceil(n/2) bytes (bits 4:
 *         element 2j in the low nibble of byte j, 2j+1 in the high nibble,
 *         two's complement; an odd tail leaves the last high nibble 0).
 * Errors: RRA_ERR_INVALID (NULL, n 0, bits not 8/4), RRA_ERR_CUDA.
 */
rra_status rra_bfp_encode(const void *x, size_t n, rra_dtype dtype, int bits, int8_t *exps,
                          uint8_t *mants, void *stream);

/*
 * Block-floating-point decode: out[i] = m_i * 2^(e-q) (exact in fp32), or,
 * with accumulate != 0, out[i] = out[i] + m_i * 2^(e-q) (fp32, round to
 * nearest even).  Layout as for rra_bfp_encode; out is device fp32[n].
 */
rra_status rra_bfp_decode(const int8_t *exps, const uint8_t *mants, size_t n, int bits,
                          float *out, int accumulate, void *stream);

/*
 * Sparse encode of x[0..n) as ONE message ([cccl] §2.1: send only the
 * nonzero values and their indices when the sparsity exceeds the
 * threshold).  An element is zero iff its bit pattern, widened to fp32, is
 * +0.0 (so -0.0 is kept and the round trip is exact).
 *  hdr    device uint32[2]: hdr[0] = 1 (sparse) or 0 (dense), hdr[1] = nnz.
 *  vals   device, n elements of dtype capacity.  Sparse: the nnz nonzero
 *         values in index order.  Dense: a copy of x.
 *  idx    device, n int32 capacity.  Sparse: the nnz indices, ascending.
 * Sparse iff nnz < (1 - threshold) * n (evaluated in double).  Three
 * passes: a count per 1024-element chunk, an exclusive scan of the counts,
 * and an emit pass that writes each chunk's nonzeros at its offset (or copies
 * x when the message is dense; idx is then left as it was).
 * Uses scratch (one uint32 per 1024 elements, one per 4096 chunks) from a
 * workspace per device and stream that the library allocates with
 * cudaMalloc on the first call that needs more than it holds (so that first
 * call must not be made during stream capture).  Encodes on different streams may overlap: each stream
 * has its own workspace.  Errors: RRA_ERR_INVALID, RRA_ERR_NOMEM,
 * RRA_ERR_CUDA.
 */
rra_status rra_sparse_encode(const void *x, size_t n, rra_dtype dtype, float threshold,
                             uint32_t *hdr, void *vals, int32_t *idx, void *stream);

/* Largest n that rra_sparse_encode_noalloc accepts: its fixed scratch holds
 * one 32-bit count per 1024 elements and one total per 4096 counts. */
#define RRA_NOALLOC_MAX_COUNT (65536ull * 4096ull)

/*
 * rra_sparse_encode for callers that cannot allocate device memory (the
 * pages have no counterpart; it is a deployment variant of the sparse
 * encoder).  Such callers are processes whose device memory is handed out by
 * their own allocator or budgeted up front, latency-critical loops that
 * cannot take an allocation's implicit device synchronisation, and libraries
 * that must not call the CUDA allocator behind their host framework's back.
 * Same arguments, output and errors as rra_sparse_encode, except:
 *  - it never allocates: no cudaMalloc, cudaFree or allocating library call.
 *    Its scratch is a fixed array inside the library (about 1 MiB of
 *    device memory on every GPU that loads the library, held until the
 *    process exits).
 *  - n may not exceed RRA_NOALLOC_MAX_COUNT (2^28 elements); larger n returns
 *    RRA_ERR_INVALID without doing anything (use rra_sparse_encode then).
 *  - the first call on a device looks up the scratch array's device address
 *    (cudaGetSymbolAddress) with that device current, and keeps it for the
 *    rest of the process; after cudaDeviceReset the function must not be
 *    called again.
 *  - all calls on a device share the one scratch array.  A call writes
 *    every scratch word it reads before reading it, so nothing needs
 *    clearing, before the first call or between calls; calls that overlap
 *    on the GPU (different streams without ordering between them) race on
 *    the scratch and give undefined results for those calls.
 */
rra_status rra_sparse_encode_noalloc(const void *x, size_t n, rra_dtype dtype, float threshold,
                                     uint32_t *hdr, void *vals, int32_t *idx, void *stream);

/*
 * Sparse decode into fp32 acc[0..n) (hdr, vals, idx as written by
 * rra_sparse_encode: indices ascending; the format is read on the device).
 * A sparse message is restored (or added) in one pass over acc, 4096
 * elements at a time, using a scratch of n/4096 + 1 words per device
 * and stream that the library allocates on first use and grows as needed
 * (so the first call on a stream, or the first with a larger n, must not be
 * made during stream capture; decodes on different streams may overlap);
 * an index out of order or outside [0, n) is ignored.
 *  accumulate == 0: acc = the restored message (+0.0 where a sparse message
 *                   lists nothing).
 *  accumulate != 0: acc[i] = acc[i] + v at every position the message
 *                   carries (all of them when dense, the listed ones when
 *                   sparse); other positions are left as they are.
 */
rra_status rra_sparse_decode(const uint32_t *hdr, const void *vals, const int32_t *idx,
                             size_t n, rra_dtype dtype, float *acc, int accumulate,
                             void *stream);

/* Difference encoding ([cccl] §2.1): diff[i] = cur[i] - prev[i] in fp32,
 * round to nearest even.  diff may alias cur or prev. */
rra_status rra_diff_encode(const float *cur, const float *prev, float *diff, size_t n,
                           void *stream);

/*
 * Byte counters of the last collective call on this communicator ([ring]
 * "练习": per-rank byte counter): sent[r] / recv[r] = wire bytes rank r
 * wrote into / read from receive slots, counted on the device.  Lossless
 * ring: 2 (N-1) n * 4 bytes per rank when N divides T.  Synchronises the
 * stream of that call.  sent, recv: HOST arrays of N entries.  A call that
 * returned an error did not launch and does not count as the last call.
 * Errors: RRA_ERR_INVALID, RRA_ERR_CUDA, or a latched device error.
 */
rra_status rra_get_bytes(rra_comm *comm, uint64_t *sent, uint64_t *recv);

/* Synchronise the last call's stream, return the latched device-side error
 * (RRA_ERR_TIMEOUT, ...) or RRA_OK, and clear it. */
rra_status rra_comm_status(rra_comm *comm);

/* Time limit of every device-side wait (mailbox and copy waits), in
 * nanoseconds; 0 restores the default (2 s).  On expiry the kernel latches
 * RRA_ERR_TIMEOUT and returns instead of waiting further ([ring] "练习":
 * a stuck rank raises a deadline error instead of hanging). */
rra_status rra_set_timeout(rra_comm *comm, uint64_t ns);

/*
 * Launch tuning of the fused kernels (the in-kernel pipeline that replaces
 * the pages' "chunk size" knob, CCCL §3.3: automatic by default, manual
 * override allowed).  Each value 0 = automatic.
 *  blocks_per_sm  resident blocks per SM to launch (1..32; clamped to what
 *                 the occupancy calculator allows).
 *  mailbox_depth  messages in flight per ring edge (1..8; slices of more
 *                 than 256 elements always use at least 2, because a rank
 *                 frees the slot it streams from only after its own send).
 *  stage_depth    input slices each rank stages ahead with bulk copies (1..16).
 *  slice_groups   elements per ring message in units of 256 (1, 2, 4 or 8;
 *                 the sparse codec uses 1, 2 or 4).
 * Depths and widths that do not fit the shared memory are reduced
 * automatically.  Errors: RRA_ERR_INVALID for NULL or values out of range.
 */
rra_status rra_comm_set_tuning(rra_comm *comm, int blocks_per_sm, int mailbox_depth,
                               int stage_depth, int slice_groups);

/* The launch shape of the last ring call (rra_ring_allreduce,
 * rra_reduce_scatter, rra_allreduce_auto's ring leg): resident blocks per SM,
 * mailbox slots per ring edge, staging depth, 256-element groups per slice.
 * Errors: RRA_ERR_INVALID for NULL arguments. */
rra_status rra_comm_last_shape(rra_comm *comm, int *blocks_per_sm, int *mailbox_depth,
                               int *stage_depth, int *slice_groups);

/*
 * Measured launch-shape tuning of the ring allreduce (the pages' pipeline
 * chunk size, CCCL §2.2 and §3.3, which suggest 1-4 MB pieces and leave the
 * choice to the workload).  Runs the allreduce described by the arguments
 * (same meaning as rra_ring_allreduce) once per candidate shape -- slice
 * widths 8, 4, 2, 1 x 256 elements, staging depths 1-4, 2-4 or all
 * resident blocks per SM -- times each on `stream` with CUDA events, and
 * remembers the fastest for this communicator and this call's (codec, input
 * kind, output dtype, alignment, count).  Later ring allreduce calls with
 * the same key use it, unless rra_comm_set_tuning set a manual shape.  The
 * final call runs with the chosen shape, so `out` holds its result on
 * return.  Results are bit-identical for every shape; only time differs.
 * Synchronous: it waits on events, so it must not be called while `stream`
 * is being captured (RRA_ERR_INVALID).  Errors: as rra_ring_allreduce;
 * a device time-out in any candidate is returned and nothing is stored.
 */
rra_status rra_autotune(rra_comm *comm, const void *const *in, void *const *out, size_t count,
                        rra_dtype in_t, rra_dtype out_t, const rra_codec *codec, void *stream);

/* Size-based choice between ring and tree ([ring] section "真实世界中的生产模式":
 * pick ring or tree by message size, from measurement; section "练习": add
 * the tree variant, switch by size and measure the crossover).  The default
 * crossover follows the measurement on GB300 (lossless fp32 in place, 1 KiB
 * to 1 GiB per rank): for N = 2 and 4 the ring is never slower from 256 MiB
 * per rank on (RRA_DEFAULT_CROSSOVER); for N = 8 and 64 the tree was the
 * faster at every measured size, and for N = 16 the ring led by 2 % from 256
 * MiB per rank, so from N = 5 on the default sends every message up to 1 GiB
 * per rank to the tree (RRA_DEFAULT_CROSSOVER_WIDE, one byte above the
 * largest size measured). */
#define RRA_DEFAULT_CROSSOVER (256ull << 20)
#define RRA_DEFAULT_CROSSOVER_WIDE ((1ull << 30) + 1)
#define RRA_ALGO_RING 0
#define RRA_ALGO_TREE 1

/* In-place allreduce of buf[r][0..count) that runs rra_tree_allreduce when
 * count * sizeof(dtype) is below the communicator's crossover and dtype is
 * fp32 (the tree sums fp32 only), otherwise the lossless rra_ring_allreduce
 * in place.  The two algorithms add in different orders, so their results
 * may differ in the last bits; *algorithm (if not NULL) reports which ran
 * (RRA_ALGO_RING / RRA_ALGO_TREE).  Errors: as the chosen operation. */
rra_status rra_allreduce_auto(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                              void *stream, int *algorithm);

/* Crossover of rra_allreduce_auto in bytes per rank (0 restores the
 * default: RRA_DEFAULT_CROSSOVER for N <= 4, RRA_DEFAULT_CROSSOVER_WIDE
 * otherwise).  Errors: RRA_ERR_INVALID for NULL. */
rra_status rra_set_crossover(rra_comm *comm, size_t bytes_per_rank);
rra_status rra_get_crossover(rra_comm *comm, size_t *bytes_per_rank);

/* Measure the crossover on this GPU: times the in-place ring and tree
 * allreduce of buf at 256 * 4^k fp32 elements per rank (k = 0, 1, ..., up
 * to count) and sets the communicator's crossover to the smallest measured
 * size from which on the ring is never slower (one byte above the largest
 * size if the tree always wins).  buf's contents are overwritten.  fp32
 * only.  Synchronous; not during a stream capture (RRA_ERR_INVALID).  The
 * result is also stored in *bytes_per_rank if not NULL. */
rra_status rra_autotune_crossover(rra_comm *comm, void *const *buf, size_t count,
                                  rra_dtype dtype, void *stream, size_t *bytes_per_rank);

/*
 * Adaptive codec choice ([cccl] §5, future directions: watch the gradients'
 * statistics -- sparsity, value distribution -- and switch the compression
 * to match, instead of one static threshold).
 *
 * Statistics of the N input buffers in[r][0..count): every ring chunk of
 * every buffer is cut into 128-element blocks from its start, as the ring's
 * first hop encodes them.
 *  elements      N * count.
 *  nonzero       elements whose fp32 value is not +0.0 (-0.0 counts).
 *  bfp4_flushed  nonzero elements whose BFP4 code would be 0
 *                (|x| <= 2^(e-3), e the block exponent).
 *  bfp8_flushed  the same for BFP8 (|x| <= 2^(e-7)).
 */
typedef struct {
    uint64_t elements, nonzero, bfp4_flushed, bfp8_flushed;
} rra_codec_stats;

/* Measure the statistics (one read of every input on `stream`, then a
 * synchronous read-back: not inside a stream capture, RRA_ERR_INVALID).
 * Errors: RRA_ERR_INVALID (NULL, count 0 or above max_count, bad dtype),
 * RRA_ERR_CUDA. */
rra_status rra_codec_measure(rra_comm *comm, const void *const *in, size_t count,
                             rra_dtype dtype, rra_codec_stats *out, void *stream);

/* Measure, then fill *codec (every other field zero/NULL) by this rule:
 * RRA_CODEC_SPARSE with `sparsity_threshold` when the share of zero elements
 * exceeds it; else BFP4 when it flushes at most `max_flushed_fraction` of
 * the nonzero elements to code 0; else BFP8.  *stats (if not NULL) receives
 * the measurement.  Errors: RRA_ERR_INVALID for a threshold outside [0, 1) or
 * a fraction outside [0, 1]; otherwise as rra_codec_measure. */
rra_status rra_codec_advise(rra_comm *comm, const void *const *in, size_t count, rra_dtype dtype,
                            float sparsity_threshold, float max_flushed_fraction,
                            rra_codec *codec, rra_codec_stats *stats, void *stream);

/*
 * Operator-aware choice ([cccl] §2.1, third layer: the allreduce may
 * compress boldly, since the reduction averages the errors out; allgather
 * and broadcast carry parameters and whole tensors and take lossless or
 * higher-precision lossy compression, or none).  op: RRA_OP_ALLREDUCE,
 * RRA_OP_ALLGATHER or RRA_OP_BROADCAST; root: the broadcast root (ignored
 * otherwise).
 * rra_codec_measure_op measures what that operation encodes: the allreduce
 * every chunk of every buffer (as rra_codec_measure); the compressed
 * allgather chunk r of in[r] alone; the compressed broadcast in[root] alone,
 * blocks from its start.
 * rra_codec_advise_op: RRA_OP_ALLREDUCE is rra_codec_advise.  Otherwise,
 * RRA_CODEC_SPARSE for the allgather when the share of zero elements exceeds
 * `sparsity_threshold` (lossless); else, when `allow_lossy` is nonzero and
 * BFP8 flushes at most `max_flushed_fraction` of the nonzero elements to
 * code 0, BFP8; else RRA_CODEC_NONE.  BFP4 is never advised for these ops.
 * Errors: RRA_ERR_INVALID (an unknown op, a root outside 0..N-1 for the
 * broadcast, or as rra_codec_advise / rra_codec_measure), RRA_ERR_CUDA.
 */
#define RRA_OP_ALLREDUCE 0
#define RRA_OP_ALLGATHER 1
#define RRA_OP_BROADCAST 2
rra_status rra_codec_measure_op(rra_comm *comm, int op, int root, const void *const *in,
                                size_t count, rra_dtype dtype, rra_codec_stats *out, void *stream);
rra_status rra_codec_advise_op(rra_comm *comm, int op, int root, const void *const *in,
                               size_t count, rra_dtype dtype, float sparsity_threshold,
                               float max_flushed_fraction, int allow_lossy, rra_codec *codec,
                               rra_codec_stats *stats, void *stream);

/* Test-only fault injection: in the next collective call, simulated rank
 * "rank" does not publish the message it sends at ring step "step" (1-based,
 * counted over both passes; the compressed allgather sends first at step N,
 * the owner's), for the first slice each block handles, so its receiver's
 * wait runs out and the call ends with RRA_ERR_TIMEOUT.  In the broadcasts
 * and the tree, where a rank publishes each slice once for every rank that
 * reads it: the plain broadcast withholds the rank's publish when it has a
 * child at tree level "step" (1-based); the tree withholds a rank's reduced
 * partial at step = its sending level + 1 (the position of its lowest set
 * bit, plus one), and its broadcast publish at step = L + 1 + a level at
 * which it has a child (L = ceil(log2 N)); the compressed broadcast at any
 * step >= 1.  rank < 0 disables.  The setting applies to one call only. */
rra_status rra_debug_withhold(rra_comm *comm, int rank, int step);

/* Human-readable name of a status code (static string). */
const char *rra_status_string(rra_status s);

#ifdef __cplusplus
}
#endif
#endif /* RRA_H */

// rra_host.cu -- the C ABI declared in include/rra.h: argument checks, the
// communicator (device byte counters, status word, time limit, launch
// configuration), path selection (bulk-copy fast path vs generic path) and
// kernel launches.  No allocation happens on the collective paths.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <vector>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "rra.h"
#include "rra_device.cuh"
#include "rra_kernels.h"

namespace rra {
const void *ring_fn_none(int in_t, bool fast, int groups, int rmap);
const void *ring_fn_bfp8(int in_t, bool fast, int groups, int rmap);
const void *ring_fn_bfp4(int in_t, bool fast, int groups, int rmap);
const void *ring_fn_sparse(int in_t, bool fast, int groups, int rmap);
const void *ring_fn_sparse_chunk(int in_t, bool fast, int groups, int rmap);
const void *ring_fn_bfp8_ef(int in_t, bool fast, int groups, int rmap);
const void *ring_fn_bfp4_ef(int in_t, bool fast, int groups, int rmap);
} // namespace rra

using namespace rra;

struct rra_comm {
    int N = 0;
    int device = 0;
    size_t max_count = 0;
    unsigned long long *counters = nullptr; // [2 sets][sent N | recv N]
    unsigned *status = nullptr;
    uint64_t timeout_ns = 2000000000ull;
    int withhold_rank = -1;
    int withhold_step = 0;
    unsigned gen = 0;          // counter set of the next call = gen & 1
    int last_set = -1;         // counter set written by the last call
    cudaStream_t last_stream = nullptr;
    bool have_last = false;
    int smem_optin = 0;
    int smem_per_sm = 0;
    rra::Tune tune;      // manual tuning (rra_comm_set_tuning); zeros: automatic
    // measured best ring shapes (rra_autotune), by (op, codec, input kind,
    // output dtype, staged path, count)
    std::map<std::array<long long, 6>, rra::Tune> tuned;
    rra::Tune last{};      // shape of the last ring launch (blocks = blocks per SM)
    size_t crossover = 0;  // rra_allreduce_auto: tree below this many bytes per rank
    unsigned long long *stats = nullptr; // [4] codec statistics (inside `counters`)
    // per-chunk sparse codec: message nonzero counts, [N*N] accumulated by
    // the count pass, [N*N] its result, and its block ticket
    unsigned long long *sp_acc = nullptr, *sp_out = nullptr;
    unsigned *sp_ticket = nullptr;
    // per-chunk sparse codec: spill area for the pairs of a group beyond the
    // 128 a slot holds; no launch needs more than the slots of all resident
    // blocks, i.e. the shared memory of every SM
    unsigned char *sp_spill = nullptr;
    size_t sp_spill_bytes = 0;
    std::map<long long, int> occ; // (kernel key, smem) -> blocks per SM
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

bool valid_dtype(int t) { return t == RRA_F32 || t == RRA_F16 || t == RRA_BF16; }
size_t esize(int t) { return t == RRA_F32 ? 4 : 2; }
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    if (abytes == 0 || bbytes == 0)
        return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

rra_status check_device(const rra_comm *c)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RRA_ERR_CUDA;
    return dev == c->device ? RRA_OK : RRA_ERR_INVALID;
}

// Counters for this call; block 0 of the launch clears the other set so the
// next call starts from zero without a separate memset.
void counter_sets(rra_comm *c, unsigned long long **sent, unsigned long long **recv,
                  unsigned long long **zero)
{
    const int set = (int)(c->gen & 1u);
    *sent = c->counters + (size_t)set * 2 * c->N;
    *recv = *sent + c->N;
    *zero = c->counters + (size_t)(set ^ 1) * 2 * c->N;
    c->last_set = set;
    c->gen++;
}

// A launch that failed cleared nothing and counted nothing: step back to the
// previous call's set, so the next call still starts from a cleared set and
// rra_get_bytes still reports the last launched call.
void undo_counter_sets(rra_comm *c, int prev_set)
{
    c->gen--;
    c->last_set = prev_set;
}

void note_call(rra_comm *c, cudaStream_t st)
{
    c->last_stream = st;
    c->have_last = true;
    c->withhold_rank = -1; // fault injection applies to one call only
}

int warps_for(int N) { return std::min(N, kMaxWarps); }

// Largest dynamic shared memory already allowed for each kernel (per device),
// so the attribute is set once per kernel rather than on every launch.
std::mutex g_attr_mu;
std::map<std::pair<int, const void *>, int> g_attr_smem;

cudaError_t allow_smem(const void *fn, int smem)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    int &have = g_attr_smem[{dev, fn}];
    if (smem <= have)
        return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        have = smem;
    return e;
}

int grid_for(rra_comm *c, long long key, const void *fn, int warps, int smem, long long items,
             int blocks_cap = 0, int *per_sm = nullptr)
{
    const long long k = key * (1LL << 20) + smem;
    int occ = 0;
    auto it = c->occ.find(k);
    if (it != c->occ.end()) {
        occ = it->second;
    } else {
        // raise (never lower) the kernel's shared-memory limit before asking
        allow_smem(fn, smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, warps * 32, (size_t)smem) !=
                cudaSuccess ||
            occ < 1)
            occ = 1;
        c->occ[k] = occ;
    }
    if (blocks_cap)
        occ = std::min(occ, blocks_cap);
    if (per_sm)
        *per_sm = occ;
    long long g = (long long)num_sms() * occ;
    if (items < g)
        g = items;
    return (int)std::max(1LL, g);
}

const void *ring_fn(int codec, int in_t, bool fast, int groups, int rmap, bool ef)
{
    if (ef)
        return codec == kCodecBfp8 ? ring_fn_bfp8_ef(in_t, fast, groups, rmap)
               : codec == kCodecBfp4 ? ring_fn_bfp4_ef(in_t, fast, groups, rmap)
                                     : nullptr;
    if (codec == kCodecNone)
        return ring_fn_none(in_t, fast, groups, rmap);
    if (codec == kCodecSparse)
        return ring_fn_sparse(in_t, fast, groups, rmap);
    if (codec == kCodecSparseChunk)
        return ring_fn_sparse_chunk(in_t, fast, groups, rmap);
    if (codec == kCodecBfp8)
        return ring_fn_bfp8(in_t, fast, groups, rmap);
    return ring_fn_bfp4(in_t, fast, groups, rmap);
}

// Sparse group sub-message: a 16-byte header, fp32 values, then the indices
// of a sparse group.  A group goes sparse only with nnz < lim, so at most
// lim - 1 pairs; the dense form holds 256 values.
int sparse_icap(int lim) { return std::max(lim - 1, 0); }
int sparse_sub_bytes(int lim) { return align_up(16 + std::max(kTile * 4, 8 * sparse_icap(lim)), 16); }

// Bytes of one mailbox slot for a slice of 256 * groups elements.  The
// per-chunk sparse slot: 32 header bytes, then a 1024-byte region per group
// (256 fp32 values, or 128 (value, index) pairs; more pairs spill to global
// memory).
int slot_bytes_for(int codec, int groups, int sparse_lim)
{
    switch (codec) {
    case kCodecNone: return kTile * 4 * groups;
    case kCodecBfp8: return 16 + kTile * groups;
    case kCodecBfp4: return 16 + kTile / 2 * groups;
    case kCodecSparseChunk: return 32 + kTile * 4 * groups;
    default: return sparse_sub_bytes(sparse_lim) * groups;
    }
}

// Slice width (groups of 8 elements per lane) and staging depth: wider
// slices amortise each step's handshakes over more elements; the first
// candidate that leaves room for about 24 resident warps per SM wins (three
// blocks of up to 8 warps, two wider ones), else the first that fits at all.
struct LaunchShape {
    int groups, K, D, smem;
    bool fast;
};

bool pick_shape(rra_comm *c, const Tune &t, int N, long long n, int kc, int ies, bool diff,
                bool fast, int warps, int sparse_lim, LaunchShape *out)
{
    const int sms = num_sms();
    static const int kGD[][2] = {{8, 2}, {8, 1}, {4, 2}, {4, 1}, {2, 4},
                                 {2, 2}, {2, 1}, {1, 4}, {1, 2}, {1, 1}};
    // resident blocks to leave room for: about 24 warps per SM (three blocks
    // of up to 8 warps, two of 12 to 16)
    const int want = warps >= 12 ? 2 : 3;
    const bool sparse = kc == kCodecSparse || kc == kCodecSparseChunk;
    const int sparse_kind = kc == kCodecSparse ? 1 : kc == kCodecSparseChunk ? 2 : 0;
    // Lossless rings of 12 or more ranks (a launch-shape sweep at N = 12,
    // 16, 32 and 64 found this 5-19 % faster than the rule below at N = 16 to
    // 64 and as fast at N = 12): two slots per edge and one stage; as many
    // blocks as give 16 resident warps per SM (one block of 16 warps, two of
    // 12 to 15), then the widest slice that fits them and leaves every SM a
    // slice position.  BFP rings of more ranks than warps keep the rule
    // below: a variant of this one that also accepts one slice position per
    // two SMs was 9-30 % faster at 4 Mi elements per rank and N = 32 and 64,
    // but 7-8 % slower at N = 24 and at 16 Mi elements per rank, N = 32.
    const bool wide = kc == kCodecNone && warps >= 12;
    if (wide && fast && !t.G && !t.K && !t.D) {
        const int nb = warps >= 16 ? 1 : 2;
        for (int G : {8, 4, 2, 1}) {
            if (G > 1 && (n + (long long)kTile * G - 1) / ((long long)kTile * G) < sms)
                continue;
            const int slot = slot_bytes_for(kc, G, sparse_lim);
            const int stage = kTile * G * (diff ? 8 : ies);
            const Layout L = make_layout(N, 2, 1, slot, stage, warps, true, 0, false);
            if (nb * (L.total + 1024) <= c->smem_per_sm && L.total <= c->smem_optin) {
                *out = LaunchShape{G, 2, 1, L.total, true};
                return true;
            }
        }
    }
    // a requested slice width is tried first on its own; passes 2 and 3 are
    // the automatic choice
    for (int pass = t.G ? 0 : 2; pass < 4; ++pass) {
        for (const auto &gd : kGD) {
            const int G = gd[0];
            if (pass < 2 && G != t.G)
                continue;
            if (sparse && G > 4) // sparse slices of 1, 2 or 4 groups are instantiated
                continue;
            int D = t.D ? t.D : gd[1];
            // a short chunk is cut into narrower slices while a wider one
            // would leave SMs without a slice position to work on
            if (pass >= 2 && G > 1 && (n + (long long)kTile * G - 1) / ((long long)kTile * G) < sms)
                continue;
            if (!fast)
                D = 1;
            const int slot = slot_bytes_for(kc, G, sparse_lim);
            const int stage = kTile * G * (diff ? 8 : ies);
            // wider messages need two slots per ring edge: a rank frees the
            // slot it streams from only after its own send of the same step,
            // so with one slot every rank would wait for its successor
            for (int K = t.K ? t.K : 2; K >= (G == 1 ? 1 : 2); --K) {
                const Layout L =
                    make_layout(N, K, D, slot, stage, warps, fast, sparse_kind, kc == kCodecBfp8);
                const bool several = pass % 2 == 0; // leave room for `want` blocks per SM
                const int need = several ? want * (L.total + 1024) : L.total;
                const int have = several ? c->smem_per_sm : c->smem_optin;
                if (need <= have && L.total <= c->smem_optin) {
                    *out = LaunchShape{G, K, D, L.total, fast};
                    return true;
                }
            }
        }
    }
    return false;
}

// force: an explicit launch shape (autotuning); otherwise the manual tuning,
// else a measured shape for this call's key, else the automatic choice.
rra_status ring_common(rra_comm *comm, int mode, const void *const *in, void *const *out,
                       size_t count, rra_dtype in_t, rra_dtype out_t, const rra_codec *codec,
                       void *stream, const Tune *force = nullptr,
                       std::array<long long, 6> *key_out = nullptr)
{
    if (!comm || !in || !out || count == 0 || count > comm->max_count || !valid_dtype(in_t) ||
        !valid_dtype(out_t))
        return RRA_ERR_INVALID;
    rra_status s = check_device(comm);
    if (s != RRA_OK)
        return s;
    const int N = comm->N;
    rra_codec cd{};
    cd.kind = RRA_CODEC_NONE;
    if (codec)
        cd = *codec;
    int kc;
    if (cd.kind == RRA_CODEC_NONE)
        kc = kCodecNone;
    else if (cd.kind == RRA_CODEC_BFP) {
        if (cd.bits == 8)
            kc = kCodecBfp8;
        else if (cd.bits == 4)
            kc = kCodecBfp4;
        else
            return RRA_ERR_INVALID;
    } else if (cd.kind == RRA_CODEC_SPARSE) {
        if (!(cd.sparsity_threshold >= 0.0f && cd.sparsity_threshold < 1.0f))
            return RRA_ERR_INVALID;
        if (cd.sparse_granularity == RRA_SPARSE_PER_CHUNK)
            kc = kCodecSparseChunk;
        else if (cd.sparse_granularity == RRA_SPARSE_PER_SLICE)
            kc = kCodecSparse;
        else
            return RRA_ERR_INVALID;
    } else {
        return RRA_ERR_INVALID;
    }
    if (cd.diff_prev && in_t != RRA_F32)
        return RRA_ERR_INVALID;
    // error feedback: only a lossy codec has an error to carry
    const bool ef = cd.residual != nullptr;
    if (ef && kc != kCodecBfp8 && kc != kCodecBfp4)
        return RRA_ERR_UNSUPPORTED;
    // Region of out[r] the call writes: all of it for the allreduce and the
    // allgather, chunk r alone for the reduce-scatter (so its outputs may
    // share one buffer).
    const size_t oes = esize(out_t);
    const size_t nchunk = (count + N - 1) / N;
    auto region = [&](int r, const char **p, size_t *bytes) {
        const char *b = static_cast<const char *>(out[r]);
        if (mode != kModeReduceScatter) {
            *p = b;
            *bytes = count * oes;
            return;
        }
        size_t lo = std::min(count, (size_t)r * nchunk), hi = std::min(count, lo + nchunk);
        *p = b + lo * oes;
        *bytes = (hi - lo) * oes;
    };
    for (int r = 0; r < N; ++r) {
        if (!in[r] || !out[r] || (cd.diff_prev && !cd.diff_prev[r]))
            return RRA_ERR_INVALID;
        const char *pr;
        size_t br;
        region(r, &pr, &br);
        if (cd.diff_base && overlap(pr, br, cd.diff_base, count * 4))
            return RRA_ERR_INVALID;
        for (int q = 0; q < r; ++q) {
            const char *pq;
            size_t bq;
            region(q, &pq, &bq);
            if (overlap(pr, br, pq, bq))
                return RRA_ERR_INVALID;
        }
    }
    // residuals are read and written: they may share no byte with any
    // buffer of the call, nor with each other
    if (ef) {
        const size_t rb = count * 4, ib = count * esize(in_t);
        for (int r = 0; r < N; ++r) {
            const void *e = cd.residual[r];
            if (!e || (cd.diff_base && overlap(e, rb, cd.diff_base, rb)))
                return RRA_ERR_INVALID;
            for (int q = 0; q < N; ++q) {
                const char *pq;
                size_t bq;
                region(q, &pq, &bq);
                if (overlap(e, rb, pq, bq) || overlap(e, rb, in[q], ib) ||
                    (cd.diff_prev && overlap(e, rb, cd.diff_prev[q], rb)) ||
                    (q < r && overlap(e, rb, cd.residual[q], rb)))
                    return RRA_ERR_INVALID;
            }
        }
    }

    RingArgs a;
    std::memset(&a, 0, sizeof a);
    a.N = N;
    a.mode = mode;
    a.in_t = in_t;
    a.out_t = out_t;
    a.T = (long long)count;
    a.n = (a.T + N - 1) / N;
    a.tiles = (a.n + kTile - 1) / kTile;
    a.average = cd.average ? 1 : 0;
    a.has_prev = cd.diff_prev ? 1 : 0;
    a.base = cd.diff_base;
    a.one_minus_thr = 1.0 - (double)cd.sparsity_threshold;
    // the same test for a full slice as an integer limit: nnz < lim
    a.sp_full_lim = 0;
    while (a.sp_full_lim <= kTile && (double)a.sp_full_lim < a.one_minus_thr * (double)kTile)
        ++a.sp_full_lim;
    a.sp_icap = sparse_icap(a.sp_full_lim);
    a.sp_sub = sparse_sub_bytes(a.sp_full_lim);
    // per-chunk sparse messages index a chunk with int32
    if (kc == kCodecSparseChunk && a.n > 0x7fffffffLL)
        return RRA_ERR_UNSUPPORTED;
    a.sp_nnz = comm->sp_out;
    a.timeout_ns = comm->timeout_ns;
    a.status = comm->status;
    a.withhold_rank = comm->withhold_rank;
    a.withhold_step = comm->withhold_step;

    const size_t ies = esize(in_t);
    bool fast = (a.n * ies) % 16 == 0 && (a.T * ies) % 16 == 0;
    bool vec_out = (a.n * oes) % 16 == 0;
    for (int r = 0; r < N; ++r) {
        a.in[r] = in[r];
        a.out[r] = out[r];
        a.prev[r] = cd.diff_prev ? cd.diff_prev[r] : nullptr;
        fast = fast && al16(in[r]) && (!cd.diff_prev || al16(cd.diff_prev[r]));
        vec_out = vec_out && al16(out[r]);
    }
    a.vec_out = vec_out ? 1 : 0;
    a.vec_base = (cd.diff_base && al16(cd.diff_base) && (a.n * 4) % 16 == 0) ? 1 : 0;
    bool vec_resid = ef && (a.n * 4) % 16 == 0;
    for (int r = 0; ef && r < N; ++r) {
        a.resid[r] = cd.residual[r];
        vec_resid = vec_resid && al16(cd.residual[r]);
    }
    a.vec_resid = vec_resid ? 1 : 0;

    const int warps = warps_for(N);
    const int kin = cd.diff_prev ? kF32Diff : (int)in_t; // kernel input kind
    const std::array<long long, 6> tkey = {mode, kc + (ef ? 100 : 0), kin, (long long)out_t,
                                           fast ? 1 : 0, (long long)count};
    if (key_out)
        *key_out = tkey;
    Tune t = comm->tune;
    if (force) {
        t = *force;
    } else if (!t.any()) {
        const auto it = comm->tuned.find(tkey);
        if (it != comm->tuned.end())
            t = it->second;
    }
    LaunchShape sh;
    if (!pick_shape(comm, t, N, a.n, kc, (int)ies, cd.diff_prev != nullptr, fast, warps,
                    a.sp_full_lim, &sh)) {
        fast = false;
        if (!pick_shape(comm, t, N, a.n, kc, (int)ies, cd.diff_prev != nullptr, false, warps,
                        a.sp_full_lim, &sh))
            return RRA_ERR_UNSUPPORTED;
    }
    const int groups = sh.groups, smem = sh.smem;
    a.K = sh.K;
    a.D = sh.D;
    a.slot_bytes = slot_bytes_for(kc, groups, a.sp_full_lim);
    a.stage_bytes = kTile * groups * (cd.diff_prev ? 8 : (int)ies);
    a.sp_spill = comm->sp_spill;
    a.slots_off = make_layout(N, a.K, a.D, a.slot_bytes, a.stage_bytes, warps, fast,
                              kc == kCodecSparse ? 1 : kc == kCodecSparseChunk ? 2 : 0,
                              kc == kCodecBfp8)
                      .slots;
    a.tiles = (a.n + kTile * groups - 1) / (kTile * groups);
    // every warp plays exactly one rank when N fits the block
    const int rmap = warps != N ? kRanksShared : (warps <= 8 ? kRankPerWarp8 : kRankPerWarp16);
    const void *fn = ring_fn(kc, kin, fast, groups, rmap, ef);
    if (!fn)
        return RRA_ERR_UNSUPPORTED;
    const long long key = (ef ? 1000000 : 0) + 100000 + kc * 10000 + kin * 1000 +
                          (fast ? 100 : 0) + rmap * 10 + groups;
    int per_sm = 0;
    const int grid = grid_for(comm, key, fn, warps, smem, a.tiles, t.blocks, &per_sm);
    if (kc == kCodecSparseChunk &&
        (size_t)grid * N * a.K * (size_t)(a.slot_bytes - 32) > comm->sp_spill_bytes)
        return RRA_ERR_UNSUPPORTED; // cannot happen: the slots of all blocks fit the SMs
    comm->last = Tune{per_sm, a.K, a.D, groups};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (kc == kCodecSparseChunk) {
        // the count pass: the nonzero count of every message, so that each
        // chunk's format is decided before its first slice is sent
        SpCountArgs ca;
        std::memset(&ca, 0, sizeof ca);
        ca.N = N;
        ca.h_lo = mode == kModeAllgather ? N : 1;
        ca.h_hi = mode == kModeReduceScatter ? N - 1 : N;
        ca.T = a.T;
        ca.n = a.n;
        ca.acc = comm->sp_acc;
        ca.out = comm->sp_out;
        ca.ticket = comm->sp_ticket;
        for (int r = 0; r < N; ++r) {
            ca.in[r] = in[r];
            ca.prev[r] = a.prev[r];
        }
        bool vec = (a.n * (long long)ies) % 16 == 0;
        for (int r = 0; r < N; ++r)
            vec = vec && al16(in[r]) && (!cd.diff_prev || al16(cd.diff_prev[r]));
        if (ca.h_lo <= ca.h_hi && launch_sparse_chunk_count(ca, kin, vec, st) != cudaSuccess)
            return RRA_ERR_CUDA;
    }
    const int prev_set = comm->last_set;
    counter_sets(comm, &a.sent, &a.recv, &a.zero);
    if (launch_ring(fn, a, grid, warps, smem, st) != cudaSuccess) {
        undo_counter_sets(comm, prev_set);
        return RRA_ERR_CUDA;
    }
    note_call(comm, st);
    return RRA_OK;
}

// which: 0 allgather, 1 broadcast, 2 tree allreduce; bits 8 or 4: the
// broadcast carries the root's BFP codes (0: plain copies)
rra_status copy_common(rra_comm *comm, int which, void *const *buf, size_t count,
                       rra_dtype dtype, int root, void *stream, int bits = 0)
{
    if (!comm || !buf || count == 0 || count > comm->max_count || !valid_dtype(dtype))
        return RRA_ERR_INVALID;
    rra_status s = check_device(comm);
    if (s != RRA_OK)
        return s;
    const int N = comm->N;
    if (which == 1 && (root < 0 || root >= N))
        return RRA_ERR_INVALID;
    if (which == 2 && dtype != RRA_F32)
        return RRA_ERR_UNSUPPORTED;
    const size_t es = esize(dtype);
    for (int r = 0; r < N; ++r) {
        if (!buf[r])
            return RRA_ERR_INVALID;
        for (int q = 0; q < r; ++q)
            if (overlap(buf[r], count * es, buf[q], count * es))
                return RRA_ERR_INVALID;
    }
    CopyArgs a;
    std::memset(&a, 0, sizeof a);
    a.N = N;
    a.es = (int)es;
    a.root = root;
    a.T = (long long)count;
    a.n = (a.T + N - 1) / N;
    a.timeout_ns = comm->timeout_ns;
    a.status = comm->status;
    a.withhold_rank = comm->withhold_rank;
    a.withhold_step = comm->withhold_step;
    a.bits = bits;
    a.dt = (int)dtype;
    bool fast = (a.T * (long long)es) % 16 == 0 && (which != 0 || (a.n * (long long)es) % 16 == 0);
    for (int r = 0; r < N; ++r) {
        a.buf[r] = buf[r];
        fast = fast && al16(buf[r]);
    }
    const int warps = warps_for(N);
    const bool one = warps == N;
    // allgather: ring edges, every rank stages its chunk; broadcast: a slot
    // FIFO per rank (each edge copied by its receiver), the root stages; tree:
    // no slots, every rank stages (and accumulates in) its slice, which its
    // reduce parent and broadcast children read; a reduce-ready and a
    // broadcast-ready barrier per rank and stage
    const int edges = which == 2 ? 2 * N : N;
    const int stagers = which == 1 ? 1 : N;
    const long long range = which == 0 ? a.n : a.T; // elements per rank walked in slices
    const int sms = num_sms();
    // widest slice that leaves every SM work and room for three, two or one
    // blocks per SM; ring edges need two slots (a rank holds its slot while it
    // forwards), tree edges can make do with one
    int G = 0, smem = 0;
    static const int kG[] = {4, 2, 1};
    for (int pass = 0; pass < 3 && !G; ++pass) {
        const int per_sm = 3 - pass;
        for (int g : kG) {
            if (comm->tune.G && g != comm->tune.G)
                continue;
            if (!comm->tune.G && g > 1 && (range + (long long)kTile * g - 1) / ((long long)kTile * g) < sms)
                continue;
            const int bytes = kTile * g * (int)es;
            const int slot = which == 2 ? 0 : bits ? 16 + kTile * g * bits / 8 : bytes; // BFP: codes
            bool found = false;
            for (int K = comm->tune.K ? comm->tune.K : 2; K >= (which == 0 ? 2 : 1) && !found; --K)
                for (int D = fast ? (comm->tune.D ? comm->tune.D : (which == 2 ? 3 : 2)) : 1;
                     D >= 1 && !found; --D) {
                    // the tree's barrier FIFOs follow its stages
                    const int KK = which == 2 ? D : K;
                    const CollLayout L =
                        coll_layout(N, edges, KK, stagers, D, slot, bytes, fast || which == 2);
                    if (per_sm * (L.total + 1024) <= comm->smem_per_sm &&
                        L.total <= comm->smem_optin) {
                        G = g;
                        a.K = KK;
                        a.D = D;
                        smem = L.total;
                        found = true;
                    }
                }
            if (G)
                break;
        }
    }
    if (!G)
        return RRA_ERR_UNSUPPORTED;
    a.slot_bytes = a.stage_bytes = kTile * G * (int)es;
    if (bits)
        a.slot_bytes = 16 + kTile * G * bits / 8;
    if (which == 2)
        a.slot_bytes = 0;
    a.tiles = (range + (long long)kTile * G - 1) / ((long long)kTile * G);
    const void *fn = bits ? bcast_bfp_fn(bits, G, fast, one) : coll_fn(which, (int)es, G, fast, one);
    if (!fn)
        return RRA_ERR_UNSUPPORTED;
    const long long key = 50000 + bits * 10000 + which * 1000 + (int)es * 100 + G * 10 +
                          (fast ? 2 : 0) + (one ? 1 : 0);
    const int grid = grid_for(comm, key, fn, warps, smem, a.tiles, comm->tune.blocks);
    const int prev_set = comm->last_set;
    counter_sets(comm, &a.sent, &a.recv, &a.zero);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_coll(fn, a, grid, warps, smem, st) != cudaSuccess) {
        undo_counter_sets(comm, prev_set);
        return RRA_ERR_CUDA;
    }
    note_call(comm, st);
    return RRA_OK;
}

// Scratch of the standalone sparse encoder, one per (device, stream), grown
// on demand.  Encodes on different streams never share one, and the lock is
// held until the launches are queued, so no growth by another thread frees a
// buffer under a launch.
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, std::pair<uint32_t *, long long>> g_ws;

} // namespace

namespace rra {
cudaError_t launch_coll(const void *fn, const CopyArgs &a, int grid, int warps, int smem,
                        cudaStream_t st)
{
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess)
        return e;
    void *args[] = {const_cast<CopyArgs *>(&a)};
    return cudaLaunchKernel(fn, dim3(grid), dim3(warps * 32), args, (size_t)smem, st);
}

cudaError_t launch_ring(const void *fn, const RingArgs &a, int grid, int warps, int smem,
                        cudaStream_t st)
{
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess)
        return e;
    void *args[] = {const_cast<RingArgs *>(&a)};
    return cudaLaunchKernel(fn, dim3(grid), dim3(warps * 32), args, (size_t)smem, st);
}
} // namespace rra

extern "C" {

const char *rra_status_string(rra_status s)
{
    switch (s) {
    case RRA_OK: return "RRA_OK";
    case RRA_ERR_INVALID: return "RRA_ERR_INVALID";
    case RRA_ERR_UNSUPPORTED: return "RRA_ERR_UNSUPPORTED";
    case RRA_ERR_CUDA: return "RRA_ERR_CUDA";
    case RRA_ERR_TIMEOUT: return "RRA_ERR_TIMEOUT";
    case RRA_ERR_NOMEM: return "RRA_ERR_NOMEM";
    }
    return "RRA_ERR_UNKNOWN";
}

rra_status rra_comm_create(int nranks, size_t max_count, rra_dtype max_dtype, rra_comm **out)
{
    if (!out || nranks < 1 || nranks > RRA_MAX_RANKS || max_count == 0 || !valid_dtype(max_dtype))
        return RRA_ERR_INVALID;
    *out = nullptr;
    rra_comm *c = new rra_comm();
    c->N = nranks;
    c->max_count = max_count;
    if (cudaGetDevice(&c->device) != cudaSuccess) {
        delete c;
        return RRA_ERR_CUDA;
    }
    cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    cudaDeviceGetAttribute(&c->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, c->device);
    // two counter sets (sent and recv per rank), then 4 codec statistics
    const size_t cbytes = sizeof(unsigned long long) * (4 * (size_t)nranks + 4);
    if (cudaMalloc(&c->counters, cbytes) != cudaSuccess) {
        delete c;
        return RRA_ERR_NOMEM;
    }
    if (cudaMalloc(&c->status, sizeof(unsigned)) != cudaSuccess) {
        cudaFree(c->counters);
        delete c;
        return RRA_ERR_NOMEM;
    }
    c->stats = c->counters + 4 * (size_t)nranks;
    // per-chunk sparse message counts: accumulator, result, ticket
    const size_t nn = (size_t)nranks * (size_t)nranks;
    const size_t sbytes = sizeof(unsigned long long) * (2 * nn + 1);
    if (cudaMalloc(&c->sp_acc, sbytes) != cudaSuccess) {
        cudaFree(c->counters);
        cudaFree(c->status);
        delete c;
        return RRA_ERR_NOMEM;
    }
    c->sp_out = c->sp_acc + nn;
    c->sp_ticket = reinterpret_cast<unsigned *>(c->sp_out + nn);
    c->sp_spill_bytes = (size_t)num_sms() * (size_t)c->smem_per_sm;
    if (cudaMalloc(&c->sp_spill, c->sp_spill_bytes) != cudaSuccess) {
        cudaFree(c->counters);
        cudaFree(c->status);
        cudaFree(c->sp_acc);
        delete c;
        return RRA_ERR_NOMEM;
    }
    if (cudaMemset(c->sp_acc, 0, sbytes) != cudaSuccess ||
        cudaMemset(c->counters, 0, cbytes) != cudaSuccess ||
        cudaMemset(c->status, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(c->counters);
        cudaFree(c->status);
        cudaFree(c->sp_acc);
        cudaFree(c->sp_spill);
        delete c;
        return RRA_ERR_CUDA;
    }
    *out = c;
    return RRA_OK;
}

rra_status rra_comm_destroy(rra_comm *comm)
{
    if (!comm)
        return RRA_OK;
    cudaDeviceSynchronize();
    cudaFree(comm->counters);
    cudaFree(comm->status);
    cudaFree(comm->sp_acc);
    cudaFree(comm->sp_spill);
    delete comm;
    return RRA_OK;
}

rra_status rra_ring_allreduce(rra_comm *comm, const void *const *in, void *const *out,
                              size_t count, rra_dtype in_t, rra_dtype out_t,
                              const rra_codec *codec, void *stream)
{
    return ring_common(comm, kModeAllreduce, in, out, count, in_t, out_t, codec, stream);
}

rra_status rra_reduce_scatter(rra_comm *comm, const void *const *in, void *const *out,
                              size_t count, rra_dtype in_t, rra_dtype out_t,
                              const rra_codec *codec, void *stream)
{
    return ring_common(comm, kModeReduceScatter, in, out, count, in_t, out_t, codec, stream);
}

rra_status rra_allgather(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                         void *stream)
{
    return copy_common(comm, 0, buf, count, dtype, 0, stream);
}

rra_status rra_allgather_codec(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                               const rra_codec *codec, void *stream)
{
    if (!codec || codec->kind == RRA_CODEC_NONE) {
        if (codec && (codec->diff_prev || codec->diff_base || codec->average || codec->residual))
            return RRA_ERR_INVALID;
        return rra_allgather(comm, buf, count, dtype, stream);
    }
    // the allgather moves each owner's own elements: no difference stream,
    // base, averaging or residual applies
    if (codec->diff_prev || codec->diff_base || codec->average || codec->residual)
        return RRA_ERR_INVALID;
    return ring_common(comm, kModeAllgather, reinterpret_cast<const void *const *>(buf), buf,
                       count, dtype, dtype, codec, stream);
}

rra_status rra_broadcast(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                         int root, void *stream)
{
    return copy_common(comm, 1, buf, count, dtype, root, stream);
}

rra_status rra_broadcast_codec(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                               int root, const rra_codec *codec, void *stream)
{
    if (codec && (codec->diff_prev || codec->diff_base || codec->average || codec->residual))
        return RRA_ERR_INVALID;
    if (!codec || codec->kind == RRA_CODEC_NONE)
        return rra_broadcast(comm, buf, count, dtype, root, stream);
    if (codec->kind == RRA_CODEC_SPARSE)
        return RRA_ERR_UNSUPPORTED;
    if (codec->kind != RRA_CODEC_BFP || (codec->bits != 8 && codec->bits != 4))
        return RRA_ERR_INVALID;
    return copy_common(comm, 1, buf, count, dtype, root, stream, codec->bits);
}

rra_status rra_tree_allreduce(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                              void *stream)
{
    return copy_common(comm, 2, buf, count, dtype, 0, stream);
}

rra_status rra_bfp_encode(const void *x, size_t n, rra_dtype dtype, int bits, int8_t *exps,
                          uint8_t *mants, void *stream)
{
    if (!x || n == 0 || !exps || !mants || !valid_dtype(dtype) || (bits != 8 && bits != 4))
        return RRA_ERR_INVALID;
    return launch_bfp_encode(x, (long long)n, dtype, bits, exps, mants,
                             reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RRA_OK
               : RRA_ERR_CUDA;
}

rra_status rra_bfp_decode(const int8_t *exps, const uint8_t *mants, size_t n, int bits,
                          float *out, int accumulate, void *stream)
{
    if (!exps || !mants || !out || n == 0 || (bits != 8 && bits != 4))
        return RRA_ERR_INVALID;
    return launch_bfp_decode(exps, mants, (long long)n, bits, out, accumulate,
                             reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RRA_OK
               : RRA_ERR_CUDA;
}

rra_status rra_sparse_encode(const void *x, size_t n, rra_dtype dtype, float threshold,
                             uint32_t *hdr, void *vals, int32_t *idx, void *stream)
{
    if (!x || n == 0 || !hdr || !vals || !idx || !valid_dtype(dtype) ||
        !(threshold >= 0.0f && threshold < 1.0f) || n > 0x7fffffffull)
        return RRA_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RRA_ERR_CUDA;
    const long long words = sparse_encode_scratch_words((long long)n);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto &ws = g_ws[{dev, st}];
    if (ws.second < words) {
        if (ws.first) {
            cudaDeviceSynchronize(); // an encode in flight may still use it
            cudaFree(ws.first);
            ws.first = nullptr;
            ws.second = 0;
        }
        long long want = std::max(words, 1LL << 16);
        if (cudaMalloc(&ws.first, (size_t)want * sizeof(uint32_t)) != cudaSuccess) {
            ws.first = nullptr;
            return RRA_ERR_NOMEM;
        }
        ws.second = want;
    }
    return launch_sparse_encode(x, (long long)n, dtype, 1.0 - (double)threshold, hdr, vals, idx,
                                ws.first, st) == cudaSuccess
               ? RRA_OK
               : RRA_ERR_CUDA;
}

rra_status rra_sparse_decode(const uint32_t *hdr, const void *vals, const int32_t *idx,
                             size_t n, rra_dtype dtype, float *acc, int accumulate,
                             void *stream)
{
    if (!hdr || !vals || !idx || !acc || n == 0 || !valid_dtype(dtype))
        return RRA_ERR_INVALID;
    return launch_sparse_decode(hdr, vals, idx, (long long)n, dtype, acc, accumulate,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RRA_OK
               : RRA_ERR_CUDA;
}

rra_status rra_diff_encode(const float *cur, const float *prev, float *diff, size_t n,
                           void *stream)
{
    if (!cur || !prev || !diff || n == 0)
        return RRA_ERR_INVALID;
    return launch_diff_encode(cur, prev, diff, (long long)n,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RRA_OK
               : RRA_ERR_CUDA;
}

rra_status rra_get_bytes(rra_comm *comm, uint64_t *sent, uint64_t *recv)
{
    if (!comm || !sent || !recv)
        return RRA_ERR_INVALID;
    const int N = comm->N;
    if (!comm->have_last) {
        std::fill(sent, sent + N, 0);
        std::fill(recv, recv + N, 0);
        return RRA_OK;
    }
    if (cudaStreamSynchronize(comm->last_stream) != cudaSuccess)
        return RRA_ERR_CUDA;
    const unsigned long long *src = comm->counters + (size_t)comm->last_set * 2 * N;
    if (cudaMemcpy(sent, src, sizeof(uint64_t) * N, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(recv, src + N, sizeof(uint64_t) * N, cudaMemcpyDeviceToHost) != cudaSuccess)
        return RRA_ERR_CUDA;
    unsigned st = 0;
    if (cudaMemcpy(&st, comm->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess)
        return RRA_ERR_CUDA;
    return st ? (rra_status)st : RRA_OK;
}

rra_status rra_comm_status(rra_comm *comm)
{
    if (!comm)
        return RRA_ERR_INVALID;
    if (comm->have_last && cudaStreamSynchronize(comm->last_stream) != cudaSuccess)
        return RRA_ERR_CUDA;
    unsigned st = 0;
    if (cudaMemcpy(&st, comm->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess)
        return RRA_ERR_CUDA;
    if (st && cudaMemset(comm->status, 0, sizeof(unsigned)) != cudaSuccess)
        return RRA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return RRA_ERR_CUDA;
    return st ? (rra_status)st : RRA_OK;
}

rra_status rra_set_timeout(rra_comm *comm, uint64_t ns)
{
    if (!comm)
        return RRA_ERR_INVALID;
    comm->timeout_ns = ns ? ns : kDefaultTimeoutNs;
    return RRA_OK;
}

rra_status rra_comm_set_tuning(rra_comm *comm, int blocks_per_sm, int mailbox_depth,
                               int stage_depth, int slice_groups)
{
    if (!comm || blocks_per_sm < 0 || blocks_per_sm > 32 || mailbox_depth < 0 ||
        mailbox_depth > 8 || stage_depth < 0 || stage_depth > 16 ||
        !(slice_groups == 0 || slice_groups == 1 || slice_groups == 2 || slice_groups == 4 ||
          slice_groups == 8))
        return RRA_ERR_INVALID;
    comm->tune.blocks = blocks_per_sm;
    comm->tune.K = mailbox_depth;
    comm->tune.D = stage_depth;
    comm->tune.G = slice_groups;
    return RRA_OK;
}

rra_status rra_debug_withhold(rra_comm *comm, int rank, int step)
{
    if (!comm || rank >= comm->N)
        return RRA_ERR_INVALID;
    comm->withhold_rank = rank < 0 ? -1 : rank;
    comm->withhold_step = step;
    return RRA_OK;
}

rra_status rra_comm_last_shape(rra_comm *comm, int *blocks_per_sm, int *mailbox_depth,
                               int *stage_depth, int *slice_groups)
{
    if (!comm || !blocks_per_sm || !mailbox_depth || !stage_depth || !slice_groups)
        return RRA_ERR_INVALID;
    *blocks_per_sm = comm->last.blocks;
    *mailbox_depth = comm->last.K;
    *stage_depth = comm->last.D;
    *slice_groups = comm->last.G;
    return RRA_OK;
}

rra_status rra_autotune(rra_comm *comm, const void *const *in, void *const *out, size_t count,
                        rra_dtype in_t, rra_dtype out_t, const rra_codec *codec, void *stream)
{
    if (!comm)
        return RRA_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess)
        return RRA_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone)
        return RRA_ERR_INVALID; // it waits on events: not inside a capture
    // the automatic shape first: checks the arguments, warms up, gives the key
    std::array<long long, 6> key{};
    const Tune autoshape{};
    rra_status s = ring_common(comm, kModeAllreduce, in, out, count, in_t, out_t, codec, stream,
                               &autoshape, &key);
    if (s != RRA_OK)
        return s;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0)
            cudaEventDestroy(e0);
        return RRA_ERR_CUDA;
    }
    // best of a few calls of one shape (fewer for long calls)
    auto time_shape = [&](const Tune &t, float *best_ms) -> rra_status {
        *best_ms = 1e30f;
        for (int rep = 0; rep < 4; ++rep) {
            if (cudaEventRecord(e0, st) != cudaSuccess)
                return RRA_ERR_CUDA;
            const rra_status r =
                ring_common(comm, kModeAllreduce, in, out, count, in_t, out_t, codec, stream, &t);
            if (r != RRA_OK)
                return r;
            float ms = 0.0f;
            if (cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
                return RRA_ERR_CUDA;
            if (rep > 0) // the first call of a shape warms it up
                *best_ms = std::min(*best_ms, ms);
            if (rep >= 2 && ms > 2.0f)
                break;
        }
        return RRA_OK;
    };
    Tune best{};
    float best_ms = 1e30f;
    std::vector<std::array<int, 4>> seen;
    static const int kG[] = {8, 4, 2, 1}, kD[] = {1, 2, 3, 4}, kB[] = {0, 2, 3, 4};
    for (int G : kG)
        for (int D : kD)
            for (int B : kB) {
                if (s != RRA_OK)
                    break;
                const Tune cand{B, 0, D, G};
                float ms = 0.0f;
                s = time_shape(cand, &ms);
                if (s == RRA_ERR_UNSUPPORTED) { // this shape does not fit: skip it
                    s = RRA_OK;
                    continue;
                }
                if (s != RRA_OK)
                    break;
                // different requests can land on the same launch shape
                const std::array<int, 4> got = {comm->last.blocks, comm->last.K, comm->last.D,
                                                comm->last.G};
                if (std::find(seen.begin(), seen.end(), got) != seen.end())
                    continue;
                seen.push_back(got);
                if (ms < best_ms) {
                    best_ms = ms;
                    best = Tune{got[0], got[1], got[2], got[3]};
                }
            }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (s != RRA_OK)
        return s;
    // a candidate that timed out latches the status word: report it, keep nothing
    s = rra_comm_status(comm);
    if (s != RRA_OK)
        return s;
    comm->tuned[key] = best;
    // leave the outputs of a call with the chosen shape
    return ring_common(comm, kModeAllreduce, in, out, count, in_t, out_t, codec, stream);
}

rra_status rra_set_crossover(rra_comm *comm, size_t bytes_per_rank)
{
    if (!comm)
        return RRA_ERR_INVALID;
    comm->crossover = bytes_per_rank;
    return RRA_OK;
}

namespace {
// The communicator's crossover: the one set or measured, else the default
// for its rank count.
size_t crossover_of(const rra_comm *comm)
{
    if (comm->crossover)
        return comm->crossover;
    return comm->N <= 4 ? (size_t)RRA_DEFAULT_CROSSOVER : (size_t)RRA_DEFAULT_CROSSOVER_WIDE;
}
} // namespace

rra_status rra_get_crossover(rra_comm *comm, size_t *bytes_per_rank)
{
    if (!comm || !bytes_per_rank)
        return RRA_ERR_INVALID;
    *bytes_per_rank = crossover_of(comm);
    return RRA_OK;
}

rra_status rra_allreduce_auto(rra_comm *comm, void *const *buf, size_t count, rra_dtype dtype,
                              void *stream, int *algorithm)
{
    if (!comm || !buf || !valid_dtype(dtype))
        return RRA_ERR_INVALID;
    const size_t cross = crossover_of(comm);
    // the tree sums fp32 only; other dtypes always take the ring
    const bool tree = dtype == RRA_F32 && count * esize(dtype) < cross;
    if (algorithm)
        *algorithm = tree ? RRA_ALGO_TREE : RRA_ALGO_RING;
    if (tree)
        return copy_common(comm, 2, buf, count, dtype, 0, stream);
    return ring_common(comm, kModeAllreduce, reinterpret_cast<const void *const *>(buf), buf,
                       count, dtype, dtype, nullptr, stream);
}

rra_status rra_autotune_crossover(rra_comm *comm, void *const *buf, size_t count,
                                  rra_dtype dtype, void *stream, size_t *bytes_per_rank)
{
    if (!comm || !buf || dtype != RRA_F32 || count == 0 || count > comm->max_count)
        return RRA_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess)
        return RRA_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone)
        return RRA_ERR_INVALID;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0)
            cudaEventDestroy(e0);
        return RRA_ERR_CUDA;
    }
    rra_status s = RRA_OK;
    auto time_op = [&](bool tree, size_t n, float *best_ms) -> rra_status {
        *best_ms = 1e30f;
        for (int rep = 0; rep < 4; ++rep) {
            if (cudaEventRecord(e0, st) != cudaSuccess)
                return RRA_ERR_CUDA;
            const rra_status r =
                tree ? copy_common(comm, 2, buf, n, dtype, 0, stream)
                     : ring_common(comm, kModeAllreduce, reinterpret_cast<const void *const *>(buf),
                                   buf, n, dtype, dtype, nullptr, stream);
            if (r != RRA_OK)
                return r;
            float ms = 0.0f;
            if (cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
                return RRA_ERR_CUDA;
            if (rep > 0)
                *best_ms = std::min(*best_ms, ms);
        }
        return RRA_OK;
    };
    // sizes 1 KiB * 4^k per rank up to count: the crossover is the smallest
    // measured size from which on the ring is never slower than the tree
    std::vector<std::pair<size_t, bool>> ring_wins;
    for (size_t n = 256; s == RRA_OK; n = n * 4 > count && n < count ? count : n * 4) {
        float tr = 0.0f, tt = 0.0f;
        s = time_op(false, n, &tr);
        if (s == RRA_OK)
            s = time_op(true, n, &tt);
        if (s == RRA_OK)
            ring_wins.push_back({n * 4, tr <= tt});
        if (n >= count)
            break;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (s == RRA_OK)
        s = rra_comm_status(comm);
    if (s != RRA_OK)
        return s;
    size_t cross = ring_wins.back().second ? ring_wins.back().first : ring_wins.back().first + 1;
    for (size_t i = ring_wins.size(); i-- > 0;) {
        if (!ring_wins[i].second)
            break;
        cross = ring_wins[i].first;
    }
    comm->crossover = cross;
    if (bytes_per_rank)
        *bytes_per_rank = cross;
    return RRA_OK;
}

rra_status rra_codec_measure_op(rra_comm *comm, int op, int root, const void *const *in,
                                size_t count, rra_dtype dtype, rra_codec_stats *out, void *stream)
{
    if (!comm || !in || !out || count == 0 || count > comm->max_count || !valid_dtype(dtype) ||
        op < RRA_OP_ALLREDUCE || op > RRA_OP_BROADCAST ||
        (op == RRA_OP_BROADCAST && (root < 0 || root >= comm->N)))
        return RRA_ERR_INVALID;
    rra_status s = check_device(comm);
    if (s != RRA_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess)
        return RRA_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone)
        return RRA_ERR_INVALID; // it reads the result back on the host
    for (int r = 0; r < comm->N; ++r)
        if (!in[r])
            return RRA_ERR_INVALID;
    const int N = comm->N;
    const long long T = (long long)count, n = (T + N - 1) / N;
    const size_t es = esize(dtype);
    unsigned long long h[4];
    if (cudaMemsetAsync(comm->stats, 0, sizeof h, st) != cudaSuccess)
        return RRA_ERR_CUDA;
    // the statistics kernel counts every chunk of every buffer it is given;
    // the allgather's owner chunks and the broadcast's root buffer are each
    // given as a one-buffer, one-chunk problem
    auto run = [&](int nb, long long t, const void *const *bufs) -> bool {
        StatsArgs a;
        std::memset(&a, 0, sizeof a);
        a.N = nb;
        a.T = t;
        a.n = (t + nb - 1) / nb;
        a.stats = comm->stats;
        for (int r = 0; r < nb; ++r)
            a.in[r] = bufs[r];
        return launch_codec_stats(a, dtype, st) == cudaSuccess;
    };
    bool ok = true;
    if (op == RRA_OP_ALLREDUCE) {
        ok = run(N, T, in);
    } else if (op == RRA_OP_BROADCAST) {
        ok = run(1, T, in + root);
    } else {
        for (int r = 0; r < N && ok; ++r) {
            const long long lo = std::min(T, r * n), hi = std::min(T, lo + n);
            if (hi > lo) {
                const void *p = static_cast<const char *>(in[r]) + lo * (long long)es;
                ok = run(1, hi - lo, &p);
            }
        }
    }
    if (!ok ||
        cudaMemcpyAsync(h, comm->stats, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return RRA_ERR_CUDA;
    out->elements = h[0];
    out->nonzero = h[1];
    out->bfp4_flushed = h[2];
    out->bfp8_flushed = h[3];
    return RRA_OK;
}

rra_status rra_codec_measure(rra_comm *comm, const void *const *in, size_t count,
                             rra_dtype dtype, rra_codec_stats *out, void *stream)
{
    return rra_codec_measure_op(comm, RRA_OP_ALLREDUCE, 0, in, count, dtype, out, stream);
}

rra_status rra_codec_advise(rra_comm *comm, const void *const *in, size_t count, rra_dtype dtype,
                            float sparsity_threshold, float max_flushed_fraction,
                            rra_codec *codec, rra_codec_stats *stats, void *stream)
{
    if (!codec || !(sparsity_threshold >= 0.0f && sparsity_threshold < 1.0f) ||
        !(max_flushed_fraction >= 0.0f && max_flushed_fraction <= 1.0f))
        return RRA_ERR_INVALID;
    rra_codec_stats st{};
    const rra_status s = rra_codec_measure(comm, in, count, dtype, &st, stream);
    if (s != RRA_OK)
        return s;
    if (stats)
        *stats = st;
    std::memset(codec, 0, sizeof *codec);
    codec->sparsity_threshold = sparsity_threshold;
    // sparse when the zeros exceed the threshold (the sparse codec still
    // decides per group); else the narrowest BFP that flushes at most the
    // allowed share of the nonzero values to code 0
    const double zeros = (double)(st.elements - st.nonzero);
    if (st.elements && zeros > (double)sparsity_threshold * (double)st.elements) {
        codec->kind = RRA_CODEC_SPARSE;
        codec->bits = 8;
    } else if ((double)st.bfp4_flushed <= (double)max_flushed_fraction * (double)st.nonzero) {
        codec->kind = RRA_CODEC_BFP;
        codec->bits = 4;
    } else {
        codec->kind = RRA_CODEC_BFP;
        codec->bits = 8;
    }
    return RRA_OK;
}

rra_status rra_codec_advise_op(rra_comm *comm, int op, int root, const void *const *in,
                               size_t count, rra_dtype dtype, float sparsity_threshold,
                               float max_flushed_fraction, int allow_lossy, rra_codec *codec,
                               rra_codec_stats *stats, void *stream)
{
    if (op == RRA_OP_ALLREDUCE)
        return rra_codec_advise(comm, in, count, dtype, sparsity_threshold,
                                max_flushed_fraction, codec, stats, stream);
    if (!codec || !(sparsity_threshold >= 0.0f && sparsity_threshold < 1.0f) ||
        !(max_flushed_fraction >= 0.0f && max_flushed_fraction <= 1.0f))
        return RRA_ERR_INVALID;
    rra_codec_stats st{};
    const rra_status s =
        rra_codec_measure_op(comm, op, root, in, count, dtype, &st, stream);
    if (s != RRA_OK)
        return s;
    if (stats)
        *stats = st;
    std::memset(codec, 0, sizeof *codec);
    codec->sparsity_threshold = sparsity_threshold;
    codec->kind = RRA_CODEC_NONE;
    // conservative: lossless sparse codes first (allgather only), then the
    // higher-precision lossy width, and only when it is allowed and flushes
    // at most the given share of the nonzero values; else no compression
    const double zeros = (double)(st.elements - st.nonzero);
    if (op == RRA_OP_ALLGATHER && st.elements &&
        zeros > (double)sparsity_threshold * (double)st.elements) {
        codec->kind = RRA_CODEC_SPARSE;
        codec->bits = 8;
    } else if (allow_lossy &&
               (double)st.bfp8_flushed <= (double)max_flushed_fraction * (double)st.nonzero) {
        codec->kind = RRA_CODEC_BFP;
        codec->bits = 8;
    }
    return RRA_OK;
}

} // extern "C"

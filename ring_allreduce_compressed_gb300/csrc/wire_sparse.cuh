// wire_sparse.cuh -- the sparse values + indices wire formats of the fused
// ring ("CCCL通信压缩库" §2.1: above a sparsity threshold send only the
// nonzero values and their indices; the receiver puts the values back at
// their indices).  Included by ring_sparse.cu only, after ring_kernel.cuh.
//
// Both formats share the receiver's side (§2.2: receive, decompress, then
// reduce): a received group is restored into its dense form -- the listed
// values at their indices, +0.0 everywhere else -- and the whole restored
// group is added to the receiver's partial.  A group in registers is
// therefore just its 8 restored values per lane.  Forwarding re-emits the
// identical message from them: a sparse message lists exactly the values
// whose fp32 bits are not +0.0, and those are exactly the restored values
// with nonzero bits.
#pragma once

#include "ring_kernel.cuh"

namespace rra {

struct SparseWarp {
    // inclusive prefix sum of cnt over the lanes of the warp
    __device__ __forceinline__ static int incl_scan(int lane, int cnt)
    {
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += t;
        }
        return incl;
    }
    // bit i set where element 8*lane + i (< len) has fp32 bits other than +0.0
    __device__ __forceinline__ static uint32_t nonzero_mask(const float (&v)[8], int lane,
                                                            int len)
    {
        uint32_t nzm = 0;
        if (len >= kTile) { // a full group: every lane's 8 positions are inside it
#pragma unroll
            for (int i = 0; i < 8; ++i)
                nzm |= (__float_as_uint(v[i]) != 0u ? 1u : 0u) << i;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (8 * lane + i < len && __float_as_uint(v[i]) != 0u)
                    nzm |= 1u << i;
        }
        return nzm;
    }
    // lane's values at the positions of nzm into vals[pos..] and their
    // indices ix0 + 8*lane + i into idx[pos..], pos = the lane's exclusive
    // prefix (ascending order across the warp)
    __device__ __forceinline__ static void write_pairs(float *vals, int *idx, int pos, int lane,
                                                       int ix0, const float (&v)[8], uint32_t nzm)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if ((nzm >> i) & 1u) {
                vals[pos] = v[i];
                idx[pos] = ix0 + 8 * lane + i;
                ++pos;
            }
    }
    // Decompress cnt (value, index) pairs of one 256-element group whose
    // first element has index ix0 into the warp's scratch (zeros, then the
    // values at their indices) and read the lane's 8 restored values back.
    // Warp-collective.
    __device__ __forceinline__ static void restore(const float *vals, const int *idx, int cnt,
                                                   int ix0, int lane, unsigned char *scratch,
                                                   float (&f)[8])
    {
        float *sval = reinterpret_cast<float *>(scratch);
        float4 *mine = reinterpret_cast<float4 *>(sval) + 2 * lane;
        mine[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        mine[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
        for (int k = lane; k < cnt; k += 32)
            sval[(idx[k] - ix0) & (kTile - 1)] = vals[k]; // in range for any slot contents
        __syncwarp();
        const float4 x = mine[0], y = mine[1];
        f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
        f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
        __syncwarp();
    }
    __device__ __forceinline__ static void add8(float (&v)[8], const float (&f)[8])
    {
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const float2 r = __fadd2_rn(make_float2(v[i], v[i + 1]), make_float2(f[i], f[i + 1]));
            v[i] = r.x;
            v[i + 1] = r.y;
        }
    }
};

// Sparse values + indices, one message per 256 elements (the per-slice
// option, RRA_SPARSE_PER_SLICE).  Every 256-element group of a slice is its
// own sub-message with its own sparse/dense decision, so a slice of G groups
// carries G sub-messages of a.sp_sub bytes each: {uint32 fmt, uint32 nnz}
// padded to 16 bytes, fp32 values, then (sparse form) int32 indices,
// group-relative and ascending, from byte 16 + 4*icap.  A group is sent
// sparse only with nnz < a.sp_full_lim, so icap = a.sp_icap = lim - 1 pairs
// always fit; the dense fallback (fmt 0) holds values[0..len) in place.
template <> struct WireCodec<kCodecSparse> {
    static constexpr bool kVarBytes = true;
    struct Reg {
        uint32_t fmt, nnz;
        float f[8]; // restored values
    };
    __device__ __forceinline__ static unsigned char *sub(const unsigned char *slot, int gi,
                                                         const RingArgs &a)
    {
        return const_cast<unsigned char *>(slot) + gi * a.sp_sub;
    }
    __device__ __forceinline__ static float *vals(unsigned char *s)
    {
        return reinterpret_cast<float *>(s + 16);
    }
    __device__ __forceinline__ static int *idxs(unsigned char *s, const RingArgs &a)
    {
        return reinterpret_cast<int *>(s + 16 + 4 * a.sp_icap);
    }
    // elements of group gi in a slice of V
    __device__ __forceinline__ static int group_len(int V, int gi)
    {
        return min(max(V - gi * kTile, 0), kTile);
    }
    // wire bytes of one sub-message: the 8-byte header, then nnz (value,
    // index) pairs (sparse) or the group's values (dense); an empty group
    // past the slice's end sends nothing
    __device__ __forceinline__ static uint32_t sub_bytes(uint32_t fmt, uint32_t nnz, int len)
    {
        return len > 0 ? 8u + (fmt ? 8u * nnz : 4u * (uint32_t)len) : 0u;
    }
    // wire bytes of the sub-messages of a slice of V elements
    __device__ __forceinline__ static uint32_t bytes(int V, const unsigned char *slot,
                                                     const RingArgs &a, const Msg &)
    {
        uint32_t b = 0;
        for (int gi = 0; gi * kTile < V; ++gi) {
            const uint2 h = *reinterpret_cast<const uint2 *>(sub(slot, gi, a));
            b += sub_bytes(h.x, h.y, group_len(V, gi));
        }
        return b;
    }
    // wire bytes of a loaded group gi of a slice of V elements
    __device__ __forceinline__ static uint32_t group_bytes(const Reg &m, int V, int gi, const Msg &)
    {
        return sub_bytes(m.fmt, m.nnz, group_len(V, gi));
    }
    // Write the sub-message of the lane values v (nonzero at the bits of
    // nzm): sparse when fmt is set, dense otherwise.  Warp-collective.
    __device__ __forceinline__ static void emit(unsigned char *s, int lane, const float (&v)[8],
                                                uint32_t nzm, uint32_t fmt, int total,
                                                const RingArgs &a)
    {
        if (lane == 0)
            *reinterpret_cast<uint2 *>(s) = make_uint2(fmt, (uint32_t)total);
        if (fmt) {
            const int cnt = __popc(nzm);
            const int incl = SparseWarp::incl_scan(lane, cnt);
            SparseWarp::write_pairs(vals(s), idxs(s, a), incl - cnt, lane, 0, v, nzm);
        } else {
            float4 *p = reinterpret_cast<float4 *>(vals(s)) + 2 * lane;
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
    // Read sub-message gi and restore it.  Warp-collective.
    __device__ __forceinline__ static void load(const unsigned char *slot, int gi, int lane,
                                                unsigned char *scratch, const RingArgs &a,
                                                Reg &m, const Msg &)
    {
        unsigned char *s = sub(slot, gi, a);
        const uint2 h = *reinterpret_cast<const uint2 *>(s);
        m.fmt = h.x;
        m.nnz = h.y;
        if (!m.fmt) {
            const float4 *p = reinterpret_cast<const float4 *>(vals(s)) + 2 * lane;
            const float4 x = p[0], y = p[1];
            m.f[0] = x.x; m.f[1] = x.y; m.f[2] = x.z; m.f[3] = x.w;
            m.f[4] = y.x; m.f[5] = y.y; m.f[6] = y.z; m.f[7] = y.w;
            return;
        }
        SparseWarp::restore(vals(s), idxs(s, a), min((int)h.y, a.sp_icap), 0, lane, scratch, m.f);
    }
    // Forward a received group unchanged: the same format, count, values
    // and ascending indices.  Warp-collective.
    __device__ __forceinline__ static void store(unsigned char *slot, int gi, int lane,
                                                 const Reg &m, const RingArgs &a, const Msg &)
    {
        const uint32_t nzm = m.fmt ? SparseWarp::nonzero_mask(m.f, lane, kTile) : 0xffu;
        emit(sub(slot, gi, a), lane, m.f, nzm, m.fmt, (int)m.nnz, a);
    }
    // The header of a dense group also carries its nonzero count.  The
    // receiver restores every value exactly, so the decoded values are v
    // itself: DEC changes nothing.
    template <bool DEC>
    __device__ __forceinline__ static uint32_t encode(float (&v)[8], unsigned char *slot, int gi,
                                                      int lane, int V, const RingArgs &a,
                                                      unsigned char *, const Msg &)
    {
        const int Vg = group_len(V, gi);
        const uint32_t nzm = SparseWarp::nonzero_mask(v, lane, Vg);
        const int total = (int)__reduce_add_sync(kFull, (unsigned)__popc(nzm));
        // full groups compare with the precomputed integer limit; a ragged
        // group evaluates nnz < (1 - threshold) * len in double
        const uint32_t fmt = Vg == kTile ? (total < a.sp_full_lim ? 1u : 0u)
                                         : ((double)total < a.one_minus_thr * (double)Vg ? 1u : 0u);
        emit(sub(slot, gi, a), lane, v, nzm, fmt, total, a);
        return sub_bytes(fmt, (uint32_t)total, Vg);
    }
    __device__ __forceinline__ static void decode_add(const Reg &m, float (&v)[8], int,
                                                      unsigned char *)
    {
        SparseWarp::add8(v, m.f);
    }
    __device__ __forceinline__ static void values(const Reg &m, float (&v)[8], int,
                                                  unsigned char *)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = m.f[i];
    }
};

// Sparse values + indices, one message per ring chunk and hop (the
// default, RRA_SPARSE_PER_CHUNK).  The format of every message -- sparse iff
// the chunk's partial at that hop has nnz < (1 - threshold) * len -- comes
// from the count pass before the ring starts; the ring then streams each
// chunk's message slice by slice, every slice carrying its piece in the
// chunk's format:
//  dense   the piece's fp32 values;
//  sparse  the piece's (value, index) pairs in ascending index order, the
//          indices int32 and relative to the chunk start.
// The chunk's first slice also carries the message header {fmt, nnz}.
// Slot layout (G groups of 256): bytes 0..8 the header {fmt, nnz} (first
// slice only), bytes 16 + 4*gi the pair count of a sparse group gi, and the
// 1024-byte region of group gi from 32 + 1024*gi: 256 fp32 values (dense),
// or up to 128 pairs, values from byte 0 and indices from byte 512 of the
// region (sparse).  A sparse chunk has fewer nonzeros than half its
// elements, but one group of it may have more: pairs 128..255 of a group go
// to the same layout in the slot's spill area in global memory
// (a.sp_spill), which is written and read only then.  The pair counts only
// frame the piece on chip; the receiver could read them off the ascending
// indices, and they are not wire bytes.
template <> struct WireCodec<kCodecSparseChunk> {
    static constexpr bool kVarBytes = true;
    static constexpr int kHdr = 32;
    static constexpr int kRegion = kTile * 4;  // bytes of one group's region
    static constexpr int kCap = kTile / 2;     // pairs of a group held in the slot
    struct Reg {
        uint32_t cnt; // pairs of a sparse group
        float f[8];   // restored values
    };
    __device__ __forceinline__ static unsigned char *region(const unsigned char *slot, int gi)
    {
        return const_cast<unsigned char *>(slot) + kHdr + gi * kRegion;
    }
    __device__ __forceinline__ static uint32_t *counts(const unsigned char *slot)
    {
        return reinterpret_cast<uint32_t *>(const_cast<unsigned char *>(slot) + 16);
    }
    // group gi's spill region of this slot (rare path: a group of more than
    // 128 nonzeros in a sparse chunk)
    __device__ __forceinline__ static unsigned char *spill(const unsigned char *slot, int gi,
                                                           const RingArgs &a)
    {
        extern __shared__ __align__(128) unsigned char smem[];
        const long long si = (slot - (smem + a.slots_off)) / a.slot_bytes;
        return a.sp_spill + ((long long)blockIdx.x * a.N * a.K + si) * (a.slot_bytes - kHdr) +
               gi * kRegion;
    }
    __device__ __forceinline__ static int group_len(int V, int gi)
    {
        return min(max(V - gi * kTile, 0), kTile);
    }
    // the message header's 8 bytes travel with the chunk's first slice
    __device__ __forceinline__ static uint32_t header_bytes(int V, int gi, const Msg &mg)
    {
        return gi == 0 && mg.base == 0 && V > 0 ? 8u : 0u;
    }
    __device__ __forceinline__ static uint32_t bytes(int V, const unsigned char *slot,
                                                     const RingArgs &, const Msg &mg)
    {
        uint32_t b = header_bytes(V, 0, mg);
        if (!mg.sparse())
            return b + 4u * (uint32_t)V;
        for (int gi = 0; gi * kTile < V; ++gi)
            b += 8u * counts(slot)[gi];
        return b;
    }
    __device__ __forceinline__ static uint32_t group_bytes(const Reg &m, int V, int gi,
                                                           const Msg &mg)
    {
        return header_bytes(V, gi, mg) +
               (mg.sparse() ? 8u * m.cnt : 4u * (uint32_t)group_len(V, gi));
    }
    // Write group gi of the piece from the lane values v (sparse: the
    // nonzero ones, ascending).  Returns the wire bytes.  Warp-collective.
    __device__ __forceinline__ static uint32_t emit(unsigned char *slot, int gi, int lane,
                                                    const float (&v)[8], int V, const RingArgs &a,
                                                    const Msg &mg)
    {
        const int Vg = group_len(V, gi);
        unsigned char *rg = region(slot, gi);
        const uint32_t hb = header_bytes(V, gi, mg);
        if (hb && lane == 0)
            *reinterpret_cast<uint2 *>(slot) =
                make_uint2((uint32_t)mg.sparse(), (uint32_t)a.sp_nnz[mg.key()]);
        if (!mg.sparse()) {
            float4 *p = reinterpret_cast<float4 *>(rg) + 2 * lane;
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
            return hb + 4u * (uint32_t)Vg;
        }
        const uint32_t nzm = SparseWarp::nonzero_mask(v, lane, Vg);
        const int cnt = __popc(nzm);
        const int incl = SparseWarp::incl_scan(lane, cnt);
        const int total = __shfl_sync(kFull, incl, 31);
        const int ix0 = mg.base + gi * kTile;
        if (total <= kCap) {
            SparseWarp::write_pairs(reinterpret_cast<float *>(rg),
                                    reinterpret_cast<int *>(rg + kRegion / 2), incl - cnt, lane,
                                    ix0, v, nzm);
        } else {
            unsigned char *sp = spill(slot, gi, a);
            int pos = incl - cnt;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((nzm >> i) & 1u) {
                    unsigned char *b = pos < kCap ? rg : sp;
                    const int k = pos < kCap ? pos : pos - kCap;
                    reinterpret_cast<float *>(b)[k] = v[i];
                    reinterpret_cast<int *>(b + kRegion / 2)[k] = ix0 + 8 * lane + i;
                    ++pos;
                }
        }
        if (lane == 0)
            counts(slot)[gi] = (uint32_t)total;
        return hb + 8u * (uint32_t)total;
    }
    __device__ __forceinline__ static void load(const unsigned char *slot, int gi, int lane,
                                                unsigned char *scratch, const RingArgs &a,
                                                Reg &m, const Msg &mg)
    {
        const unsigned char *rg = region(slot, gi);
        if (!mg.sparse()) {
            const float4 *p = reinterpret_cast<const float4 *>(rg) + 2 * lane;
            const float4 x = p[0], y = p[1];
            m.f[0] = x.x; m.f[1] = x.y; m.f[2] = x.z; m.f[3] = x.w;
            m.f[4] = y.x; m.f[5] = y.y; m.f[6] = y.z; m.f[7] = y.w;
            m.cnt = 0;
            return;
        }
        // decompress: zeros, then every listed value at its index
        const int cnt = (int)min(counts(slot)[gi], (uint32_t)kTile);
        m.cnt = (uint32_t)cnt;
        const int ix0 = mg.base + gi * kTile;
        float *sval = reinterpret_cast<float *>(scratch);
        float4 *mine = reinterpret_cast<float4 *>(sval) + 2 * lane;
        mine[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        mine[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
        const float *vs = reinterpret_cast<const float *>(rg);
        const int *is = reinterpret_cast<const int *>(rg + kRegion / 2);
        for (int k = lane; k < min(cnt, kCap); k += 32)
            sval[(is[k] - ix0) & (kTile - 1)] = vs[k]; // in range for any slot contents
        if (cnt > kCap) {
            const unsigned char *sp = spill(slot, gi, a);
            const float *vo = reinterpret_cast<const float *>(sp);
            const int *io = reinterpret_cast<const int *>(sp + kRegion / 2);
            for (int k = lane; k < cnt - kCap; k += 32)
                sval[(io[k] - ix0) & (kTile - 1)] = vo[k];
        }
        __syncwarp();
        const float4 x = mine[0], y = mine[1];
        m.f[0] = x.x; m.f[1] = x.y; m.f[2] = x.z; m.f[3] = x.w;
        m.f[4] = y.x; m.f[5] = y.y; m.f[6] = y.z; m.f[7] = y.w;
        __syncwarp();
    }
    // forward the owner's piece unchanged (allgather pass): its restored
    // values list exactly the same nonzeros
    __device__ __forceinline__ static void store(unsigned char *slot, int gi, int lane,
                                                 const Reg &m, const RingArgs &a, const Msg &mg)
    {
        emit(slot, gi, lane, m.f, kTile * (gi + 1), a, mg);
    }
    // the receiver restores every value exactly: DEC changes nothing
    template <bool DEC>
    __device__ __forceinline__ static uint32_t encode(float (&v)[8], unsigned char *slot, int gi,
                                                      int lane, int V, const RingArgs &a,
                                                      unsigned char *, const Msg &mg)
    {
        return emit(slot, gi, lane, v, V, a, mg);
    }

    // ---- the same operations for a step whose messages are all dense
    __device__ __forceinline__ static uint32_t bytes(int V, const unsigned char *,
                                                     const RingArgs &, const DenseMsg &mg)
    {
        return header_bytes(V, 0, mg) + 4u * (uint32_t)V;
    }
    __device__ __forceinline__ static uint32_t group_bytes(const Reg &, int V, int gi,
                                                           const DenseMsg &mg)
    {
        return header_bytes(V, gi, mg) + 4u * (uint32_t)group_len(V, gi);
    }
    __device__ __forceinline__ static uint32_t emit(unsigned char *slot, int gi, int lane,
                                                    const float (&v)[8], int V, const RingArgs &a,
                                                    const DenseMsg &mg)
    {
        const uint32_t hb = header_bytes(V, gi, mg);
        if (hb && lane == 0)
            *reinterpret_cast<uint2 *>(slot) = make_uint2(0u, (uint32_t)a.sp_nnz[mg.key()]);
        float4 *p = reinterpret_cast<float4 *>(region(slot, gi)) + 2 * lane;
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
        return hb + 4u * (uint32_t)group_len(V, gi);
    }
    __device__ __forceinline__ static void load(const unsigned char *slot, int gi, int lane,
                                                unsigned char *, const RingArgs &, Reg &m,
                                                const DenseMsg &)
    {
        const float4 *p = reinterpret_cast<const float4 *>(region(slot, gi)) + 2 * lane;
        const float4 x = p[0], y = p[1];
        m.f[0] = x.x; m.f[1] = x.y; m.f[2] = x.z; m.f[3] = x.w;
        m.f[4] = y.x; m.f[5] = y.y; m.f[6] = y.z; m.f[7] = y.w;
        m.cnt = 0;
    }
    __device__ __forceinline__ static void store(unsigned char *slot, int gi, int lane,
                                                 const Reg &m, const RingArgs &a,
                                                 const DenseMsg &mg)
    {
        emit(slot, gi, lane, m.f, kTile * (gi + 1), a, mg);
    }
    template <bool DEC>
    __device__ __forceinline__ static uint32_t encode(float (&v)[8], unsigned char *slot, int gi,
                                                      int lane, int V, const RingArgs &a,
                                                      unsigned char *, const DenseMsg &mg)
    {
        return emit(slot, gi, lane, v, V, a, mg);
    }
    __device__ __forceinline__ static void decode_add(const Reg &m, float (&v)[8], int,
                                                      unsigned char *)
    {
        SparseWarp::add8(v, m.f);
    }
    __device__ __forceinline__ static void values(const Reg &m, float (&v)[8], int,
                                                  unsigned char *)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = m.f[i];
    }
};

} // namespace rra

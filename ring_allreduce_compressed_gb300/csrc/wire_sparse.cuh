// wire_sparse.cuh -- the sparse values + indices wire format of the fused
// ring ("CCCL通信压缩库" §2.1: values and indices above a sparsity
// threshold, restored by index at the receiver; reading: one decision per
// 256 elements).  Included by ring_sparse.cu only, after ring_kernel.cuh.
#pragma once

#include "ring_kernel.cuh"

namespace rra {

// Sparse values + indices.  Every 256-element group of a slice is its own
// sub-message (reading: one sparse/dense decision per 256 elements), so a
// slice of G groups carries G sub-messages of a.sp_sub bytes each:
// {uint32 fmt, uint32 nnz} padded to 16 bytes, fp32 values, then (sparse
// form) int32 indices, slice-relative and ascending, from byte 16 + 4*icap.
// A group is sent sparse only with nnz < a.sp_full_lim, so icap =
// a.sp_icap = lim - 1 pairs always fit; the dense fallback (fmt 0) holds
// values[0..len) in place.  Compaction: per-lane presence masks and a warp
// inclusive scan of their popcounts give every lane's first output position.
// A received group is held in registers in its decoded form: the lane's 8
// values (+0.0 where the message has none) and a presence mask, from which
// the identical sub-message can be written again when it is forwarded.
template <> struct WireCodec<kCodecSparse> {
    static constexpr bool kVarBytes = true;
    struct Reg {
        uint32_t fmt, nnz, pres;
        float f[8];
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
                                                     const RingArgs &a)
    {
        uint32_t b = 0;
        for (int gi = 0; gi * kTile < V; ++gi) {
            const uint2 h = *reinterpret_cast<const uint2 *>(sub(slot, gi, a));
            b += sub_bytes(h.x, h.y, group_len(V, gi));
        }
        return b;
    }
    // wire bytes of a loaded group gi of a slice of V elements
    __device__ __forceinline__ static uint32_t group_bytes(const Reg &m, int V, int gi)
    {
        return sub_bytes(m.fmt, m.nnz, group_len(V, gi));
    }
    // Write the sub-message whose lane values are v and whose present
    // positions are the bits of nzm: sparse (ascending indices) when fmt is
    // set, dense otherwise.  Warp-collective.
    __device__ __forceinline__ static void emit(unsigned char *s, int lane, const float (&v)[8],
                                                uint32_t nzm, uint32_t fmt, int cnt, int incl,
                                                int total, const RingArgs &a)
    {
        if (lane == 0)
            *reinterpret_cast<uint2 *>(s) = make_uint2(fmt, (uint32_t)total);
        if (fmt) {
            int pos = incl - cnt;
            float *vv = vals(s);
            int *x = idxs(s, a);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((nzm >> i) & 1u) {
                    vv[pos] = v[i];
                    x[pos] = 8 * lane + i;
                    ++pos;
                }
        } else {
            float4 *p = reinterpret_cast<float4 *>(vals(s)) + 2 * lane;
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
    __device__ __forceinline__ static int warp_incl_scan(int lane, int cnt)
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
    // Read sub-message gi into its decoded register form.  Sparse groups
    // are scattered into the warp's scratch (values + presence bytes) and
    // read back at the lane's 8 positions.  Warp-collective.
    __device__ __forceinline__ static void load(const unsigned char *slot, int gi, int lane,
                                                unsigned char *scratch, const RingArgs &a,
                                                Reg &m)
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
            m.pres = 0xffu;
            return;
        }
        const int nnz = min((int)h.y, a.sp_icap);
        float *sval = reinterpret_cast<float *>(scratch);
        unsigned char *spres = scratch + kTile * 4;
        *reinterpret_cast<uint2 *>(spres + 8 * lane) = make_uint2(0u, 0u);
        __syncwarp();
        const int *ix_in = idxs(s, a);
        for (int k = lane; k < nnz; k += 32) {
            const int ix = ix_in[k] & (kTile - 1); // in range for any slot contents
            sval[ix] = vals(s)[k];
            spres[ix] = 1;
        }
        __syncwarp();
        const uint2 pb = *reinterpret_cast<const uint2 *>(spres + 8 * lane);
        const float4 *sv = reinterpret_cast<const float4 *>(sval) + 2 * lane;
        const float4 x = sv[0], y = sv[1];
        const float t[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        uint32_t pres = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = ((i < 4 ? pb.x : pb.y) >> (8 * (i & 3))) & 0xffu;
            pres |= (byte ? 1u : 0u) << i;
            m.f[i] = byte ? t[i] : 0.0f;
        }
        m.pres = pres;
        __syncwarp();
    }
    // Forward a received group unchanged: the same format, count, values
    // and ascending indices.  Warp-collective.
    __device__ __forceinline__ static void store(unsigned char *slot, int gi, int lane,
                                                 const Reg &m, const RingArgs &a)
    {
        unsigned char *s = sub(slot, gi, a);
        if (!m.fmt) {
            emit(s, lane, m.f, 0xffu, 0u, 0, 0, (int)m.nnz, a);
            return;
        }
        const int cnt = __popc(m.pres);
        const int incl = warp_incl_scan(lane, cnt);
        emit(s, lane, m.f, m.pres, 1u, cnt, incl, (int)m.nnz, a);
    }
    // The header of a dense group also carries its nonzero count.  The
    // receiver restores every value exactly (absent ones are +0.0), so the
    // decoded values are v itself: DEC changes nothing.
    template <bool DEC>
    __device__ __forceinline__ static uint32_t encode(float (&v)[8], unsigned char *slot, int gi,
                                                      int lane, int V, const RingArgs &a,
                                                      unsigned char *)
    {
        const int Vg = group_len(V, gi);
        uint32_t nzm = 0;
        if (Vg == kTile) { // a full group: every lane's 8 positions are inside it
#pragma unroll
            for (int i = 0; i < 8; ++i)
                nzm |= (__float_as_uint(v[i]) != 0u ? 1u : 0u) << i;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (8 * lane + i < Vg && __float_as_uint(v[i]) != 0u)
                    nzm |= 1u << i;
        }
        const int cnt = __popc(nzm);
        const int total = (int)__reduce_add_sync(kFull, (unsigned)cnt);
        // full groups compare with the precomputed integer limit; a ragged
        // group evaluates nnz < (1 - threshold) * len in double
        const uint32_t fmt = Vg == kTile ? (total < a.sp_full_lim ? 1u : 0u)
                                         : ((double)total < a.one_minus_thr * (double)Vg ? 1u : 0u);
        // only a sparse group needs every lane's output position
        const int incl = fmt ? warp_incl_scan(lane, cnt) : 0;
        emit(sub(slot, gi, a), lane, v, nzm, fmt, cnt, incl, total, a);
        return sub_bytes(fmt, (uint32_t)total, Vg);
    }
    __device__ __forceinline__ static void decode_add(const Reg &m, float (&v)[8], int,
                                                      unsigned char *)
    {
        if (m.pres == 0xffu) { // every position present (always so for a dense group)
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 r = __fadd2_rn(make_float2(v[i], v[i + 1]),
                                            make_float2(m.f[i], m.f[i + 1]));
                v[i] = r.x;
                v[i + 1] = r.y;
            }
            return;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = ((m.pres >> i) & 1u) ? __fadd_rn(v[i], m.f[i]) : v[i];
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

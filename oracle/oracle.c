/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the chunked ring
 * allreduce with gradient-compression codecs.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The GPU library never
 * links, includes or calls this file, and this file includes nothing from the
 * GPU library: its enums, constants, conversions and wire formats are written
 * out here on their own, from the definitions below.
 *
 * Build:  gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (no FMA contraction, no reassociation: every float operation is one IEEE
 * binary32 operation rounded to nearest-even, in the order written).
 *
 * Sources (web pages, cited by title and section):
 *  [P2] "从零实现集合通信" (collective ops from scratch, aibook lesson 76):
 *       section "两趟实现 ring allreduce" (two-pass ring; per-rank byte and
 *       step table: ring 2T(N-1)/N, tree T log2 N, broadcast T, allgather and
 *       reduce_scatter T(N-1)/N), section "练习" (tree variant, byte counter).
 *  [P4] "CCCL通信压缩库：突破LLM训练通信墙的工程实践":
 *       §2.1 (sparse values+indices format above a sparsity threshold; block
 *       floating point, one shared exponent per block of e.g. 128 elements,
 *       8- or 4-bit mantissas; difference against the previous round),
 *       §2.2 (the tensor is cut into chunks that are compressed, sent,
 *       decompressed and reduced one after the other),
 *       §3.3 (compression types block_fp16_to_8bit / block_fp16_to_4bit /
 *       sparse / diff; sparsity_threshold 0.5).
 *
 * Readings taken where the pages are silent (each one is listed, with its
 * reason, in the design notes of the repository):
 *  R1  ring steps are numbered s = 1..N-1: at reduce-scatter step s rank r
 *      sends chunk (r-s) mod N; at allgather step s it sends (r-s+1) mod N.
 *  R3  n = ceil(T/N); chunk c = [c*n, min(T,(c+1)*n)), possibly short/empty.
 *  R4  lossless messages carry fp32 (the accumulator type).
 *  B1  block exponent e = floor(log2 max|x|), clamped below at -126.
 *  B2  q = bits-2; m = clamp(rne(x * 2^(q-e)), -(2^(bits-1)-1), +(...));
 *      decode m * 2^(e-q).
 *  B5  planar BFP message: exps[ceil(len/128)] then mants (int8[len], or
 *      uint8[ceil(len/2)] with element 2j in the low nibble).
 *  B6  every reduce-scatter hop re-encodes the sender's fp32 partial; the
 *      owner encodes its full sum once; the allgather forwards those codes
 *      unchanged; every rank (owner included) outputs decode(codes).
 *  S1  an element is "zero" iff its fp32 bit pattern is +0.0.
 *  S2  sparse iff nnz < (1 - threshold) * len (in double); tie -> dense.
 *  S3  the sparse codec sends one message per ring chunk and hop (slice 0:
 *      the format is chosen from the nonzero count of the whole chunk's
 *      partial, as [P4] §2.1 analyses the sparsity of the tensor about to
 *      be sent), or, as an option, one message per slice of `slice`
 *      elements.  A message is an 8-byte header {fmt, nnz}, then fp32
 *      values[nnz] and int32 indices[nnz] ascending, relative to the
 *      message start (sparse), or fp32[len] (dense).
 *  S4  decompress, then reduce ([P4] §2.2: receive, decompress, reduce;
 *      §2.1: the receiver restores the nonzero values to their positions by
 *      index): a sparse message is restored into a piece of +0.0 values,
 *      and the receiver adds the whole restored piece, acc[i] = acc[i] + v.
 *  D1  diff: d = cur - prev (fp32); the ring runs on d.
 *  D2  epilogue: out = base + (v / N) when a base (previous result) is given
 *      and averaging is on; v / N with averaging only; v otherwise.
 *  RS  reduce-scatter: the owner's output is its fp32 sum (not re-encoded).
 *  AG  compressed allgather ([P4] §2.1, operator-aware layer: allgather
 *      and broadcast take lossless compression or a higher-precision lossy
 *      one; §3.3: low-precision compression for all_gather after
 *      all_reduce): the owner of chunk c encodes its own elements of chunk c
 *      (widened to fp32) once, as one ring message; the allgather steps of
 *      R1 forward those codes unchanged; every rank, the owner included,
 *      stores decode(codes) in the buffer's dtype (RNE), so all buffers end
 *      identical.  Sparse codes restore every element exactly.
 *  F4op  what each operation encodes, for its statistics: the allreduce
 *      every chunk of every buffer; the compressed allgather chunk r of
 *      buffer r; the compressed broadcast the root's buffer, blocks from its
 *      start.
 *  AB  compressed broadcast (the same layer of [P4] §2.1 and §3.3), BFP:
 *      the root encodes its whole buffer (widened to fp32) once, as one
 *      message with blocks of 128 from the buffer start; every edge of the
 *      binomial tree carries those codes unchanged; every rank, the root
 *      included, stores decode(codes) in the buffer's dtype (RNE).
 *  EF  error feedback ([P4] §5, future directions), BFP only: each rank
 *      keeps an fp32 residual e_r[T]; whatever value v it encodes (its
 *      reduce-scatter messages, and as owner its chunk's full sum) is encoded
 *      as u = v + e, after which e = u - decode(Q(u)).  Every element of
 *      e_r is updated exactly once per allreduce.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

/* Allocation that ends the process with a message instead of returning NULL:
 * the oracle is a test program, and running out of host memory is fatal to
 * it.  Zero-byte requests get one byte, so a pointer is never NULL. */
static void *xcalloc(size_t count, size_t size)
{
    void *p = calloc(count ? count : 1, size ? size : 1);
    if (!p) {
        fprintf(stderr, "oracle: out of host memory (%zu x %zu bytes)\n", count, size);
        abort();
    }
    return p;
}

static void *xmalloc(size_t bytes) { return xcalloc(bytes, 1); }

/* ------------------------------------------------------------------ */
/* element types and IEEE conversions, written from the binary16 /     */
/* bfloat16 definitions (sign, exponent, significand)                  */
/* ------------------------------------------------------------------ */

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };
enum { OR_CODEC_NONE = 0, OR_CODEC_BFP = 1, OR_CODEC_SPARSE = 2 };
enum { OR_BFP_BLOCK = 128 };

size_t oracle_dtype_size(int t) { return t == OR_F32 ? 4 : 2; }

/* binary16 -> binary32: exact. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    float v;
    if (ex == 0)
        v = ldexpf((float)man, -24); /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + man), ex - 25); /* 1.man * 2^(ex-15) */
    return sign ? -v : v;
}

/* binary32 -> binary16, round to nearest even. */
uint16_t oracle_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    float a = fabsf(x);
    if (isnan(x))
        return sign | 0x7e00;
    /* largest finite half is 65504; the midpoint to 65536 is 65520 and
     * rounds to even, i.e. up, so everything from 65520 on overflows */
    if (a >= 65520.0f)
        return sign | 0x7c00;
    if (a < ldexpf(1.0f, -14)) {
        /* subnormal range: spacing 2^-24 */
        float q = nearbyintf(ldexpf(a, 24)); /* exact scaling, then RNE */
        return sign | (uint16_t)q;           /* q == 1024 encodes 2^-14 */
    }
    int E;
    frexpf(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1; /* floor(log2 a) */
    float m = nearbyintf(ldexpf(a, 10 - e)); /* in [1024, 2048] */
    if (m == 2048.0f) {
        m = 1024.0f;
        e += 1;
    }
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)m - 1024);
}

/* bfloat16 -> binary32: the top half of the binary32 pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float v;
    memcpy(&v, &u, 4);
    return v;
}

/* binary32 -> bfloat16, round to nearest even. */
uint16_t oracle_f32_to_bf16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    float a = fabsf(x);
    if (isnan(x))
        return sign | 0x7fc0;
    if (isinf(x))
        return sign | 0x7f80;
    if (a < ldexpf(1.0f, -126)) {
        /* subnormal range of bfloat16: spacing 2^-133 */
        float q = nearbyintf(ldexpf(a, 133));
        return sign | (uint16_t)q; /* q == 128 encodes 2^-126 */
    }
    int E;
    frexpf(a, &E);
    int e = E - 1;
    float m = nearbyintf(ldexpf(a, 7 - e)); /* in [128, 256] */
    if (m == 256.0f) {
        m = 128.0f;
        e += 1;
    }
    if (e > 127)
        return sign | 0x7f80; /* rounded past the largest finite value */
    return sign | (uint16_t)((e + 127) << 7) | (uint16_t)((int)m - 128);
}

static float load_as_f32(const void *buf, size_t i, int t)
{
    if (t == OR_F32)
        return ((const float *)buf)[i];
    if (t == OR_F16)
        return oracle_f16_to_f32(((const uint16_t *)buf)[i]);
    return oracle_bf16_to_f32(((const uint16_t *)buf)[i]);
}

static void store_from_f32(void *buf, size_t i, int t, float v)
{
    if (t == OR_F32)
        ((float *)buf)[i] = v;
    else if (t == OR_F16)
        ((uint16_t *)buf)[i] = oracle_f32_to_f16(v);
    else
        ((uint16_t *)buf)[i] = oracle_f32_to_bf16(v);
}

/* ------------------------------------------------------------------ */
/* block floating point  [P4 §2.1, §3.3]                                */
/* ------------------------------------------------------------------ */

/* B1: floor(log2 max|x_i|) over the block, -126 for a zero or subnormal max. */
int oracle_bfp_block_exponent(const float *x, size_t len)
{
    float amax = 0.0f;
    for (size_t i = 0; i < len; i++)
        if (fabsf(x[i]) > amax)
            amax = fabsf(x[i]);
    if (amax < ldexpf(1.0f, -126))
        return -126;
    int E;
    frexpf(amax, &E);
    return E - 1;
}

static int bfp_limit(int bits) { return (1 << (bits - 1)) - 1; } /* 127 or 7 */

/* B2: one element's integer code for block exponent e. */
int oracle_bfp_code(float x, int e, int bits)
{
    int q = bits - 2;
    float scaled = ldexpf(x, q - e); /* exact power-of-two scaling */
    float r = nearbyintf(scaled);    /* round to nearest even */
    int M = bfp_limit(bits);
    if (r > (float)M)
        r = (float)M;
    if (r < -(float)M)
        r = -(float)M;
    return (int)r;
}

float oracle_bfp_value(int m, int e, int bits) { return ldexpf((float)m, e - (bits - 2)); }

size_t oracle_bfp_bytes(size_t len, int bits)
{
    size_t nb = (len + OR_BFP_BLOCK - 1) / OR_BFP_BLOCK;
    return nb + (bits == 8 ? len : (len + 1) / 2);
}

/* B5: planar encode of x[0..n) into exps[ceil(n/128)] and mants. */
void oracle_bfp_encode(const float *x, size_t n, int bits, int8_t *exps, uint8_t *mants)
{
    size_t nb = (n + OR_BFP_BLOCK - 1) / OR_BFP_BLOCK;
    if (bits == 4)
        memset(mants, 0, (n + 1) / 2);
    for (size_t b = 0; b < nb; b++) {
        size_t lo = b * OR_BFP_BLOCK;
        size_t len = n - lo < OR_BFP_BLOCK ? n - lo : OR_BFP_BLOCK;
        int e = oracle_bfp_block_exponent(x + lo, len);
        exps[b] = (int8_t)e;
        for (size_t i = lo; i < lo + len; i++) {
            int m = oracle_bfp_code(x[i], e, bits);
            if (bits == 8) {
                mants[i] = (uint8_t)(int8_t)m;
            } else {
                uint8_t nib = (uint8_t)(m & 0xf);
                if (i % 2 == 0)
                    mants[i / 2] |= nib;
                else
                    mants[i / 2] |= (uint8_t)(nib << 4);
            }
        }
    }
}

static int bfp_code_at(const uint8_t *mants, size_t i, int bits)
{
    if (bits == 8)
        return (int)(int8_t)mants[i];
    int nib = (i % 2 == 0) ? (mants[i / 2] & 0xf) : (mants[i / 2] >> 4);
    return nib >= 8 ? nib - 16 : nib; /* two's-complement 4-bit value */
}

void oracle_bfp_decode(const int8_t *exps, const uint8_t *mants, size_t n, int bits, float *out,
                       int accumulate)
{
    for (size_t i = 0; i < n; i++) {
        float v = oracle_bfp_value(bfp_code_at(mants, i, bits), exps[i / OR_BFP_BLOCK], bits);
        out[i] = accumulate ? out[i] + v : v;
    }
}

/* ------------------------------------------------------------------ */
/* sparse values + indices  [P4 §2.1, §3.3]                             */
/* ------------------------------------------------------------------ */

/* S1: nonzero means "bit pattern is not +0.0". */
static int is_nonzero(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    return u != 0u;
}

/* S2 */
int oracle_sparse_is_sparse(size_t nnz, size_t len, double threshold)
{
    return (double)nnz < (1.0 - threshold) * (double)len;
}

/* Standalone encode of x[0..n) (values kept in the input dtype t):
 * hdr[0] = 1 sparse / 0 dense, hdr[1] = nnz.  Sparse: vals[0..nnz) and
 * idx[0..nnz) ascending.  Dense: vals[0..n) = x. */
void oracle_sparse_encode(const void *x, size_t n, int t, double threshold, uint32_t *hdr,
                          void *vals, int32_t *idx)
{
    size_t es = oracle_dtype_size(t);
    size_t nnz = 0;
    for (size_t i = 0; i < n; i++)
        if (is_nonzero(load_as_f32(x, i, t)))
            nnz++;
    int sparse = oracle_sparse_is_sparse(nnz, n, threshold);
    hdr[0] = (uint32_t)sparse;
    hdr[1] = (uint32_t)nnz;
    if (!sparse) {
        memcpy(vals, x, n * es);
        return;
    }
    size_t k = 0;
    for (size_t i = 0; i < n; i++) {
        if (is_nonzero(load_as_f32(x, i, t))) {
            memcpy((char *)vals + k * es, (const char *)x + i * es, es);
            idx[k] = (int32_t)i;
            k++;
        }
    }
}

/* Standalone decode into fp32 acc[0..n).  accumulate = 0: acc = restored
 * message (+0.0 where the sparse message lists nothing).  accumulate = 1:
 * acc[i] = acc[i] + v at every position the message carries (all positions
 * for a dense message, the listed ones for a sparse message). */
void oracle_sparse_decode(const uint32_t *hdr, const void *vals, const int32_t *idx, size_t n,
                          int t, float *acc, int accumulate)
{
    if (hdr[0] == 0) {
        for (size_t i = 0; i < n; i++) {
            float v = load_as_f32(vals, i, t);
            acc[i] = accumulate ? acc[i] + v : v;
        }
        return;
    }
    if (!accumulate)
        for (size_t i = 0; i < n; i++)
            acc[i] = 0.0f;
    for (size_t k = 0; k < hdr[1]; k++) {
        float v = load_as_f32(vals, k, t);
        size_t i = (size_t)idx[k];
        acc[i] = accumulate ? acc[i] + v : v;
    }
}

/* ------------------------------------------------------------------ */
/* difference encoding  [P4 §2.1 "current minus previous round"]        */
/* ------------------------------------------------------------------ */

void oracle_diff_encode(const float *cur, const float *prev, float *diff, size_t n)
{
    for (size_t i = 0; i < n; i++)
        diff[i] = cur[i] - prev[i];
}

/* ------------------------------------------------------------------ */
/* ring messages: one chunk's worth of data on one edge of the ring    */
/* ------------------------------------------------------------------ */

typedef struct {
    int kind;         /* codec */
    int bits;         /* bfp */
    double threshold; /* sparse */
    size_t slice;     /* sparse: elements per message; 0 = one message per chunk */
} codec_t;

typedef struct {
    size_t len;     /* elements covered */
    size_t bytes;   /* wire size */
    float *f;       /* NONE: fp32 values; SPARSE: restored values (+0.0 where none) */
    int8_t *exps;   /* BFP */
    uint8_t *mants; /* BFP */
    size_t nexps;   /* BFP: ceil(len/128) */
    size_t nmants;  /* BFP: len (8-bit) or ceil(len/2) (4-bit) */
} message;

static void msg_free(message *m)
{
    free(m->f);
    free(m->exps);
    free(m->mants);
    memset(m, 0, sizeof *m);
}

/* Build the message a rank sends for the fp32 data x[0..len). */
static void msg_encode(message *m, const codec_t *cd, const float *x, size_t len)
{
    msg_free(m);
    m->len = len;
    if (cd->kind == OR_CODEC_NONE) {
        m->f = xmalloc((len ? len : 1) * sizeof(float));
        memcpy(m->f, x, len * sizeof(float));
        m->bytes = 4 * len;
    } else if (cd->kind == OR_CODEC_BFP) {
        size_t nb = (len + OR_BFP_BLOCK - 1) / OR_BFP_BLOCK;
        size_t mb = cd->bits == 8 ? len : (len + 1) / 2;
        m->exps = xmalloc(nb ? nb : 1);
        m->mants = xmalloc(mb ? mb : 1);
        m->nexps = nb;
        m->nmants = mb;
        oracle_bfp_encode(x, len, cd->bits, m->exps, m->mants);
        m->bytes = nb + mb;
    } else {
        /* S3: the chunk's message (slice 0), or one message per slice.
         * The sender lists the nonzero values and their indices (S1); the
         * message is sparse iff S2 holds for its length.  The receiver's
         * restored copy (S4) is built from what is sent: the listed values
         * put back by index into zeros, or the dense values. */
        const size_t step = cd->slice ? cd->slice : (len ? len : 1);
        float *pv = xmalloc((len ? len : 1) * sizeof(float));
        int32_t *pi = xmalloc((len ? len : 1) * sizeof(int32_t));
        m->f = xcalloc(len ? len : 1, sizeof(float));
        m->bytes = 0;
        for (size_t lo = 0; lo < len; lo += step) {
            size_t sl = len - lo < step ? len - lo : step;
            size_t nnz = 0;
            for (size_t i = lo; i < lo + sl; i++)
                if (is_nonzero(x[i])) {
                    pv[nnz] = x[i];
                    pi[nnz] = (int32_t)(i - lo);
                    nnz++;
                }
            if (oracle_sparse_is_sparse(nnz, sl, cd->threshold)) {
                for (size_t k = 0; k < nnz; k++)
                    m->f[lo + (size_t)pi[k]] = pv[k];
                m->bytes += 8 + 8 * nnz;
            } else {
                for (size_t i = lo; i < lo + sl; i++)
                    m->f[i] = x[i];
                m->bytes += 8 + 4 * sl;
            }
        }
        free(pv);
        free(pi);
    }
}

static void msg_copy(message *dst, const message *src)
{
    msg_free(dst);
    *dst = *src;
    size_t len = src->len ? src->len : 1;
    if (src->f) {
        dst->f = xmalloc(len * sizeof(float));
        memcpy(dst->f, src->f, src->len * sizeof(float));
    }
    if (src->exps) {
        dst->exps = xmalloc(src->nexps ? src->nexps : 1);
        memcpy(dst->exps, src->exps, src->nexps);
    }
    if (src->mants) {
        dst->mants = xmalloc(src->nmants ? src->nmants : 1);
        memcpy(dst->mants, src->mants, src->nmants);
    }
}

/* Decoded value of element i of a message (sparse: its restored value,
 * +0.0 where the message lists nothing). */
static float msg_value(const message *m, const codec_t *cd, size_t i)
{
    if (cd->kind == OR_CODEC_BFP)
        return oracle_bfp_value(bfp_code_at(m->mants, i, cd->bits), m->exps[i / OR_BFP_BLOCK],
                                cd->bits);
    return m->f[i];
}

/* ------------------------------------------------------------------ */
/* chunking  [P2 "两趟实现 ring allreduce"]                              */
/* ------------------------------------------------------------------ */

static int mod(long a, int n) { return (int)(((a % n) + n) % n); }

static void chunk_range(size_t T, int N, int c, size_t *lo, size_t *len)
{
    size_t n = (T + (size_t)N - 1) / (size_t)N; /* R3 */
    size_t a = (size_t)c * n;
    size_t b = a + n;
    if (a > T)
        a = T;
    if (b > T)
        b = T;
    *lo = a;
    *len = b - a;
}

/* ------------------------------------------------------------------ */
/* the two-pass ring  [P2 "两趟实现 ring allreduce"; P4 §1, §2.2]        */
/* ------------------------------------------------------------------ */

enum { OR_MODE_ALLREDUCE = 0, OR_MODE_REDUCE_SCATTER = 1 };

/*
 * Each rank r keeps a local fp32 copy of its whole buffer.  Reduce-scatter,
 * steps s = 1..N-1: every rank r encodes its local chunk (r-s) mod N into a
 * message for rank r+1; then every rank r decodes the message it got (chunk
 * (r-s-1) mod N) and adds it into its local copy of that chunk.  After the
 * last step rank r holds the full sum of chunk r.
 * Allgather, steps s = 1..N-1: rank r sends chunk (r-s+1) mod N (for s = 1
 * its own finished chunk, encoded once; afterwards the message it received
 * the step before, unchanged) and rank r+1 keeps it and decodes it.
 * Byte counters: sent[r] and recv[r+1] grow by each message's wire size.
 *
 * Returns 0 on success, -1 on a bad argument.
 */
/* Encode n fp32 values v into m with error feedback ("CCCL通信压缩库" §5,
 * future directions: the precision a compression loses in one round is
 * carried into the next round).  The value encoded is u = v + e (fp32); the
 * residual becomes e = u - decode(Q(u)).  e is updated in place. */
static void msg_encode_ef(message *m, const codec_t *cd, const float *v, float *e, size_t n)
{
    float *u = xmalloc((n ? n : 1) * sizeof(float));
    for (size_t i = 0; i < n; i++)
        u[i] = v[i] + e[i];
    msg_encode(m, cd, u, n);
    for (size_t i = 0; i < n; i++) {
        const float d = msg_value(m, cd, i);
        e[i] = u[i] - d;
    }
    free(u);
}

int oracle_ring_ef(int mode, int N, size_t T, const void *const *in, int in_t, void *const *out,
                   int out_t, int codec, int bits, double threshold, size_t slice,
                   const float *const *diff_prev, const float *diff_base, int average,
                   float *const *resid, uint64_t *sent, uint64_t *recv)
{
    if (N < 1 || (codec == OR_CODEC_BFP && bits != 8 && bits != 4) || (diff_prev && in_t != OR_F32))
        return -1;
    if (resid && codec != OR_CODEC_BFP) /* only a lossy codec has an error to feed back */
        return -1;
    codec_t cd = {codec, bits, threshold, slice};
    for (int r = 0; r < N; r++)
        sent[r] = recv[r] = 0;

    /* local working copies (D1: the ring runs on cur - prev when diffing) */
    float **local = xmalloc((size_t)N * sizeof(float *));
    for (int r = 0; r < N; r++) {
        local[r] = xmalloc((T ? T : 1) * sizeof(float));
        for (size_t i = 0; i < T; i++)
            local[r][i] = diff_prev ? ((const float *)in[r])[i] - diff_prev[r][i]
                                    : load_as_f32(in[r], i, in_t);
    }
    message *outbox = xcalloc((size_t)N, sizeof(message));

    /* ---- pass 1: reduce-scatter ---- */
    for (int s = 1; s <= N - 1; s++) {
        for (int r = 0; r < N; r++) {
            int c = mod((long)r - s, N);
            size_t lo, len;
            chunk_range(T, N, c, &lo, &len);
            int dst = mod((long)r + 1, N);
            if (resid) /* every message a rank encodes takes its residual */
                msg_encode_ef(&outbox[dst], &cd, local[r] + lo, resid[r] + lo, len);
            else
                msg_encode(&outbox[dst], &cd, local[r] + lo, len);
            sent[r] += outbox[dst].bytes;
            recv[dst] += outbox[dst].bytes;
        }
        for (int r = 0; r < N; r++) {
            int c = mod((long)r - s - 1, N);
            size_t lo, len;
            chunk_range(T, N, c, &lo, &len);
            for (size_t i = 0; i < len; i++) {
                float v = msg_value(&outbox[r], &cd, i);
                local[r][lo + i] = local[r][lo + i] + v; /* S4 */
            }
        }
    }

    /* value each rank ends with, per element, before the epilogue */
    float **res = xmalloc((size_t)N * sizeof(float *));
    for (int r = 0; r < N; r++)
        res[r] = xmalloc((T ? T : 1) * sizeof(float));

    /* held[r]: the codes of the chunk rank r sends at the next allgather step */
    message *held = xcalloc((size_t)N, sizeof(message));
    int *has = xcalloc((size_t)N * (size_t)N, sizeof(int));

    for (int r = 0; r < N; r++) {
        size_t lo, len;
        chunk_range(T, N, r, &lo, &len);
        if (mode == OR_MODE_REDUCE_SCATTER || codec == OR_CODEC_NONE) {
            for (size_t i = 0; i < len; i++)
                res[r][lo + i] = local[r][lo + i];
        }
        if (mode == OR_MODE_ALLREDUCE) {
            /* B6: the owner encodes its full sum once */
            if (resid)
                msg_encode_ef(&held[r], &cd, local[r] + lo, resid[r] + lo, len);
            else
                msg_encode(&held[r], &cd, local[r] + lo, len);
            if (codec != OR_CODEC_NONE)
                for (size_t i = 0; i < len; i++) {
                    res[r][lo + i] = msg_value(&held[r], &cd, i);
                }
        }
        has[r * N + r] = 1;
    }

    /* ---- pass 2: allgather ---- */
    if (mode == OR_MODE_ALLREDUCE) {
        for (int s = 1; s <= N - 1; s++) {
            for (int r = 0; r < N; r++) {
                int dst = mod((long)r + 1, N);
                msg_copy(&outbox[dst], &held[r]);
                sent[r] += outbox[dst].bytes;
                recv[dst] += outbox[dst].bytes;
            }
            for (int r = 0; r < N; r++) {
                int c = mod((long)r - s, N);
                size_t lo, len;
                chunk_range(T, N, c, &lo, &len);
                for (size_t i = 0; i < len; i++) {
                    res[r][lo + i] = msg_value(&outbox[r], &cd, i);
                }
                msg_copy(&held[r], &outbox[r]);
                has[r * N + c] = 1;
            }
        }
    }

    /* ---- epilogue (D2) and output cast ---- */
    for (int r = 0; r < N; r++) {
        for (int c = 0; c < N; c++) {
            if (!has[r * N + c])
                continue; /* reduce-scatter leaves other chunks untouched */
            size_t lo, len;
            chunk_range(T, N, c, &lo, &len);
            for (size_t i = lo; i < lo + len; i++) {
                float w = res[r][i];
                if (average)
                    w = w / (float)N;
                if (diff_base)
                    w = diff_base[i] + w;
                store_from_f32(out[r], i, out_t, w);
            }
        }
    }

    for (int r = 0; r < N; r++) {
        msg_free(&outbox[r]);
        msg_free(&held[r]);
        free(local[r]);
        free(res[r]);
    }
    free(outbox);
    free(held);
    free(has);
    free(local);
    free(res);
    return 0;
}

int oracle_ring(int mode, int N, size_t T, const void *const *in, int in_t, void *const *out,
                int out_t, int codec, int bits, double threshold, size_t slice,
                const float *const *diff_prev, const float *diff_base, int average,
                uint64_t *sent, uint64_t *recv)
{
    return oracle_ring_ef(mode, N, T, in, in_t, out, out_t, codec, bits, threshold, slice,
                          diff_prev, diff_base, average, NULL, sent, recv);
}

/* ------------------------------------------------------------------ */
/* allgather as its own op  [P2 table: T(N-1)/N per rank, N-1 steps]    */
/* ------------------------------------------------------------------ */

/* In place: on entry chunk r of buf[r] is rank r's contribution; on exit
 * every buffer holds every chunk.  Element bytes are copied exactly. */
int oracle_allgather(int N, size_t T, void *const *buf, int t, uint64_t *sent, uint64_t *recv)
{
    if (N < 1)
        return -1;
    size_t es = oracle_dtype_size(t);
    for (int r = 0; r < N; r++)
        sent[r] = recv[r] = 0;
    for (int s = 1; s <= N - 1; s++) {
        /* every rank sends first, then every rank stores what it got */
        size_t n = (T + (size_t)N - 1) / (size_t)N;
        char **msg = xmalloc((size_t)N * sizeof(char *));
        for (int r = 0; r < N; r++) {
            int c = mod((long)r - s + 1, N);
            size_t lo, len;
            chunk_range(T, N, c, &lo, &len);
            int dst = mod((long)r + 1, N);
            msg[dst] = xmalloc(n * es + 1);
            memcpy(msg[dst], (char *)buf[r] + lo * es, len * es);
            sent[r] += len * es;
            recv[dst] += len * es;
        }
        for (int r = 0; r < N; r++) {
            int c = mod((long)r - s, N);
            size_t lo, len;
            chunk_range(T, N, c, &lo, &len);
            memcpy((char *)buf[r] + lo * es, msg[r], len * es);
        }
        for (int r = 0; r < N; r++)
            free(msg[r]);
        free(msg);
    }
    return 0;
}

/* Compressed allgather (reading AG), in place: chunk r of buf[r] is rank
 * r's contribution; codec BFP (bits 8 or 4) or sparse (threshold; one
 * message per chunk, or per slice of `slice` elements, S3).  Rank r sends
 * at allgather step s the codes of chunk (r - s + 1) mod N, so it forwards
 * every chunk but chunk r + 1; the byte counters add the message bytes. */
int oracle_allgather_codec(int N, size_t T, void *const *buf, int t, int codec, int bits,
                           double threshold, size_t slice, uint64_t *sent, uint64_t *recv)
{
    if (N < 1 || (codec != OR_CODEC_BFP && codec != OR_CODEC_SPARSE) ||
        (codec == OR_CODEC_BFP && bits != 8 && bits != 4))
        return -1;
    codec_t cd = {codec, bits, threshold, slice};
    for (int r = 0; r < N; r++)
        sent[r] = recv[r] = 0;
    /* held[r]: the codes rank r sends at the next step; first its own chunk */
    message *held = xcalloc((size_t)N, sizeof(message));
    message *inbox = xcalloc((size_t)N, sizeof(message));
    float *x = xmalloc((T ? T : 1) * sizeof(float));
    for (int r = 0; r < N; r++) {
        size_t lo, len;
        chunk_range(T, N, r, &lo, &len);
        for (size_t i = 0; i < len; i++)
            x[i] = load_as_f32(buf[r], lo + i, t);
        msg_encode(&held[r], &cd, x, len);
    }
    /* the owner's own chunk becomes the decoded codes as well */
    for (int r = 0; r < N; r++) {
        size_t lo, len;
        chunk_range(T, N, r, &lo, &len);
        for (size_t i = 0; i < len; i++) {
            store_from_f32(buf[r], lo + i, t, msg_value(&held[r], &cd, i));
        }
    }
    for (int s = 1; s <= N - 1; s++) {
        for (int r = 0; r < N; r++) {
            int dst = mod((long)r + 1, N);
            msg_copy(&inbox[dst], &held[r]);
            sent[r] += inbox[dst].bytes;
            recv[dst] += inbox[dst].bytes;
        }
        for (int r = 0; r < N; r++) {
            int c = mod((long)r - s, N); /* the chunk rank r receives at step s */
            size_t lo, len;
            chunk_range(T, N, c, &lo, &len);
            for (size_t i = 0; i < len; i++) {
                store_from_f32(buf[r], lo + i, t, msg_value(&inbox[r], &cd, i));
            }
            msg_copy(&held[r], &inbox[r]);
        }
    }
    for (int r = 0; r < N; r++) {
        msg_free(&held[r]);
        msg_free(&inbox[r]);
    }
    free(held);
    free(inbox);
    free(x);
    return 0;
}

/* ------------------------------------------------------------------ */
/* broadcast and tree allreduce  [P2 table: broadcast T over a log2(N)  */
/* tree; tree allreduce T log2 N, 2 log2 N steps; "练习" tree variant]  */
/* ------------------------------------------------------------------ */

static int ceil_log2(int N)
{
    int L = 0;
    while ((1 << L) < N)
        L++;
    return L;
}

/* Binomial broadcast from root: at level k = 0..ceil(log2 N)-1 every
 * relative rank q < 2^k with q + 2^k < N sends the whole buffer to q + 2^k
 * (relative rank q is absolute rank (q + root) mod N). */
int oracle_broadcast(int N, size_t T, void *const *buf, int t, int root, uint64_t *sent,
                     uint64_t *recv)
{
    if (N < 1 || root < 0 || root >= N)
        return -1;
    size_t es = oracle_dtype_size(t);
    for (int r = 0; r < N; r++)
        sent[r] = recv[r] = 0;
    int L = ceil_log2(N);
    for (int k = 0; k < L; k++) {
        for (int q = 0; q < (1 << k); q++) {
            int qd = q + (1 << k);
            if (qd >= N)
                continue;
            int src = (q + root) % N, dst = (qd + root) % N;
            memcpy(buf[dst], buf[src], T * es);
            sent[src] += T * es;
            recv[dst] += T * es;
        }
    }
    return 0;
}

/* Compressed broadcast (reading AB): the root's codes travel the binomial
 * tree above; every rank, the root included, stores the decoded buffer.
 * BFP only (bits 8 or 4); every edge carries the whole message. */
int oracle_broadcast_codec(int N, size_t T, void *const *buf, int t, int root, int bits,
                           uint64_t *sent, uint64_t *recv)
{
    if (N < 1 || root < 0 || root >= N || (bits != 8 && bits != 4))
        return -1;
    codec_t cd = {OR_CODEC_BFP, bits, 0.0, 0};
    for (int r = 0; r < N; r++)
        sent[r] = recv[r] = 0;
    float *x = xmalloc((T ? T : 1) * sizeof(float));
    for (size_t i = 0; i < T; i++)
        x[i] = load_as_f32(buf[root], i, t);
    message m;
    memset(&m, 0, sizeof m);
    msg_encode(&m, &cd, x, T);
    int L = ceil_log2(N);
    for (int k = 0; k < L; k++) {
        for (int q = 0; q < (1 << k); q++) {
            int qd = q + (1 << k);
            if (qd >= N)
                continue;
            sent[(q + root) % N] += m.bytes;
            recv[(qd + root) % N] += m.bytes;
        }
    }
    for (int r = 0; r < N; r++)
        for (size_t i = 0; i < T; i++)
            store_from_f32(buf[r], i, t, msg_value(&m, &cd, i));
    msg_free(&m);
    free(x);
    return 0;
}

/* Binomial reduce to rank 0: at level k every rank r with r mod 2^(k+1) = 0
 * and r + 2^k < N adds rank r+2^k's partial into its own (fp32); then the
 * binomial broadcast above from root 0.  In place, fp32 only. */
int oracle_tree_allreduce(int N, size_t T, float *const *buf, uint64_t *sent, uint64_t *recv)
{
    if (N < 1)
        return -1;
    for (int r = 0; r < N; r++)
        sent[r] = recv[r] = 0;
    int L = ceil_log2(N);
    for (int k = 0; k < L; k++) {
        int step = 1 << k;
        for (int r = 0; r < N; r += 2 * step) {
            int src = r + step;
            if (src >= N)
                continue;
            for (size_t i = 0; i < T; i++)
                buf[r][i] = buf[r][i] + buf[src][i];
            sent[src] += 4 * T;
            recv[r] += 4 * T;
        }
    }
    uint64_t *s2 = xcalloc((size_t)N, sizeof(uint64_t));
    uint64_t *r2 = xcalloc((size_t)N, sizeof(uint64_t));
    oracle_broadcast(N, T, (void *const *)buf, OR_F32, 0, s2, r2);
    for (int r = 0; r < N; r++) {
        sent[r] += s2[r];
        recv[r] += r2[r];
    }
    free(s2);
    free(r2);
    return 0;
}

/* ------------------------------------------------------------------ */
/* per-element dtype helpers for the Python side                       */
/* ------------------------------------------------------------------ */

void oracle_cast_to_f32(const void *x, size_t n, int t, float *out)
{
    for (size_t i = 0; i < n; i++)
        out[i] = load_as_f32(x, i, t);
}

void oracle_cast_from_f32(const float *x, size_t n, int t, void *out)
{
    for (size_t i = 0; i < n; i++)
        store_from_f32(out, i, t, x[i]);
}

/* ------------------------------------------------------------------------ */
/* codec statistics for the adaptive choice  [P4 §5 future directions:       */
/* watch sparsity and value distribution, switch compression accordingly]    */
/* ------------------------------------------------------------------------ */

/* Over the N input buffers of T elements (each cut into chunks of ceil(T/N)
 * and each chunk into 128-element BFP blocks from its start, as the ring's
 * first hop encodes them):
 *   stats[0] = N * T                      elements
 *   stats[1] = elements whose fp32 bits are not +0.0
 *   stats[2] = of those, the ones whose BFP4 code is 0 (|x| <= 2^(e-3))
 *   stats[3] = of those, the ones whose BFP8 code is 0 (|x| <= 2^(e-7))
 * A code rounds to 0 exactly when |x| * 2^(q-e) <= 1/2 (ties to even), with
 * e the block exponent and q = bits - 2. */
/* adds the statistics of buf[lo, lo + len), cut into blocks from lo */
static void stats_range(const void *buf, size_t lo, size_t len, int in_t, float *blk,
                        uint64_t *stats)
{
    for (size_t b = 0; b < len; b += OR_BFP_BLOCK) {
        const size_t m = len - b < OR_BFP_BLOCK ? len - b : OR_BFP_BLOCK;
        for (size_t i = 0; i < m; i++)
            blk[i] = load_as_f32(buf, lo + b + i, in_t);
        const int e = oracle_bfp_block_exponent(blk, m);
        for (size_t i = 0; i < m; i++) {
            uint32_t u;
            memcpy(&u, &blk[i], 4);
            stats[0]++;
            if (u == 0u)
                continue;
            stats[1]++;
            if (fabsf(blk[i]) <= ldexpf(1.0f, e - 3))
                stats[2]++;
            if (fabsf(blk[i]) <= ldexpf(1.0f, e - 7))
                stats[3]++;
        }
    }
}

int oracle_codec_stats_op(int op, int root, int N, size_t T, const void *const *in, int in_t,
                          uint64_t *stats);

int oracle_codec_stats(int N, size_t T, const void *const *in, int in_t, uint64_t *stats)
{
    return oracle_codec_stats_op(0, 0, N, T, in, in_t, stats);
}

/* The statistics of what an operation encodes (reading F4-op): op 0, the
 * allreduce's first hop: every chunk of every buffer; op 1, the compressed
 * allgather: chunk r of buffer r only (the rest is overwritten); op 2, the
 * compressed broadcast: the root's whole buffer, blocks from its start. */
int oracle_codec_stats_op(int op, int root, int N, size_t T, const void *const *in, int in_t,
                          uint64_t *stats)
{
    if (N < 1 || op < 0 || op > 2 || (op == 2 && (root < 0 || root >= N)))
        return -1;
    for (int k = 0; k < 4; k++)
        stats[k] = 0;
    float *blk = xmalloc(OR_BFP_BLOCK * sizeof(float));
    if (op == 2) {
        stats_range(in[root], 0, T, in_t, blk, stats);
    } else {
        for (int r = 0; r < N; r++)
            for (int c = 0; c < N; c++) {
                if (op == 1 && c != r)
                    continue;
                size_t lo, len;
                chunk_range(T, N, c, &lo, &len);
                stats_range(in[r], lo, len, in_t, blk, stats);
            }
    }
    free(blk);
    return 0;
}

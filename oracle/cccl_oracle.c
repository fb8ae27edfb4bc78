/*
 * cccl_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU definition of what the compressed
 * collective hot path computes.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  The GPU library shares no code,
 * header, table or helper with this file, and this file includes none of the
 * GPU library's headers.
 *
 * Source of the method: "CCCL: In-GPU Compression-Coupled Collective
 * Communication" (arXiv 2604.17172):
 *   - section 4.1 "Compression Principle": a bf16 value splits into sign,
 *     8-bit exponent and fraction; sign and fraction travel raw, only the
 *     skewed exponent is re-encoded;
 *   - section 4.3 "Localized Frequency Tables": every block derives its own
 *     exponent table from its own data, and every exponent symbol gets a
 *     fixed-length bit code;
 *   - section 4.4 "Reducing Global Memory Access": each block writes straight
 *     into its final place in one preallocated output;
 *   - section 5 "Handling data alignment": data outside whole chunks travels
 *     uncompressed;
 *   - section 5 (CopyReducePacks) and Figure 2: the reduce step of an
 *     allreduce is receive -> decompress -> reduce -> compress -> send.
 *
 * The pages fix no bitstream.  This file DEFINES one (every field, every
 * choice); the readings taken where the pages are silent are listed in the
 * design notes of the repository.  In short:
 *   - chunks of 4096 elements; the exponent table of a chunk is its exact
 *     minimum exponent `base` plus a code width k (0..7): element i stores
 *     code = e_i - base when that is below S = 2^k - 1, else the sentinel S
 *     and its raw exponent goes to an escape list (in bit-plane order: the
 *     order in which the elements' bits appear in the planes);
 *   - k minimises 512*k + pad16(#escapes); ties go to the smaller k; the
 *     chunk is stored raw when no k beats the 4096 bytes of exponents;
 *   - the last chunk, when shorter than 4096 elements, is stored raw;
 *   - the reduce adds in binary32, rank 0 first, and rounds once to bf16
 *     (round to nearest even; every NaN becomes 0x7FC0).
 *
 * Element types.  Section 4.1 states the split for floating-point values
 * and works it out for bf16 (8-bit exponent).  fp16 (5-bit exponent) and fp32
 * (8-bit exponent) take the same split, only the field widths change:
 *   - bf16: exponent = bits 7..14; the byte plane holds sign and the 7
 *     fraction bits;
 *   - fp16: exponent = bits 10..14; the byte plane holds the low 8 fraction
 *     bits, and three more bit-planes hold fraction bits 8 and 9 and the sign;
 *   - fp32: exponent = bits 23..30; the upper 16 bits are a bf16 pattern
 *     and go exactly as bf16 does (byte plane: sign and fraction bits 16..22),
 *     the lower 16 fraction bits follow the byte plane verbatim as 4096 u16.
 * The code width k runs 1..(exponent bits - 1); a chunk is stored raw when its
 * exponent part is not smaller than its exponents stored verbatim (512 bytes
 * per exponent bit).  The sum reduce accumulates in binary32 and rounds once
 * to the element type (fp32: no final rounding); the NaN of each type is
 * 0x7FC0, 0x7E00 or 0x7FC00000.
 *
 * Little endian throughout.  All stored integers are written byte by byte.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status codes (same numbering as the library's, defined independently) */
#define ORC_OK 0
#define ORC_ERR_INVALID_ARG 1
#define ORC_ERR_CAPACITY 2
#define ORC_ERR_CORRUPT 3

#define CHUNK_ELEMS 4096u
#define STREAM_HEADER_BYTES 64u
#define CHUNK_HEADER_BYTES 16u
#define STREAM_MAGIC 0x31424343u /* "CCB1" */
#define STREAM_VERSION 1u
#define STREAM_VERSION_WINDOW 2u /* the window-base variant: same layout, other table choice */
#define DTYPE_BF16 1u
#define DTYPE_FP16 2u
#define DTYPE_FP32 3u
#define MODE_PACKED 0u
#define MODE_RAW 1u
#define SM_PLANE_BYTES 4096u /* one sign+fraction byte per element */
#define BIT_PLANE_BYTES 512u /* one bit per element */

/* ------------------------------------------------------------------ */
/* little-endian byte access                                           */
/* ------------------------------------------------------------------ */
static void put_u16(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)((v >> 8) & 0xFF);
}
static void put_u32(uint8_t *p, uint32_t v)
{
    for (int b = 0; b < 4; b++)
        p[b] = (uint8_t)((v >> (8 * b)) & 0xFF);
}
static void put_u64(uint8_t *p, uint64_t v)
{
    for (int b = 0; b < 8; b++)
        p[b] = (uint8_t)((v >> (8 * b)) & 0xFF);
}
static uint32_t get_u16(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8);
}
static uint32_t get_u32(const uint8_t *p)
{
    uint32_t v = 0;
    for (int b = 3; b >= 0; b--)
        v = (v << 8) | p[b];
    return v;
}
static uint64_t get_u64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int b = 7; b >= 0; b--)
        v = (v << 8) | p[b];
    return v;
}

static size_t pad16(size_t x)
{
    return (x + 15) / 16 * 16;
}

/* ------------------------------------------------------------------ */
/* element types (section 4.1's split; see the notes at the top)       */
/* ------------------------------------------------------------------ */
typedef struct {
    unsigned code;       /* dtype field of the stream header */
    unsigned elem_bytes; /* 2 or 4 */
    unsigned exp_bits;   /* width of the exponent field */
    unsigned exp_shift;  /* lowest bit of the exponent field */
    size_t resid_bytes;  /* sign and fraction section of a packed chunk */
    uint32_t nan;        /* the one NaN a reduce writes */
} dtype_desc;

static const dtype_desc DT_BF16 = {DTYPE_BF16, 2, 8, 7, SM_PLANE_BYTES, 0x7FC0u};
static const dtype_desc DT_FP16 = {DTYPE_FP16, 2, 5, 10, SM_PLANE_BYTES + 3 * BIT_PLANE_BYTES, 0x7E00u};
static const dtype_desc DT_FP32 = {DTYPE_FP32, 4, 8, 23, SM_PLANE_BYTES + 2 * CHUNK_ELEMS, 0x7FC00000u};

static const dtype_desc *dtype_of(int code)
{
    if (code == DTYPE_BF16)
        return &DT_BF16;
    if (code == DTYPE_FP16)
        return &DT_FP16;
    if (code == DTYPE_FP32)
        return &DT_FP32;
    return NULL;
}

/* element i of a host array of the type, as its bit pattern */
static uint32_t elem(const dtype_desc *dt, const void *x, size_t i)
{
    if (dt->elem_bytes == 2)
        return ((const uint16_t *)x)[i];
    return ((const uint32_t *)x)[i];
}
static void set_elem(const dtype_desc *dt, void *x, size_t i, uint32_t v)
{
    if (dt->elem_bytes == 2)
        ((uint16_t *)x)[i] = (uint16_t)v;
    else
        ((uint32_t *)x)[i] = v;
}

/* number of exponent symbols, 2^exp_bits */
static unsigned n_symbols(const dtype_desc *dt)
{
    return 1u << dt->exp_bits;
}
/* largest code width: a width of exp_bits never beats the raw exponents */
static unsigned max_width(const dtype_desc *dt)
{
    return dt->exp_bits - 1;
}
/* a chunk's exponents stored verbatim, exp_bits bits per element; the packed
 * exponent part (planes + escapes) must be smaller than this */
static size_t raw_exponent_bytes(const dtype_desc *dt)
{
    return (size_t)BIT_PLANE_BYTES * dt->exp_bits;
}

/* ------------------------------------------------------------------ */
/* stream geometry                                                     */
/* ------------------------------------------------------------------ */
size_t oracle_n_chunks(size_t n)
{
    return (n + CHUNK_ELEMS - 1) / CHUNK_ELEMS;
}

/* number of elements in chunk c of an n-element buffer */
static size_t chunk_len(size_t n, size_t c)
{
    size_t start = c * CHUNK_ELEMS;
    size_t left = n - start;
    return left < CHUNK_ELEMS ? left : CHUNK_ELEMS;
}

/* byte offset of the first chunk: stream header, then the offset table
 * (one u64 per chunk) padded to 16 bytes */
size_t oracle_data_start(size_t n)
{
    return STREAM_HEADER_BYTES + pad16(8 * oracle_n_chunks(n));
}

/* size of a raw chunk of n_c elements, header included */
static size_t raw_chunk_bytes(const dtype_desc *dt, size_t n_c)
{
    return CHUNK_HEADER_BYTES + pad16(dt->elem_bytes * n_c);
}

/* size of a packed chunk, header included */
static size_t packed_chunk_bytes(const dtype_desc *dt, unsigned k, size_t n_esc)
{
    return CHUNK_HEADER_BYTES + dt->resid_bytes + (size_t)BIT_PLANE_BYTES * k + pad16(n_esc);
}

/* Largest stream n elements can produce: every chunk raw.  A packed chunk is
 * chosen only when it is strictly smaller than the raw one. */
static size_t compress_bound(const dtype_desc *dt, size_t n)
{
    size_t bytes = oracle_data_start(n);
    for (size_t c = 0; c < oracle_n_chunks(n); c++)
        bytes += raw_chunk_bytes(dt, chunk_len(n, c));
    return bytes;
}
size_t oracle_compress_bound(size_t n)
{
    return compress_bound(&DT_BF16, n);
}
/* 0 for an unknown dtype */
size_t oracle_compress_bound_typed(int dtype, size_t n)
{
    const dtype_desc *dt = dtype_of(dtype);
    return dt ? compress_bound(dt, n) : 0;
}

/* ------------------------------------------------------------------ */
/* splitting an element (section 4.1)                                  */
/* ------------------------------------------------------------------ */
static unsigned exponent_of(const dtype_desc *dt, uint32_t v)
{
    return (v >> dt->exp_shift) & (n_symbols(dt) - 1);
}
/* bf16: sign bit moved to bit 7, the 7 fraction bits kept in bits 0..6 */
static unsigned sign_fraction_of(uint16_t b)
{
    return ((b >> 8) & 0x80u) | (b & 0x7Fu);
}
static uint16_t join_bf16(unsigned sign_fraction, unsigned exponent)
{
    return (uint16_t)(((sign_fraction & 0x80u) << 8) | ((exponent & 0xFFu) << 7) | (sign_fraction & 0x7Fu));
}
/* fp16: the bits of an element held by its three residual bit-planes */
static const unsigned FP16_PLANE_BITS[3] = {8, 9, 15};

/* the byte-plane byte of an element */
static unsigned plane_byte_of(const dtype_desc *dt, uint32_t v)
{
    if (dt->code == DTYPE_FP16)
        return v & 0xFFu; /* fraction bits 0..7 */
    if (dt->code == DTYPE_FP32)
        return sign_fraction_of((uint16_t)(v >> 16)); /* the upper half's bf16 byte */
    return sign_fraction_of((uint16_t)v);
}

/* Where bit p of the code of element i sits inside bit-plane p: word index
 * (0..127, u32 little-endian words) and bit index (0..31).
 * With j = i / 256, l = (i / 8) % 32, s = i % 8:
 *   word = (j / 4) * 32 + l
 *   bit  = 8 * (s % 4) + 2 * (j % 4) + s / 4
 * This is a fixed permutation of the 4096 elements; it is this format's own
 * choice (the pages fix no bit order). */
void oracle_plane_position(unsigned i, unsigned *word, unsigned *bit)
{
    unsigned j = i / 256, l = (i / 8) % 32, s = i % 8;
    *word = (j / 4) * 32 + l;
    *bit = 8 * (s % 4) + 2 * (j % 4) + s / 4;
}

/* The element at bit `bit` of plane word `word` (inverse of the above):
 * with q = word / 32, l = word % 32, b = bit / 8, m = bit % 8:
 *   i = 256 * (4 q + m / 2) + 8 l + 4 (m % 2) + b */
unsigned oracle_plane_element(unsigned word, unsigned bit)
{
    unsigned q = word / 32, l = word % 32, b = bit / 8, m = bit % 8;
    return 256 * (4 * q + m / 2) + 8 * l + 4 * (m % 2) + b;
}

/* set / read element i's bit in the 512-byte bit-plane `plane` */
static void set_plane_bit(uint8_t *plane, unsigned i)
{
    unsigned word, bit;
    oracle_plane_position(i, &word, &bit);
    plane[4 * (size_t)word + bit / 8] = (uint8_t)(plane[4 * (size_t)word + bit / 8] | (1u << (bit % 8)));
}
static unsigned plane_bit(const uint8_t *plane, unsigned i)
{
    unsigned word, bit;
    oracle_plane_position(i, &word, &bit);
    return (plane[4 * (size_t)word + bit / 8] >> (bit % 8)) & 1u;
}

/* Sign and fraction of the n_c elements (everything but the exponent),
 * verbatim: the byte plane, then fp16's three bit-planes or fp32's lower
 * halves. */
static void write_residual(const dtype_desc *dt, const void *x, size_t n_c, uint8_t *body)
{
    for (size_t i = 0; i < n_c; i++)
        body[i] = (uint8_t)plane_byte_of(dt, elem(dt, x, i));
    if (dt->code == DTYPE_FP16) {
        for (unsigned i = 0; i < n_c; i++)
            for (unsigned t = 0; t < 3; t++)
                if ((elem(dt, x, i) >> FP16_PLANE_BITS[t]) & 1u)
                    set_plane_bit(body + SM_PLANE_BYTES + (size_t)BIT_PLANE_BYTES * t, i);
    } else if (dt->code == DTYPE_FP32) {
        for (size_t i = 0; i < n_c; i++)
            put_u16(body + SM_PLANE_BYTES + 2 * i, elem(dt, x, i) & 0xFFFFu);
    }
}

/* element i of a packed chunk from its residual and its exponent e */
static uint32_t join_elem(const dtype_desc *dt, const uint8_t *body, unsigned i, unsigned e)
{
    if (dt->code == DTYPE_FP16) {
        uint32_t v = body[i] | (e << 10);
        for (unsigned t = 0; t < 3; t++)
            v |= plane_bit(body + SM_PLANE_BYTES + (size_t)BIT_PLANE_BYTES * t, i) << FP16_PLANE_BITS[t];
        return v;
    }
    if (dt->code == DTYPE_FP32)
        return ((uint32_t)join_bf16(body[i], e) << 16) | get_u16(body + SM_PLANE_BYTES + 2 * (size_t)i);
    return join_bf16(body[i], e);
}

/* ------------------------------------------------------------------ */
/* encoding choice of one full chunk (section 4.3)                     */
/* ------------------------------------------------------------------ */
typedef struct {
    unsigned raw;   /* 1: stored raw */
    unsigned k;     /* code width, 0..max_width */
    unsigned base;  /* minimum exponent of the chunk */
    size_t n_esc;   /* escapes at width k */
    size_t bytes;   /* chunk size, header included */
} chunk_choice;

/* Count of elements whose exponent offset from base is >= threshold. */
static size_t count_at_or_above(const dtype_desc *dt, const void *x, size_t n_c, unsigned base, unsigned threshold)
{
    size_t count = 0;
    for (size_t i = 0; i < n_c; i++)
        if (exponent_of(dt, elem(dt, x, i)) - base >= threshold)
            count++;
    return count;
}

static chunk_choice choose_encoding(const dtype_desc *dt, const void *x, size_t n_c)
{
    chunk_choice best;
    best.raw = 1;
    best.k = 0;
    best.base = 0;
    best.n_esc = 0;
    best.bytes = raw_chunk_bytes(dt, n_c);
    if (n_c != CHUNK_ELEMS) /* a partial chunk travels raw (section 5) */
        return best;

    unsigned emin = n_symbols(dt) - 1, emax = 0;
    for (size_t i = 0; i < n_c; i++) {
        unsigned e = exponent_of(dt, elem(dt, x, i));
        if (e < emin)
            emin = e;
        if (e > emax)
            emax = e;
    }

    /* size of the exponent part of a packed chunk: k bit-planes + escapes */
    int have = 0;
    unsigned best_k = 0;
    size_t best_size = 0, best_esc = 0;
    if (emax == emin) { /* one symbol: width 0, no planes, no escapes */
        have = 1;
        best_k = 0;
        best_size = 0;
        best_esc = 0;
    } else {
        for (unsigned k = 1; k <= max_width(dt); k++) {
            unsigned sentinel = (1u << k) - 1;
            size_t n_esc = count_at_or_above(dt, x, n_c, emin, sentinel);
            size_t size = (size_t)BIT_PLANE_BYTES * k + pad16(n_esc);
            if (!have || size < best_size) { /* strict: ties keep the smaller k */
                have = 1;
                best_k = k;
                best_size = size;
                best_esc = n_esc;
            }
        }
    }
    if (best_size >= raw_exponent_bytes(dt)) /* no gain over the verbatim exponents: raw (ties too) */
        return best;
    best.raw = 0;
    best.k = best_k;
    best.base = emin;
    best.n_esc = best_esc;
    best.bytes = packed_chunk_bytes(dt, best_k, best_esc);
    return best;
}

/* Window-base variant (stream version 2).  The chunk's table is again a
 * fixed code width k and a base, but the base is the start of the window of
 * S = 2^k - 1 exponents [base, base + S - 1] that leaves the fewest
 * escapes: every exponent outside the window, below it included, is an
 * escape.  This is section 4.3's per-block frequency table taken at its
 * word: the codes go to the most frequent contiguous run of exponent
 * symbols, so that rare low outliers (zeros, subnormals, tiny magnitudes)
 * no longer stretch the range.  Ties: the smaller k, then the smaller base;
 * raw when no k beats the verbatim exponents (ties too); k = 0 when all
 * exponents are equal.  escapes(k, b) = #(e < b) + #(e >= b + S), from the
 * exponent histogram and its prefix sums. */
static chunk_choice choose_encoding_window(const dtype_desc *dt, const void *x, size_t n_c)
{
    chunk_choice best;
    best.raw = 1;
    best.k = 0;
    best.base = 0;
    best.n_esc = 0;
    best.bytes = raw_chunk_bytes(dt, n_c);
    if (n_c != CHUNK_ELEMS)
        return best;

    const unsigned n_sym = n_symbols(dt);
    size_t hist[256] = {0};
    unsigned emin = n_sym - 1, emax = 0;
    for (size_t i = 0; i < n_c; i++) {
        unsigned e = exponent_of(dt, elem(dt, x, i));
        hist[e]++;
        if (e < emin)
            emin = e;
        if (e > emax)
            emax = e;
    }
    size_t below[257]; /* below[v] = number of exponents < v */
    below[0] = 0;
    for (unsigned v = 0; v < n_sym; v++)
        below[v + 1] = below[v] + hist[v];

    int have = 0;
    unsigned best_k = 0, best_base = emin;
    size_t best_size = 0, best_esc = 0;
    if (emax == emin) {
        have = 1;
    } else {
        for (unsigned k = 1; k <= max_width(dt); k++) {
            unsigned S = (1u << k) - 1;
            size_t k_esc = 0;
            unsigned k_base = 0;
            for (unsigned b = 0; b < n_sym; b++) {
                unsigned top = b + S < n_sym ? b + S : n_sym; /* first exponent above the window */
                size_t n_esc = below[b] + (n_c - below[top]);
                if (b == 0 || n_esc < k_esc) { /* strict: ties keep the smaller base */
                    k_esc = n_esc;
                    k_base = b;
                }
            }
            size_t size = (size_t)BIT_PLANE_BYTES * k + pad16(k_esc);
            if (!have || size < best_size) {
                have = 1;
                best_k = k;
                best_base = k_base;
                best_size = size;
                best_esc = k_esc;
            }
        }
    }
    if (best_size >= raw_exponent_bytes(dt))
        return best;
    best.raw = 0;
    best.k = best_k;
    best.base = best_base;
    best.n_esc = best_esc;
    best.bytes = packed_chunk_bytes(dt, best_k, best_esc);
    return best;
}

/* Encoding statistics of one chunk without writing it (for tests). */
int oracle_chunk_choice_typed(int dtype, const void *x, size_t n_c, unsigned *raw, unsigned *k, unsigned *base,
                              size_t *n_esc, size_t *bytes)
{
    const dtype_desc *dt = dtype_of(dtype);
    if (dt == NULL || n_c == 0 || n_c > CHUNK_ELEMS)
        return ORC_ERR_INVALID_ARG;
    chunk_choice ch = choose_encoding(dt, x, n_c);
    *raw = ch.raw;
    *k = ch.k;
    *base = ch.base;
    *n_esc = ch.n_esc;
    *bytes = ch.bytes;
    return ORC_OK;
}
int oracle_chunk_choice(const uint16_t *x, size_t n_c, unsigned *raw, unsigned *k, unsigned *base, size_t *n_esc,
                        size_t *bytes)
{
    return oracle_chunk_choice_typed(DTYPE_BF16, x, n_c, raw, k, base, n_esc, bytes);
}

/* ------------------------------------------------------------------ */
/* chunk encoder                                                       */
/* ------------------------------------------------------------------ */
/* Writes one chunk (header + body + zero padding) at out; out must hold
 * ch.bytes bytes.  Returns the number of bytes written. */
static size_t write_chunk(const dtype_desc *dt, const void *x, size_t n_c, chunk_choice ch, uint8_t *out)
{
    memset(out, 0, ch.bytes);
    out[0] = (uint8_t)(ch.raw ? MODE_RAW : MODE_PACKED);
    out[1] = (uint8_t)ch.k;
    out[2] = (uint8_t)ch.base;
    out[3] = 0;
    put_u16(out + 4, (uint32_t)n_c);
    put_u16(out + 6, (uint32_t)ch.n_esc);
    put_u32(out + 8, (uint32_t)ch.bytes);
    put_u32(out + 12, 0);
    uint8_t *body = out + CHUNK_HEADER_BYTES;

    if (ch.raw) {
        for (size_t i = 0; i < n_c; i++) {
            if (dt->elem_bytes == 2)
                put_u16(body + 2 * i, elem(dt, x, i));
            else
                put_u32(body + 4 * i, elem(dt, x, i));
        }
        return ch.bytes;
    }

    /* sign and fraction */
    write_residual(dt, x, n_c, body);

    /* bit-planes */
    uint8_t *planes = body + dt->resid_bytes;
    uint8_t *escapes = planes + (size_t)BIT_PLANE_BYTES * ch.k;
    if (ch.k > 0) {
        unsigned sentinel = (1u << ch.k) - 1;
        for (unsigned i = 0; i < n_c; i++) {
            unsigned code = exponent_of(dt, elem(dt, x, i)) - ch.base;
            if (code >= sentinel)
                code = sentinel;
            for (unsigned p = 0; p < ch.k; p++)
                if ((code >> p) & 1u)
                    set_plane_bit(planes + (size_t)BIT_PLANE_BYTES * p, i);
        }
        /* escapes: raw exponents of the elements whose code is the sentinel,
         * in bit-plane order (word by word, bit by bit) */
        unsigned element_at[CHUNK_ELEMS];
        for (unsigned pos = 0; pos < CHUNK_ELEMS; pos++)
            element_at[pos] = CHUNK_ELEMS; /* none: only if the layout were not a permutation */
        for (unsigned i = 0; i < n_c; i++) {
            unsigned word, bit;
            oracle_plane_position(i, &word, &bit);
            if (word < 128 && bit < 32)
                element_at[32 * word + bit] = i;
        }
        size_t n_esc = 0;
        for (unsigned pos = 0; pos < CHUNK_ELEMS; pos++) {
            if (element_at[pos] >= n_c)
                continue;
            unsigned e = exponent_of(dt, elem(dt, x, element_at[pos]));
            if (e - ch.base >= sentinel)
                escapes[n_esc++] = (uint8_t)e;
        }
        (void)n_esc; /* equals ch.n_esc by construction of the count */
    }
    return ch.bytes;
}

/* One chunk on its own, header included (for sampled checks of big streams).
 * out must hold 16 + 4096 * element bytes. */
int oracle_encode_chunk_typed(int dtype, const void *x, size_t n_c, uint8_t *out, size_t *bytes)
{
    const dtype_desc *dt = dtype_of(dtype);
    if (dt == NULL || n_c == 0 || n_c > CHUNK_ELEMS)
        return ORC_ERR_INVALID_ARG;
    chunk_choice ch = choose_encoding(dt, x, n_c);
    *bytes = write_chunk(dt, x, n_c, ch, out);
    return ORC_OK;
}
int oracle_encode_chunk(const uint16_t *x, size_t n_c, uint8_t *out, size_t *bytes)
{
    return oracle_encode_chunk_typed(DTYPE_BF16, x, n_c, out, bytes);
}

/* ------------------------------------------------------------------ */
/* stream encoder                                                      */
/* ------------------------------------------------------------------ */
static int compress_stream(const dtype_desc *dt, const void *x, size_t n, uint8_t *out, size_t capacity,
                           size_t *out_bytes, int window)
{
    if (n == 0 || x == NULL || out == NULL)
        return ORC_ERR_INVALID_ARG;
    size_t n_chunks = oracle_n_chunks(n);
    size_t start = oracle_data_start(n);
    if (capacity < start)
        return ORC_ERR_CAPACITY;
    const uint8_t *xb = (const uint8_t *)x;

    /* placement: each chunk starts where the previous one ended */
    size_t pos = start;
    memset(out, 0, start);
    for (size_t c = 0; c < n_chunks; c++) {
        size_t n_c = chunk_len(n, c);
        const void *xc = xb + c * CHUNK_ELEMS * dt->elem_bytes;
        chunk_choice ch = window ? choose_encoding_window(dt, xc, n_c) : choose_encoding(dt, xc, n_c);
        if (pos + ch.bytes > capacity)
            return ORC_ERR_CAPACITY;
        put_u64(out + STREAM_HEADER_BYTES + 8 * c, pos);
        write_chunk(dt, xc, n_c, ch, out + pos);
        pos += ch.bytes;
    }

    put_u32(out + 0, STREAM_MAGIC);
    put_u16(out + 4, window ? STREAM_VERSION_WINDOW : STREAM_VERSION);
    put_u16(out + 6, dt->code);
    put_u32(out + 8, CHUNK_ELEMS);
    put_u32(out + 12, 0);
    put_u64(out + 16, n);
    put_u64(out + 24, n_chunks);
    put_u64(out + 32, pos);
    /* bytes 40..63 stay zero */
    *out_bytes = pos;
    return ORC_OK;
}

int oracle_compress(const uint16_t *x, size_t n, uint8_t *out, size_t capacity, size_t *out_bytes)
{
    return compress_stream(&DT_BF16, x, n, out, capacity, out_bytes, 0);
}

/* The window-base variant: the same stream layout, version 2. */
int oracle_compress_window(const uint16_t *x, size_t n, uint8_t *out, size_t capacity, size_t *out_bytes)
{
    return compress_stream(&DT_BF16, x, n, out, capacity, out_bytes, 1);
}

/* Any element type; window selects the window-base variant. */
int oracle_compress_typed(int dtype, const void *x, size_t n, uint8_t *out, size_t capacity, size_t *out_bytes,
                          int window)
{
    const dtype_desc *dt = dtype_of(dtype);
    if (dt == NULL)
        return ORC_ERR_INVALID_ARG;
    return compress_stream(dt, x, n, out, capacity, out_bytes, window != 0);
}

/* ------------------------------------------------------------------ */
/* stream decoder                                                      */
/* ------------------------------------------------------------------ */
/* Decodes one chunk of n_c elements from `chunk` (chunk_size bytes) into
 * elements 0 .. n_c - 1 of x. */
static int read_chunk(const dtype_desc *dt, const uint8_t *chunk, size_t chunk_size, size_t n_c, void *x)
{
    if (chunk_size < CHUNK_HEADER_BYTES)
        return ORC_ERR_CORRUPT;
    unsigned mode = chunk[0], k = chunk[1], base = chunk[2];
    size_t stored_n = get_u16(chunk + 4), n_esc = get_u16(chunk + 6);
    size_t bytes = get_u32(chunk + 8);
    if (bytes != chunk_size || stored_n != n_c)
        return ORC_ERR_CORRUPT;
    const uint8_t *body = chunk + CHUNK_HEADER_BYTES;

    if (mode == MODE_RAW) {
        if (k != 0 || base != 0 || n_esc != 0 || bytes != raw_chunk_bytes(dt, n_c))
            return ORC_ERR_CORRUPT;
        for (size_t i = 0; i < n_c; i++)
            set_elem(dt, x, i, dt->elem_bytes == 2 ? get_u16(body + 2 * i) : get_u32(body + 4 * i));
        return ORC_OK;
    }
    if (mode != MODE_PACKED || n_c != CHUNK_ELEMS || k > max_width(dt) || base >= n_symbols(dt))
        return ORC_ERR_CORRUPT;
    if (k == 0 && n_esc != 0)
        return ORC_ERR_CORRUPT;
    if (bytes != packed_chunk_bytes(dt, k, n_esc))
        return ORC_ERR_CORRUPT;
    /* a chunk is packed only when that beats its raw form, so a packed
     * chunk is never as large as a raw one */
    if ((size_t)BIT_PLANE_BYTES * k + pad16(n_esc) >= raw_exponent_bytes(dt))
        return ORC_ERR_CORRUPT;

    const uint8_t *planes = body + dt->resid_bytes;
    const uint8_t *escapes = planes + (size_t)BIT_PLANE_BYTES * k;
    unsigned sentinel = (1u << k) - 1;
    size_t used = 0;
    /* visit the elements in bit-plane order, the order of the escape list */
    for (unsigned pos = 0; pos < CHUNK_ELEMS; pos++) {
        unsigned word = pos / 32, bit = pos % 32, code = 0;
        for (unsigned p = 0; p < k; p++) {
            uint8_t byte = planes[(size_t)BIT_PLANE_BYTES * p + 4 * (size_t)word + bit / 8];
            code |= ((byte >> (bit % 8)) & 1u) << p;
        }
        unsigned e;
        if (k > 0 && code == sentinel) {
            if (used >= n_esc)
                return ORC_ERR_CORRUPT;
            e = escapes[used++];
        } else {
            e = base + code;
        }
        if (e >= n_symbols(dt))
            return ORC_ERR_CORRUPT;
        unsigned i = oracle_plane_element(word, bit);
        if (i >= n_c)
            return ORC_ERR_CORRUPT;
        set_elem(dt, x, i, join_elem(dt, body, i, e));
    }
    if (used != n_esc)
        return ORC_ERR_CORRUPT;
    return ORC_OK;
}

static int decompress_stream(const dtype_desc *dt, const uint8_t *s, size_t s_bytes, void *x, size_t n)
{
    if (s == NULL || x == NULL || n == 0)
        return ORC_ERR_INVALID_ARG;
    if (s_bytes < STREAM_HEADER_BYTES)
        return ORC_ERR_CORRUPT;
    size_t n_chunks = oracle_n_chunks(n);
    size_t start = oracle_data_start(n);
    if (get_u32(s + 0) != STREAM_MAGIC ||
        (get_u16(s + 4) != STREAM_VERSION && get_u16(s + 4) != STREAM_VERSION_WINDOW) ||
        get_u16(s + 6) != dt->code || get_u32(s + 8) != CHUNK_ELEMS || get_u64(s + 16) != n ||
        get_u64(s + 24) != n_chunks)
        return ORC_ERR_CORRUPT;
    size_t total = get_u64(s + 32);
    if (total > s_bytes || total < start)
        return ORC_ERR_CORRUPT;
    uint8_t *xb = (uint8_t *)x;
    for (size_t c = 0; c < n_chunks; c++) {
        size_t off = get_u64(s + STREAM_HEADER_BYTES + 8 * c);
        size_t end = (c + 1 < n_chunks) ? get_u64(s + STREAM_HEADER_BYTES + 8 * (c + 1)) : total;
        if (c == 0 && off != start)
            return ORC_ERR_CORRUPT;
        if (off % 16 != 0 || end <= off || end > total)
            return ORC_ERR_CORRUPT;
        int st = read_chunk(dt, s + off, end - off, chunk_len(n, c), xb + c * CHUNK_ELEMS * dt->elem_bytes);
        if (st != ORC_OK)
            return st;
    }
    return ORC_OK;
}

int oracle_decompress(const uint8_t *s, size_t s_bytes, uint16_t *x, size_t n)
{
    return decompress_stream(&DT_BF16, s, s_bytes, x, n);
}

int oracle_decompress_typed(int dtype, const uint8_t *s, size_t s_bytes, void *x, size_t n)
{
    const dtype_desc *dt = dtype_of(dtype);
    if (dt == NULL)
        return ORC_ERR_INVALID_ARG;
    return decompress_stream(dt, s, s_bytes, x, n);
}

/* ------------------------------------------------------------------ */
/* reduce (section 5, CopyReducePacks; Figure 2)                       */
/* ------------------------------------------------------------------ */
static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even; every NaN -> 0x7FC0 */
uint16_t oracle_round_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return 0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* IEEE binary16 -> binary32 (exact): (-1)^s * m * 2^-24 for e = 0,
 * (-1)^s * (1024 + m) * 2^(e - 25) for 0 < e < 31, Inf or NaN for e = 31. */
float oracle_fp16_to_float(uint16_t h)
{
    unsigned s = h >> 15, e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    float mag;
    if (e == 0)
        mag = ldexpf((float)m, -24);
    else if (e == 31)
        mag = m ? NAN : INFINITY;
    else
        mag = ldexpf((float)(1024u + m), (int)e - 25);
    return s ? -mag : mag;
}

/* binary32 -> IEEE binary16, round to nearest, ties to even, with
 * subnormal results and overflow to Inf; every NaN -> 0x7E00.  The value is
 * scaled to units of the binary16 quantum of its binade (2^-24 below 2^-14,
 * 2^(E - 10) in [2^E, 2^(E+1))); that count is rounded to an integer. */
uint16_t oracle_round_fp16(float f)
{
    if (isnan(f))
        return 0x7E00;
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    double a = fabs((double)f);
    if (a >= 65520.0) /* halfway between 65504 and 2^16 and above: Inf */
        return (uint16_t)(sign | 0x7C00u);
    int E;
    if (a < ldexp(1.0, -14)) {
        E = -14; /* subnormal range: quantum 2^-24 */
    } else {
        int ex;
        frexp(a, &ex); /* a = f * 2^ex, 0.5 <= f < 1 */
        E = ex - 1;    /* 2^E <= a < 2^(E+1) */
    }
    double units = ldexp(a, 10 - E); /* a / 2^(E - 10), exact */
    double n = floor(units);
    double frac = units - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    /* n * 2^(E - 10); for E = -14 the pattern is the subnormal count itself
     * (n = 1024 is the smallest normal), otherwise the implicit bit is 1024 */
    unsigned bits;
    if (a < ldexp(1.0, -14))
        bits = (unsigned)n;
    else if (n >= 2048.0)
        bits = ((unsigned)(E + 1 + 15) << 10); /* rounded up into the next binade */
    else
        bits = ((unsigned)(E + 15) << 10) | ((unsigned)n - 1024u);
    return (uint16_t)(sign | bits);
}

/* element -> binary32 (exact for all three types) */
static float to_binary32(const dtype_desc *dt, uint32_t v)
{
    if (dt->code == DTYPE_FP16)
        return oracle_fp16_to_float((uint16_t)v);
    if (dt->code == DTYPE_FP32) {
        float f;
        memcpy(&f, &v, sizeof f);
        return f;
    }
    return bf16_to_float((uint16_t)v);
}

/* binary32 -> element: one rounding to nearest even (fp32: none); every NaN
 * becomes the type's NaN */
static uint32_t from_binary32(const dtype_desc *dt, float f)
{
    if (dt->code == DTYPE_FP16)
        return oracle_round_fp16(f);
    if (dt->code == DTYPE_FP32) {
        uint32_t u;
        if (isnan(f))
            return dt->nan;
        memcpy(&u, &f, sizeof u);
        return u;
    }
    return oracle_round_bf16(f);
}

/* Element-wise sum of R vectors: binary32 accumulator starting from rank 0's
 * value, ranks added in order 1..R-1, one final rounding. */
static void sum_ranks(const dtype_desc *dt, const void *const *xs, int R, size_t n, void *out)
{
    for (size_t i = 0; i < n; i++) {
        float acc = to_binary32(dt, elem(dt, xs[0], i));
        for (int r = 1; r < R; r++)
            acc = acc + to_binary32(dt, elem(dt, xs[r], i));
        set_elem(dt, out, i, from_binary32(dt, acc));
    }
}
void oracle_sum_ranks(const uint16_t *const *xs, int R, size_t n, uint16_t *out)
{
    sum_ranks(&DT_BF16, (const void *const *)xs, R, n, out);
}
int oracle_sum_ranks_typed(int dtype, const void *const *xs, int R, size_t n, void *out)
{
    const dtype_desc *dt = dtype_of(dtype);
    if (dt == NULL || R < 1)
        return ORC_ERR_INVALID_ARG;
    sum_ranks(dt, xs, R, n, out);
    return ORC_OK;
}

/* Min and max reduce ops (section 5: CopyReducePacks performs "the required
 * collective operation (e.g., sum, min, max)").  Element-wise over the
 * ranks, exact (the result is one of the inputs, so there is no binary32
 * stage): a NaN in any rank gives the type's NaN; otherwise the smallest
 * (largest) value, with -0 below +0.  op: 1 min, 2 max. */
static uint32_t sign_bit(const dtype_desc *dt)
{
    return 1u << (8 * dt->elem_bytes - 1);
}
static int is_nan_elem(const dtype_desc *dt, uint32_t v) /* exponent all ones, fraction not zero */
{
    uint32_t inf = (n_symbols(dt) - 1) << dt->exp_shift;
    return (v & ~sign_bit(dt)) > inf;
}
static int less_elem(const dtype_desc *dt, uint32_t a, uint32_t b) /* a < b, neither NaN, -0 < +0 */
{
    uint32_t sb = sign_bit(dt);
    int na = (a & sb) != 0, nb = (b & sb) != 0;
    if (na != nb)
        return na; /* negative (including -0) below positive (including +0) */
    if (na)
        return (a & ~sb) > (b & ~sb); /* larger magnitude is smaller */
    return a < b;
}
static void minmax_ranks(const dtype_desc *dt, int op, const void *const *xs, int R, size_t n, void *out)
{
    for (size_t i = 0; i < n; i++) {
        uint32_t acc = elem(dt, xs[0], i);
        for (int r = 1; r < R; r++) {
            uint32_t b = elem(dt, xs[r], i);
            if (is_nan_elem(dt, acc) || is_nan_elem(dt, b))
                acc = dt->nan;
            else if (op == 1 ? less_elem(dt, b, acc) : less_elem(dt, acc, b))
                acc = b;
        }
        set_elem(dt, out, i, is_nan_elem(dt, acc) ? dt->nan : acc);
    }
}

/* The reduce step: rank 0 is the local uncompressed operand when `local` is
 * given (section 5, "Selective compression across collective stages": an
 * intermediate step merges the local operand with received compressed
 * partial results, and only the remote data are decompressed), the
 * n_streams compressed streams follow in order; the ranks are decompressed,
 * reduced element-wise with op (0 sum, 1 min, 2 max) and the result is
 * compressed (version 1). */
int oracle_reduce_typed(int dtype, int op, const void *local, const uint8_t *const *ins, const size_t *in_bytes,
                        int n_streams, size_t n, uint8_t *out, size_t capacity, size_t *out_bytes)
{
    const dtype_desc *dt = dtype_of(dtype);
    const int first = local != NULL ? 1 : 0;
    const int R = n_streams + first;
    if (dt == NULL || op < 0 || op > 2 || n_streams < 0 || R < 1 || R > 64 || n == 0 || out == NULL ||
        (n_streams > 0 && (ins == NULL || in_bytes == NULL)))
        return ORC_ERR_INVALID_ARG;
    const void **xs = (const void **)calloc((size_t)R, sizeof(void *));
    void *res = malloc(n * dt->elem_bytes);
    int st = (xs && res) ? ORC_OK : ORC_ERR_INVALID_ARG;
    if (xs && first)
        xs[0] = local;
    for (int r = first; r < R && st == ORC_OK; r++) {
        void *x = malloc(n * dt->elem_bytes);
        xs[r] = x;
        if (!x)
            st = ORC_ERR_INVALID_ARG;
        else
            st = decompress_stream(dt, ins[r - first], in_bytes[r - first], x, n);
    }
    if (st == ORC_OK) {
        if (op == 0)
            sum_ranks(dt, xs, R, n, res);
        else
            minmax_ranks(dt, op, xs, R, n, res);
        st = compress_stream(dt, res, n, out, capacity, out_bytes, 0);
    }
    if (xs)
        for (int r = first; r < R; r++)
            free((void *)xs[r]);
    free((void *)xs);
    free(res);
    return st;
}

/* bf16 sum of R streams */
int oracle_reduce(const uint8_t *const *ins, const size_t *in_bytes, int R, size_t n, uint8_t *out, size_t capacity,
                  size_t *out_bytes)
{
    if (R < 1 || ins == NULL)
        return ORC_ERR_INVALID_ARG;
    return oracle_reduce_typed(DTYPE_BF16, 0, NULL, ins, in_bytes, R, n, out, capacity, out_bytes);
}

/* bf16 sum of a local operand (rank 0) and n_remote streams (ranks 1..) */
int oracle_reduce_mixed(const uint16_t *local, const uint8_t *const *ins, const size_t *in_bytes, int n_remote,
                        size_t n, uint8_t *out, size_t capacity, size_t *out_bytes)
{
    if (local == NULL)
        return ORC_ERR_INVALID_ARG;
    return oracle_reduce_typed(DTYPE_BF16, 0, local, ins, in_bytes, n_remote, n, out, capacity, out_bytes);
}

/* bf16 reduce of R streams with op 0 (sum), 1 (min) or 2 (max) */
int oracle_reduce_op(const uint8_t *const *ins, const size_t *in_bytes, int R, size_t n, int op, uint8_t *out,
                     size_t capacity, size_t *out_bytes)
{
    if (R < 1 || ins == NULL)
        return ORC_ERR_INVALID_ARG;
    return oracle_reduce_typed(DTYPE_BF16, op, NULL, ins, in_bytes, R, n, out, capacity, out_bytes);
}

/* Paged payload (Figure 3 and section 6.2: KV-cache blocks sent between
 * prefill and decode instances).  The logical buffer is the concatenation of
 * n_blocks blocks of block_elems values, block i being pool block table[i];
 * block_elems is a multiple of 4096, so no chunk straddles two blocks.
 * compress_paged compresses the gathered buffer; decompress_paged writes the
 * decompressed buffer back into the pool blocks named by the table (which
 * must be distinct). */
int oracle_compress_paged(const uint16_t *pool, size_t block_elems, const int32_t *table, size_t n_blocks,
                          uint8_t *out, size_t capacity, size_t *out_bytes)
{
    if (pool == NULL || table == NULL || n_blocks == 0 || block_elems == 0 || block_elems % CHUNK_ELEMS != 0)
        return ORC_ERR_INVALID_ARG;
    const size_t n = n_blocks * block_elems;
    uint16_t *x = (uint16_t *)malloc(n * sizeof(uint16_t));
    if (!x)
        return ORC_ERR_INVALID_ARG;
    for (size_t i = 0; i < n_blocks; i++)
        memcpy(x + i * block_elems, pool + (size_t)table[i] * block_elems, block_elems * sizeof(uint16_t));
    int st = oracle_compress(x, n, out, capacity, out_bytes);
    free(x);
    return st;
}

int oracle_decompress_paged(const uint8_t *s, size_t s_bytes, uint16_t *pool, size_t block_elems, const int32_t *table,
                            size_t n_blocks)
{
    if (pool == NULL || table == NULL || n_blocks == 0 || block_elems == 0 || block_elems % CHUNK_ELEMS != 0)
        return ORC_ERR_INVALID_ARG;
    const size_t n = n_blocks * block_elems;
    uint16_t *x = (uint16_t *)malloc(n * sizeof(uint16_t));
    if (!x)
        return ORC_ERR_INVALID_ARG;
    int st = oracle_decompress(s, s_bytes, x, n);
    if (st == ORC_OK)
        for (size_t i = 0; i < n_blocks; i++)
            memcpy(pool + (size_t)table[i] * block_elems, x + i * block_elems, block_elems * sizeof(uint16_t));
    free(x);
    return st;
}

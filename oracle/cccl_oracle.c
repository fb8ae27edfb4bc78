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
 * Little endian throughout.  All stored integers are written byte by byte.
 */
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
static size_t raw_chunk_bytes(size_t n_c)
{
    return CHUNK_HEADER_BYTES + pad16(2 * n_c);
}

/* size of a packed chunk, header included */
static size_t packed_chunk_bytes(unsigned k, size_t n_esc)
{
    return CHUNK_HEADER_BYTES + SM_PLANE_BYTES + (size_t)BIT_PLANE_BYTES * k + pad16(n_esc);
}

/* Largest stream n elements can produce: every chunk raw.  A packed chunk is
 * chosen only when it is strictly smaller than the raw one. */
size_t oracle_compress_bound(size_t n)
{
    size_t bytes = oracle_data_start(n);
    for (size_t c = 0; c < oracle_n_chunks(n); c++)
        bytes += raw_chunk_bytes(chunk_len(n, c));
    return bytes;
}

/* ------------------------------------------------------------------ */
/* bf16 components (section 4.1)                                       */
/* ------------------------------------------------------------------ */
static unsigned exponent_of(uint16_t b)
{
    return (b >> 7) & 0xFFu;
}
/* sign bit moved to bit 7, the 7 fraction bits kept in bits 0..6 */
static unsigned sign_fraction_of(uint16_t b)
{
    return ((b >> 8) & 0x80u) | (b & 0x7Fu);
}
static uint16_t join_bf16(unsigned sign_fraction, unsigned exponent)
{
    return (uint16_t)(((sign_fraction & 0x80u) << 8) | ((exponent & 0xFFu) << 7) | (sign_fraction & 0x7Fu));
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

/* ------------------------------------------------------------------ */
/* encoding choice of one full chunk (section 4.3)                     */
/* ------------------------------------------------------------------ */
typedef struct {
    unsigned raw;   /* 1: stored raw */
    unsigned k;     /* code width, 0..7 */
    unsigned base;  /* minimum exponent of the chunk */
    size_t n_esc;   /* escapes at width k */
    size_t bytes;   /* chunk size, header included */
} chunk_choice;

/* Count of elements whose exponent offset from base is >= threshold. */
static size_t count_at_or_above(const uint16_t *x, size_t n_c, unsigned base, unsigned threshold)
{
    size_t count = 0;
    for (size_t i = 0; i < n_c; i++)
        if (exponent_of(x[i]) - base >= threshold)
            count++;
    return count;
}

static chunk_choice choose_encoding(const uint16_t *x, size_t n_c)
{
    chunk_choice best;
    best.raw = 1;
    best.k = 0;
    best.base = 0;
    best.n_esc = 0;
    best.bytes = raw_chunk_bytes(n_c);
    if (n_c != CHUNK_ELEMS) /* a partial chunk travels raw (section 5) */
        return best;

    unsigned emin = 255, emax = 0;
    for (size_t i = 0; i < n_c; i++) {
        unsigned e = exponent_of(x[i]);
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
        for (unsigned k = 1; k <= 7; k++) {
            unsigned sentinel = (1u << k) - 1;
            size_t n_esc = count_at_or_above(x, n_c, emin, sentinel);
            size_t size = (size_t)BIT_PLANE_BYTES * k + pad16(n_esc);
            if (!have || size < best_size) { /* strict: ties keep the smaller k */
                have = 1;
                best_k = k;
                best_size = size;
                best_esc = n_esc;
            }
        }
    }
    if (best_size >= SM_PLANE_BYTES) /* no gain over 8-bit exponents: raw (ties too) */
        return best;
    best.raw = 0;
    best.k = best_k;
    best.base = emin;
    best.n_esc = best_esc;
    best.bytes = packed_chunk_bytes(best_k, best_esc);
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
 * raw when no k beats the 4096 bytes of exponents (ties too); k = 0 when all
 * exponents are equal.  escapes(k, b) = #(e < b) + #(e >= b + S), from the
 * exponent histogram and its prefix sums. */
static chunk_choice choose_encoding_window(const uint16_t *x, size_t n_c)
{
    chunk_choice best;
    best.raw = 1;
    best.k = 0;
    best.base = 0;
    best.n_esc = 0;
    best.bytes = raw_chunk_bytes(n_c);
    if (n_c != CHUNK_ELEMS)
        return best;

    size_t hist[256] = {0};
    unsigned emin = 255, emax = 0;
    for (size_t i = 0; i < n_c; i++) {
        unsigned e = exponent_of(x[i]);
        hist[e]++;
        if (e < emin)
            emin = e;
        if (e > emax)
            emax = e;
    }
    size_t below[257]; /* below[v] = number of exponents < v */
    below[0] = 0;
    for (unsigned v = 0; v < 256; v++)
        below[v + 1] = below[v] + hist[v];

    int have = 0;
    unsigned best_k = 0, best_base = emin;
    size_t best_size = 0, best_esc = 0;
    if (emax == emin) {
        have = 1;
    } else {
        for (unsigned k = 1; k <= 7; k++) {
            unsigned S = (1u << k) - 1;
            size_t k_esc = 0;
            unsigned k_base = 0;
            for (unsigned b = 0; b < 256; b++) {
                unsigned top = b + S < 256 ? b + S : 256; /* first exponent above the window */
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
    if (best_size >= SM_PLANE_BYTES)
        return best;
    best.raw = 0;
    best.k = best_k;
    best.base = best_base;
    best.n_esc = best_esc;
    best.bytes = packed_chunk_bytes(best_k, best_esc);
    return best;
}

/* Encoding statistics of one chunk without writing it (for tests). */
int oracle_chunk_choice(const uint16_t *x, size_t n_c, unsigned *raw, unsigned *k, unsigned *base,
                        size_t *n_esc, size_t *bytes)
{
    if (n_c == 0 || n_c > CHUNK_ELEMS)
        return ORC_ERR_INVALID_ARG;
    chunk_choice ch = choose_encoding(x, n_c);
    *raw = ch.raw;
    *k = ch.k;
    *base = ch.base;
    *n_esc = ch.n_esc;
    *bytes = ch.bytes;
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* chunk encoder                                                       */
/* ------------------------------------------------------------------ */
/* Writes one chunk (header + body + zero padding) at out; out must hold
 * ch.bytes bytes.  Returns the number of bytes written. */
static size_t write_chunk(const uint16_t *x, size_t n_c, chunk_choice ch, uint8_t *out)
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
        for (size_t i = 0; i < n_c; i++)
            put_u16(body + 2 * i, x[i]);
        return ch.bytes;
    }

    /* sign+fraction plane */
    for (size_t i = 0; i < n_c; i++)
        body[i] = (uint8_t)sign_fraction_of(x[i]);

    /* bit-planes */
    uint8_t *planes = body + SM_PLANE_BYTES;
    uint8_t *escapes = planes + (size_t)BIT_PLANE_BYTES * ch.k;
    if (ch.k > 0) {
        unsigned sentinel = (1u << ch.k) - 1;
        for (unsigned i = 0; i < n_c; i++) {
            unsigned code = exponent_of(x[i]) - ch.base;
            if (code >= sentinel)
                code = sentinel;
            unsigned word, bit;
            oracle_plane_position(i, &word, &bit);
            for (unsigned p = 0; p < ch.k; p++) {
                if ((code >> p) & 1u) {
                    size_t byte = (size_t)BIT_PLANE_BYTES * p + 4 * (size_t)word + bit / 8;
                    planes[byte] = (uint8_t)(planes[byte] | (1u << (bit % 8)));
                }
            }
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
            unsigned e = exponent_of(x[element_at[pos]]);
            if (e - ch.base >= sentinel)
                escapes[n_esc++] = (uint8_t)e;
        }
        (void)n_esc; /* equals ch.n_esc by construction of the count */
    }
    return ch.bytes;
}

/* One chunk on its own, header included (for sampled checks of big streams).
 * out must hold 16 + 8192 bytes. */
int oracle_encode_chunk(const uint16_t *x, size_t n_c, uint8_t *out, size_t *bytes)
{
    if (n_c == 0 || n_c > CHUNK_ELEMS)
        return ORC_ERR_INVALID_ARG;
    chunk_choice ch = choose_encoding(x, n_c);
    *bytes = write_chunk(x, n_c, ch, out);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* stream encoder                                                      */
/* ------------------------------------------------------------------ */
static int compress_stream(const uint16_t *x, size_t n, uint8_t *out, size_t capacity, size_t *out_bytes,
                           int window)
{
    if (n == 0 || x == NULL || out == NULL)
        return ORC_ERR_INVALID_ARG;
    size_t n_chunks = oracle_n_chunks(n);
    size_t start = oracle_data_start(n);
    if (capacity < start)
        return ORC_ERR_CAPACITY;

    /* placement: each chunk starts where the previous one ended */
    size_t pos = start;
    memset(out, 0, start);
    for (size_t c = 0; c < n_chunks; c++) {
        size_t n_c = chunk_len(n, c);
        chunk_choice ch = window ? choose_encoding_window(x + c * CHUNK_ELEMS, n_c)
                                 : choose_encoding(x + c * CHUNK_ELEMS, n_c);
        if (pos + ch.bytes > capacity)
            return ORC_ERR_CAPACITY;
        put_u64(out + STREAM_HEADER_BYTES + 8 * c, pos);
        write_chunk(x + c * CHUNK_ELEMS, n_c, ch, out + pos);
        pos += ch.bytes;
    }

    put_u32(out + 0, STREAM_MAGIC);
    put_u16(out + 4, window ? STREAM_VERSION_WINDOW : STREAM_VERSION);
    put_u16(out + 6, DTYPE_BF16);
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
    return compress_stream(x, n, out, capacity, out_bytes, 0);
}

/* The window-base variant: the same stream layout, version 2. */
int oracle_compress_window(const uint16_t *x, size_t n, uint8_t *out, size_t capacity, size_t *out_bytes)
{
    return compress_stream(x, n, out, capacity, out_bytes, 1);
}

/* ------------------------------------------------------------------ */
/* stream decoder                                                      */
/* ------------------------------------------------------------------ */
/* Decodes one chunk of n_c elements from `chunk` (chunk_size bytes). */
static int read_chunk(const uint8_t *chunk, size_t chunk_size, size_t n_c, uint16_t *x)
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
        if (k != 0 || base != 0 || n_esc != 0 || bytes != raw_chunk_bytes(n_c))
            return ORC_ERR_CORRUPT;
        for (size_t i = 0; i < n_c; i++)
            x[i] = (uint16_t)get_u16(body + 2 * i);
        return ORC_OK;
    }
    if (mode != MODE_PACKED || n_c != CHUNK_ELEMS || k > 7)
        return ORC_ERR_CORRUPT;
    if (k == 0 && n_esc != 0)
        return ORC_ERR_CORRUPT;
    if (bytes != packed_chunk_bytes(k, n_esc))
        return ORC_ERR_CORRUPT;
    /* a chunk is packed only when that beats its raw form, so a packed
     * chunk is never as large as a raw one */
    if ((size_t)BIT_PLANE_BYTES * k + pad16(n_esc) >= SM_PLANE_BYTES)
        return ORC_ERR_CORRUPT;

    const uint8_t *planes = body + SM_PLANE_BYTES;
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
            if (e > 255)
                return ORC_ERR_CORRUPT;
        }
        unsigned i = oracle_plane_element(word, bit);
        if (i >= n_c)
            return ORC_ERR_CORRUPT;
        x[i] = join_bf16(body[i], e);
    }
    if (used != n_esc)
        return ORC_ERR_CORRUPT;
    return ORC_OK;
}

int oracle_decompress(const uint8_t *s, size_t s_bytes, uint16_t *x, size_t n)
{
    if (s == NULL || x == NULL || n == 0)
        return ORC_ERR_INVALID_ARG;
    if (s_bytes < STREAM_HEADER_BYTES)
        return ORC_ERR_CORRUPT;
    size_t n_chunks = oracle_n_chunks(n);
    size_t start = oracle_data_start(n);
    if (get_u32(s + 0) != STREAM_MAGIC || (get_u16(s + 4) != STREAM_VERSION && get_u16(s + 4) != STREAM_VERSION_WINDOW) || get_u16(s + 6) != DTYPE_BF16 ||
        get_u32(s + 8) != CHUNK_ELEMS || get_u64(s + 16) != n || get_u64(s + 24) != n_chunks)
        return ORC_ERR_CORRUPT;
    size_t total = get_u64(s + 32);
    if (total > s_bytes || total < start)
        return ORC_ERR_CORRUPT;
    for (size_t c = 0; c < n_chunks; c++) {
        size_t off = get_u64(s + STREAM_HEADER_BYTES + 8 * c);
        size_t end = (c + 1 < n_chunks) ? get_u64(s + STREAM_HEADER_BYTES + 8 * (c + 1)) : total;
        if (c == 0 && off != start)
            return ORC_ERR_CORRUPT;
        if (off % 16 != 0 || end <= off || end > total)
            return ORC_ERR_CORRUPT;
        int st = read_chunk(s + off, end - off, chunk_len(n, c), x + c * CHUNK_ELEMS);
        if (st != ORC_OK)
            return st;
    }
    return ORC_OK;
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

/* Element-wise sum of R bf16 vectors: binary32 accumulator starting from
 * rank 0's value, ranks added in order 1..R-1, one final rounding. */
void oracle_sum_ranks(const uint16_t *const *xs, int R, size_t n, uint16_t *out)
{
    for (size_t i = 0; i < n; i++) {
        float acc = bf16_to_float(xs[0][i]);
        for (int r = 1; r < R; r++)
            acc = acc + bf16_to_float(xs[r][i]);
        out[i] = oracle_round_bf16(acc);
    }
}

/* Decompress R streams, sum them as above, compress the sum. */
int oracle_reduce(const uint8_t *const *ins, const size_t *in_bytes, int R, size_t n, uint8_t *out, size_t capacity,
                  size_t *out_bytes)
{
    if (R < 1 || R > 64 || n == 0 || ins == NULL || in_bytes == NULL || out == NULL)
        return ORC_ERR_INVALID_ARG;
    uint16_t **xs = (uint16_t **)calloc((size_t)R, sizeof(uint16_t *));
    uint16_t *sum = (uint16_t *)malloc(n * sizeof(uint16_t));
    int st = (xs && sum) ? ORC_OK : ORC_ERR_INVALID_ARG;
    for (int r = 0; r < R && st == ORC_OK; r++) {
        xs[r] = (uint16_t *)malloc(n * sizeof(uint16_t));
        if (!xs[r])
            st = ORC_ERR_INVALID_ARG;
        else
            st = oracle_decompress(ins[r], in_bytes[r], xs[r], n);
    }
    if (st == ORC_OK) {
        oracle_sum_ranks((const uint16_t *const *)xs, R, n, sum);
        st = oracle_compress(sum, n, out, capacity, out_bytes);
    }
    if (xs)
        for (int r = 0; r < R; r++)
            free(xs[r]);
    free(xs);
    free(sum);
    return st;
}

/* Selective-compression reduce (section 5, "Selective compression across
 * collective stages"): an intermediate reduction step merges the local,
 * uncompressed operand with received compressed partial results; only the
 * remote data are decompressed.  The local operand is rank 0, the n_remote
 * streams are ranks 1..n_remote, summed and compressed as oracle_reduce. */
int oracle_reduce_mixed(const uint16_t *local, const uint8_t *const *ins, const size_t *in_bytes, int n_remote,
                        size_t n, uint8_t *out, size_t capacity, size_t *out_bytes)
{
    if (local == NULL || n_remote < 0 || n_remote > 63 || n == 0 || out == NULL ||
        (n_remote > 0 && (ins == NULL || in_bytes == NULL)))
        return ORC_ERR_INVALID_ARG;
    const int R = n_remote + 1;
    const uint16_t **xs = (const uint16_t **)calloc((size_t)R, sizeof(uint16_t *));
    uint16_t *sum = (uint16_t *)malloc(n * sizeof(uint16_t));
    int st = (xs && sum) ? ORC_OK : ORC_ERR_INVALID_ARG;
    if (xs)
        xs[0] = local;
    for (int r = 1; r < R && st == ORC_OK; r++) {
        uint16_t *x = (uint16_t *)malloc(n * sizeof(uint16_t));
        xs[r] = x;
        if (!x)
            st = ORC_ERR_INVALID_ARG;
        else
            st = oracle_decompress(ins[r - 1], in_bytes[r - 1], x, n);
    }
    if (st == ORC_OK) {
        oracle_sum_ranks(xs, R, n, sum);
        st = oracle_compress(sum, n, out, capacity, out_bytes);
    }
    if (xs)
        for (int r = 1; r < R; r++)
            free((void *)xs[r]);
    free((void *)xs);
    free(sum);
    return st;
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

/* Min and max reduce ops (section 5: CopyReducePacks performs "the required
 * collective operation (e.g., sum, min, max)").  Element-wise over the
 * ranks, exact (the result is one of the inputs, so there is no binary32
 * stage): a NaN in any rank gives 0x7FC0; otherwise the smallest (largest)
 * value, with -0 below +0.  op: 1 min, 2 max (0 is the sum of oracle_reduce). */
static int is_nan_bf16(uint16_t b)
{
    return (b & 0x7FFFu) > 0x7F80u;
}
static int less_bf16(uint16_t a, uint16_t b) /* a < b, neither NaN, -0 < +0 */
{
    int na = (a & 0x8000u) != 0, nb = (b & 0x8000u) != 0;
    if (na != nb)
        return na; /* negative (including -0) below positive (including +0) */
    if (na)
        return (a & 0x7FFFu) > (b & 0x7FFFu); /* larger magnitude is smaller */
    return a < b;
}

int oracle_reduce_op(const uint8_t *const *ins, const size_t *in_bytes, int R, size_t n, int op, uint8_t *out,
                     size_t capacity, size_t *out_bytes)
{
    if (op == 0)
        return oracle_reduce(ins, in_bytes, R, n, out, capacity, out_bytes);
    if ((op != 1 && op != 2) || R < 1 || R > 64 || n == 0 || ins == NULL || in_bytes == NULL || out == NULL)
        return ORC_ERR_INVALID_ARG;
    uint16_t *x = (uint16_t *)malloc(n * sizeof(uint16_t));
    uint16_t *acc = (uint16_t *)malloc(n * sizeof(uint16_t));
    int st = (x && acc) ? ORC_OK : ORC_ERR_INVALID_ARG;
    for (int r = 0; r < R && st == ORC_OK; r++) {
        st = oracle_decompress(ins[r], in_bytes[r], r == 0 ? acc : x, n);
        if (st != ORC_OK || r == 0)
            continue;
        for (size_t i = 0; i < n; i++) {
            uint16_t a = acc[i], b = x[i];
            if (is_nan_bf16(a) || is_nan_bf16(b))
                acc[i] = 0x7FC0;
            else if (op == 1 ? less_bf16(b, a) : less_bf16(a, b))
                acc[i] = b;
        }
    }
    if (st == ORC_OK) {
        for (size_t i = 0; i < n; i++)
            if (is_nan_bf16(acc[i]))
                acc[i] = 0x7FC0;
        st = oracle_compress(acc, n, out, capacity, out_bytes);
    }
    free(x);
    free(acc);
    return st;
}

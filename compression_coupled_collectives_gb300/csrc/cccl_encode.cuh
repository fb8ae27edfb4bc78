// cccl_encode.cuh -- encoding chunks staged in shared memory or held in
// registers (shared by the compress and fused-reduce kernels).
//
// Per chunk ("CCCL: In-GPU Compression-Coupled Collective Communication"):
//   section 4.1  split every value into its exponent and the rest (sign and
//                fraction, kept verbatim in the type's residual section);
//   section 4.3  the chunk's own table: base = minimum exponent, width k that
//                minimises 512 k + pad16(#escapes), fixed-length k-bit codes;
//   section 4.4  the chunk is written once, straight into its final place;
//   section 5    the partial last chunk is stored raw.
// Element types (bf16, fp16, fp32) and their residual sections: see the
// traits in cccl_device.cuh.
//
// Work split: a pair of warps encodes a chunk staged in shared memory, half
// the rows each (lane l owns elements 256 j + 8 l + s, i.e. bit-plane words
// 32 q + l); or a team of four warps encodes a chunk it holds in registers, a
// quarter per warp.
#pragma once

#include <type_traits>

#include "cccl_device.cuh"

namespace cccl {

struct StreamOut {
    uint8_t* out;        // stream base (16-byte aligned)
    uint64_t capacity;   // bytes writable at out (>= the compress bound)
    uint64_t* status;    // one placement word per group
    WsHeader* ws;
    uint64_t n_elems;
    uint64_t n_chunks;
    uint32_t version;    // stream header version: kVersion, or kVersionWindow
    uint32_t dtype;      // stream header element type (the trait's kCode)
};

// Encoding decision of one full chunk (warp-uniform).
struct ChunkPlan {
    uint32_t raw;    // 1: stored raw
    uint32_t k;      // code width
    uint32_t base;   // header base: minimum exponent (0 when raw)
    uint32_t n_esc;  // escapes at width k
    uint32_t bytes;  // chunk size, header included
};

// This lane's 4 pair-words of row j (elements 256 j + 8 l .. + 7) of a 16-bit
// type.
__device__ __forceinline__ uint4 lds_row(const uint8_t* chunk, uint32_t j, uint32_t lane) {
    return *reinterpret_cast<const uint4*>(chunk + 512 * j + 16 * lane);
}

// Sign+fraction bytes of 4 bf16 values held as two pair-words (section 4.1).
__device__ __forceinline__ uint32_t sign_fraction_quad(uint32_t A, uint32_t B) {
    const uint32_t lo = __byte_perm(A, B, 0x6420), hi = __byte_perm(A, B, 0x7531);
    return (lo & 0x7F7F7F7Fu) | (hi & 0x80808080u);
}
// Low bytes of 4 fp16 values (fraction bits 0..7).
__device__ __forceinline__ uint32_t low_byte_quad(uint32_t A, uint32_t B) { return __byte_perm(A, B, 0x6420); }

// Row j of this lane's 8 staged values: two exponent quads (for fp16 with the
// residual bits 5..7, see fp16_exponent_quad), and the running minimum and
// maximum of the exponents held in the high bytes of 16-bit lanes.
template <class D>
__device__ __forceinline__ void row_exponents(const uint8_t* chunk, int j, uint32_t lane, uint32_t& q0, uint32_t& q1,
                                              uint32_t& mn, uint32_t& mx) {
    if constexpr (D::kExpBits == 5) {
        const uint4 v = lds_row(chunk, j, lane);
        const uint32_t u0 = fp16_exponent_lanes(v.x), u1 = fp16_exponent_lanes(v.y);
        const uint32_t u2 = fp16_exponent_lanes(v.z), u3 = fp16_exponent_lanes(v.w);
        mn = vmin_u16x2(mn, vmin_u16x2(vmin_u16x2(u0, u1), vmin_u16x2(u2, u3)));
        mx = vmax_u16x2(mx, vmax_u16x2(vmax_u16x2(u0, u1), vmax_u16x2(u2, u3)));
        q0 = fp16_exponent_quad(v.x, v.y);
        q1 = fp16_exponent_quad(v.z, v.w);
    } else {
        uint32_t t0, t1, t2, t3;
        if constexpr (D::kElemBytes == 4) {  // the upper halves are bf16 patterns
            const uint8_t* row = chunk + 1024 * j + 32 * lane;
            const uint4 a = *reinterpret_cast<const uint4*>(row), b = *reinterpret_cast<const uint4*>(row + 16);
            t0 = upper_halves(a.x, a.y) << 1, t1 = upper_halves(a.z, a.w) << 1;
            t2 = upper_halves(b.x, b.y) << 1, t3 = upper_halves(b.z, b.w) << 1;
        } else {
            const uint4 v = lds_row(chunk, j, lane);
            t0 = v.x << 1, t1 = v.y << 1, t2 = v.z << 1, t3 = v.w << 1;
        }
        // doubling a pair-word puts each value's exponent in the high byte of
        // its 16-bit lane (a low value's sign lands in the high lane's low
        // byte, which cannot change its high byte)
        mn = vmin_u16x2(mn, vmin_u16x2(vmin_u16x2(t0, t1), vmin_u16x2(t2, t3)));
        mx = vmax_u16x2(mx, vmax_u16x2(vmax_u16x2(t0, t1), vmax_u16x2(t2, t3)));
        q0 = __byte_perm(t0, t1, 0x7531);
        q1 = __byte_perm(t2, t3, 0x7531);
    }
}

// Escape bits at width k (1..kExpBits-1) of one plane word from its planes:
// the offset is at least 2^k - 1 when a bit at or above k is set (the offset
// reaches 2^k) or when bits 0..k-1 are all set.
template <class D>
__device__ __forceinline__ uint32_t escape_word(const uint32_t* P, uint32_t k) {
    uint32_t lowAnd = 0xFFFFFFFFu, highOr = 0u;
#pragma unroll
    for (uint32_t p = 0; p < D::kExpBits; ++p) {
        if (p < k)
            lowAnd &= P[p];
        else
            highOr |= P[p];
    }
    return lowAnd | highOr;
}

// Escape counts of one plane word at every width: with low_k = AND of planes
// 0..k-1 and high_k = OR of planes k..kExpBits-1, the escapes at width k are
// exactly low_k | high_k (section 4.3's per-block table, exact).
template <class D>
__device__ __forceinline__ void add_escape_counts(const uint32_t* P, uint32_t* cnt) {
    constexpr int kTop = (int)D::kExpBits - 1;
    uint32_t high[8];
    high[kTop] = P[kTop];
#pragma unroll
    for (int k = kTop - 1; k >= 1; --k) high[k] = high[k + 1] | P[k];
    uint32_t low = P[0];
#pragma unroll
    for (int k = 1; k <= kTop; ++k) {
        cnt[k] += __popc(low | high[k]);
        if (k < kTop) low &= P[k];
    }
}

// Size of a packed full chunk, header included.
template <class D>
__host__ __device__ constexpr uint32_t packed_chunk_bytes(uint32_t k, uint32_t n_esc) {
    return (uint32_t)(16 + D::kResidBytes + kPlaneBytes * k + pad16(n_esc));
}

// ---------------------------------------------------------------------------
// Pair encoding: two warps encode one chunk staged in shared memory.  Warp h
// (0 or 1) of the pair owns plane words 32 q + l for q = 2 h, 2 h + 1 (lane
// l): rows 8 h .. 8 h + 7, elements 8 l .. 8 l + 7 of each.  The pair meets
// twice per chunk (exponent extremes; escape counts) at a named barrier of 64
// threads, through an exchange record in shared memory.
// ---------------------------------------------------------------------------
struct PairBarrier {
    uint32_t id;  // 1..15; barrier 0 is __syncthreads'
    __device__ void sync() const { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }
    __device__ bool any(bool p) const {
        uint32_t r;
        asm volatile(
            "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.or.pred po, %2, 64, pi; selp.u32 %0, 1, 0, po; }"
            : "=r"(r)
            : "r"((uint32_t)p), "r"(id)
            : "memory");
        return r != 0;
    }
};

struct PairXch {
    uint32_t mn[2], mx[2];  // per warp: smallest and largest exponent
    uint32_t cnt[2][8];     // per warp: escapes at width k (window variant: [h][0] the escapes at the
                            // chosen table, [h][1..4] the warp's best size, k, base, escapes)
};

// One warp's half of a chunk, kept in registers between sizing and writing:
// P[8 qq + p] is plane p of word 32 (2 h + qq) + l, i.e. bit p of the
// exponent offsets (e - base) of the 32 elements that word covers (bit
// 8 b + m: element 256 (4 q + m / 2) + 8 l + 4 (m % 2) + b).  For fp16,
// planes 5..7 hold fraction bit 8, fraction bit 9 and the sign.
struct HalfRegs {
    uint32_t P[16];
};

// Plan of one full chunk: as ChunkPlan, plus the escapes of the pair's
// first warp at the chosen table (where the second warp's escapes start).
struct PairPlan {
    ChunkPlan p;
    uint32_t esc_before;  // 0 for warp 0
};

// Phase A: exponent table and size of the full chunk staged at `chunk` (left
// untouched), leaving this warp's bit-planes of the exponent offsets in `r`.
// Both warps of the pair return the same plan (esc_before aside).
template <class D>
__device__ __forceinline__ PairPlan plan_chunk_pair(const uint8_t* chunk, HalfRegs& r, uint32_t h, PairXch& x,
                                                    const PairBarrier& bar) {
    constexpr uint32_t kTop = D::kExpBits - 1;
    const uint32_t lane = threadIdx.x & 31;
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) row_exponents<D>(chunk, 8 * h + jj, lane, r.P[2 * jj], r.P[2 * jj + 1], mn, mx);
    const uint32_t wmn = __reduce_min_sync(0xFFFFFFFFu, min((mn >> 8) & 0xFFu, mn >> 24));
    const uint32_t wmx = __reduce_max_sync(0xFFFFFFFFu, max((mx >> 8) & 0xFFu, mx >> 24));
    if (lane == 0) {
        x.mn[h] = wmn;
        x.mx[h] = wmx;
    }
    bar.sync();
    const uint32_t emin = min(x.mn[0], x.mn[1]), emax = max(x.mx[0], x.mx[1]);
    const uint32_t base4 = emin * 0x01010101u;
    uint32_t cnt[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // escapes at width k
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
        uint32_t* P = r.P + 8 * qq;
#pragma unroll
        for (int m = 0; m < 8; ++m) P[m] -= base4;  // no borrow: every exponent >= emin
        transpose8x8x4(P);                          // quads of offsets -> planes
        add_escape_counts<D>(P, cnt);
    }
#pragma unroll
    for (uint32_t k = 1; k <= kTop; ++k) {
        const uint32_t n = __reduce_add_sync(0xFFFFFFFFu, cnt[k]);
        if (lane == 0) x.cnt[h][k] = n;
    }
    bar.sync();
    PairPlan pp{{0u, 0u, emin, 0u, 0u}, 0u};
    ChunkPlan& pl = pp.p;
    uint32_t best = 0;
    if (emax > emin) {
        // lane k (1..kTop) sizes width k; the smallest (size, k) wins, so a
        // tie keeps the smaller width
        uint32_t n = 0, before = 0, key = 0xFFFFFFFFu;
        if (lane >= 1 && lane <= kTop) {
            const uint32_t c0 = x.cnt[0][lane];
            n = c0 + x.cnt[1][lane];
            before = h ? c0 : 0u;
            key = ((kPlaneBytes * lane + (uint32_t)pad16(n)) << 3) | lane;
        }
        key = __reduce_min_sync(0xFFFFFFFFu, key);
        pl.k = key & 7u;
        best = key >> 3;
        pl.n_esc = __shfl_sync(0xFFFFFFFFu, n, pl.k);
        pp.esc_before = __shfl_sync(0xFFFFFFFFu, before, pl.k);
    }
    pl.raw = best >= raw_exponent_bytes<D>() ? 1u : 0u;
    if (pl.raw) {
        pl.k = 0;
        pl.base = 0;
        pl.n_esc = 0;
        pp.esc_before = 0;
        pl.bytes = max_chunk_bytes<D>();
    } else {
        pl.bytes = packed_chunk_bytes<D>(pl.k, pl.n_esc);
    }
    return pp;
}

// Phase A of the window-base variant (stream version 2): for every width k
// the base is the start of the window of 2^k - 1 exponents with the fewest
// escapes (exponents outside it, below included), ties to the smaller base;
// then the smallest size wins, ties to the smaller k.  The pair shares one
// histogram and splits the widths between its warps.  `hist`: the pair's 264
// words of shared memory; `below`: this warp's own 264 words.  Leaves in `r`
// the bit-planes of the codes, escaped elements carrying all ones, which is
// what write_chunk_pair's escape test (low_k | high_k) and plane writes
// expect.
template <class D>
__device__ __forceinline__ PairPlan plan_chunk_pair_window(const uint8_t* chunk, HalfRegs& r, uint32_t h, PairXch& x,
                                                           uint32_t* hist, uint32_t* below_s,
                                                           const PairBarrier& bar) {
    constexpr uint32_t kExpMask4 = ((1u << D::kExpBits) - 1u) * 0x01010101u;  // the exponent bits of a quad
    const uint32_t lane = threadIdx.x & 31;
    *reinterpret_cast<uint4*>(hist + 128 * h + 4 * lane) = make_uint4(0u, 0u, 0u, 0u);  // this warp's half
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) row_exponents<D>(chunk, 8 * h + jj, lane, r.P[2 * jj], r.P[2 * jj + 1], mn, mx);
    const uint32_t wmn = __reduce_min_sync(0xFFFFFFFFu, min((mn >> 8) & 0xFFu, mn >> 24));
    const uint32_t wmx = __reduce_max_sync(0xFFFFFFFFu, max((mx >> 8) & 0xFFu, mx >> 24));
    if (lane == 0) {
        x.mn[h] = wmn;
        x.mx[h] = wmx;
    }
    bar.sync();  // the histogram is cleared, the extremes are in
    const uint32_t emin = min(x.mn[0], x.mn[1]), emax = max(x.mx[0], x.mx[1]);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const uint32_t q = r.P[m] & kExpMask4;
#pragma unroll
        for (int b = 0; b < 4; ++b) atomicAdd(hist + ((q >> (8 * b)) & 0xFFu), 1u);
    }
    bar.sync();  // the histogram is complete
    // below[v] = exponents smaller than v; lane l holds v = 8 l .. 8 l + 7
    const uint4 h0 = *reinterpret_cast<const uint4*>(hist + 8 * lane);
    const uint4 h1 = *reinterpret_cast<const uint4*>(hist + 8 * lane + 4);
    const uint32_t hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t below[8], run = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        below[i] = run;
        run += hv[i];
    }
    uint32_t incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= (uint32_t)d) incl += t;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) below[i] += incl - run;
    *reinterpret_cast<uint4*>(below_s + 8 * lane) = make_uint4(below[0], below[1], below[2], below[3]);
    *reinterpret_cast<uint4*>(below_s + 8 * lane + 4) = make_uint4(below[4], below[5], below[6], below[7]);
    if (lane == 31) below_s[256] = kChunkElems;
    __syncwarp();
    PairPlan pp{{0u, 0u, emin, 0u, 0u}, 0u};
    ChunkPlan& pl = pp.p;
    uint32_t best = 0;
    if (emax > emin) {
        // a window starting above the type's exponents escapes everything, so
        // scanning all 256 starts gives the same choice for narrower types.
        // Warp 0 sizes the widths 1..kSplit, warp 1 the rest; each keeps its
        // best (size, k, base, escapes) and the pair then takes the smaller
        // size, warp 0's on a tie (its widths are the smaller ones).
        constexpr uint32_t kSplit = (max_width<D>() + 1) / 2;
        const uint32_t k_lo = h == 0 ? 1u : kSplit + 1, k_hi = h == 0 ? kSplit : max_width<D>();
        best = 0xFFFFFFFFu;
        for (uint32_t k = k_lo; k <= k_hi; ++k) {
            const uint32_t S = (1u << k) - 1u;
            uint32_t key = 0xFFFFFFFFu;  // (escapes, base): fewest escapes, then the smallest base
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t b = 8 * lane + i, top = min(b + S, 256u);
                const uint32_t n = below[i] + (kChunkElems - below_s[top]);
                key = min(key, (n << 8) | b);
            }
            key = __reduce_min_sync(0xFFFFFFFFu, key);
            const uint32_t n = key >> 8, size = kPlaneBytes * k + (uint32_t)pad16(n);
            if (size < best) {  // ascending k: a tie keeps the smaller width
                best = size;
                pl.k = k;
                pl.base = key & 0xFFu;
                pl.n_esc = n;
            }
        }
        if (lane == 0) {
            x.cnt[h][1] = best;
            x.cnt[h][2] = pl.k;
            x.cnt[h][3] = pl.base;
            x.cnt[h][4] = pl.n_esc;
        }
        bar.sync();
        const uint32_t w = x.cnt[0][1] <= x.cnt[1][1] ? 0u : 1u;
        best = x.cnt[w][1];
        pl.k = x.cnt[w][2];
        pl.base = x.cnt[w][3];
        pl.n_esc = x.cnt[w][4];
    }
    pl.raw = best >= raw_exponent_bytes<D>() ? 1u : 0u;
    if (pl.raw) {
        pl.k = 0;
        pl.base = 0;
        pl.n_esc = 0;
        pl.bytes = max_chunk_bytes<D>();
        return pp;
    }
    pl.bytes = packed_chunk_bytes<D>(pl.k, pl.n_esc);
    // (fp16 goes on at k = 0 too: its residual planes 5..7 come from the
    // transposes below; the codes, all escapes at width 0, are not written)
    if (D::kExpBits != 5 && pl.k == 0) return pp;
    // codes: e - base inside the window, all ones outside (an escape).
    // Byte-wise e - base with no borrow between bytes, and the bytes where
    // e < base (the borrow out of each byte).
    const uint32_t b4 = pl.base * 0x01010101u, kb = (128u - ((1u << pl.k) - 1u)) * 0x01010101u;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const uint32_t e = r.P[m] & kExpMask4;
        const uint32_t d = ((e | 0x80808080u) - (b4 & 0x7F7F7F7Fu)) ^ ((e ^ ~b4) & 0x80808080u);
        const uint32_t lt = ((~e & b4) | (~(e ^ b4) & d)) & 0x80808080u;  // e < base
        const uint32_t esc = flags_to_mask(lt | ge_flags(d, kb));
        if constexpr (D::kExpBits == 5)
            r.P[m] = ((d | esc) & kExpMask4) | (r.P[m] & ~kExpMask4);
        else
            r.P[m] = d | esc;
    }
    uint32_t mine = 0;  // this warp's escapes at the chosen table
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
        transpose8x8x4(r.P + 8 * qq);
        if (pl.k > 0) mine += __popc(escape_word<D>(r.P + 8 * qq, pl.k));
    }
    mine = __reduce_add_sync(0xFFFFFFFFu, mine);
    if (lane == 0) x.cnt[h][0] = mine;
    bar.sync();
    pp.esc_before = h ? x.cnt[0][0] : 0u;
    return pp;
}

// The residual section of this warp's rows (8 h .. 8 h + 7) of a packed full
// chunk staged at `chunk`: the byte plane, then fp16's three bit-planes (from
// the warp's planes 5..7) or fp32's lower halves.
template <class D>
__device__ __forceinline__ void write_residual_pair(const HalfRegs& r, uint32_t h, const uint8_t* chunk, uint8_t* body) {
    const uint32_t lane = threadIdx.x & 31;
#pragma unroll 4
    for (int jj = 0; jj < 8; ++jj) {
        const uint32_t j = 8 * h + jj;
        if constexpr (D::kElemBytes == 4) {
            const uint8_t* row = chunk + 1024 * j + 32 * lane;
            const uint4 a = *reinterpret_cast<const uint4*>(row), b = *reinterpret_cast<const uint4*>(row + 16);
            *reinterpret_cast<uint2*>(body + 256 * j + 8 * lane) =
                make_uint2(sign_fraction_quad(upper_halves(a.x, a.y), upper_halves(a.z, a.w)),
                           sign_fraction_quad(upper_halves(b.x, b.y), upper_halves(b.z, b.w)));
            *reinterpret_cast<uint4*>(body + kSmPlaneBytes + 512 * j + 16 * lane) =
                make_uint4(lower_halves(a.x, a.y), lower_halves(a.z, a.w), lower_halves(b.x, b.y),
                           lower_halves(b.z, b.w));
        } else {
            const uint4 v = lds_row(chunk, j, lane);
            if constexpr (D::kExpBits == 5)
                *reinterpret_cast<uint2*>(body + 256 * j + 8 * lane) =
                    make_uint2(low_byte_quad(v.x, v.y), low_byte_quad(v.z, v.w));
            else
                *reinterpret_cast<uint2*>(body + 256 * j + 8 * lane) =
                    make_uint2(sign_fraction_quad(v.x, v.y), sign_fraction_quad(v.z, v.w));
        }
    }
    if constexpr (D::kExpBits == 5) {
#pragma unroll
        for (int qq = 0; qq < 2; ++qq)
#pragma unroll
            for (int t = 0; t < 3; ++t)
                *reinterpret_cast<uint32_t*>(body + kSmPlaneBytes + kPlaneBytes * t + 4 * (32 * (2 * h + qq) + lane)) =
                    r.P[8 * qq + 5 + t];
    }
}

// Exponent of staged element i.
template <class D>
__device__ __forceinline__ uint32_t staged_exponent(const uint8_t* chunk, uint32_t i) {
    if constexpr (D::kElemBytes == 4)
        return (reinterpret_cast<const uint32_t*>(chunk)[i] >> 23) & 0xFFu;
    else
        return (reinterpret_cast<const uint16_t*>(chunk)[i] >> (15 - D::kExpBits)) & ((1u << D::kExpBits) - 1u);
}

// Phase B: this warp's share of writing the full chunk staged at `chunk`
// (unchanged since phase A) with its planes `r` to `dst` (global, 16-byte
// aligned) following `pp`.  No barrier.  A raw chunk leaves by one bulk (TMA)
// store issued by lane 0 of warp 0, which waits until the copy has read
// `chunk` before returning; the caller must have ordered any generic writes of
// `chunk` before it with fence.proxy.async.  A packed chunk is written by
// coalesced stores: the residual section (warp h: rows 8 h .. 8 h + 7), the
// warp's words of the k planes (escaped elements carry the sentinel, all k
// bits set), then its escape bytes in bit-plane order, read back from the
// staged values, starting after esc_before.
template <class D>
__device__ __forceinline__ void write_chunk_pair(const HalfRegs& r, const PairPlan& pp, uint32_t h,
                                                 const uint8_t* chunk, uint8_t* dst) {
    const ChunkPlan& pl = pp.p;
    const uint32_t lane = threadIdx.x & 31;
    uint8_t* body = dst + kChunkHeaderBytes;
    if (h == 0 && lane == 0)
        *reinterpret_cast<uint4*>(dst) =
            make_uint4((pl.raw ? kModeRaw : kModePacked) | (pl.k << 8) | (pl.base << 16), kChunkElems | (pl.n_esc << 16),
                       pl.bytes, 0u);
    if (pl.raw) {
        if (h == 0) {
            if (lane == 0) {
                bulk_store(body, chunk, D::kElemBytes * kChunkElems);
                bulk_commit();
                bulk_wait_read();
            }
            __syncwarp();
        }
        return;
    }
    write_residual_pair<D>(r, h, chunk, body);
    const uint32_t k = pl.k;
    if (k == 0) return;
    uint32_t esc[2];
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
        const uint32_t* P = r.P + 8 * qq;
        esc[qq] = escape_word<D>(P, k);
        uint8_t* col = body + D::kResidBytes + 4 * (32 * (2 * h + qq) + lane);
#pragma unroll
        for (uint32_t p = 0; p < max_width<D>(); ++p)
            if (p < k) *reinterpret_cast<uint32_t*>(col + kPlaneBytes * p) = P[p] | esc[qq];
    }
    const uint32_t n_esc = pl.n_esc;
    if (n_esc == 0) return;
    // escapes before word (q, lane): the first warp's (esc_before), then all
    // of this warp's first quarter, then lanes < lane of quarter q (16-bit
    // fields: at most 1024 per quarter)
    const uint32_t c01 = __popc(esc[0]) | (__popc(esc[1]) << 16);
    uint32_t a = c01;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t ta = __shfl_up_sync(0xFFFFFFFFu, a, d);
        if (lane >= (uint32_t)d) a += ta;
    }
    const uint32_t t0 = __shfl_sync(0xFFFFFFFFu, a, 31) & 0xFFFFu;
    const uint32_t ea = a - c01;  // exclusive over lanes
    uint32_t idx[2] = {pp.esc_before + (ea & 0xFFFFu), pp.esc_before + t0 + (ea >> 16)};
    uint8_t* esc_out = body + D::kResidBytes + kPlaneBytes * k;
    // one escape of each quarter per step: two independent load -> store
    // chains in flight per lane
    while (__any_sync(0xFFFFFFFFu, (esc[0] | esc[1]) != 0u)) {
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            if (esc[qq]) {
                const uint32_t bit = __ffs(esc[qq]) - 1;
                esc[qq] &= esc[qq] - 1;
                const uint32_t m = bit & 7, bb = bit >> 3, q = 2 * h + qq;
                const uint32_t i = 256 * (4 * q + (m >> 1)) + 8 * lane + 4 * (m & 1) + bb;
                if (idx[qq] < n_esc) esc_out[idx[qq]] = (uint8_t)staged_exponent<D>(chunk, i);
                ++idx[qq];
            }
        }
    }
    if (h == 1 && lane < 16 && n_esc + lane < pad16(n_esc)) esc_out[n_esc + lane] = 0;
}

// ---------------------------------------------------------------------------
// Team encoding: a full chunk held in registers by a team of four warps.
// Thread (warp q of the team, lane l) holds rows 4 q .. 4 q + 3, elements
// 8 l .. 8 l + 7 of each, in the layout decode_full_chunk produces (16-bit
// types: P[4 jj + x] = elements 2 x, 2 x + 1 of row 4 q + jj; fp32:
// P[8 jj + s] = element s): exactly the 32 elements of bit-plane word
// 32 q + l, quad m = 2 jj + h being elements 4 h .. 4 h + 3 of row 4 q + jj.
// The team meets twice per chunk (exponent extremes, escape counts); after
// that every warp writes its own quarter.
// ---------------------------------------------------------------------------
struct TeamPlan {
    uint32_t raw;         // 1: stored raw
    uint32_t k;           // code width
    uint32_t base;        // header base (0 when raw)
    uint32_t n_esc;       // escapes at width k
    uint32_t bytes;       // chunk size, header included
    uint32_t esc_before;  // escapes of the quarters before this warp's, at width k
};

// Per-team exchange space in shared memory.
struct TeamXch {
    uint32_t mn[4], mx[4];  // per warp: smallest and largest exponent
    uint32_t cnt[4][8];     // per warp: escapes at width k (k = 1..7)
};

// The two upper-half pair-words (bf16 patterns) of quad m of an fp32 thread.
__device__ __forceinline__ uint32_t upper_pair0(const uint32_t* P, int m) { return upper_halves(P[4 * m], P[4 * m + 1]); }
__device__ __forceinline__ uint32_t upper_pair1(const uint32_t* P, int m) {
    return upper_halves(P[4 * m + 2], P[4 * m + 3]);
}

// Exponent quad m of this thread's values (one exponent per byte).
template <class D>
__device__ __forceinline__ uint32_t exponent_quad(const uint32_t* P, int m) {
    if constexpr (D::kElemBytes == 4)
        return __byte_perm(upper_pair0(P, m) << 1, upper_pair1(P, m) << 1, 0x7531);
    else if constexpr (D::kExpBits == 5)
        return fp16_exponent_quad(P[2 * m], P[2 * m + 1]) & 0x1F1F1F1Fu;
    else
        return __byte_perm(P[2 * m] << 1, P[2 * m + 1] << 1, 0x7531);
}

// Phase A for a team: exponent table and size of the chunk in P, leaving the
// bit-planes of this thread's word (offsets e - base; fp16: residual bits in
// planes 5..7) in `planes`.  Every thread of the team returns the same plan
// except esc_before.
template <class D, typename Barrier>
__device__ __forceinline__ TeamPlan plan_chunk_team(const Barrier& bar, const uint32_t* P, uint32_t planes[8],
                                                    TeamXch& x) {
    const uint32_t lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        if constexpr (D::kExpBits == 5) {
            const uint32_t u0 = fp16_exponent_lanes(P[2 * m]), u1 = fp16_exponent_lanes(P[2 * m + 1]);
            mn = vmin_u16x2(mn, vmin_u16x2(u0, u1));
            mx = vmax_u16x2(mx, vmax_u16x2(u0, u1));
            planes[m] = fp16_exponent_quad(P[2 * m], P[2 * m + 1]);
        } else {
            // doubling puts each value's exponent in the high byte of its 16-bit lane
            uint32_t t0, t1;
            if constexpr (D::kElemBytes == 4)
                t0 = upper_pair0(P, m) << 1, t1 = upper_pair1(P, m) << 1;
            else
                t0 = P[2 * m] << 1, t1 = P[2 * m + 1] << 1;
            mn = vmin_u16x2(mn, vmin_u16x2(t0, t1));
            mx = vmax_u16x2(mx, vmax_u16x2(t0, t1));
            planes[m] = __byte_perm(t0, t1, 0x7531);
        }
    }
    const uint32_t wmn = __reduce_min_sync(0xFFFFFFFFu, min((mn >> 8) & 0xFFu, mn >> 24));
    const uint32_t wmx = __reduce_max_sync(0xFFFFFFFFu, max((mx >> 8) & 0xFFu, mx >> 24));
    if (lane == 0) {
        x.mn[q] = wmn;
        x.mx[q] = wmx;
    }
    bar.sync();
    const uint32_t emin = min(min(x.mn[0], x.mn[1]), min(x.mn[2], x.mn[3]));
    const uint32_t emax = max(max(x.mx[0], x.mx[1]), max(x.mx[2], x.mx[3]));
    const uint32_t base4 = emin * 0x01010101u;
#pragma unroll
    for (int m = 0; m < 8; ++m) planes[m] -= base4;  // no borrow: every exponent >= emin
    transpose8x8x4(planes);                          // quads of offsets -> planes
    // escapes at width k are low_k | high_k (see add_escape_counts)
    constexpr int kTop = (int)D::kExpBits - 1;
    uint32_t high[8];
    high[kTop] = planes[kTop];
#pragma unroll
    for (int k = kTop - 1; k >= 1; --k) high[k] = high[k + 1] | planes[k];
    uint32_t low = planes[0];
#pragma unroll
    for (int k = 1; k <= kTop; ++k) {
        const uint32_t n = __reduce_add_sync(0xFFFFFFFFu, __popc(low | high[k]));
        if (lane == 0) x.cnt[q][k] = n;
        if (k < kTop) low &= planes[k];
    }
    bar.sync();
    TeamPlan pl{0u, 0u, emin, 0u, 0u, 0u};
    uint32_t best = 0;
    if (emax > emin) {
        // lane k (1..kTop) sizes width k; the smallest (size, k) wins, so a
        // tie keeps the smaller width
        uint32_t n = 0, before = 0, key = 0xFFFFFFFFu;
        if (lane >= 1 && lane <= (uint32_t)kTop) {
            const uint32_t c0 = x.cnt[0][lane], c1 = x.cnt[1][lane], c2 = x.cnt[2][lane];
            n = c0 + c1 + c2 + x.cnt[3][lane];
            before = (q > 0 ? c0 : 0u) + (q > 1 ? c1 : 0u) + (q > 2 ? c2 : 0u);
            key = ((kPlaneBytes * lane + (uint32_t)pad16(n)) << 3) | lane;
        }
        key = __reduce_min_sync(0xFFFFFFFFu, key);
        pl.k = key & 7u;
        best = key >> 3;
        pl.n_esc = __shfl_sync(0xFFFFFFFFu, n, pl.k);
        pl.esc_before = __shfl_sync(0xFFFFFFFFu, before, pl.k);
    }
    pl.raw = best >= raw_exponent_bytes<D>() ? 1u : 0u;
    if (pl.raw) {
        pl.k = 0;
        pl.base = 0;
        pl.n_esc = 0;
        pl.esc_before = 0;
        pl.bytes = max_chunk_bytes<D>();
    } else {
        pl.bytes = packed_chunk_bytes<D>(pl.k, pl.n_esc);
    }
    return pl;
}

// Phase B for a team: the chunk in P (planes from phase A), in its final
// byte layout, into `dst`, a staging buffer in shared memory (16-byte
// aligned) whose first pl.bytes bytes are all written.  No barrier: each warp
// writes the header (warp 0), its four rows of the residual section, its word
// of every bit-plane and its escapes, whose place follows from esc_before.  A
// thread with escapes first parks its exponent quads in its own 32 bytes of
// the residual section, reads the escaped bytes back from there, then
// overwrites them with the residual values.
template <class D>
__device__ __forceinline__ void stage_chunk_team(const uint32_t* P, const uint32_t planes[8], const TeamPlan& pl,
                                                 uint8_t* dst) {
    const uint32_t lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
    uint8_t* body = dst + kChunkHeaderBytes;
    if (q == 0 && lane == 0)
        *reinterpret_cast<uint4*>(dst) =
            make_uint4((pl.raw ? kModeRaw : kModePacked) | (pl.k << 8) | (pl.base << 16), kChunkElems | (pl.n_esc << 16),
                       pl.bytes, 0u);
    if (pl.raw) {
        if constexpr (D::kElemBytes == 4) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint8_t* row = body + 1024 * (4 * q + jj) + 32 * lane;
                *reinterpret_cast<uint4*>(row) = make_uint4(P[8 * jj], P[8 * jj + 1], P[8 * jj + 2], P[8 * jj + 3]);
                *reinterpret_cast<uint4*>(row + 16) =
                    make_uint4(P[8 * jj + 4], P[8 * jj + 5], P[8 * jj + 6], P[8 * jj + 7]);
            }
        } else {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                *reinterpret_cast<uint4*>(body + 512 * (4 * q + jj) + 16 * lane) =
                    make_uint4(P[4 * jj], P[4 * jj + 1], P[4 * jj + 2], P[4 * jj + 3]);
        }
        return;
    }
    const uint32_t k = pl.k, n_esc = pl.n_esc;
    uint8_t* own = body + 256 * 4 * q + 8 * lane;  // this thread's bytes of rows 4 q .. 4 q + 3
    const uint32_t esc = k ? escape_word<D>(planes, k) : 0u;
    if (n_esc != 0) {
        // escapes of the lanes before this one, from six independent ballots
        // of the count's bits (a count is at most 32)
        const uint32_t mine = __popc(esc), below = (1u << lane) - 1u;
        uint32_t idx = pl.esc_before;
#pragma unroll
        for (int b = 0; b < 6; ++b) idx += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, (mine >> b) & 1u) & below) << b;
        uint8_t* esc_out = body + D::kResidBytes + kPlaneBytes * k;
        if (esc) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                *reinterpret_cast<uint2*>(own + 256 * jj) =
                    make_uint2(exponent_quad<D>(P, 2 * jj), exponent_quad<D>(P, 2 * jj + 1));
            uint32_t rest = esc;
            while (rest) {
                const uint32_t bit = __ffs(rest) - 1;  // element (m, b) = byte b of quad m
                rest &= rest - 1;
                if (idx < n_esc) esc_out[idx] = own[((bit & 6) << 7) | ((bit & 1) << 2) | (bit >> 3)];
                ++idx;
            }
        }
        if (q == 0 && lane < 16 && n_esc + lane < pad16(n_esc)) esc_out[n_esc + lane] = 0;
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        uint8_t* plane_row = own + 256 * jj;
        if constexpr (D::kElemBytes == 4) {
            const uint32_t* R = P + 8 * jj;
            *reinterpret_cast<uint2*>(plane_row) =
                make_uint2(sign_fraction_quad(upper_halves(R[0], R[1]), upper_halves(R[2], R[3])),
                           sign_fraction_quad(upper_halves(R[4], R[5]), upper_halves(R[6], R[7])));
            *reinterpret_cast<uint4*>(body + kSmPlaneBytes + 512 * (4 * q + jj) + 16 * lane) =
                make_uint4(lower_halves(R[0], R[1]), lower_halves(R[2], R[3]), lower_halves(R[4], R[5]),
                           lower_halves(R[6], R[7]));
        } else if constexpr (D::kExpBits == 5) {
            *reinterpret_cast<uint2*>(plane_row) =
                make_uint2(low_byte_quad(P[4 * jj], P[4 * jj + 1]), low_byte_quad(P[4 * jj + 2], P[4 * jj + 3]));
        } else {
            *reinterpret_cast<uint2*>(plane_row) = make_uint2(sign_fraction_quad(P[4 * jj], P[4 * jj + 1]),
                                                              sign_fraction_quad(P[4 * jj + 2], P[4 * jj + 3]));
        }
    }
    if constexpr (D::kExpBits == 5) {
#pragma unroll
        for (int t = 0; t < 3; ++t)
            *reinterpret_cast<uint32_t*>(body + kSmPlaneBytes + kPlaneBytes * t + 4 * (32 * q + lane)) = planes[5 + t];
    }
    uint8_t* col = body + D::kResidBytes + 4 * (32 * q + lane);
#pragma unroll
    for (uint32_t p = 0; p < max_width<D>(); ++p)
        if (p < k) *reinterpret_cast<uint32_t*>(col + kPlaneBytes * p) = planes[p] | esc;
}

template <class D>
__host__ __device__ constexpr uint32_t tail_chunk_bytes(uint32_t n_c) {
    return (uint32_t)(16 + pad16(D::kElemBytes * n_c));
}

// The partial last chunk held by a team (values past n_c ignored), raw.
template <class D>
__device__ __forceinline__ void write_tail_chunk_team(const uint32_t* P, uint32_t n_c, uint8_t* dst) {
    const uint32_t lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
    const uint32_t bytes = tail_chunk_bytes<D>(n_c);
    if constexpr (D::kElemBytes == 4) {
        uint32_t* out = reinterpret_cast<uint32_t*>(dst + 16);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const uint32_t e = 256 * (4 * q + jj) + 8 * lane + x;
                if (e < n_c) out[e] = P[8 * jj + x];
            }
    } else {
        uint16_t* out = reinterpret_cast<uint16_t*>(dst + 16);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const uint32_t e = 256 * (4 * q + jj) + 8 * lane + 2 * x;
                if (e < n_c) out[e] = (uint16_t)(P[4 * jj + x] & 0xFFFFu);
                if (e + 1 < n_c) out[e + 1] = (uint16_t)(P[4 * jj + x] >> 16);
            }
    }
    if (q == 0 && lane == 0) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(kModeRaw, n_c, bytes, 0u);
        for (uint32_t b = 16 + D::kElemBytes * n_c; b < bytes; ++b) dst[b] = 0;
    }
}

// The partial last chunk (n_c < 4096 elements) is stored raw (section 5,
// "Handling data alignment").  One warp; `vals` are its n_c values.
template <class D, typename Src>
__device__ __forceinline__ void write_tail_chunk_warp(Src vals, uint32_t n_c, uint8_t* dst) {
    using Elem = typename std::conditional<D::kElemBytes == 4, uint32_t, uint16_t>::type;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t bytes = tail_chunk_bytes<D>(n_c);
    Elem* out = reinterpret_cast<Elem*>(dst + 16);
    for (uint32_t i = lane; i < n_c; i += 32) out[i] = vals(i);
    if (lane == 0) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(kModeRaw, n_c, bytes, 0u);
        for (uint32_t b = 16 + D::kElemBytes * n_c; b < bytes; ++b) dst[b] = 0;
    }
}

// Thread 0 of the warp that wrote chunk c: offset-table entry, the stream
// header (chunk 0) and the stream size (last chunk).
__device__ __forceinline__ void finish_chunk(const StreamOut& so, uint64_t c, uint64_t offset, uint32_t bytes) {
    uint8_t* out = so.out;
    *reinterpret_cast<uint64_t*>(out + kStreamHeaderBytes + 8 * c) = offset;
    if (c == 0) {
        *reinterpret_cast<uint4*>(out + 0) = make_uint4(kMagic, so.version | (so.dtype << 16), kChunkElems, 0u);
        *reinterpret_cast<uint4*>(out + 16) =
            make_uint4((uint32_t)so.n_elems, (uint32_t)(so.n_elems >> 32), (uint32_t)so.n_chunks,
                       (uint32_t)(so.n_chunks >> 32));
        *reinterpret_cast<uint64_t*>(out + 40) = 0;
        *reinterpret_cast<uint4*>(out + 48) = make_uint4(0u, 0u, 0u, 0u);
        if (so.n_chunks & 1) *reinterpret_cast<uint64_t*>(out + kStreamHeaderBytes + 8 * so.n_chunks) = 0;
    }
    if (c == so.n_chunks - 1) {
        const uint64_t total = offset + bytes;
        *reinterpret_cast<uint64_t*>(out + 32) = total;
        so.ws->total_bytes = total;
    }
}

}  // namespace cccl

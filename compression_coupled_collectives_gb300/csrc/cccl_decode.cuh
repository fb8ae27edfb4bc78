// cccl_decode.cuh -- decoding one staged chunk into registers (shared by the
// decompress and fused-reduce kernels).
//
// Inverse of the split of "CCCL: In-GPU Compression-Coupled Collective
// Communication", section 4.1: each exponent is base + code, or, where the
// code is the sentinel 2^k - 1, the next byte of the chunk's escape list
// (bit-plane order); sign and fraction come back from the residual section.
#pragma once

#include "cccl_device.cuh"

namespace cccl {

// This thread's words (decode_full_chunk's layout, below) of 4096 raw values
// at `vals` in shared memory.
template <class D>
__device__ __forceinline__ void load_raw_full(const uint8_t* vals, uint32_t* P) {
    const uint32_t lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
    if constexpr (D::kElemBytes == 4) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint8_t* row = vals + 1024 * (4 * q + jj) + 32 * lane;
            const uint4 a = *reinterpret_cast<const uint4*>(row), b = *reinterpret_cast<const uint4*>(row + 16);
            P[8 * jj] = a.x, P[8 * jj + 1] = a.y, P[8 * jj + 2] = a.z, P[8 * jj + 3] = a.w;
            P[8 * jj + 4] = b.x, P[8 * jj + 5] = b.y, P[8 * jj + 6] = b.z, P[8 * jj + 7] = b.w;
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4*>(vals + 512 * (4 * q + jj) + 16 * lane);
            P[4 * jj] = v.x;
            P[4 * jj + 1] = v.y;
            P[4 * jj + 2] = v.z;
            P[4 * jj + 3] = v.w;
        }
    }
}

// Decode the full chunk staged at `buf` (header already validated against
// the stream) into this thread's words.  Thread t (warp q = t / 32, lane l)
// gets rows 4 q .. 4 q + 3, elements 8 l .. 8 l + 7 of each: for the 16-bit
// types P[4 jj + w] = elements 2 w, 2 w + 1 of row 4 q + jj (16 words), for
// fp32 P[8 jj + s] = element s of row 4 q + jj (32 words).  The four warps of
// a team (four consecutive warps starting at a multiple of four; q = warp
// index mod 4) call it together and meet at `Barrier`; every branch on the
// header is uniform over them.  Returns false if the chunk body is malformed
// (a sentinel count that disagrees with n_esc, or an exponent the type cannot
// hold).  `special` is set when the chunk may hold an all-ones exponent (Inf
// or NaN).
template <class D, typename Barrier>
__device__ __forceinline__ bool decode_full_chunk(const Barrier& bar, uint8_t* buf, const ChunkHeader& h, uint32_t* P,
                                                  uint32_t* s_row_tot, bool& special) {
    constexpr uint32_t kTop = (1u << D::kExpBits) - 1;  // all-ones exponent
    const uint32_t t = threadIdx.x, lane = t & 31, q = (t >> 5) & 3;
    const uint8_t* body = buf + kChunkHeaderBytes;
    if (h.mode == kModeRaw) {
        load_raw_full<D>(body, P);
        special = true;
        return true;
    }
    const int k = (int)h.k;
    uint32_t S[8], code[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const uint2 v = *reinterpret_cast<const uint2*>(body + 256 * (4 * q + jj) + 8 * lane);
        S[2 * jj] = v.x;
        S[2 * jj + 1] = v.y;
    }
    uint32_t sent = 0xFFFFFFFFu;  // bit set where the code is the sentinel (all k bits set)
    const uint8_t* col = body + D::kResidBytes + 4 * (32 * q + lane);
    if constexpr (D::kExpBits == 5) {
        // codes (k <= 4) in slots 0..3 and the three residual planes in slots
        // 5..7: one transpose gives per byte code | f8 << 5 | f9 << 6 | sign << 7
        const uint8_t* rcol = body + kSmPlaneBytes + 4 * (32 * q + lane);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            code[p] = p < k ? *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p) : 0xFFFFFFFFu;
            sent &= code[p];
            if (p >= k) code[p] = 0u;
        }
#pragma unroll
        for (int r = 0; r < 3; ++r) code[5 + r] = *reinterpret_cast<const uint32_t*>(rcol + kPlaneBytes * r);
        transpose8x8x4(code);
    } else if (k >= 4) {  // one 8x8 bit transpose turns the planes into codes
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            code[p] = p < k ? *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p) : 0xFFFFFFFFu;
            sent &= code[p];
            if (p >= k) code[p] = 0u;
        }
        transpose8x8x4(code);
    } else {
#pragma unroll 1
        for (uint32_t p = 0; p < (uint32_t)k; ++p) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p);
            unpack_plane(w, p, code);
            sent &= w;
        }
    }
    uint32_t R[8];  // fp16: the residual bits 5..7 of every byte
    if constexpr (D::kExpBits == 5) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            R[m] = code[m] & 0xE0E0E0E0u;
            code[m] &= 0x0F0F0F0Fu;
        }
    }
    const uint32_t base4 = h.base * 0x01010101u;
    uint32_t E[8];
    if (k == 0) {
#pragma unroll
        for (int m = 0; m < 8; ++m) E[m] = base4;
        special = (h.base == kTop);
    } else {
        const uint32_t max_code = (1u << k) - 2u;  // largest non-sentinel code
        special = (h.base + max_code >= kTop);
        if (h.base + max_code + 1u <= kTop) {
            // no code, the sentinel included, leaves the type's exponents (or
            // carries out of its byte); escaped bytes are overwritten below
#pragma unroll
            for (int m = 0; m < 8; ++m) E[m] = code[m] + base4;
        } else {  // only a malformed stream overflows here
            bool bad = false;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t ff = ((sent >> m) & 0x01010101u) * 0xFFu;
                const uint32_t c = code[m] & ~ff;
#pragma unroll
                for (int b = 0; b < 4; ++b) bad |= ((c >> (8 * b)) & 0xFFu) + h.base > kTop;
                E[m] = (c + base4) & ~ff;
            }
            if (bar.any(bad)) return false;
        }
        if (h.n_esc == 0) {
            if (bar.any(sent != 0u)) return false;
        } else {
            // escapes are listed in bit-plane order: plane word 32 q + l, then
            // bit; this thread's sentinel bits are exactly its word's escapes.
            // Lanes before this one in the quarter, from six independent
            // ballots of the count's bits (a count is at most 32).
            const uint32_t mine = __popc(sent);
            const uint32_t below = (1u << lane) - 1u;
            uint32_t excl = 0;
#pragma unroll
            for (int b = 0; b < 6; ++b) excl += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, (mine >> b) & 1u) & below) << b;
            if (lane == 31) s_row_tot[q] = excl + mine;
            bar.sync();
            uint32_t before = 0, total = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t v = s_row_tot[r];
                if ((uint32_t)r < q) before += v;
                total += v;
            }
            if (total != h.n_esc) return false;  // CTA-uniform
            const uint8_t* esc = body + D::kResidBytes + kPlaneBytes * k;
            bool inf_nan = false, esc_bad = false;
            if (sent) {
                // patch the escaped exponents in shared memory: this thread's
                // exponent quads go over its own byte-plane bytes (already
                // in S), each escape byte lands in place, the quads come back
                uint8_t* own = buf + kChunkHeaderBytes + 256 * 4 * q + 8 * lane;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    *reinterpret_cast<uint2*>(own + 256 * jj) = make_uint2(E[2 * jj], E[2 * jj + 1]);
                uint32_t rest = sent, idx = before + excl;
                while (rest) {
                    const uint32_t bit = __ffs(rest) - 1;  // element (m, b): byte b of quad m
                    rest &= rest - 1;
                    const uint32_t e = idx < h.n_esc ? esc[idx] : 0u;
                    ++idx;
                    inf_nan |= (e == kTop);
                    if constexpr (D::kExpBits < 8) esc_bad |= (e > kTop);
                    own[((bit & 6) << 7) | ((bit & 1) << 2) | (bit >> 3)] = (uint8_t)e;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint2 v = *reinterpret_cast<const uint2*>(own + 256 * jj);
                    E[2 * jj] = v.x;
                    E[2 * jj + 1] = v.y;
                }
            }
            if constexpr (D::kExpBits < 8) {
                if (bar.any(esc_bad)) return false;
            }
            special = special || inf_nan;
        }
    }
    if constexpr (D::kExpBits == 5) {
#pragma unroll
        for (int m = 0; m < 8; ++m) join_quad_fp16(E[m], R[m], S[m], P[2 * m], P[2 * m + 1]);
    } else if constexpr (D::kElemBytes == 4) {
        // upper halves from (E, S); lower halves from the section after the
        // byte plane (row j of this thread: 16 bytes at 4096 + 512 j + 16 l)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 lo = *reinterpret_cast<const uint4*>(body + kSmPlaneBytes + 512 * (4 * q + jj) + 16 * lane);
            const uint32_t L[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t A, B;
                join_quad(E[2 * jj + hh], S[2 * jj + hh], A, B);
                uint32_t* o = P + 8 * jj + 4 * hh;
                o[0] = join_first(L[2 * hh], A);
                o[1] = join_second(L[2 * hh], A);
                o[2] = join_first(L[2 * hh + 1], B);
                o[3] = join_second(L[2 * hh + 1], B);
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m) join_quad(E[m], S[m], P[2 * m], P[2 * m + 1]);
    }
    return true;
}

// The codes of this thread's plane word (`col`: its column of plane 0) at
// width K, as 8 exponent-offset quads (fp16: with the residual bits 5..7 of
// every byte from the chunk's three residual planes), and the bits where the
// code is the sentinel (all K bits set; all ones when K = 0).  K is a
// compile-time constant: absent planes are zero and drop out of the transpose.
template <class D, int K>
__device__ __forceinline__ void quarter_codes(const uint8_t* body, const uint8_t* col, uint32_t* code,
                                              uint32_t& sent) {
    static_assert(K < (int)D::kExpBits, "widths run 0 .. exponent bits - 1");
#pragma unroll
    for (int p = 0; p < 8; ++p) code[p] = 0u;
    sent = 0xFFFFFFFFu;
#pragma unroll
    for (int p = 0; p < K; ++p) {
        code[p] = *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p);
        sent &= code[p];
    }
    if constexpr (D::kExpBits == 5) {
        // codes (K <= 4) in slots 0..3 and the three residual planes in slots
        // 5..7: one transpose gives per byte code | f8 << 5 | f9 << 6 | sign << 7
        const uint32_t off = (uint32_t)(col - body) - D::kResidBytes + kSmPlaneBytes;
#pragma unroll
        for (int r = 0; r < 3; ++r) code[5 + r] = *reinterpret_cast<const uint32_t*>(body + off + kPlaneBytes * r);
    }
    if constexpr (D::kExpBits == 8 && K >= 1 && K <= 4) {
        // planes 4..7 are zero: transpose the four 4x4 blocks of rows 0..3
        // first (the block swaps of the last two rounds), then the round
        // that moves the right blocks down reduces to splitting each byte's
        // nibbles (the blocks commute with that swap)
#pragma unroll
        for (int m = 0; m < 4; m += 2) block_swap(code[m], code[m + 1], 1, 0x55555555u);
#pragma unroll
        for (int m = 0; m < 2; ++m) block_swap(code[m], code[m + 2], 2, 0x33333333u);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            code[m + 4] = (code[m] >> 4) & 0x0F0F0F0Fu;
            code[m] &= 0x0F0F0F0Fu;
        }
    } else if (K > 0 || D::kExpBits == 5) {
        transpose8x8x4(code);
    }
}

// Escapes held in quarters 0 .. q - 1 of a packed chunk with k >= 1: the
// sentinel codes (all k bits set) of plane words 0 .. 32 q - 1, counted by
// one warp alone.  `planes` is the first plane of the staged chunk.
__device__ __forceinline__ uint32_t escapes_before_quarter(const uint8_t* planes, uint32_t k, uint32_t q) {
    const uint32_t lane = threadIdx.x & 31;
    uint32_t n = 0;
    for (uint32_t qq = 0; qq < q; ++qq) {
        const uint8_t* col = planes + 4 * (32 * qq + lane);
        uint32_t s = *reinterpret_cast<const uint32_t*>(col);
        for (uint32_t p = 1; p < k; ++p) s &= *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p);
        n += __popc(s);
    }
    return __reduce_add_sync(0xFFFFFFFFu, n);
}

// One warp decodes its quarter of the full chunk staged at `buf` (header `h`
// already checked against the stream), with no barrier: warp q (threadIdx.x
// / 32 mod 4), lane l gets rows 4 q .. 4 q + 3, elements 8 l .. 8 l + 7 of
// each, in decode_full_chunk's layout.  The warp finds where its escapes
// start in the chunk's list by counting the sentinel codes of the quarters
// before it itself.  Returns the number of sentinel codes in the quarter: the
// caller checks that the four quarters' counts add up to the header's n_esc.
// `bad` is set when a code or an escape leaves the type's exponents,
// `special` when the quarter may hold an all-ones exponent (Inf or NaN).
// Every lane returns the same count and flags.
template <class D>
__device__ __forceinline__ uint32_t decode_quarter(uint8_t* buf, const ChunkHeader& h, uint32_t* P, bool& special,
                                                   bool& bad) {
    constexpr uint32_t kTop = (1u << D::kExpBits) - 1;  // all-ones exponent
    const uint32_t t = threadIdx.x, lane = t & 31, q = (t >> 5) & 3;
    const uint8_t* body = buf + kChunkHeaderBytes;
    if (h.mode == kModeRaw) {
        load_raw_full<D>(body, P);
        special = true;
        return 0;
    }
    const uint32_t k = h.k;
    uint32_t S[8], code[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const uint2 v = *reinterpret_cast<const uint2*>(body + 256 * (4 * q + jj) + 8 * lane);
        S[2 * jj] = v.x;
        S[2 * jj + 1] = v.y;
    }
    uint32_t sent = 0xFFFFFFFFu;  // bit set where the code is the sentinel (all k bits set)
    const uint8_t* planes = body + D::kResidBytes;
    const uint8_t* col = planes + 4 * (32 * q + lane);
    // one copy of the plane loads and the transpose per width, so that the
    // planes a width does not have fold away
    switch (k) {
        case 1: quarter_codes<D, 1>(body, col, code, sent); break;
        case 2: quarter_codes<D, 2>(body, col, code, sent); break;
        case 3: quarter_codes<D, 3>(body, col, code, sent); break;
        case 4: quarter_codes<D, 4>(body, col, code, sent); break;
        case 5: if constexpr (max_width<D>() >= 5) quarter_codes<D, 5>(body, col, code, sent); break;
        case 6: if constexpr (max_width<D>() >= 6) quarter_codes<D, 6>(body, col, code, sent); break;
        case 7: if constexpr (max_width<D>() >= 7) quarter_codes<D, 7>(body, col, code, sent); break;
        default: quarter_codes<D, 0>(body, col, code, sent); break;
    }
    uint32_t R[8];  // fp16: the residual bits 5..7 of every byte
    if constexpr (D::kExpBits == 5) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            R[m] = code[m] & 0xE0E0E0E0u;
            code[m] &= 0x0F0F0F0Fu;
        }
    }
    const uint32_t base4 = h.base * 0x01010101u;
    uint32_t E[8];
    uint32_t mine = 0;  // this thread's sentinel codes
    if (k == 0) {
#pragma unroll
        for (int m = 0; m < 8; ++m) E[m] = base4;
        special = special || (h.base == kTop);
    } else {
        const uint32_t max_code = (1u << k) - 2u;  // largest non-sentinel code
        special = special || (h.base + max_code >= kTop);
        if (h.base + max_code + 1u <= kTop) {
            // no code, the sentinel included, leaves the type's exponents (or
            // carries out of its byte); escaped bytes are overwritten below
#pragma unroll
            for (int m = 0; m < 8; ++m) E[m] = code[m] + base4;
        } else {  // only a malformed stream overflows here
            bool over = false;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t ff = ((sent >> m) & 0x01010101u) * 0xFFu;
                const uint32_t c = code[m] & ~ff;
#pragma unroll
                for (int b = 0; b < 4; ++b) over |= ((c >> (8 * b)) & 0xFFu) + h.base > kTop;
                E[m] = (c + base4) & ~ff;
            }
            bad = bad || __any_sync(0xFFFFFFFFu, over);
        }
        mine = __popc(sent);
        if (h.n_esc != 0 && __any_sync(0xFFFFFFFFu, sent != 0u)) {  // uniform over the warp
            // escapes are listed in bit-plane order: plane word 32 q + l, then
            // bit; this thread's sentinel bits are exactly its word's escapes.
            // Lanes before this one, from six independent ballots of the
            // count's bits (a count is at most 32).
            const uint32_t below = (1u << lane) - 1u;
            uint32_t idx = q ? escapes_before_quarter(planes, k, q) : 0u;
#pragma unroll
            for (int b = 0; b < 6; ++b) idx += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, (mine >> b) & 1u) & below) << b;
            const uint8_t* esc = planes + kPlaneBytes * k;
            bool inf_nan = false, esc_bad = false;
            if (sent) {
                // patch the escaped exponents in shared memory: this thread's
                // exponent quads go over its own byte-plane bytes (already
                // in S), each escape byte lands in place, the quads come back
                uint8_t* own = buf + kChunkHeaderBytes + 256 * 4 * q + 8 * lane;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    *reinterpret_cast<uint2*>(own + 256 * jj) = make_uint2(E[2 * jj], E[2 * jj + 1]);
                uint32_t rest = sent;
                while (rest) {
                    const uint32_t bit = __ffs(rest) - 1;  // element (m, b): byte b of quad m
                    rest &= rest - 1;
                    const uint32_t e = idx < h.n_esc ? esc[idx] : 0u;
                    ++idx;
                    inf_nan |= (e == kTop);
                    if constexpr (D::kExpBits < 8) esc_bad |= (e > kTop);
                    own[((bit & 6) << 7) | ((bit & 1) << 2) | (bit >> 3)] = (uint8_t)e;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint2 v = *reinterpret_cast<const uint2*>(own + 256 * jj);
                    E[2 * jj] = v.x;
                    E[2 * jj + 1] = v.y;
                }
            }
            special = special || __any_sync(0xFFFFFFFFu, inf_nan);
            if constexpr (D::kExpBits < 8) bad = bad || __any_sync(0xFFFFFFFFu, esc_bad);
        }
    }
    if constexpr (D::kExpBits == 5) {
#pragma unroll
        for (int m = 0; m < 8; ++m) join_quad_fp16(E[m], R[m], S[m], P[2 * m], P[2 * m + 1]);
    } else if constexpr (D::kElemBytes == 4) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 lo = *reinterpret_cast<const uint4*>(body + kSmPlaneBytes + 512 * (4 * q + jj) + 16 * lane);
            const uint32_t L[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t A, B;
                join_quad(E[2 * jj + hh], S[2 * jj + hh], A, B);
                uint32_t* o = P + 8 * jj + 4 * hh;
                o[0] = join_first(L[2 * hh], A);
                o[1] = join_second(L[2 * hh], A);
                o[2] = join_first(L[2 * hh + 1], B);
                o[3] = join_second(L[2 * hh + 1], B);
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m) join_quad(E[m], S[m], P[2 * m], P[2 * m + 1]);
    }
    // the quarter's sentinel count, for the caller's check; no branch waits on it
    return __reduce_add_sync(0xFFFFFFFFu, mine);
}

}  // namespace cccl

namespace cccl {

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

}  // namespace cccl

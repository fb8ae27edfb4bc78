// cccl_decode.cuh -- decoding one staged chunk into registers (shared by the
// decompress and fused-reduce kernels).
//
// Inverse of the split of "CCCL: In-GPU Compression-Coupled Collective
// Communication", section 4.1: each exponent is base + code, or, where the
// code is the sentinel 2^k - 1, the next byte of the chunk's escape list
// (bit-plane order); sign and fraction come back from their byte.
#pragma once

#include "cccl_device.cuh"

namespace cccl {

// Decode the full chunk staged at `buf` (header already validated against
// the stream) into this thread's 16 words of bf16 pairs: thread t (warp
// q = t / 32, lane l) gets rows 4 q .. 4 q + 3, elements 8 l .. 8 l + 7 of
// each, as P[4 jj + w] = elements 2 w, 2 w + 1 of row 4 q + jj.  The four
// warps of a team (four consecutive warps starting at a multiple of four;
// q = warp index mod 4) call it together and meet at `Barrier`; every branch
// on the header is uniform over them.  Returns false if the chunk body is malformed (a sentinel
// count that disagrees with n_esc, or base + code above 255).  `special` is
// set when the chunk may hold an exponent of 255 (Inf or NaN).
template <typename Barrier>
__device__ __forceinline__ bool decode_full_chunk(const Barrier& bar, const uint8_t* buf, const ChunkHeader& h,
                                                  uint32_t P[16], uint32_t* s_row_tot, bool& special) {
    const uint32_t t = threadIdx.x, lane = t & 31, q = (t >> 5) & 3;
    const uint8_t* body = buf + kChunkHeaderBytes;
    if (h.mode == kModeRaw) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4*>(body + 512 * (4 * q + jj) + 16 * lane);
            P[4 * jj] = v.x;
            P[4 * jj + 1] = v.y;
            P[4 * jj + 2] = v.z;
            P[4 * jj + 3] = v.w;
        }
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
    const uint8_t* col = body + kSmPlaneBytes + 4 * (32 * q + lane);
    if (k >= 4) {  // one 8x8 bit transpose turns the planes into codes
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
    const uint32_t base4 = h.base * 0x01010101u;
    uint32_t E[8];
    if (k == 0) {
#pragma unroll
        for (int m = 0; m < 8; ++m) E[m] = base4;
        special = (h.base == 255);
    } else {
        const uint32_t max_code = (1u << k) - 2u;  // largest non-sentinel code
        special = (h.base + max_code >= 255u);
        if (h.base + max_code + 1u <= 255u) {
            // no code, the sentinel included, carries out of its byte;
            // escaped bytes are overwritten below
#pragma unroll
            for (int m = 0; m < 8; ++m) E[m] = code[m] + base4;
        } else {  // only a malformed stream overflows here
            bool bad = false;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t ff = ((sent >> m) & 0x01010101u) * 0xFFu;
                const uint32_t c = code[m] & ~ff;
#pragma unroll
                for (int b = 0; b < 4; ++b) bad |= ((c >> (8 * b)) & 0xFFu) + h.base > 255u;
                E[m] = (c + base4) & ~ff;
            }
            if (bar.any(bad)) return false;
        }
        if (h.n_esc == 0) {
            if (bar.any(sent != 0u)) return false;
        } else {
            // escapes are listed in bit-plane order: plane word 32 q + l, then
            // bit; this thread's sentinel bits are exactly its word's escapes
            const uint32_t mine = __popc(sent);
            uint32_t incl = mine;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= (uint32_t)d) incl += t2;
            }
            if (lane == 31) s_row_tot[q] = incl;
            bar.sync();
            uint32_t before = 0, total = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t v = s_row_tot[r];
                if ((uint32_t)r < q) before += v;
                total += v;
            }
            if (total != h.n_esc) return false;  // CTA-uniform
            const uint8_t* esc = body + kSmPlaneBytes + kPlaneBytes * k;
            bool inf_nan = false;
            // every lane takes its next escaped element until none is left
            uint32_t rest = sent, idx = before + incl - mine;
            while (__any_sync(0xFFFFFFFFu, rest != 0u)) {
                if (rest) {
                    const uint32_t bit = __ffs(rest) - 1;
                    rest &= rest - 1;
                    const uint32_t e = idx < h.n_esc ? esc[idx] : 0u;
                    ++idx;
                    inf_nan |= (e == 255u);
                    const uint32_t m = bit & 7, sh = 8 * (bit >> 3);
                    const uint32_t keep = ~(0xFFu << sh), put = e << sh;
#pragma unroll
                    for (int mm = 0; mm < 8; ++mm)
                        if ((uint32_t)mm == m) E[mm] = (E[mm] & keep) | put;
                }
            }
            special = special || inf_nan;
        }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) join_quad(E[m], S[m], P[2 * m], P[2 * m + 1]);
    return true;
}

}  // namespace cccl

namespace cccl {

// bf16 pair -> binary32 pair (exact)
__device__ __forceinline__ uint64_t widen_pair(uint32_t p) {
    return (uint64_t)(p << 16) | ((uint64_t)(p & 0xFFFF0000u) << 32);
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Decode quarter q (rows 4 q .. 4 q + 3) of the full chunk staged at `buf`
// (header already validated against the stream) into this lane's 16 words of
// bf16 pairs, in the layout of decode_full_chunk for warp q, by one warp
// alone: no other warp takes part, so the warps decoding the other quarters
// never wait for each other.  The warp reads the sentinel bits of all four
// quarters (escapes are listed in bit-plane order, so quarter q's first
// escape follows every escape of quarters < q) and checks the chunk's total
// against n_esc.  Returns false (warp-uniform) if the chunk body is
// malformed; `special` is set when the quarter may hold an exponent of 255.
__device__ __forceinline__ bool decode_quarter_warp(const uint8_t* buf, const ChunkHeader& h, uint32_t q,
                                                    uint32_t P[16], bool& special) {
    const uint32_t lane = threadIdx.x & 31;
    const uint8_t* body = buf + kChunkHeaderBytes;
    if (h.mode == kModeRaw) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4*>(body + 512 * (4 * q + jj) + 16 * lane);
            P[4 * jj] = v.x;
            P[4 * jj + 1] = v.y;
            P[4 * jj + 2] = v.z;
            P[4 * jj + 3] = v.w;
        }
        special = true;
        return true;
    }
    const uint32_t k = h.k, base = h.base, base4 = base * 0x01010101u;
    uint32_t S[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const uint2 v = *reinterpret_cast<const uint2*>(body + 256 * (4 * q + jj) + 8 * lane);
        S[2 * jj] = v.x;
        S[2 * jj + 1] = v.y;
    }
    const uint8_t* planes = body + kSmPlaneBytes;
    uint32_t code[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    uint32_t E[8];
    if (k == 0) {  // one exponent for the whole chunk (no escapes: checked with the header)
#pragma unroll
        for (int m = 0; m < 8; ++m) E[m] = base4;
        special = (base == 255);
    } else {
        // sentinel (escape) bits of this lane's word in every quarter
        uint32_t sq[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
#pragma unroll
        for (uint32_t p = 0; p < 8; ++p) {
            if (p < k) {
                const uint32_t* row = reinterpret_cast<const uint32_t*>(planes + kPlaneBytes * p) + lane;
#pragma unroll
                for (int x = 0; x < 4; ++x) sq[x] &= row[32 * x];
                code[p] = row[32 * q];
            }
        }
        const uint32_t sent = q == 0 ? sq[0] : q == 1 ? sq[1] : q == 2 ? sq[2] : sq[3];
        if (k >= 4) {
            transpose8x8x4(code);  // planes -> codes
        } else {
            uint32_t w[3] = {code[0], code[1], code[2]};
#pragma unroll
            for (int m = 0; m < 8; ++m) code[m] = 0u;
#pragma unroll
            for (uint32_t p = 0; p < 3; ++p)
                if (p < k) unpack_plane(w[p], p, code);
        }
        const uint32_t max_code = (1u << k) - 2u;  // largest non-sentinel code
        special = (base + max_code >= 255u);
        bool bad = false;
        if (base + max_code + 1u <= 255u) {
            // no code, the sentinel included, carries out of its byte;
            // escaped bytes are overwritten below
#pragma unroll
            for (int m = 0; m < 8; ++m) E[m] = code[m] + base4;
        } else {  // only a malformed stream overflows here
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t ff = ((sent >> m) & 0x01010101u) * 0xFFu;
                const uint32_t c = code[m] & ~ff;
#pragma unroll
                for (int b = 0; b < 4; ++b) bad |= ((c >> (8 * b)) & 0xFFu) + base > 255u;
                E[m] = (c + base4) & ~ff;
            }
        }
        // per-quarter sentinel totals (16-bit fields) and this lane's place in quarter q
        const uint32_t c01 = __popc(sq[0]) | (__popc(sq[1]) << 16), c23 = __popc(sq[2]) | (__popc(sq[3]) << 16);
        const uint32_t mine = __popc(sent);
        const uint32_t t01 = __reduce_add_sync(0xFFFFFFFFu, c01), t23 = __reduce_add_sync(0xFFFFFFFFu, c23);
        uint32_t incl = mine;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += t;
        }
        const uint32_t T0 = t01 & 0xFFFFu, T1 = t01 >> 16, T2 = t23 & 0xFFFFu, T3 = t23 >> 16;
        if (__any_sync(0xFFFFFFFFu, bad) || T0 + T1 + T2 + T3 != h.n_esc) return false;  // warp-uniform
        const uint32_t before = (q > 0 ? T0 : 0u) + (q > 1 ? T1 : 0u) + (q > 2 ? T2 : 0u);
        const uint8_t* esc = planes + kPlaneBytes * k;
        bool inf_nan = false;
        // every lane takes its next escaped element until none is left
        uint32_t rest = sent, idx = before + incl - mine;
        while (__any_sync(0xFFFFFFFFu, rest != 0u)) {
            if (rest) {
                const uint32_t bit = __ffs(rest) - 1;
                rest &= rest - 1;
                const uint32_t e = idx < h.n_esc ? esc[idx] : 0u;
                ++idx;
                inf_nan |= (e == 255u);
                const uint32_t m = bit & 7, sh = 8 * (bit >> 3);
                const uint32_t keep = ~(0xFFu << sh), put = e << sh;
#pragma unroll
                for (int mm = 0; mm < 8; ++mm)
                    if ((uint32_t)mm == m) E[mm] = (E[mm] & keep) | put;
            }
        }
        special = special || inf_nan;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) join_quad(E[m], S[m], P[2 * m], P[2 * m + 1]);
    return true;
}

}  // namespace cccl

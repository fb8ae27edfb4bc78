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
__device__ __forceinline__ bool decode_full_chunk(const Barrier& bar, uint8_t* buf, const ChunkHeader& h,
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
            const uint8_t* esc = body + kSmPlaneBytes + kPlaneBytes * k;
            bool inf_nan = false;
            if (sent) {
                // patch the escaped exponents in shared memory: this thread's
                // exponent quads go over its own sign+fraction bytes (already
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
                    inf_nan |= (e == 255u);
                    own[((bit & 6) << 7) | ((bit & 1) << 2) | (bit >> 3)] = (uint8_t)e;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint2 v = *reinterpret_cast<const uint2*>(own + 256 * jj);
                    E[2 * jj] = v.x;
                    E[2 * jj + 1] = v.y;
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

}  // namespace cccl

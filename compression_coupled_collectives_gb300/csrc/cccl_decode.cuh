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
// the stream) into this thread's 16 words of bf16 pairs, in the layout of
// encode_full_chunk.  All 128 threads call it; every branch on the header
// is CTA-uniform.  Returns false if the chunk body is malformed (a sentinel
// count that disagrees with n_esc, or base + code above 255).  `special` is
// set when the chunk may hold an exponent of 255 (Inf or NaN).
__device__ __forceinline__ bool decode_full_chunk(const uint8_t* buf, const ChunkHeader& h, uint32_t P[16],
                                                  uint32_t* s_row_tot, bool& special) {
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;
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
#pragma unroll 1
    for (uint32_t p = 0; p < (uint32_t)k; ++p) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p);
        unpack_plane(w, p, code);
        sent &= w;
    }
    const uint32_t base4 = h.base * 0x01010101u;
    uint32_t E[8];
    if (k == 0) {
#pragma unroll
        for (int m = 0; m < 8; ++m) E[m] = base4;
        special = (h.base == 255);
    } else {
        uint32_t FF[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            FF[m] = ((sent >> m) & 0x01010101u) * 0xFFu;
            E[m] = ((code[m] & ~FF[m]) + base4) & ~FF[m];
        }
        const uint32_t max_code = (1u << k) - 2u;  // largest non-sentinel code
        special = (h.base + max_code >= 255u);
        if (h.base + max_code > 255u) {  // only a malformed stream overflows here
            bool bad = false;
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (!((FF[m] >> (8 * b)) & 1u) && ((code[m] >> (8 * b)) & 0xFFu) + h.base > 255u) bad = true;
            if (__syncthreads_or(bad)) return false;
        }
        if (h.n_esc == 0) {
            if (__syncthreads_or(sent != 0u)) return false;
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
            __syncthreads();
            uint32_t before = 0, total = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t v = s_row_tot[r];
                if ((uint32_t)r < q) before += v;
                total += v;
            }
            if (total != h.n_esc) return false;  // CTA-uniform
            const uint32_t first = before + incl - mine;
            const uint8_t* esc = body + kSmPlaneBytes + kPlaneBytes * k;
            bool inf_nan = false;
            if (sent) {
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const uint32_t bit = 8 * b + m;
                        if ((sent >> bit) & 1u) {
                            const uint32_t idx = first + __popc(sent & ((1u << bit) - 1u));
                            const uint32_t e = idx < h.n_esc ? esc[idx] : 0u;
                            E[m] |= e << (8 * b);
                            inf_nan |= (e == 255u);
                        }
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

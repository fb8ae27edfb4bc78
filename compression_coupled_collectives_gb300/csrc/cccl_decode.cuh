// cccl_decode.cuh -- decoding one staged chunk into registers (shared by the
// decompress and fused-reduce kernels).
//
// Inverse of the split of "CCCL: In-GPU Compression-Coupled Collective
// Communication", section 4.1: each exponent is base + code, or, where the
// code is the sentinel 2^k - 1, the next byte of the chunk's escape list
// (ascending element order); sign and fraction come back from their byte.
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
    uint32_t S[8], code[8], W[7];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const uint2 v = *reinterpret_cast<const uint2*>(body + 256 * (4 * q + jj) + 8 * lane);
        S[2 * jj] = v.x;
        S[2 * jj + 1] = v.y;
    }
#pragma unroll
    for (int p = 0; p < 7; ++p)
        W[p] = (p < k) ? *reinterpret_cast<const uint32_t*>(body + kSmPlaneBytes + kPlaneBytes * p + 4 * (32 * q + lane))
                       : 0u;
    unpack_planes_k(k, W, code);
    const uint32_t base4 = h.base * 0x01010101u;
    uint32_t E[8];
    if (k == 0) {
#pragma unroll
        for (int m = 0; m < 8; ++m) E[m] = base4;
        special = (h.base == 255);
    } else {
        uint32_t sent = 0xFFFFFFFFu;  // bit set where the code is the sentinel (all k bits set)
#pragma unroll
        for (int p = 0; p < 7; ++p)
            if (p < k) sent &= W[p];
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
            uint32_t cnt[4], rb[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) cnt[jj] = (uint32_t)__popc(sent & (0x03030303u << (2 * jj)));
            const uint32_t total = escape_row_bases(cnt, rb, s_row_tot);
            if (total != h.n_esc) return false;
            const uint8_t* esc = body + kSmPlaneBytes + kPlaneBytes * k;
            bool inf_nan = false;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint32_t idx = rb[jj];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int m = 2 * jj + hh;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        if ((FF[m] >> (8 * b)) & 1u) {
                            const uint32_t e = idx < h.n_esc ? esc[idx] : 0u;
                            ++idx;
                            E[m] |= e << (8 * b);
                            inf_nan |= (e == 255u);
                        }
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

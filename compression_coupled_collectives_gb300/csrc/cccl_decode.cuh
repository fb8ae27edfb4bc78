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

// Accumulator layout (16 KiB of binary32): row j, lane l, elements 4 h .. 4 h
// + 3 of the lane's 8 at acc + 1024 j + 512 h + 16 l, so that each 16-byte
// access of a warp covers 512 contiguous bytes (no bank conflicts).
__device__ __forceinline__ void accumulate_row(uint8_t* acc, uint32_t j, uint32_t lane, const uint32_t P[4],
                                               bool first) {
    ulonglong2* a0 = reinterpret_cast<ulonglong2*>(acc + 1024 * j + 16 * lane);
    ulonglong2* a1 = reinterpret_cast<ulonglong2*>(acc + 1024 * j + 512 + 16 * lane);
    ulonglong2 v0 = make_ulonglong2(widen_pair(P[0]), widen_pair(P[1]));
    ulonglong2 v1 = make_ulonglong2(widen_pair(P[2]), widen_pair(P[3]));
    if (!first) {
        const ulonglong2 o0 = *a0, o1 = *a1;
        v0 = make_ulonglong2(add_f32x2(o0.x, v0.x), add_f32x2(o0.y, v0.y));
        v1 = make_ulonglong2(add_f32x2(o1.x, v1.x), add_f32x2(o1.y, v1.y));
    }
    *a0 = v0;
    *a1 = v1;
}

// One warp: decode the full chunk staged at `buf` (header already validated)
// and add its values into the binary32 accumulator `acc` (shared memory,
// 16 KiB, layout of accumulate_row), or store them there when `first`.  Adds follow
// rank order because the caller feeds ranks in order.  Returns false if the
// chunk body is malformed; `special` is set when the chunk may hold an
// exponent of 255.  Escapes are listed in bit-plane order: lane l's
// sentinel bits in quarter q are exactly those of plane word 32 q + l.
__device__ __forceinline__ bool decode_accumulate_warp(const uint8_t* buf, const ChunkHeader& h, uint8_t* acc,
                                                       bool first, bool& special) {
    const uint32_t lane = threadIdx.x & 31;
    const uint8_t* body = buf + kChunkHeaderBytes;
    if (h.mode == kModeRaw) {
#pragma unroll 4
        for (uint32_t j = 0; j < 16; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(body + 512 * j + 16 * lane);
            const uint32_t P[4] = {v.x, v.y, v.z, v.w};
            accumulate_row(acc, j, lane, P, first);
        }
        special = true;
        return true;
    }
    const uint32_t k = h.k, base = h.base, base4 = base * 0x01010101u;
    const uint8_t* planes = body + kSmPlaneBytes;
    // sentinel (escape) bits of this lane's four plane words
    uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    if (k > 0) {
        s0 = s1 = s2 = s3 = 0xFFFFFFFFu;
        for (uint32_t p = 0; p < k; ++p) {
            const uint32_t* row = reinterpret_cast<const uint32_t*>(planes + kPlaneBytes * p) + lane;
            s0 &= row[0];
            s1 &= row[32];
            s2 &= row[64];
            s3 &= row[96];
        }
    }
    const uint32_t max_code = k ? (1u << k) - 2u : 0u;  // largest non-sentinel code
    special = (base + max_code >= 255u);
    // escapes before word (q, lane): all of quarters < q, lanes < lane of quarter q
    uint32_t qb0 = 0, qb1 = 0, qb2 = 0, qb3 = 0;
    if (h.n_esc == 0) {
        if (__any_sync(0xFFFFFFFFu, (s0 | s1 | s2 | s3) != 0u)) return false;
    } else {
        const uint32_t c01 = __popc(s0) | (__popc(s1) << 16), c23 = __popc(s2) | (__popc(s3) << 16);
        uint32_t a = c01, b = c23;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t ta = __shfl_up_sync(0xFFFFFFFFu, a, d), tb = __shfl_up_sync(0xFFFFFFFFu, b, d);
            if (lane >= (uint32_t)d) {
                a += ta;
                b += tb;
            }
        }
        const uint32_t ta = __shfl_sync(0xFFFFFFFFu, a, 31), tb = __shfl_sync(0xFFFFFFFFu, b, 31);
        const uint32_t t0 = ta & 0xFFFFu, t1 = ta >> 16, t2 = tb & 0xFFFFu, t3 = tb >> 16;
        if (t0 + t1 + t2 + t3 != h.n_esc) return false;  // warp-uniform
        const uint32_t ea = a - c01, eb = b - c23;
        qb0 = ea & 0xFFFFu;
        qb1 = t0 + (ea >> 16);
        qb2 = t0 + t1 + (eb & 0xFFFFu);
        qb3 = t0 + t1 + t2 + (eb >> 16);
    }
    const uint8_t* esc = planes + kPlaneBytes * k;
    // base + code stays within its byte for every non-sentinel code unless
    // base + max_code > 255 (then only a malformed stream carries)
    const bool carry_free = base + (k ? (1u << k) - 1u : 0u) <= 255u;
    bool bad = false, inf_nan = false;
#pragma unroll 1
    for (uint32_t q = 0; q < 4; ++q) {
        const uint32_t sent = q == 0 ? s0 : q == 1 ? s1 : q == 2 ? s2 : s3;
        const uint32_t first_esc = q == 0 ? qb0 : q == 1 ? qb1 : q == 2 ? qb2 : qb3;
        uint32_t code[8];
        const uint8_t* col = planes + 4 * (32 * q + lane);
        if (k >= 4) {  // one 8x8 bit transpose turns the planes into codes
#pragma unroll
            for (int p = 0; p < 8; ++p)
                code[p] = (uint32_t)p < k ? *reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p) : 0u;
            transpose8x8x4(code);
        } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) code[m] = 0;
            for (uint32_t p = 0; p < k; ++p)
                unpack_plane(*reinterpret_cast<const uint32_t*>(col + kPlaneBytes * p), p, code);
        }
        uint32_t E[8];
        if (carry_free) {
#pragma unroll
            for (int m = 0; m < 8; ++m) E[m] = code[m] + base4;  // escaped bytes are patched below
        } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t ff = ((sent >> m) & 0x01010101u) * 0xFFu;  // escaped bytes
                const uint32_t c = code[m] & ~ff;
#pragma unroll
                for (int b = 0; b < 4; ++b) bad |= ((c >> (8 * b)) & 0xFFu) + base > 255u;
                E[m] = (c + base4) & ~ff;
            }
        }
        // escapes: every lane takes its next escaped element until none is left
        uint32_t rest = sent, idx = first_esc;
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
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint2 sv = *reinterpret_cast<const uint2*>(body + 256 * (4 * q + jj) + 8 * lane);
            uint32_t P[4];
            join_quad(E[2 * jj], sv.x, P[0], P[1]);
            join_quad(E[2 * jj + 1], sv.y, P[2], P[3]);
            accumulate_row(acc, 4 * q + jj, lane, P, first);
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad)) return false;
    special = special || __any_sync(0xFFFFFFFFu, inf_nan);
    return true;
}

}  // namespace cccl

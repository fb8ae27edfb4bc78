// cccl_encode.cuh -- encoding chunks staged in shared memory and placing a
// group of them in the output stream (shared by the compress and fused-reduce
// kernels).
//
// Per chunk ("CCCL: In-GPU Compression-Coupled Collective Communication"):
//   section 4.1  split every bf16 into its exponent and a sign+fraction byte;
//   section 4.3  the chunk's own table: base = minimum exponent, width k that
//                minimises 512 k + pad16(#escapes), fixed-length k-bit codes;
//   section 4.4  the chunk is written once, straight into its final place;
//   section 5    the partial last chunk is stored raw.
//
// Work split: one warp encodes one whole chunk (lane l owns the elements
// 256 j + 8 l + s of all 16 rows j, i.e. bit-plane words 32 q + l for
// q < 4), so a chunk needs only warp-level reductions.  A CTA of G warps
// encodes G consecutive chunks and places them with ONE decoupled look-back
// over groups; the chunks' offsets inside the group come from a local scan.
#pragma once

#include "cccl_device.cuh"

namespace cccl {

struct StreamOut {
    uint8_t* out;        // stream base (16-byte aligned)
    uint64_t capacity;   // bytes writable at out (>= the compress bound)
    uint64_t* status;    // one placement word per group
    WsHeader* ws;
    uint64_t n_elems;
    uint64_t n_chunks;
};

// Encoding decision of one full chunk (warp-uniform).
struct ChunkPlan {
    uint32_t raw;    // 1: stored raw
    uint32_t k;      // code width
    uint32_t base;   // minimum exponent
    uint32_t n_esc;  // escapes at width k
    uint32_t kfull;  // narrowest width without escapes (0 when one symbol; 8, 9: none)
    uint32_t bytes;  // chunk size, header included
};

// This lane's 4 pair-words of row j (elements 256 j + 8 l .. + 7).
__device__ __forceinline__ uint4 lds_row(const uint8_t* chunk, uint32_t j, uint32_t lane) {
    return *reinterpret_cast<const uint4*>(chunk + 512 * j + 16 * lane);
}

// Number of this lane's elements among 8 quads whose offset is >= 2^k - 1.
__device__ __forceinline__ uint32_t count_escapes8(const uint32_t* off, uint32_t k) {
    const uint32_t kb = (128u - ((1u << k) - 1u)) * 0x01010101u;
    uint32_t f[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) f[m] = ge_flags(off[m], kb);
    return count_flags8(f);
}

// Phase A: exponent table and size of the full chunk at `chunk` (8192 bytes
// of bf16 in shared memory).  One warp; every lane returns the same plan.
__device__ __forceinline__ ChunkPlan plan_chunk_warp(const uint8_t* chunk) {
    const uint32_t lane = threadIdx.x & 31;
    uint32_t off[32];  // exponents of this lane's 128 elements (quads), later offsets
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 v = lds_row(chunk, 4 * q + jj, lane);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t mag = w[i] & 0x7FFF7FFFu;  // |x| orders like the exponent
                mn = vmin_u16x2(mn, mag);
                mx = vmax_u16x2(mx, mag);
            }
            uint32_t sm_unused;
            split_quad(w[0], w[1], off[8 * q + 2 * jj], sm_unused);
            split_quad(w[2], w[3], off[8 * q + 2 * jj + 1], sm_unused);
        }
    }
    const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, min(mn & 0xFFFFu, mn >> 16) >> 7);
    const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16) >> 7);
    const uint32_t base4 = emin * 0x01010101u;
#pragma unroll
    for (int m = 0; m < 32; ++m) off[m] -= base4;  // no borrow: every exponent >= emin

    ChunkPlan pl{0u, 0u, emin, 0u, 0u, 0u};
    const uint32_t range = emax - emin;
    uint32_t best = 0;
    if (range > 0) {
        const uint32_t kfull = 32 - __clz(range + 1);  // 2..9
        pl.kfull = kfull;
        int bk = -1;
        uint32_t bsize = 0xFFFFFFFFu, besc = 0;
        if (kfull <= 7) {
            bk = (int)kfull;
            bsize = kPlaneBytes * kfull;
        }
        // widths below k1 can only win when 512 k + pad16(n_esc(k1)) does not
        // exceed the best size (n_esc never shrinks as k shrinks)
        const uint32_t k1 = min(kfull - 1, 7u);
        uint32_t c1 = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) c1 += count_escapes8(off + 8 * q, k1);
        const uint32_t n1 = __reduce_add_sync(0xFFFFFFFFu, c1);
        const uint32_t s1 = kPlaneBytes * k1 + (uint32_t)pad16(n1);
        if (s1 <= bsize) {  // k1 < kfull: a tie keeps the smaller width
            bk = (int)k1;
            bsize = s1;
            besc = n1;
        }
        for (int kk = (int)k1 - 1; kk >= 1; --kk) {
            if (kPlaneBytes * kk + (uint32_t)pad16(n1) > bsize) continue;  // bound grows with kk
            // kk is the widest remaining candidate: evaluate kk down to 1
            for (int k2 = kk; k2 >= 1; --k2) {
                uint32_t ck = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) ck += count_escapes8(off + 8 * q, (uint32_t)k2);
                const uint32_t nk = __reduce_add_sync(0xFFFFFFFFu, ck);
                const uint32_t sk = kPlaneBytes * k2 + (uint32_t)pad16(nk);
                if (sk <= bsize) {
                    bk = k2;
                    bsize = sk;
                    besc = nk;
                }
            }
            break;
        }
        pl.k = (uint32_t)bk;
        pl.n_esc = besc;
        best = bsize;
    }
    pl.raw = best >= kSmPlaneBytes ? 1u : 0u;
    if (pl.raw) {
        pl.k = 0;
        pl.base = 0;
        pl.n_esc = 0;
        pl.bytes = kMaxChunkBytes;
    } else {
        pl.bytes = (uint32_t)(16 + kSmPlaneBytes + kPlaneBytes * pl.k + pad16(pl.n_esc));
    }
    return pl;
}

// 4 flag bytes (0x80 each) -> 4 bits in element order
__device__ __forceinline__ uint32_t gather_msb4(uint32_t f) { return ((f & 0x80808080u) * 0x00204081u) >> 28; }

// Phase B: write the full chunk at `chunk` (shared memory) to `dst` (global,
// 16-byte aligned) following `pl`.  One warp.
__device__ __forceinline__ void write_chunk_warp(const uint8_t* chunk, const ChunkPlan& pl, uint8_t* dst) {
    const uint32_t lane = threadIdx.x & 31;
    if (lane == 0)
        *reinterpret_cast<uint4*>(dst) =
            make_uint4((pl.raw ? kModeRaw : kModePacked) | (pl.k << 8) | (pl.base << 16), kChunkElems | (pl.n_esc << 16),
                       pl.bytes, 0u);
    uint8_t* body = dst + kChunkHeaderBytes;
    if (pl.raw) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            *reinterpret_cast<uint4*>(body + 512 * j + 16 * lane) = lds_row(chunk, j, lane);
        return;
    }
    const uint32_t k = pl.k;
    const uint32_t base4 = pl.base * 0x01010101u;
    const bool escapes = pl.n_esc > 0;
    const uint32_t sent = (1u << k) - 1u;
    const uint32_t kb = (128u - sent) * 0x01010101u;
    uint8_t* esc_out = body + kSmPlaneBytes + kPlaneBytes * k;
    uint32_t esc_done = 0;  // escapes written for the rows before (warp-uniform)
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        uint32_t E[8], S[8];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 v = lds_row(chunk, 4 * q + jj, lane);
            split_quad(v.x, v.y, E[2 * jj], S[2 * jj]);
            split_quad(v.z, v.w, E[2 * jj + 1], S[2 * jj + 1]);
            *reinterpret_cast<uint2*>(body + 256 * (4 * q + jj) + 8 * lane) = make_uint2(S[2 * jj], S[2 * jj + 1]);
        }
        if (k == 0) continue;
        uint32_t code[8], emask = 0;  // emask: escaped elements, bit 8 jj + s
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t off = E[m] - base4;
            if (escapes) {
                const uint32_t f = ge_flags(off, kb);
                const uint32_t ff = flags_to_mask(f);
                code[m] = (off & ~ff) | ((sent * 0x01010101u) & ff);
                emask |= gather_msb4(f) << (4 * m);
            } else {
                code[m] = off;
            }
        }
        uint32_t W[7];
        pack_planes_k((int)k, code, W);
#pragma unroll
        for (int p = 0; p < 7; ++p)
            if ((uint32_t)p < k)
                *reinterpret_cast<uint32_t*>(body + kSmPlaneBytes + kPlaneBytes * p + 4 * (32 * q + lane)) = W[p];
        if (escapes && __any_sync(0xFFFFFFFFu, emask != 0u)) {
            // ascending element order: row j = 4q + jj, then lane, then s
            const uint32_t c01 = __popc(emask & 0xFFu) | (__popc(emask & 0xFF00u) << 16);
            const uint32_t c23 = __popc(emask & 0xFF0000u) | (__popc(emask >> 24) << 16);
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
            const uint32_t row_tot[4] = {ta & 0xFFFFu, ta >> 16, tb & 0xFFFFu, tb >> 16};
            const uint32_t ea = a - c01, eb = b - c23;  // exclusive over lanes
            uint32_t row_base[4];
            row_base[0] = esc_done + (ea & 0xFFFFu);
            row_base[1] = esc_done + row_tot[0] + (ea >> 16);
            row_base[2] = esc_done + row_tot[0] + row_tot[1] + (eb & 0xFFFFu);
            row_base[3] = esc_done + row_tot[0] + row_tot[1] + row_tot[2] + (eb >> 16);
            esc_done += row_tot[0] + row_tot[1] + row_tot[2] + row_tot[3];
            uint32_t rest = emask;
            while (rest) {
                const uint32_t bit = __ffs(rest) - 1;
                rest &= rest - 1;
                const uint32_t jj = bit >> 3, m = bit >> 2, b = bit & 3;
                uint32_t rbase = 0, eword = 0;  // select without run-time register indexing
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if ((uint32_t)r == jj) rbase = row_base[r];
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if ((uint32_t)r == m) eword = E[r];
                const uint32_t idx = rbase + __popc(emask & ((1u << bit) - 1u) & (0xFFu << (8 * jj)));
                if (idx < pl.n_esc) esc_out[idx] = (uint8_t)(eword >> (8 * b));
            }
        }
    }
    if (escapes && lane < 16 && pl.n_esc + lane < pad16(pl.n_esc)) esc_out[pl.n_esc + lane] = 0;
}

// The partial last chunk (n_c < 4096 elements) is stored raw (section 5,
// "Handling data alignment").  One warp; `vals` are its n_c values.
template <typename Src>
__device__ __forceinline__ void write_tail_chunk_warp(Src vals, uint32_t n_c, uint8_t* dst) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t bytes = (uint32_t)(16 + pad16(2 * n_c));
    uint16_t* out = reinterpret_cast<uint16_t*>(dst + 16);
    for (uint32_t i = lane; i < n_c; i += 32) out[i] = vals(i);
    if (lane == 0) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(kModeRaw, n_c, bytes, 0u);
        for (uint32_t b = 16 + 2 * n_c; b < bytes; ++b) dst[b] = 0;
    }
}

__host__ __device__ constexpr uint32_t tail_chunk_bytes(uint32_t n_c) { return (uint32_t)(16 + pad16(2 * n_c)); }

// Group placement.  Every thread of the CTA calls it after each warp w has
// stored its chunk's size (0 for a chunk past the end) in s_bytes[w].  Warp 0
// scans the sizes and runs the look-back for group g; returns (to every
// thread) the byte offset of warp w's chunk, or kFlagPoison.
// A CTA whose chunks could not be sized (`failed`, CTA-uniform) publishes a
// poisoned placement so that the groups after it give up at once.
template <int G>
__device__ __forceinline__ uint64_t place_group(const StreamOut& so, uint64_t g, const uint32_t* s_bytes,
                                                uint64_t* s_offset, bool failed) {
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (__syncthreads_or(failed)) {
        if (threadIdx.x == 0) st_relaxed_u64(&so.status[g], kFlagPoison);
        return kFlagPoison;
    }
    if (w == 0) {
        const uint32_t mine = lane < (uint32_t)G ? s_bytes[lane] : 0u;
        uint32_t incl = mine;
#pragma unroll
        for (int d = 1; d < G; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += t;
        }
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, G - 1);
        const uint64_t go = lookback_offset_wide(so.status, g, total, data_start(so.n_chunks), so.ws);
        if (lane < (uint32_t)G) s_offset[lane] = go == kFlagPoison ? kFlagPoison : go + (incl - mine);
    }
    __syncthreads();
    return s_offset[w];
}

// Thread 0 of the warp that wrote chunk c: offset-table entry, the stream
// header (chunk 0) and the stream size (last chunk).
__device__ __forceinline__ void finish_chunk(const StreamOut& so, uint64_t c, uint64_t offset, uint32_t bytes) {
    uint8_t* out = so.out;
    *reinterpret_cast<uint64_t*>(out + kStreamHeaderBytes + 8 * c) = offset;
    if (c == 0) {
        *reinterpret_cast<uint4*>(out + 0) = make_uint4(kMagic, kVersion | (kDtypeBf16 << 16), kChunkElems, 0u);
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

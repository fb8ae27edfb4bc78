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
    uint32_t base;   // header base: minimum exponent (0 when raw)
    uint32_t n_esc;  // escapes at width k
    uint32_t emin;   // minimum exponent (kept for raw chunks too)
    uint32_t k1;     // width whose escape bits are kept in ChunkRegs::esc
    uint32_t bytes;  // chunk size, header included
};

// One lane's share of a full chunk, kept in registers between sizing and
// writing: its 128 elements as 32 quads of exponent offsets from the chunk
// minimum, quad 8 q + m holding row 4 q + m / 2, elements 4 (m % 2) .. +3 of
// the lane's 8.  esc[q] holds the escape bits at width k1 in bit-plane layout
// (bit 8 b + m: byte b of quad 8 q + m).  The sign+fraction bytes wait in
// shared memory instead: sizing writes them over the first half of the
// chunk's own (consumed) input slot, in stream order.
struct ChunkRegs {
    uint32_t off[32];
    uint32_t esc[4];
};

// This lane's 4 pair-words of row j (elements 256 j + 8 l .. + 7).
__device__ __forceinline__ uint4 lds_row(const uint8_t* chunk, uint32_t j, uint32_t lane) {
    return *reinterpret_cast<const uint4*>(chunk + 512 * j + 16 * lane);
}

// Escape bits (bit-plane layout) of 8 quads of offsets at width k, and their
// number: the bits of element (m, b) sit at 8 b + m.
__device__ __forceinline__ uint32_t escape_bits8(const uint32_t* off, uint32_t k) {
    const uint32_t kb = (128u - ((1u << k) - 1u)) * 0x01010101u;
    uint32_t acc = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) acc |= ge_flags(off[m], kb) >> (7 - m);
    return acc;
}

// Phase A: exponent table and size of the full chunk at `chunk` (8192 bytes
// of bf16 in shared memory), leaving the offsets in `r` and the chunk's
// sign+fraction plane over the first 4096 bytes of `chunk`.  One warp; every
// lane returns the same plan.
__device__ __forceinline__ ChunkPlan plan_chunk_warp(uint8_t* chunk, ChunkRegs& r) {
    const uint32_t lane = threadIdx.x & 31;
    // pass 1: exponent extremes
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint4 v = lds_row(chunk, j, lane);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // doubling drops each value's sign; a low lane's sign lands in the
            // high lane's last fraction bit, which cannot move its exponent
            const uint32_t mag2 = w[i] << 1;
            mn = vmin_u16x2(mn, mag2);
            mx = vmax_u16x2(mx, mag2);
        }
    }
    const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, min(mn & 0xFFFFu, mn >> 16) >> 8);
    const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16) >> 8);
    const uint32_t base4 = emin * 0x01010101u;
    // pass 2: split every row; its sign+fraction bytes go to their place in
    // the stream's byte plane (row j -> bytes 256 j ..), over input already read
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint4 v = lds_row(chunk, j, lane);
        uint32_t s0, s1;
        split_quad(v.x, v.y, r.off[2 * j], s0);
        split_quad(v.z, v.w, r.off[2 * j + 1], s1);
        r.off[2 * j] -= base4;  // no borrow: every exponent >= emin
        r.off[2 * j + 1] -= base4;
        __syncwarp();  // all lanes have read row j (and row j / 2 before it)
        *reinterpret_cast<uint2*>(chunk + 256 * j + 8 * lane) = make_uint2(s0, s1);
    }

    ChunkPlan pl{0u, 0u, emin, 0u, emin, 0u, 0u};
    const uint32_t range = emax - emin;
    uint32_t best = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) r.esc[q] = 0;
    if (range > 0) {
        const uint32_t kfull = 32 - __clz(range + 1);  // 2..9
        int bk = -1;
        uint32_t bsize = 0xFFFFFFFFu, besc = 0;
        if (kfull <= 7) {
            bk = (int)kfull;
            bsize = kPlaneBytes * kfull;
        }
        // widths below k1 can only win when 512 k + pad16(n_esc(k1)) does not
        // exceed the best size (n_esc never shrinks as k shrinks)
        const uint32_t k1 = min(kfull - 1, 7u);
        pl.k1 = k1;
        uint32_t c1 = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            r.esc[q] = escape_bits8(r.off + 8 * q, k1);
            c1 += __popc(r.esc[q]);
        }
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
                for (int q = 0; q < 4; ++q) ck += __popc(escape_bits8(r.off + 8 * q, (uint32_t)k2));
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

// Escape bytes of a packed chunk, in bit-plane order: plane word 32 q + l,
// then bit.  e0..e3: this lane's escape bits of quarters 0..3, i.e. exactly
// the sentinel bits of its plane words; offw: this lane's 32 offset words,
// word m at offw[32 m] (shared memory, one column per lane).
__device__ __forceinline__ void write_escapes(uint32_t e0, uint32_t e1, uint32_t e2, uint32_t e3, const uint32_t* offw,
                                              uint32_t base, uint32_t n_esc, uint8_t* esc_out) {
    const uint32_t lane = threadIdx.x & 31;
    // escapes before word (q, lane): all of quarters < q, then lanes < lane of quarter q
    const uint32_t c01 = __popc(e0) | (__popc(e1) << 16), c23 = __popc(e2) | (__popc(e3) << 16);
    uint32_t a = c01, b = c23;  // 16-bit fields: at most 1024 per quarter
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t ta = __shfl_up_sync(0xFFFFFFFFu, a, d), tb = __shfl_up_sync(0xFFFFFFFFu, b, d);
        if (lane >= (uint32_t)d) {
            a += ta;
            b += tb;
        }
    }
    const uint32_t ta = __shfl_sync(0xFFFFFFFFu, a, 31), tb = __shfl_sync(0xFFFFFFFFu, b, 31);
    const uint32_t t0 = ta & 0xFFFFu, t1 = ta >> 16, t2 = tb & 0xFFFFu;
    const uint32_t ea = a - c01, eb = b - c23;  // exclusive over lanes
    const uint32_t qb[4] = {ea & 0xFFFFu, t0 + (ea >> 16), t0 + t1 + (eb & 0xFFFFu), t0 + t1 + t2 + (eb >> 16)};
    const uint32_t em[4] = {e0, e1, e2, e3};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t rest = em[q];
        while (rest) {
            const uint32_t bit = __ffs(rest) - 1;
            rest &= rest - 1;
            const uint32_t idx = qb[q] + __popc(em[q] & ((1u << bit) - 1u));
            const uint32_t ow = offw[32 * (8 * q + (bit & 7))];
            if (idx < n_esc) esc_out[idx] = (uint8_t)(((ow >> (8 * (bit >> 3))) & 0xFFu) + base);
        }
    }
}

// Phase B: write the full chunk held in `r` (offsets) and `chunk` (its
// sign+fraction plane, in shared memory) to `dst` (global, 16-byte aligned)
// following `pl`.  One warp.  A packed chunk's byte plane leaves by one bulk
// (TMA) store issued by lane 0, which waits until it has read `chunk` before
// returning; a raw chunk's values are rebuilt in registers.  Uses the second
// half of `chunk` (consumed input) as scratch.
__device__ __forceinline__ void write_chunk_warp(const ChunkRegs& r, const ChunkPlan& pl, uint8_t* chunk,
                                                 uint8_t* dst) {
    const uint32_t lane = threadIdx.x & 31;
    uint8_t* body = dst + kChunkHeaderBytes;
    if (lane == 0)
        *reinterpret_cast<uint4*>(dst) =
            make_uint4((pl.raw ? kModeRaw : kModePacked) | (pl.k << 8) | (pl.base << 16), kChunkElems | (pl.n_esc << 16),
                       pl.bytes, 0u);
    if (pl.raw) {  // rebuild the values from the offsets and the sign+fraction plane
        const uint32_t base4 = pl.emin * 0x01010101u;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint2 sv = *reinterpret_cast<const uint2*>(chunk + 256 * j + 8 * lane);
            uint4 v;
            join_quad(r.off[2 * j] + base4, sv.x, v.x, v.y);
            join_quad(r.off[2 * j + 1] + base4, sv.y, v.z, v.w);
            *reinterpret_cast<uint4*>(body + 512 * j + 16 * lane) = v;
        }
        return;
    }
    // the sign+fraction plane was written by generic stores: order them before
    // the bulk copy's reads
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        bulk_store(body, chunk, kSmPlaneBytes);
        bulk_commit();
    }
    const uint32_t k = pl.k;
    if (k > 0) {
        const bool escapes = pl.n_esc > 0;
        uint32_t em[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // escaped elements carry the sentinel (all k bits set): OR their
            // bits into every plane; the offset bits of the others are their codes
            if (escapes) em[q] = (k == pl.k1) ? r.esc[q] : escape_bits8(r.off + 8 * q, k);
            uint8_t* col = body + kSmPlaneBytes + 4 * (32 * q + lane);
            if (k >= 4) {  // one 8x8 bit transpose makes every plane
                uint32_t W[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) W[m] = r.off[8 * q + m];
                transpose8x8x4(W);
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    if ((uint32_t)p < k) *reinterpret_cast<uint32_t*>(col + kPlaneBytes * p) = W[p] | em[q];
            } else {
#pragma unroll 1
                for (uint32_t p = 0; p < k; ++p)
                    *reinterpret_cast<uint32_t*>(col + kPlaneBytes * p) = pack_plane(r.off + 8 * q, p) | em[q];
            }
        }
        if (escapes) {
            uint32_t* offw = reinterpret_cast<uint32_t*>(chunk + kSmPlaneBytes) + lane;
#pragma unroll
            for (int m = 0; m < 32; ++m) offw[32 * m] = r.off[m];
            __syncwarp();
            uint8_t* esc_out = body + kSmPlaneBytes + kPlaneBytes * k;
            write_escapes(em[0], em[1], em[2], em[3], offw, pl.emin, pl.n_esc, esc_out);
            if (lane < 16 && pl.n_esc + lane < pad16(pl.n_esc)) esc_out[pl.n_esc + lane] = 0;
        }
    }
    if (lane == 0) bulk_wait_read();
    __syncwarp();
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

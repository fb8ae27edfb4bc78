// cccl_encode.cuh -- encoding one chunk held in registers and placing it in
// the output stream (shared by the compress and fused-reduce kernels).
//
// Per chunk ("CCCL: In-GPU Compression-Coupled Collective Communication"):
//   section 4.1  split every bf16 into its exponent and a sign+fraction byte;
//   section 4.3  the chunk's own table: base = minimum exponent, width k that
//                minimises 512 k + pad16(#escapes), fixed-length k-bit codes;
//   section 4.4  the chunk is written once, straight into its final place,
//                found by a decoupled look-back over the chunks before it;
//   section 5    the partial last chunk is stored raw.
#pragma once

#include "cccl_device.cuh"

namespace cccl {

struct EncodeSmem {
    uint32_t wmin[4], wmax[4];  // per-warp exponent extremes
    uint32_t cnt[4][8];         // per-warp escape counts, by width
    uint32_t row_tot[16];       // escapes per 256-element row
    uint64_t offset;            // this chunk's byte offset (or kFlagPoison)
};

struct StreamOut {
    uint8_t* out;        // stream base (16-byte aligned)
    uint64_t capacity;   // bytes writable at out (>= the compress bound)
    uint64_t* status;    // one placement word per chunk
    WsHeader* ws;
    uint64_t n_elems;
    uint64_t n_chunks;
};

// Thread 0 only: offset-table entry, the stream header (chunk 0) and the
// stream size (last chunk).
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

// Number of this thread's elements whose offset is >= 2^k - 1.
__device__ __forceinline__ uint32_t count_escapes(const uint32_t off[8], uint32_t k) {
    const uint32_t kb = (128u - ((1u << k) - 1u)) * 0x01010101u;
    uint32_t f[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) f[m] = ge_flags(off[m], kb);
    return count_flags8(f);
}

// Encode a full chunk c whose 16 words of bf16 pairs per thread are in P
// (word 4 jj + w of thread (q, l) = elements 256 (4q + jj) + 8 l + 2w, +1).
// All 128 threads call it.
__device__ __forceinline__ void encode_full_chunk(const uint32_t P[16], uint64_t c, const StreamOut& so,
                                                  EncodeSmem& sm) {
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;

    // -- split and exponent extremes (section 4.1)
    uint32_t E[8], S[8];
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int w = 0; w < 16; ++w) {
        const uint32_t mag = P[w] & 0x7FFF7FFFu;  // |x| orders like the exponent
        mn = vmin_u16x2(mn, mag);
        mx = vmax_u16x2(mx, mag);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) split_quad(P[2 * m], P[2 * m + 1], E[m], S[m]);
    uint32_t emin = min(mn & 0xFFFFu, mn >> 16) >> 7;
    uint32_t emax = max(mx & 0xFFFFu, mx >> 16) >> 7;
    emin = __reduce_min_sync(0xFFFFFFFFu, emin);
    emax = __reduce_max_sync(0xFFFFFFFFu, emax);
    if (lane == 0) {
        sm.wmin[q] = emin;
        sm.wmax[q] = emax;
    }
    __syncthreads();
    emin = min(min(sm.wmin[0], sm.wmin[1]), min(sm.wmin[2], sm.wmin[3]));
    emax = max(max(sm.wmax[0], sm.wmax[1]), max(sm.wmax[2], sm.wmax[3]));
    const uint32_t range = emax - emin;
    const uint32_t base4 = emin * 0x01010101u;
    uint32_t off[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) off[m] = E[m] - base4;  // no borrow: every exponent >= emin

    // -- choose the width (section 4.3).  Candidates are 1..min(kfull, 7),
    // kfull being the narrowest width without escapes; a width below K1 can
    // only win if 512 k + pad16(n_esc(K1)) does not exceed the best size,
    // since n_esc never shrinks as k shrinks.
    int k = 0;
    uint32_t n_esc = 0, best = 0;
    int kfull = 0;
    if (range > 0) {
        kfull = 32 - __clz(range + 1);  // 2..9
        int bk = -1;
        uint32_t bsize = 0xFFFFFFFFu, besc = 0;
        if (kfull <= 7) {
            bk = kfull;
            bsize = kPlaneBytes * kfull;
        }
        const int k1 = min(kfull - 1, 7);
        const uint32_t c1 = __reduce_add_sync(0xFFFFFFFFu, count_escapes(off, k1));
        if (lane == 0) sm.cnt[q][k1] = c1;
        __syncthreads();
        const uint32_t n1 = sm.cnt[0][k1] + sm.cnt[1][k1] + sm.cnt[2][k1] + sm.cnt[3][k1];
        const uint32_t s1 = kPlaneBytes * k1 + (uint32_t)pad16(n1);
        if (s1 <= bsize) {  // k1 < kfull: a tie keeps the smaller width
            bk = k1;
            bsize = s1;
            besc = n1;
        }
        int kmax = 0;
        for (int kk = k1 - 1; kk >= 1; --kk) {
            if (kPlaneBytes * kk + (uint32_t)pad16(n1) <= bsize) {
                kmax = kk;
                break;
            }
        }
        if (kmax >= 1) {  // CTA-uniform: only chunks with few escapes get here
            for (int kk = 1; kk <= kmax; ++kk) {
                const uint32_t ck = __reduce_add_sync(0xFFFFFFFFu, count_escapes(off, kk));
                if (lane == 0) sm.cnt[q][kk] = ck;
            }
            __syncthreads();
            for (int kk = kmax; kk >= 1; --kk) {
                const uint32_t nk = sm.cnt[0][kk] + sm.cnt[1][kk] + sm.cnt[2][kk] + sm.cnt[3][kk];
                const uint32_t sk = kPlaneBytes * kk + (uint32_t)pad16(nk);
                if (sk <= bsize) {
                    bk = kk;
                    bsize = sk;
                    besc = nk;
                }
            }
        }
        k = bk;
        n_esc = besc;
        best = bsize;
    }
    const bool raw = best >= kSmPlaneBytes;
    const uint32_t bytes = raw ? kMaxChunkBytes : (uint32_t)(16 + kSmPlaneBytes + kPlaneBytes * k + pad16(n_esc));

    // -- placement (section 4.4): warp 0 looks back while the others pack
    if (q == 0) {
        const uint64_t o = lookback_offset(so.status, (uint32_t)c, bytes, data_start(so.n_chunks), so.ws);
        if (lane == 0) sm.offset = o;
    }

    uint32_t W[7] = {0, 0, 0, 0, 0, 0, 0};
    uint32_t FF[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t rb[4] = {0, 0, 0, 0};
    if (!raw && k > 0) {
        uint32_t code[8];
        if (k < kfull) {  // escapes possible: code = sentinel where off >= S
            const uint32_t sent = (1u << k) - 1u;
            const uint32_t kb = (128u - sent) * 0x01010101u;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                FF[m] = flags_to_mask(ge_flags(off[m], kb));
                code[m] = (off[m] & ~FF[m]) | ((sent * 0x01010101u) & FF[m]);
            }
        } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) code[m] = off[m];
        }
        pack_planes_k(k, code, W);
        if (n_esc > 0) {
            uint32_t cnt[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) cnt[jj] = (uint32_t)__popc((FF[2 * jj] & 0x80808080u) | ((FF[2 * jj + 1] & 0x80808080u) >> 1));
            escape_row_bases(cnt, rb, sm.row_tot);
        }
    }
    __syncthreads();
    const uint64_t o = sm.offset;
    if (o == kFlagPoison) return;  // a predecessor failed: the stream is void
    if (o + bytes > so.capacity) {  // cannot happen for a correct placement; never write past the buffer
        if (t == 0) record_error(so.ws, kStatusCorrupt);
        return;
    }
    uint8_t* ch = so.out + o;

    if (t == 0) {
        const uint32_t mode = raw ? kModeRaw : kModePacked;
        const uint32_t hk = raw ? 0u : (uint32_t)k, hb = raw ? 0u : emin, he = raw ? 0u : n_esc;
        *reinterpret_cast<uint4*>(ch) = make_uint4(mode | (hk << 8) | (hb << 16), kChunkElems | (he << 16), bytes, 0u);
    }
    if (raw) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<uint4*>(ch + 16 + 512 * (4 * q + jj) + 16 * lane) =
                make_uint4(P[4 * jj], P[4 * jj + 1], P[4 * jj + 2], P[4 * jj + 3]);
    } else {
        uint8_t* body = ch + 16;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<uint2*>(body + 256 * (4 * q + jj) + 8 * lane) = make_uint2(S[2 * jj], S[2 * jj + 1]);
#pragma unroll
        for (int p = 0; p < 7; ++p)
            if (p < k) *reinterpret_cast<uint32_t*>(body + kSmPlaneBytes + kPlaneBytes * p + 4 * (32 * q + lane)) = W[p];
        if (n_esc > 0) {
            uint8_t* esc = body + kSmPlaneBytes + kPlaneBytes * k;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint32_t idx = rb[jj];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 2 * jj + h;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        if ((FF[m] >> (8 * b)) & 0x80u) {
                            if (idx < n_esc) esc[idx] = (uint8_t)(E[m] >> (8 * b));
                            ++idx;
                        }
                    }
                }
            }
            if (t == 0)
                for (uint32_t i = n_esc; i < pad16(n_esc); ++i) esc[i] = 0;
        }
    }
    if (t == 0) finish_chunk(so, c, o, bytes);
}

// The partial last chunk (n_c < 4096 elements) is stored raw (section 5,
// "Handling data alignment").  P holds its elements in the usual layout;
// elements at or past n_c are ignored.  All 128 threads call it.
__device__ __forceinline__ void encode_tail_chunk(const uint32_t P[16], uint64_t c, uint32_t n_c, const StreamOut& so,
                                                  EncodeSmem& sm) {
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;
    const uint32_t bytes = (uint32_t)(16 + pad16(2 * n_c));
    if (q == 0) {
        const uint64_t o = lookback_offset(so.status, (uint32_t)c, bytes, data_start(so.n_chunks), so.ws);
        if (lane == 0) sm.offset = o;
    }
    __syncthreads();
    const uint64_t o = sm.offset;
    if (o == kFlagPoison) return;
    if (o + bytes > so.capacity) {
        if (t == 0) record_error(so.ws, kStatusCorrupt);
        return;
    }
    uint8_t* ch = so.out + o;
    uint16_t* vals = reinterpret_cast<uint16_t*>(ch + 16);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint32_t i = 256 * (4 * q + jj) + 8 * lane + s;
            if (i < n_c) vals[i] = (uint16_t)(P[4 * jj + s / 2] >> (16 * (s & 1)));
        }
    }
    if (t == 0) {
        *reinterpret_cast<uint4*>(ch) = make_uint4(kModeRaw, n_c, bytes, 0u);
        for (uint32_t b = 16 + 2 * n_c; b < bytes; ++b) ch[b] = 0;
        finish_chunk(so, c, o, bytes);
    }
}

}  // namespace cccl

// cccl_device.cuh -- device building blocks shared by the compress, decompress
// and fused-reduce kernels (sm_103a).
//
// Thread layout of a 4096-element chunk: 4 quarters q of 32 lanes l; lane l
// of quarter q owns the 32 elements
//   i = 256 j + 8 l + s,   j = 4 q + jj (jj < 4),  s < 8,
// i.e. four 16-byte rows of the chunk (bf16); a warp's 32 lanes cover 512
// contiguous bytes per row, so global loads and stores are fully coalesced
// 16-byte accesses.  The stream's bit-plane word 32 q + l holds exactly these
// 32 elements (bit 8 (s % 4) + 2 jj + s / 4), so packing and unpacking the
// exponent codes never leaves the thread.  A decode or encode team is four
// warps, one quarter each; a compress pair is two warps, two quarters each.
//
// Inside a thread, 4 elements travel in one 32-bit word, one byte each
// ("quads", element s = 4 h + b in byte b): m = 2 jj + h indexes the 8
// quads.  All exponent work is byte-SIMD on these words.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace cccl {

constexpr uint32_t kChunkElems = 4096;
constexpr uint32_t kStreamHeaderBytes = 64;
constexpr uint32_t kChunkHeaderBytes = 16;
constexpr uint32_t kSmPlaneBytes = 4096;
constexpr uint32_t kPlaneBytes = 512;
constexpr uint32_t kMaxChunkBytes = kChunkHeaderBytes + 2 * kChunkElems;  // 8208: a raw full chunk
constexpr uint32_t kMagic = 0x31424343u;                                  // "CCB1"
constexpr uint32_t kVersion = 1;
constexpr uint32_t kVersionWindow = 2;  // window-base variant: same layout, other table choice

// Element types: section 4.1's split (the exponent re-encoded, sign and
// fraction kept verbatim), worked out for bf16 and taken with the field widths
// of fp16 (5-bit exponent) and fp32 (8-bit exponent).  A packed chunk's body
// is the type's residual section (kResidBytes: sign and fraction), then k
// exponent planes, then the escapes.
//   bf16: byte plane = sign << 7 | fraction bits 0..6;
//   fp16: byte plane = fraction bits 0..7, then three bit-planes holding
//         fraction bit 8, fraction bit 9 and the sign;
//   fp32: the upper half is a bf16 pattern and is coded as one; the byte
//         plane is its sign+fraction byte, followed by the 4096 lower halves.
// Widths run 1..kExpBits - 1; a chunk is packed only when its exponent part
// is smaller than the exponents stored verbatim (512 bytes per exponent bit).
struct Bf16 {
    static constexpr uint32_t kCode = 1, kElemBytes = 2, kExpBits = 8;
    static constexpr uint32_t kResidBytes = kSmPlaneBytes;
};
struct Fp16 {
    static constexpr uint32_t kCode = 2, kElemBytes = 2, kExpBits = 5;
    static constexpr uint32_t kResidBytes = kSmPlaneBytes + 3 * kPlaneBytes;
};
struct Fp32 {
    static constexpr uint32_t kCode = 3, kElemBytes = 4, kExpBits = 8;
    static constexpr uint32_t kResidBytes = kSmPlaneBytes + 2 * kChunkElems;
};
constexpr uint32_t kDtypeBf16 = Bf16::kCode;
template <class D>
__host__ __device__ constexpr uint32_t max_width() { return D::kExpBits - 1; }
template <class D>
__host__ __device__ constexpr uint32_t raw_exponent_bytes() { return kPlaneBytes * D::kExpBits; }
template <class D>
__host__ __device__ constexpr uint32_t max_chunk_bytes() { return kChunkHeaderBytes + D::kElemBytes * kChunkElems; }
// 32-bit words of one thread's 32 elements
template <class D>
__host__ __device__ constexpr int thread_words() { return (int)D::kElemBytes * 8; }

template <class D>
__device__ __forceinline__ bool known_version_word(uint32_t w1) {
    return w1 == (kVersion | (D::kCode << 16)) || w1 == (kVersionWindow | (D::kCode << 16));
}
constexpr uint32_t kModePacked = 0;
constexpr uint32_t kModeRaw = 1;

// device status codes (same values as cccl_status)
constexpr uint32_t kStatusInvalidArg = 1;  // a block table entry outside its pool
constexpr uint32_t kStatusCorrupt = 3;
constexpr uint32_t kStatusTimeout = 4;

// Workspace: 16-byte header, then one placement word per chunk.
struct WsHeader {
    uint32_t ticket;       // next chunk index to hand out (compress, reduce)
    uint32_t error;        // 0 or the largest device status seen
    uint64_t total_bytes;  // stream size, written by the last chunk
};

// Where chunk c's 4096 values live: c * 4096 in a contiguous buffer (no
// table), or in block table[c / chunks_per_block] of a pool of equal blocks
// (a paged KV-cache payload).  Returns kBadChunk for a table entry outside
// the pool.
struct Paging {
    const int32_t* table;       // device block table, or nullptr
    uint64_t chunks_per_block;  // block_elems / 4096
    uint64_t pool_blocks;
};
constexpr uint64_t kBadChunk = ~0ull;
__device__ __forceinline__ uint64_t chunk_elem_offset(const Paging& pg, uint64_t c) {
    if (pg.table == nullptr) return c * kChunkElems;
    const uint64_t blk = c / pg.chunks_per_block, j = c - blk * pg.chunks_per_block;
    const int32_t e = pg.table[blk];
    if (e < 0 || (uint64_t)e >= pg.pool_blocks) return kBadChunk;
    return ((uint64_t)e * pg.chunks_per_block + j) * kChunkElems;
}

// Placement word of the decoupled look-back: flag in bits 62..63.
constexpr uint64_t kFlagAggregate = 1ull << 62;  // value = this chunk's bytes
constexpr uint64_t kFlagPrefix = 2ull << 62;     // value = end offset of this chunk
constexpr uint64_t kFlagPoison = 3ull << 62;     // a predecessor failed; give up
constexpr uint64_t kValueMask = (1ull << 62) - 1;

// Bounded waits: every spin gives up after kWaitLimitNs of GPU time (read
// from %globaltimer), records kStatusTimeout and returns; nothing waits
// forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__host__ __device__ constexpr uint64_t pad16(uint64_t x) { return (x + 15) & ~uint64_t(15); }
__host__ __device__ constexpr uint64_t data_start(uint64_t n_chunks) { return kStreamHeaderBytes + pad16(8 * n_chunks); }

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t vmin_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void record_error(WsHeader* ws, uint32_t status) { atomicMax(&ws->error, status); }
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// bulk (TMA) copy global -> shared, completion on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// One thread: expect `bytes` on `bar` and start the copy (bytes % 16 == 0,
// both addresses 16-byte aligned, checked by the caller).
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// One thread: bulk (TMA) copy shared -> global (bytes % 16 == 0, both
// addresses 16-byte aligned); completion tracked by bulk groups.
__device__ __forceinline__ void bulk_store(void* dst_gmem, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the committed bulk stores of this thread have read their source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until the committed bulk stores of this thread have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Barriers over the threads that decode or encode one chunk together: the
// whole CTA, or a named barrier over the 4 warps of a team (every
// participating warp executes it as a whole).
struct CtaBarrier {
    __device__ void sync() const { __syncthreads(); }
    __device__ bool any(bool p) const { return __syncthreads_or(p) != 0; }
};
struct TeamBarrier {
    uint32_t id;  // 1..15; barrier 0 is __syncthreads'
    __device__ void sync() const { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
    __device__ bool any(bool p) const {
        uint32_t r;
        asm volatile(
            "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.or.pred po, %2, 128, pi; selp.u32 %0, 1, 0, po; }"
            : "=r"(r)
            : "r"((uint32_t)p), "r"(id)
            : "memory");
        return r != 0;
    }
};

// Non-blocking: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`; false if kWaitLimitNs ran out.
// Each try suspends the warp in hardware (up to kSuspendHintNs) until the
// phase completes, so a waiting warp costs no issue slots.
constexpr uint32_t kSuspendHintNs = 100000;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_addr(bar);
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(kSuspendHintNs)
            : "memory");
        if (ok) return true;
        const uint64_t now = globaltimer_ns();
        if (it == 0)
            t0 = now;
        else if (now - t0 > kWaitLimitNs)
            return false;
    }
}

// ---------------------------------------------------------------------------
// bf16 split / join on quads (section 4.1: sign and fraction travel raw,
// only the 8-bit exponent is re-encoded)
// ---------------------------------------------------------------------------
// e: four exponents, one per byte; sm: the four sign+fraction bytes
// ((b >> 8) & 0x80 | b & 0x7F).  Joined into two words of two bf16 each
// (elements 4h+0, 4h+1 in A; 4h+2, 4h+3 in B).
__device__ __forceinline__ void join_quad(uint32_t e, uint32_t sm, uint32_t& A, uint32_t& B) {
    const uint32_t lo = (sm & 0x7F7F7F7Fu) | ((e << 7) & 0x80808080u);
    const uint32_t hi = (sm & 0x80808080u) | ((e >> 1) & 0x7F7F7F7Fu);
    A = __byte_perm(lo, hi, 0x5140);
    B = __byte_perm(lo, hi, 0x7362);
}

// fp16 quads.  A, B: two words of two fp16 each (elements 4h+0, 4h+1 in A;
// 4h+2, 4h+3 in B).  Per value the high byte is sign | exponent (5 bits) |
// fraction bits 9, 8; the quad moves the exponent to bits 0..4 and keeps the
// other three bits above it: fraction bit 8 in bit 5, bit 9 in bit 6, the
// sign in bit 7.  Subtracting a base <= every exponent leaves bits 5..7 alone.
__device__ __forceinline__ uint32_t fp16_exponent_quad(uint32_t A, uint32_t B) {
    const uint32_t H = __byte_perm(A, B, 0x7531);
    return ((H >> 2) & 0x1F1F1F1Fu) | ((H & 0x03030303u) << 5) | (H & 0x80808080u);
}
// The two fp16 exponents of a pair-word in the high byte of each 16-bit lane.
__device__ __forceinline__ uint32_t fp16_exponent_lanes(uint32_t A) { return (A >> 2) & 0x1F001F00u; }
// Inverse: low fraction bytes L, exponents E (one per byte, <= 31) and the
// quad bits 5..7 in R -> two pair-words.
__device__ __forceinline__ void join_quad_fp16(uint32_t E, uint32_t R, uint32_t L, uint32_t& A, uint32_t& B) {
    const uint32_t H = (R & 0x80808080u) | (E << 2) | ((R >> 5) & 0x03030303u);
    A = __byte_perm(L, H, 0x5140);
    B = __byte_perm(L, H, 0x7362);
}
// fp32 halves: the upper (bf16) halves, and the lower halves, of two values
// as one pair-word each; and back.
__device__ __forceinline__ uint32_t upper_halves(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }
__device__ __forceinline__ uint32_t lower_halves(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5410); }
__device__ __forceinline__ uint32_t join_first(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x5410); }
__device__ __forceinline__ uint32_t join_second(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x7632); }

// Byte flags (0x80 per byte) of the bytes of `off` that are >= S, 1 <= S <= 127;
// kb = (128 - S) * 0x01010101.  No carry crosses a byte.
__device__ __forceinline__ uint32_t ge_flags(uint32_t off, uint32_t kb) {
    return (off | ((off & 0x7F7F7F7Fu) + kb)) & 0x80808080u;
}
// 0x80 flags -> 0xFF byte masks
__device__ __forceinline__ uint32_t flags_to_mask(uint32_t f) { return f | (f - (f >> 7)); }

// ---------------------------------------------------------------------------
// bit-planes: plane p word = over quads m and bytes b, bit p of code(m, b) at
// bit 8 b + m.  Moving bit 8 b + p to 8 b + m is a rotation by (p - m) mod 32
// that never wraps (8 b + m and 8 b + p both lie in 0..31), so one funnel
// rotate and one masked OR per (quad, plane) serve every width at run time.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t rotr(uint32_t x, uint32_t n) { return __funnelshift_r(x, x, n); }

// All 8 planes at once: 8 quads hold, per byte lane b, an 8x8 bit matrix
// (row m = quad m, column p = bit p); transposing it turns codes into plane
// words and back (plane p = row p).  Recursive block transpose in three
// rounds (4x4, 2x2, 1x1 blocks), the same for every byte lane since no
// exchange crosses a byte.
// Exchange the off-diagonal s x s blocks of rows a and b (a before b):
// the bits of a selected by ~M move down by s into b's M bits and b's M bits
// move up into a's ~M bits (each a single bit-select).
__device__ __forceinline__ void block_swap(uint32_t& a, uint32_t& b, uint32_t s, uint32_t M) {
    const uint32_t na = (a & M) | ((b << s) & ~M);
    const uint32_t nb = ((a >> s) & M) | (b & ~M);
    a = na;
    b = nb;
}
__device__ __forceinline__ void transpose8x8x4(uint32_t* v) {
#pragma unroll
    for (int m = 0; m < 4; ++m) block_swap(v[m], v[m + 4], 4, 0x0F0F0F0Fu);
#pragma unroll
    for (int m = 0; m < 8; m += 4) {
        block_swap(v[m], v[m + 2], 2, 0x33333333u);
        block_swap(v[m + 1], v[m + 3], 2, 0x33333333u);
    }
#pragma unroll
    for (int m = 0; m < 8; m += 2) block_swap(v[m], v[m + 1], 1, 0x55555555u);
}

// OR plane word w (plane p) into 8 quads of codes.
__device__ __forceinline__ void unpack_plane(uint32_t w, uint32_t p, uint32_t* code) {
    const uint32_t mask = 0x01010101u << p;
#pragma unroll
    for (int m = 0; m < 8; ++m) code[m] |= rotr(w, ((uint32_t)m - p) & 31u) & mask;
}

// ---------------------------------------------------------------------------
// decoupled look-back (one warp) over placement units (groups of chunks).
// Units are numbered in the order their CTAs took a ticket, so every
// predecessor is already running and publishes its size without waiting on
// anything later: the wait always ends.  Each round trip reads 256
// predecessors (8 independent loads per lane), so a look-back that must walk
// past the units still in flight needs few round trips.
// Returns the byte offset of unit g, or kFlagPoison if a predecessor failed
// or the bounded wait ran out (then kStatusTimeout is recorded).
// ---------------------------------------------------------------------------
constexpr int kLookbackPerLane = 8;
constexpr uint32_t kLookbackWindow = 32 * kLookbackPerLane;

// Publish unit g's size: its end offset when g == 0, else its aggregate.
__device__ __forceinline__ void publish_unit_size(uint64_t* status, uint64_t g, uint32_t bytes, uint64_t start) {
    st_relaxed_u64(&status[g], g == 0 ? (kFlagPrefix | (start + bytes)) : (kFlagAggregate | bytes));
}

// `published`: the unit's size was already published with publish_unit_size.
// `max_nap_ns`: the longest back-off between polls of an unfinished window
// (a caller off the critical path polls less often, leaving issue slots to
// the warps that share its SM sub-partition).
__device__ __forceinline__ uint64_t lookback_offset_wide(uint64_t* status, uint64_t g, uint32_t bytes, uint64_t start,
                                                         WsHeader* ws, bool published = false,
                                                         uint32_t max_nap_ns = 512) {
    const uint32_t lane = threadIdx.x & 31;
    if (!published && lane == 0) publish_unit_size(status, g, bytes, start);
    if (g == 0) return start;
    uint64_t excl = 0;
    int64_t end = (int64_t)g;  // predecessors still to account for: [0, end)
    uint32_t ns = 32;
    uint64_t t0 = 0;
    while (true) {
        uint64_t v[kLookbackPerLane];
#pragma unroll
        for (int i = 0; i < kLookbackPerLane; ++i) {
            const int64_t idx = end - 1 - (int64_t)(lane + 32 * i);
            v[i] = idx >= 0 ? ld_relaxed_u64(&status[idx]) : kFlagPrefix;  // before unit 0: prefix 0
        }
        // nearest terminal (prefix or poison) entry, counted from unit end - 1
        uint32_t first = kLookbackWindow;
#pragma unroll
        for (int i = 0; i < kLookbackPerLane; ++i) {
            const uint32_t t = __ballot_sync(0xFFFFFFFFu, (v[i] >> 62) >= 2);
            if (first == kLookbackWindow && t) first = 32 * i + __ffs(t) - 1;
        }
        bool pending = false;
#pragma unroll
        for (int i = 0; i < kLookbackPerLane; ++i)
            pending |= (lane + 32 * i < first) && (v[i] >> 62) == 0;
        if (__any_sync(0xFFFFFFFFu, pending)) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (now - t0 > kWaitLimitNs) {
                if (lane == 0) {
                    record_error(ws, kStatusTimeout);
                    st_relaxed_u64(&status[g], kFlagPoison);
                }
                return kFlagPoison;
            }
            __nanosleep(ns);
            if (ns < max_nap_ns) ns <<= 1;
            continue;
        }
        uint32_t part = 0;  // aggregates are unit sizes (< 2^17 each)
#pragma unroll
        for (int i = 0; i < kLookbackPerLane; ++i)
            if (lane + 32 * i < first) part += (uint32_t)(v[i] & kValueMask);
        excl += __reduce_add_sync(0xFFFFFFFFu, part);
        if (first < kLookbackWindow) {
            uint64_t tv = 0;
#pragma unroll
            for (int i = 0; i < kLookbackPerLane; ++i) {
                const uint64_t cand = __shfl_sync(0xFFFFFFFFu, v[i], first & 31);
                if ((uint32_t)i == (first >> 5)) tv = cand;
            }
            if ((tv >> 62) == 3) {
                if (lane == 0) st_relaxed_u64(&status[g], kFlagPoison);
                return kFlagPoison;
            }
            excl += tv & kValueMask;
            break;
        }
        end -= kLookbackWindow;
    }
    if (lane == 0) st_relaxed_u64(&status[g], kFlagPrefix | (excl + bytes));
    return excl;
}

// ---------------------------------------------------------------------------
// stream header / chunk header validation (shared by decompress and reduce)
// ---------------------------------------------------------------------------
struct ChunkView {
    uint64_t offset;  // byte offset of the chunk in its stream
    uint32_t bytes;   // chunk size (<= the type's raw full chunk once validated)
    uint32_t ok;      // 1 if the stream header and this chunk's table entries are valid
};

__device__ __forceinline__ uint64_t ld_u64_aligned(const uint8_t* p) { return *reinterpret_cast<const uint64_t*>(p); }
__device__ __forceinline__ uint32_t ld_u32_aligned(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// One thread: check the stream header against (n_elems, in_bytes); returns
// the stream's total size, or 0 if the header is unusable.  Every read stays
// inside in_bytes.
template <class D>
__device__ __forceinline__ uint64_t stream_total(const uint8_t* s, uint64_t in_bytes, uint64_t n_elems,
                                                 uint64_t n_chunks) {
    const uint64_t start = data_start(n_chunks);
    if (in_bytes < start) return 0;
    const uint32_t w0 = ld_u32_aligned(s + 0), w1 = ld_u32_aligned(s + 4), w2 = ld_u32_aligned(s + 8);
    if (w0 != kMagic || !known_version_word<D>(w1) || w2 != kChunkElems) return 0;
    if (ld_u64_aligned(s + 16) != n_elems || ld_u64_aligned(s + 24) != n_chunks) return 0;
    const uint64_t total = ld_u64_aligned(s + 32);
    if (total > in_bytes || total < start) return 0;
    return total;
}

// One thread: locate chunk c through the offset table of a stream whose
// header stream_total accepted (`total` its result, nonzero).  Every read
// stays inside total.
template <class D>
__device__ __forceinline__ ChunkView locate_chunk_at(const uint8_t* s, uint64_t total, uint64_t n_chunks, uint64_t c) {
    ChunkView v{0, 0, 0};
    const uint64_t start = data_start(n_chunks);
    const uint64_t off = ld_u64_aligned(s + kStreamHeaderBytes + 8 * c);
    const uint64_t end = (c + 1 < n_chunks) ? ld_u64_aligned(s + kStreamHeaderBytes + 8 * (c + 1)) : total;
    if (c == 0 && off != start) return v;
    if ((off & 15) != 0 || end <= off || end > total || off < start) return v;
    // the bulk copy needs a size that is a multiple of 16; every valid chunk is
    if (end - off > max_chunk_bytes<D>() || ((end - off) & 15) != 0) return v;
    v.offset = off;
    v.bytes = (uint32_t)(end - off);
    v.ok = 1;
    return v;
}

// Both: check the header, then locate chunk c.
template <class D>
__device__ __forceinline__ ChunkView locate_chunk(const uint8_t* s, uint64_t in_bytes, uint64_t n_elems,
                                                  uint64_t n_chunks, uint64_t c) {
    const uint64_t total = stream_total<D>(s, in_bytes, n_elems, n_chunks);
    if (total == 0) return ChunkView{0, 0, 0};
    return locate_chunk_at<D>(s, total, n_chunks, c);
}

// Decoded chunk header (16 bytes at the start of a staged chunk).
struct ChunkHeader {
    uint32_t mode, k, base, n_c, n_esc, bytes;
};
__device__ __forceinline__ ChunkHeader read_chunk_header(const uint8_t* h) {
    const uint32_t w0 = ld_u32_aligned(h), w1 = ld_u32_aligned(h + 4), w2 = ld_u32_aligned(h + 8);
    ChunkHeader ch;
    ch.mode = w0 & 0xFF;
    ch.k = (w0 >> 8) & 0xFF;
    ch.base = (w0 >> 16) & 0xFF;
    ch.n_c = w1 & 0xFFFF;
    ch.n_esc = w1 >> 16;
    ch.bytes = w2;
    return ch;
}
// Same rules as the format: raw chunks carry no table; a packed chunk is a
// full chunk whose exponent part is smaller than its exponents stored
// verbatim, and whose base is an exponent of the type.
template <class D>
__device__ __forceinline__ bool chunk_header_valid(const ChunkHeader& h, uint32_t staged_bytes, uint32_t n_c) {
    if (h.bytes != staged_bytes || h.n_c != n_c) return false;
    if (h.mode == kModeRaw)
        return h.k == 0 && h.base == 0 && h.n_esc == 0 && h.bytes == 16 + pad16(D::kElemBytes * n_c);
    if (h.mode != kModePacked || n_c != kChunkElems || h.k > max_width<D>() || h.base >= (1u << D::kExpBits))
        return false;
    if (h.k == 0 && h.n_esc != 0) return false;
    if (h.bytes != 16 + D::kResidBytes + kPlaneBytes * h.k + pad16(h.n_esc)) return false;
    return kPlaneBytes * h.k + pad16(h.n_esc) < raw_exponent_bytes<D>();
}

}  // namespace cccl

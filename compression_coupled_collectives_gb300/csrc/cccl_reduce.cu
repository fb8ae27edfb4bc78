// cccl_reduce.cu -- the fused reduce kernel: the reduce step of a compressed
// allreduce as one pass, decompress -> binary32 accumulate in rank order ->
// one rounding to the element type -> compress ("CCCL: In-GPU
// Compression-Coupled Collective Communication", section 5, "Integration into
// the NCCL data path" (CopyReducePacks); Figure 2).  Also min and max.
//
// Persistent and pipelined, one CTA per SM with three roles:
//   teams (warps 0..4T-1)  T independent teams of 4 warps.  Per group of T
//                        consecutive output chunks, team t takes chunk t.
//                        Each warp of the team decodes its quarter of chunk c
//                        of every rank, in rank order, on its own (no team
//                        barrier per rank: the warp counts the escapes of the
//                        quarters before its own itself), keeping 32 binary32
//                        sums per thread in registers.  The team then meets,
//                        rounds once to the element type (bf16, fp16; fp32
//                        needs none), sizes the chunk (two more meetings) and
//                        writes it, in its final byte layout, into one of its
//                        staging buffers in shared memory;
//   loader (warp 4T)     checks every rank's stream header once; takes a
//                        ticket per group, one group ahead; locates every
//                        rank's chunk through its offset table and reads and
//                        checks its header; streams the chunks to the teams
//                        by bulk (TMA) copies, through one ring of staged rank
//                        chunks per team, each team's in rank order, to
//                        whichever team has a slot free; and while the
//                        copies of a group wait for slots, locates the next
//                        group;
//   placer (warp 4T+1)   places each sized group with one decoupled
//                        look-back, then copies the group's staged chunks to
//                        their final places with one bulk (TMA) store each
//                        and writes their offset-table entries.
// So the teams never wait for a placement: the look-back of group i and the
// copies out overlap the decoding of group i + 1, and the copies of later
// rank chunks are in flight meanwhile.  A team meets four times per output
// chunk whatever the number of ranks: after the group's description, after
// its decodes (to agree on timeouts and on Inf/NaN), and twice to size the
// chunk.
// Tickets hand out groups in order to CTAs that are already running, and a
// group is sized without waiting on any later group: every look-back ends.
#include "cccl_decode.cuh"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kMaxTeams = 4;
// The kernel's shape for element type T: T's fields, plus the number of
// decode teams per CTA (= output chunks per group), the depth of each team's
// ring of staged rank chunks and its number of output staging buffers.
// launch_reduce_t picks one per call.
template <class T, int kTeamsV, int kRingSlotsV, int kSBufsV = 2>
struct ReduceShape : T {
    static constexpr int kTeams = kTeamsV;
    static constexpr int kRingSlots = kRingSlotsV;
    static constexpr int kSBufs = kSBufsV;
};
template <class D>
__host__ __device__ constexpr int teams() { return D::kTeams; }
template <class D>
__host__ __device__ constexpr int loader_warp() { return 4 * teams<D>(); }   // also the locator
template <class D>
__host__ __device__ constexpr int copier_warp() { return loader_warp<D>() + 1; }  // idle with one loader warp
template <class D>
__host__ __device__ constexpr int placer_warp() { return copier_warp<D>() + 1; }
// group descriptions in flight: the loader describes group i + 1 while the
// teams may still read those of groups i - 1 and i
constexpr int kMetaBufs = 3;
template <class D>
__host__ __device__ constexpr int reduce_threads() { return 32 * (placer_warp<D>() + 1); }
constexpr uint64_t kNoGroup = ~0ull;
// staged rank chunks per team (8.2 KB each for the 16-bit types, 16.4 KB for fp32)
template <class D>
__host__ __device__ constexpr int rslots() { return D::kRingSlots; }
constexpr int kMaxRSlots = 6;
// output staging buffers per team, cycled by group: with two, a team stages
// the chunk of group i while the placer still copies out the one of group
// i - 1; one is enough when a group's decodes outlast the placer's work
template <class D>
__host__ __device__ constexpr int sbufs() { return D::kSBufs; }
constexpr int kMaxSBufs = 2;
// size records (a group's sizes, tally and index), cycled by group: one more
// than the staging buffers, so that a team publishes the size of group i
// before it waits for the placer to free a staging buffer (the record of
// group i - zslots() is free by then: the team waited for the placer to be
// done with group i - 1 - sbufs() in its previous iteration)
template <class D>
__host__ __device__ constexpr int zslots() { return sbufs<D>() + 1; }
constexpr int kMaxZSlots = kMaxSBufs + 1;
template <class D>
__host__ __device__ constexpr size_t ring_bytes() { return (size_t)teams<D>() * rslots<D>() * max_chunk_bytes<D>(); }
template <class D>
__host__ __device__ constexpr size_t staging_bytes() {
    return (size_t)teams<D>() * sbufs<D>() * max_chunk_bytes<D>();
}
template <class D>
__host__ __device__ constexpr size_t reduce_smem() { return ring_bytes<D>() + staging_bytes<D>(); }

// binary32 pair -> bf16 pair, round to nearest even (hi lane from the upper word)
__device__ __forceinline__ uint32_t round_pair_bf16(uint64_t v) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "r"((uint32_t)(v >> 32)), "r"((uint32_t)v));
    return d;
}
// binary32 pair -> IEEE fp16 pair, round to nearest even, subnormal results
// kept, overflow to Inf (hi lane from the upper word)
__device__ __forceinline__ uint32_t round_pair_fp16(uint64_t v) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "r"((uint32_t)(v >> 32)), "r"((uint32_t)v));
    return d;
}

// 16-bit types: 0xFFFF in every lane that holds a NaN (magnitude above the
// all-ones exponent with a zero fraction: 0x7F80 bf16, 0x7C00 fp16)
template <class D>
__device__ __forceinline__ uint32_t nan_lanes_pair(uint32_t x) {
    constexpr uint32_t kAdd = (0x7FFFu - ((1u << D::kExpBits) - 1u) * (1u << (15 - D::kExpBits))) * 0x00010001u;
    return ((((x & 0x7FFF7FFFu) + kAdd) & 0x80008000u) >> 15) * 0xFFFFu;
}
// the NaN every reduce writes: 0x7FC0 bf16, 0x7E00 fp16, 0x7FC00000 fp32
template <class D>
__host__ __device__ constexpr uint32_t canonical_nan() {
    return D::kElemBytes == 4 ? 0x7FC00000u : (D::kExpBits == 5 ? 0x7E00u : 0x7FC0u);
}
// every NaN lane -> the canonical NaN
template <class D>
__device__ __forceinline__ uint32_t canonical_nan_pair(uint32_t d) {
    const uint32_t mask = nan_lanes_pair<D>(d);
    return (d & ~mask) | (canonical_nan<D>() * 0x00010001u & mask);
}
__device__ __forceinline__ uint32_t canonical_nan_word(uint32_t v) {
    return (v & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : v;
}

// Element-wise min (op 1) or max (op 2), exact: a NaN in either operand gives
// the canonical NaN; otherwise the IEEE total order, -0 below +0, through the
// usual sign-magnitude key (negative: all bits flipped; positive: sign bit
// set), compared as unsigned.
__device__ __forceinline__ uint32_t order_key_pair(uint32_t x) {
    return x ^ ((((x >> 15) & 0x00010001u) * 0x7FFFu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t from_order_key_pair(uint32_t k) {
    return k ^ ((((~k >> 15) & 0x00010001u) * 0x7FFFu) | 0x80008000u);
}
template <class D>
__device__ __forceinline__ uint32_t minmax_pair(uint32_t a, uint32_t b, uint32_t op) {
    const uint32_t ka = order_key_pair(a), kb = order_key_pair(b);
    const uint32_t r = from_order_key_pair(op == 1 ? vmin_u16x2(ka, kb) : vmax_u16x2(ka, kb));
    const uint32_t nan = nan_lanes_pair<D>(a) | nan_lanes_pair<D>(b);
    return (r & ~nan) | (canonical_nan<D>() * 0x00010001u & nan);
}
__device__ __forceinline__ uint32_t minmax_word(uint32_t a, uint32_t b, uint32_t op) {
    const uint32_t ka = a ^ ((uint32_t)((int32_t)a >> 31) | 0x80000000u);
    const uint32_t kb = b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
    const uint32_t k = op == 1 ? min(ka, kb) : max(ka, kb);
    const uint32_t r = k ^ ((uint32_t)((int32_t)~k >> 31) | 0x80000000u);
    const bool nan = (a & 0x7FFFFFFFu) > 0x7F800000u || (b & 0x7FFFFFFFu) > 0x7F800000u;
    return nan ? 0x7FC00000u : r;
}

// Warp-uniform reads of the abort flag and of a bounded wait's outcome.
__device__ __forceinline__ bool warp_any(bool p) { return __any_sync(0xFFFFFFFFu, p); }
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity));
}

// A rank chunk's header, checked by the loader, packed for the teams: base
// in bits 0..7, k in 8..10, raw in bit 11 (also for the uncompressed local
// operand), n_esc in bits 16..31.
__device__ __forceinline__ uint32_t pack_desc(const ChunkHeader& h) {
    return h.base | (h.k << 8) | ((h.mode == kModeRaw ? 1u : 0u) << 11) | (h.n_esc << 16);
}
constexpr uint32_t kDescRaw = 1u << 11;
__device__ __forceinline__ ChunkHeader unpack_desc(uint32_t d) {
    ChunkHeader h;
    h.base = d & 0xFFu;
    h.k = (d >> 8) & 7u;
    h.mode = (d & kDescRaw) ? kModeRaw : kModePacked;
    h.n_esc = d >> 16;
    h.n_c = 0;
    h.bytes = 0;
    return h;
}

// What the loader hands the teams for one group.
struct ReduceMeta {
    uint64_t g;                          // group index, or kNoGroup: no more groups
    uint32_t ok;                         // every (chunk, rank) was located and its header is valid
    uint32_t n_out;                      // output chunks in the group
    uint64_t off[kMaxTeams][kMaxRanks];  // rank r's chunk teams * g + t: offset in its stream
    uint32_t bytes[kMaxTeams][kMaxRanks];  //   its size
    uint32_t desc[kMaxTeams][kMaxRanks];   //   and its header (pack_desc)
};

struct ReduceSmem {
    uint64_t meta_ready[kMetaBufs];      // loader -> teams: meta[b] describes the next group (1 arrival)
    uint64_t decoded[kMetaBufs];         // teams, loader -> loader: meta[b] read (each team warp and the loader)
    uint64_t sized[kMaxZSlots];          // teams -> placer: the group's sizes are in (one arrival per team)
    uint64_t staged[kMaxSBufs];          // teams -> placer: the group's chunks are staged (one per team warp)
    uint64_t stored[kMaxSBufs];          // placer -> teams: the group's staging buffers were read (1 arrival)
    uint64_t full[kMaxTeams][kMaxRSlots];   // a rank chunk landed in the slot (transaction count)
    uint64_t free_[kMaxTeams][kMaxRSlots];  // every warp of the team is done with the slot (4 arrivals)
    unsigned long long tally[kMaxZSlots];   // sized teams (high word) and their bytes (low word)
    uint32_t size[kMaxZSlots][kMaxTeams];
    uint32_t failed[kMaxZSlots][kMaxTeams];  // the team's chunk could not be reduced
    uint64_t gid[kMaxZSlots];               // group sized in record z, or kNoGroup
    int32_t esc_diff[kMaxTeams][kMaxRanks]; // per rank: sentinel codes found minus the header's escapes
    uint32_t corrupt[kMaxTeams][2];         // a rank chunk body is malformed (by iteration parity)
    TeamXch xch[kMaxTeams];                 // the encoder's exchange space
    volatile uint32_t abort;                // a bounded wait ran out: every role stops
    ReduceMeta meta[kMetaBufs];
    uint64_t total[kMaxRanks];              // rank r's stream size from its checked header (0: unusable)
};

__device__ __forceinline__ void set_abort(const StreamOut& so, ReduceSmem& sm) {
    record_error(so.ws, kStatusTimeout);
    sm.abort = 1;
}

// --------------------------------------------------------------------------- loader
// Group j's description, into meta[j % kMetaBufs]: every rank's chunk located
// through its offset table, its header read once and checked.  `next` holds
// (lane 0) the ticket taken one group ahead; `last` is set once the tickets
// run out (the description then says kNoGroup).  False if a bounded wait ran
// out.
template <class D>
__device__ __forceinline__ bool locate_group(const ReduceInputs& inputs, int R, const StreamOut& so, ReduceSmem& sm,
                                             int j, uint64_t& next, bool& last) {
    constexpr int kTeams = teams<D>();
    constexpr uint32_t kRawBytes = D::kElemBytes * kChunkElems;
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t n_groups = (so.n_chunks + kTeams - 1) / kTeams;
    const int b = j % kMetaBufs;
    // meta[b] was last read, by the teams and the loader, for group j - kMetaBufs
    if (j >= kMetaBufs && !warp_wait(&sm.decoded[b], (uint32_t)((j - kMetaBufs) / kMetaBufs) & 1u)) {
        if (lane == 0) set_abort(so, sm);
        return false;
    }
    const uint64_t g = __shfl_sync(0xFFFFFFFFu, next, 0);
    if (lane == 0 && g < n_groups) next = atomicAdd(&so.ws->ticket, 1u);
    ReduceMeta& m = sm.meta[b];
    if (g >= n_groups) {
        if (lane == 0) {
            m.g = kNoGroup;
            mbar_arrive(&sm.meta_ready[b]);
        }
        last = true;
        return true;
    }
    const uint64_t c0 = g * kTeams;
    const uint32_t n_out = (uint32_t)min((uint64_t)kTeams, so.n_chunks - c0);
    bool ok = true;
    for (uint32_t idx = lane; idx < n_out * (uint32_t)R; idx += 32) {
        const uint32_t t = idx / (uint32_t)R, r = idx % (uint32_t)R;
        if (r == 0 && inputs.local != nullptr) {  // uncompressed: chunk c is values 4096 c ..
            const uint64_t c = c0 + t, left = so.n_elems - c * kChunkElems;
            m.off[t][r] = (uint64_t)kRawBytes * c;
            m.bytes[t][r] = D::kElemBytes * (uint32_t)(left < kChunkElems ? left : kChunkElems);
            m.desc[t][r] = kDescRaw;
            continue;
        }
        const uint64_t total = sm.total[r];
        ChunkView v{0, 0, 0};
        if (total != 0) v = locate_chunk_at<D>(inputs.in[r], total, so.n_chunks, c0 + t);
        // the chunk header, read here once (the same bytes the bulk copy
        // stages) and checked against the offset table and the chunk's
        // element count
        if (v.ok) {
            const uint64_t left = so.n_elems - (c0 + t) * kChunkElems;
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(inputs.in[r] + v.offset));
            ChunkHeader h;
            h.mode = w.x & 0xFF;
            h.k = (w.x >> 8) & 0xFF;
            h.base = (w.x >> 16) & 0xFF;
            h.n_c = w.y & 0xFFFF;
            h.n_esc = w.y >> 16;
            h.bytes = w.z;
            if (!chunk_header_valid<D>(h, v.bytes, left < kChunkElems ? (uint32_t)left : kChunkElems)) v.ok = 0;
            m.desc[t][r] = pack_desc(h);
        }
        m.off[t][r] = v.offset;
        m.bytes[t][r] = v.bytes;
        ok = ok && v.ok;
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (lane == 0) {
        m.g = g;
        m.ok = ok ? 1u : 0u;
        m.n_out = n_out;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.meta_ready[b]);
    return true;
}

// The loader warp: per group, in ticket order, its description (locate_group)
// and the bulk (TMA) copies of its rank chunks into the teams' rings, each
// team's in rank order, to whichever team has a slot free.  While the copies
// of group i wait for ring slots, it locates group i + 1, so the description
// of the next group is ready before its slots are.
template <class D>
__device__ __forceinline__ void reduce_loader(const ReduceInputs& inputs, int R, const StreamOut& so, uint8_t* ring,
                                              ReduceSmem& sm) {
    constexpr int kRSlots = rslots<D>();
    constexpr int kTeams = teams<D>();
    constexpr uint32_t kRawBytes = D::kElemBytes * kChunkElems;
    const uint32_t lane = threadIdx.x & 31;
    // every rank's stream header, checked once
    for (int r = (int)lane; r < R; r += 32)
        sm.total[r] = (r == 0 && inputs.local != nullptr)
                          ? 1u
                          : stream_total<D>(inputs.in[r], inputs.in_bytes[r], so.n_elems, so.n_chunks);
    __syncwarp();
    // lane 0: the ticket for the next group, taken one group ahead so that
    // its latency hides behind this group's work
    uint64_t next = 0;
    if (lane == 0) next = atomicAdd(&so.ws->ticket, 1u);
    bool last = false;                        // the tickets have run out
    int located = locate_group<D>(inputs, R, so, sm, 0, next, last) ? 0 : -1;  // last group described
    uint32_t ut[kTeams] = {};  // rank chunks issued to each team
    bool stop = located < 0;
    for (int i = 0; !stop && !warp_any(sm.abort); ++i) {
        const int b = i % kMetaBufs;
        const ReduceMeta& m = sm.meta[b];
        if (m.g == kNoGroup) break;
        const uint32_t n_out = m.n_out;
        // nothing to stream for a group that could not be located: the teams poison it
        uint32_t left = m.ok ? n_out * (uint32_t)R : 0u;
        uint32_t issued[kTeams] = {};  // this group's rank chunks issued to each team
        uint64_t t_blocked = 0;
        uint32_t nap = 32;
        while (left > 0) {
            bool progress = false;
#pragma unroll
            for (int t = 0; t < kTeams; ++t) {
                if (t >= (int)n_out) break;
                while (issued[t] < (uint32_t)R) {
                    const uint32_t s = ut[t] % kRSlots;
                    // the slot's previous rank chunk is consumed
                    if (ut[t] >= (uint32_t)kRSlots && !mbar_test(&sm.free_[t][s], (ut[t] / kRSlots - 1) & 1u)) break;
                    const uint32_t r = issued[t];
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        uint8_t* slot = ring + ((size_t)t * kRSlots + s) * max_chunk_bytes<D>();
                        if (r != 0 || inputs.local == nullptr)
                            bulk_load(slot, inputs.in[r] + m.off[t][r], m.bytes[t][r], &sm.full[t][s]);
                        else if (m.bytes[t][r] == kRawBytes)  // a full local chunk, staged raw
                            bulk_load(slot, static_cast<const uint8_t*>(inputs.local) + m.off[t][r], kRawBytes,
                                      &sm.full[t][s]);
                        else  // the partial local chunk is read in place by the team
                            mbar_arrive(&sm.full[t][s]);
                    }
                    __syncwarp();
                    ++ut[t];
                    ++issued[t];
                    --left;
                    progress = true;
                }
            }
            if (progress) {
                t_blocked = 0;
                nap = 32;
                continue;
            }
            // every team with chunks left waits for a slot: describe the next
            // group meanwhile, else back off, bounded
            if (!last && located == i) {
                if (!locate_group<D>(inputs, R, so, sm, i + 1, next, last)) {
                    stop = true;
                    break;
                }
                located = i + 1;
                continue;
            }
            if (warp_any(sm.abort)) {
                stop = true;
                break;
            }
            const uint64_t now = __shfl_sync(0xFFFFFFFFu, globaltimer_ns(), 0);
            if (t_blocked == 0) {
                t_blocked = now;
            } else if (now - t_blocked > kWaitLimitNs) {
                if (lane == 0) set_abort(so, sm);
                stop = true;
                break;
            }
            __nanosleep(nap);
            if (nap < 256) nap <<= 1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.decoded[b]);  // the loader is done with meta[b]
        if (!stop && !last && located == i) {
            if (!locate_group<D>(inputs, R, so, sm, i + 1, next, last)) break;
            located = i + 1;
        }
    }
    // no copy may still be landing when the CTA exits
    for (int t = 0; t < kTeams; ++t)
        for (uint32_t v = ut[t] > (uint32_t)kRSlots ? ut[t] - kRSlots : 0u; v < ut[t]; ++v)
            mbar_wait(&sm.full[t][v % kRSlots], (v / kRSlots) & 1u);
}

// --------------------------------------------------------------------------- locator and copier
// The loader's work split over two warps, for inputs that are nearly
// incompressible: their raw rank chunks decode so fast that the teams wait
// for data whenever the copies stop while a group is being located.  The
// locator describes each group (locate_group), up to two groups ahead of the
// teams; the copier issues the bulk copies, rank by rank over the teams, each
// copy once its slot is free (a suspending wait, no polling).
template <class D>
__device__ __forceinline__ void reduce_locator(const ReduceInputs& inputs, int R, const StreamOut& so,
                                               ReduceSmem& sm) {
    const uint32_t lane = threadIdx.x & 31;
    for (int r = (int)lane; r < R; r += 32)
        sm.total[r] = (r == 0 && inputs.local != nullptr)
                          ? 1u
                          : stream_total<D>(inputs.in[r], inputs.in_bytes[r], so.n_elems, so.n_chunks);
    __syncwarp();
    uint64_t next = 0;
    if (lane == 0) next = atomicAdd(&so.ws->ticket, 1u);
    bool last = false;
    for (int i = 0; !last && !warp_any(sm.abort); ++i)
        if (!locate_group<D>(inputs, R, so, sm, i, next, last)) break;
}

template <class D>
__device__ __forceinline__ void reduce_copier(const ReduceInputs& inputs, int R, const StreamOut& so, uint8_t* ring,
                                              ReduceSmem& sm) {
    constexpr int kRSlots = rslots<D>();
    constexpr int kTeams = teams<D>();
    constexpr uint32_t kRawBytes = D::kElemBytes * kChunkElems;
    const uint32_t lane = threadIdx.x & 31;
    uint32_t ut[kTeams] = {};
    bool stop = false;
    for (int i = 0; !stop && !warp_any(sm.abort); ++i) {
        const int b = i % kMetaBufs;
        if (!warp_wait(&sm.meta_ready[b], (uint32_t)(i / kMetaBufs) & 1u)) {
            if (lane == 0) set_abort(so, sm);
            break;
        }
        const ReduceMeta& m = sm.meta[b];
        if (m.g == kNoGroup) break;
        const uint32_t n_out = m.n_out;
        if (m.ok) {
            for (int r = 0; r < R && !stop; ++r) {
#pragma unroll
                for (int t = 0; t < kTeams; ++t) {
                    if (t >= (int)n_out) break;
                    const uint32_t s = ut[t] % kRSlots;
                    if (ut[t] >= (uint32_t)kRSlots && !warp_wait(&sm.free_[t][s], (ut[t] / kRSlots - 1) & 1u)) {
                        if (lane == 0) set_abort(so, sm);
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        uint8_t* slot = ring + ((size_t)t * kRSlots + s) * max_chunk_bytes<D>();
                        if (r != 0 || inputs.local == nullptr)
                            bulk_load(slot, inputs.in[r] + m.off[t][r], m.bytes[t][r], &sm.full[t][s]);
                        else if (m.bytes[t][r] == kRawBytes)
                            bulk_load(slot, static_cast<const uint8_t*>(inputs.local) + m.off[t][r], kRawBytes,
                                      &sm.full[t][s]);
                        else
                            mbar_arrive(&sm.full[t][s]);
                    }
                    __syncwarp();
                    ++ut[t];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.decoded[b]);
    }
    for (int t = 0; t < kTeams; ++t)
        for (uint32_t v = ut[t] > (uint32_t)kRSlots ? ut[t] - kRSlots : 0u; v < ut[t]; ++v)
            mbar_wait(&sm.full[t][v % kRSlots], (v / kRSlots) & 1u);
}

// --------------------------------------------------------------------------- teams
// One team's rank operand r of its chunk into V (decode_full_chunk's layout),
// from the staged rank chunk or, for the partial local chunk, in place.
template <class D>
__device__ __forceinline__ void read_raw_partial(const uint8_t* vals_bytes, uint32_t n_c, uint32_t* V) {
    const uint32_t lane = threadIdx.x & 31, wq = (threadIdx.x >> 5) & 3;
    if constexpr (D::kElemBytes == 4) {
        const uint32_t* vals = reinterpret_cast<const uint32_t*>(vals_bytes);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const uint32_t e = 256 * (4 * wq + jj) + 8 * lane + x;
                V[8 * jj + x] = e < n_c ? vals[e] : 0u;
            }
    } else {
        const uint16_t* vals = reinterpret_cast<const uint16_t*>(vals_bytes);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const uint32_t e = 256 * (4 * wq + jj) + 8 * lane + 2 * x;
                const uint32_t lo = e < n_c ? vals[e] : 0u, hi = e + 1 < n_c ? vals[e + 1] : 0u;
                V[4 * jj + x] = lo | (hi << 16);
            }
    }
}

// acc (16 binary32 pairs, or for min/max 16 words of raw values: the 16-bit
// types keep a pair-word per entry, fp32 two words) op= V, in rank order.
// acc (a binary32 pair, low element in the low word) + the pair-word p of the
// 16-bit type, each element widened exactly and added with one rounding to
// nearest even: the mixed-precision add takes the 16-bit operand as it is.
template <class D>
__device__ __forceinline__ uint64_t add_pair_widened(uint64_t acc, uint32_t p) {
    if constexpr (D::kExpBits == 5)
        asm("{ .reg .b16 l, h; .reg .f32 a, b; mov.b32 {l, h}, %1; mov.b64 {a, b}, %0;"
            " add.rn.f32.f16 a, l, a; add.rn.f32.f16 b, h, b; mov.b64 %0, {a, b}; }"
            : "+l"(acc)
            : "r"(p));
    else
        asm("{ .reg .b16 l, h; .reg .f32 a, b; mov.b32 {l, h}, %1; mov.b64 {a, b}, %0;"
            " add.rn.f32.bf16 a, l, a; add.rn.f32.bf16 b, h, b; mov.b64 %0, {a, b}; }"
            : "+l"(acc)
            : "r"(p));
    return acc;
}
template <class D>
__device__ __forceinline__ void accumulate(uint64_t* acc, const uint32_t* V, uint32_t op, bool first) {
    if constexpr (D::kElemBytes == 4) {
        if (op != 0) {
#pragma unroll
            for (int x = 0; x < 16; ++x)
                acc[x] = first ? ((uint64_t)V[2 * x] | ((uint64_t)V[2 * x + 1] << 32))
                               : ((uint64_t)minmax_word((uint32_t)acc[x], V[2 * x], op) |
                                  ((uint64_t)minmax_word((uint32_t)(acc[x] >> 32), V[2 * x + 1], op) << 32));
        } else if (first) {
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = (uint64_t)V[2 * x] | ((uint64_t)V[2 * x + 1] << 32);
        } else {
#pragma unroll
            for (int x = 0; x < 16; ++x)
                acc[x] = add_f32x2(acc[x], (uint64_t)V[2 * x] | ((uint64_t)V[2 * x + 1] << 32));
        }
    } else {
        if (op != 0) {
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = first ? V[x] : minmax_pair<D>((uint32_t)acc[x], V[x], op);
        } else if (first) {
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = add_pair_widened<D>(0x8000000080000000ull, V[x]);  // x + (-0) = x
        } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = add_pair_widened<D>(acc[x], V[x]);
        }
    }
}

// The reduced chunk into P: one rounding of the binary32 sums to the type
// (fp32: none), or the min / max values as they are; NaNs made canonical
// when a rank may have held an Inf or a NaN (`special`: the team's verdict).
template <class D>
__device__ __forceinline__ void finish_values(const uint64_t* acc, uint32_t op, bool special, uint32_t* P) {
    if constexpr (D::kElemBytes == 4) {
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            P[2 * x] = (uint32_t)acc[x];
            P[2 * x + 1] = (uint32_t)(acc[x] >> 32);
        }
        if (special) {
#pragma unroll
            for (int x = 0; x < 32; ++x) P[x] = canonical_nan_word(P[x]);
        }
    } else {
#pragma unroll
        for (int x = 0; x < 16; ++x)
            P[x] = op != 0 ? (uint32_t)acc[x] : (D::kExpBits == 5 ? round_pair_fp16(acc[x]) : round_pair_bf16(acc[x]));
        if (special) {
#pragma unroll
            for (int x = 0; x < 16; ++x) P[x] = canonical_nan_pair<D>(P[x]);
        }
    }
}

// --------------------------------------------------------------------------- placer
// Per group: the look-back gives the group's offset; the teams' staged chunks
// then leave by one bulk (TMA) store each, issued by lane t for team t, which
// also writes the chunk's offset-table entry (and the stream header or size).
template <class D>
__device__ __forceinline__ void reduce_placer(const StreamOut& so, const uint8_t* staging, ReduceSmem& sm) {
    constexpr int kSB = sbufs<D>();
    constexpr int kZ = zslots<D>();
    constexpr int kTeams = teams<D>();
    const uint32_t lane = threadIdx.x & 31;
    for (int i = 0; !warp_any(sm.abort); ++i) {
        const int b = i % kSB, z = i % kZ;
        const uint32_t ph = (uint32_t)(i / kSB) & 1u;
        if (!warp_wait(&sm.sized[z], (uint32_t)(i / kZ) & 1u)) {
            if (lane == 0) set_abort(so, sm);
            break;
        }
        const uint64_t g = sm.gid[z];
        if (g == kNoGroup) break;
        const uint32_t mine = lane < (uint32_t)kTeams ? sm.size[z][lane] : 0u;
        const bool failed = warp_any(lane < (uint32_t)kTeams && sm.failed[z][lane] != 0);
        uint32_t incl = mine;
#pragma unroll
        for (int d = 1; d < kTeams; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += t;
        }
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, kTeams - 1);
        uint64_t go;
        if (failed) {
            if (lane == 0) st_relaxed_u64(&so.status[g], kFlagPoison);
            go = kFlagPoison;
        } else {
            go = lookback_offset_wide(so.status, g, total, data_start(so.n_chunks), so.ws, true);
        }
        if (lane == 0) sm.tally[z] = 0;  // next added to for group i + kZ, after `stored` below
        if (!warp_wait(&sm.staged[b], ph)) {
            if (lane == 0) set_abort(so, sm);
            break;
        }
        if (go != kFlagPoison && lane < (uint32_t)kTeams && mine > 0) {
            const uint64_t off = go + (incl - mine);
            if (off + mine > so.capacity) {  // cannot happen for a correct placement
                record_error(so.ws, kStatusCorrupt);
            } else {
                bulk_store(so.out + off, staging + ((size_t)lane * kSB + b) * max_chunk_bytes<D>(), mine);
                bulk_commit();
                finish_chunk(so, g * kTeams + lane, off, mine);
                bulk_wait_read();
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.stored[b]);
    }
    bulk_wait_all();  // every copy out has completed
}

template <class D>
__device__ __forceinline__ void reduce_team(int R, const void* local, uint32_t op, const StreamOut& so,
                                            uint8_t* ring_base, uint8_t* staging_base, ReduceSmem& sm) {
    constexpr int kRSlots = rslots<D>();
    constexpr int kW = thread_words<D>();
    constexpr int kSB = sbufs<D>();
    constexpr int kZ = zslots<D>();
    constexpr uint32_t kSlotBytes = max_chunk_bytes<D>();
    constexpr int kTeams = teams<D>();
    const uint32_t lane = threadIdx.x & 31, team = threadIdx.x >> 7, tt = threadIdx.x & 127, wq = tt >> 5;
    const TeamBarrier bar{1u + team};
    uint8_t* ring = ring_base + (size_t)team * kRSlots * kSlotBytes;
    const uint64_t n_full = so.n_elems / kChunkElems;
    uint32_t s = 0, ph = 0;  // this team's next ring slot and its phase (the loader's order)
    for (int i = 0;; ++i) {
        const int b = i % kMetaBufs, sb = i % kSB, z = i % kZ;
        const bool ready = mbar_wait(&sm.meta_ready[b], (uint32_t)(i / kMetaBufs) & 1u);
        if (bar.any(!ready || sm.abort)) {
            if (tt == 0) set_abort(so, sm);
            return;  // the whole team
        }
        // every thread has read iteration i - 1's flag: clear it for i + 1
        if (tt == 0) sm.corrupt[team][(i + 1) & 1] = 0;
        const ReduceMeta& m = sm.meta[b];
        const uint64_t g = m.g;
        if (g == kNoGroup) {
            // tell the placer (record z is free: see zslots)
            if (tt == 96) {
                if (team == 0) sm.gid[z] = kNoGroup;
                mbar_arrive(&sm.sized[z]);
            }
            return;
        }
        const uint64_t c = g * kTeams + team;
        const bool mine = team < m.n_out;  // uniform over the team
        const uint64_t left = mine ? so.n_elems - c * kChunkElems : 0;
        const uint32_t n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;
        uint32_t fail = m.ok ? 0u : kStatusCorrupt;
        bool timed_out = false, special = false;
        uint64_t acc[16];
        if (mine && m.ok) {
            for (int r = 0; r < R; ++r) {
                uint8_t* buf = ring + (size_t)s * kSlotBytes;
                if (!warp_wait(&sm.full[team][s], ph)) {
                    timed_out = true;
                    break;
                }
                uint32_t V[kW];
                if (fail == 0 && r == 0 && local != nullptr) {
                    // the uncompressed local operand: staged raw, or read in place
                    if (n_c == kChunkElems)
                        load_raw_full<D>(buf, V);
                    else
                        read_raw_partial<D>(
                            static_cast<const uint8_t*>(local) + (size_t)D::kElemBytes * c * kChunkElems, n_c, V);
                    special = true;
                    accumulate<D>(acc, V, op, true);
                } else if (fail == 0) {
                    const ChunkHeader h = unpack_desc(m.desc[team][r]);  // checked by the loader
                    if (n_c < kChunkElems) {  // partial last chunk: raw values, read those that exist
                        read_raw_partial<D>(buf + kChunkHeaderBytes, n_c, V);
                        special = true;
                    } else {
                        bool body_bad = false;
                        const uint32_t n = decode_quarter<D>(buf, h, V, special, body_bad);
                        if (lane == 0 && h.mode != kModeRaw) {
                            atomicAdd(&sm.esc_diff[team][r], (int32_t)n - (wq == 0 ? (int32_t)h.n_esc : 0));
                            if (body_bad) sm.corrupt[team][i & 1] = 1;
                        }
                    }
                    accumulate<D>(acc, V, op, r == 0);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.free_[team][s]);  // this warp is done with the slot
                if (++s == (uint32_t)kRSlots) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (lane == 0) mbar_arrive(&sm.decoded[b]);
        // the team meets: a timed-out wait stops it; Inf or NaN anywhere
        // makes the rounding canonicalise NaNs
        if (bar.any(timed_out)) {
            if (tt == 0) set_abort(so, sm);
            return;
        }
        const bool any_special = bar.any(special);
        // each rank chunk's quarters must hold exactly its n_esc escapes
        if (tt < (uint32_t)R) {
            if (sm.esc_diff[team][tt] != 0) sm.corrupt[team][i & 1] = 1;
            sm.esc_diff[team][tt] = 0;
        }
        TeamPlan pl{};
        uint32_t P[kW], planes[8];
        uint32_t bytes = 0;
        if (mine && fail == 0) {
            finish_values<D>(acc, op, any_special, P);
            if (c < n_full) {
                pl = plan_chunk_team<D>(bar, P, planes, sm.xch[team]);  // two meetings: the flag is in
                if (sm.corrupt[team][i & 1]) fail = kStatusCorrupt;
                bytes = pl.bytes;
            } else {
                bytes = tail_chunk_bytes<D>(n_c);
            }
        }
        if (fail) bytes = 0;
        if (tt == 96) {  // lane 0 of warp 3
            sm.size[z][team] = bytes;
            sm.failed[z][team] = fail;
            if (team == 0) sm.gid[z] = g;
            if (fail) {
                record_error(so.ws, fail);
            } else {
                // the last team to size the group publishes its size at once,
                // so later groups' look-backs need not wait for the placer
                const unsigned long long old = atomicAdd(&sm.tally[z], (1ull << 32) | bytes);
                if ((old >> 32) == kTeams - 1)
                    publish_unit_size(so.status, g, (uint32_t)old + bytes, data_start(so.n_chunks));
            }
            mbar_arrive(&sm.sized[z]);
        }
        // the placer is done with group i - kSB: its staging buffers
        const bool free_buf = i < kSB || warp_wait(&sm.stored[sb], (uint32_t)((i - kSB) / kSB) & 1u);
        if (!free_buf && lane == 0) set_abort(so, sm);
        if (free_buf && bytes > 0) {
            uint8_t* dst = staging_base + ((size_t)team * kSB + sb) * kSlotBytes;
            if (c < n_full)
                stage_chunk_team<D>(P, planes, pl, dst);
            else
                write_tail_chunk_team<D>(P, n_c, dst);
            fence_proxy_async_smem();  // the placer's bulk store reads these bytes
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.staged[sb]);
    }
}

// kSum: the operator is the sum (op 0), compiled without the min and max
// paths (a smaller kernel); otherwise op comes from the inputs.
template <class D, bool kSum>
__global__ void __launch_bounds__(reduce_threads<D>(), 1)
    reduce_kernel(ReduceInputs inputs, int R, StreamOut so, bool two_loaders) {
    constexpr int kTeams = teams<D>();
    static_assert(kTeams <= kMaxTeams && rslots<D>() <= kMaxRSlots && sbufs<D>() <= kMaxSBufs &&
                      zslots<D>() <= kMaxZSlots,
                  "the shared-memory bookkeeping arrays are sized for these bounds");
    static_assert(reduce_smem<D>() + sizeof(ReduceSmem) <= 227 * 1024, "shared memory per CTA");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ ReduceSmem sm;
    uint8_t* ring = smem;
    uint8_t* staging = smem + ring_bytes<D>();
    const uint32_t w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int b = 0; b < kMetaBufs; ++b) {
            mbar_init(&sm.meta_ready[b], 1);
            mbar_init(&sm.decoded[b], 4 * kTeams + 1);
        }
        for (int b = 0; b < sbufs<D>(); ++b) {
            mbar_init(&sm.staged[b], 4 * kTeams);
            mbar_init(&sm.stored[b], 1);
        }
        for (int z = 0; z < zslots<D>(); ++z) {
            mbar_init(&sm.sized[z], kTeams);
            sm.tally[z] = 0;
        }
        for (int t = 0; t < kTeams; ++t) {
            for (int s = 0; s < rslots<D>(); ++s) {
                mbar_init(&sm.full[t][s], 1);
                mbar_init(&sm.free_[t][s], 4);
            }
            sm.corrupt[t][0] = sm.corrupt[t][1] = 0;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    for (uint32_t x = threadIdx.x; x < kMaxTeams * kMaxRanks; x += blockDim.x) (&sm.esc_diff[0][0])[x] = 0;
    __syncthreads();
    if (w == loader_warp<D>()) {
        if (two_loaders)
            reduce_locator<D>(inputs, R, so, sm);
        else
            reduce_loader<D>(inputs, R, so, ring, sm);
    } else if (w == copier_warp<D>()) {
        if (two_loaders) reduce_copier<D>(inputs, R, so, ring, sm);
    } else if (w == placer_warp<D>())
        reduce_placer<D>(so, staging, sm);
    else if (w < 4 * (uint32_t)kTeams)
        reduce_team<D>(R, inputs.local, kSum ? 0u : inputs.op, so, ring, staging, sm);
    // (a warp with no role has nothing to do)
}

// Per-device record of the shared-memory limit set for reduce_kernel<D, *>
// (both operator variants), by element type code, team count and staging
// buffers per team.  A plain static array: a
// function-local static of a template would become one object shared by
// every copy of this library loaded into the process, and a second copy
// would then take its own kernel's limit as set.
static PerDeviceOnce g_reduce_smem_limit[4][kMaxTeams + 1][kMaxSBufs + 1];

template <class D>
cudaError_t launch_reduce_shape(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                                void* ws, cudaStream_t stream, bool two_loaders) {
    PerDeviceOnce& smem_limit = g_reduce_smem_limit[D::kCode][D::kTeams][D::kSBufs];
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = smem_limit.run(dev, [] {
            cudaError_t r = cudaFuncSetAttribute(reduce_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)reduce_smem<D>());
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(reduce_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)reduce_smem<D>());
            return r;
        });
    if (e != cudaSuccess) return e;
    StreamOut so;
    so.out = out;
    so.capacity = capacity;
    so.ws = static_cast<WsHeader*>(ws);
    so.status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    so.n_elems = n_elems;
    so.n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    so.version = kVersion;
    so.dtype = D::kCode;
    const uint64_t n_groups = (so.n_chunks + teams<D>() - 1) / teams<D>();
    const unsigned grid = (unsigned)(n_groups < (uint64_t)sms ? n_groups : (uint64_t)sms);
    if (inputs.op == 0)
        reduce_kernel<D, true><<<grid, reduce_threads<D>(), reduce_smem<D>(), stream>>>(inputs, R, so, two_loaders);
    else
        reduce_kernel<D, false><<<grid, reduce_threads<D>(), reduce_smem<D>(), stream>>>(inputs, R, so, two_loaders);
    return cudaGetLastError();
}

// Compressed bf16 inputs are bound by decoding: four teams (96 registers per
// thread) with one loader warp run fastest; from six ranks on, a group's
// decodes outlast the placer's look-back and stores, so each team keeps one
// staging buffer and five ring slots, else two and four.
// Nearly incompressible inputs (their streams at least 90% of the raw size:
// mostly raw chunks, cheap to decode) are bound by data arrival: three teams
// (128 registers) with six slots each, and a second loader warp that only
// issues copies, keep the rings fuller.  fp16 keeps three teams (its decode
// spills at 96 registers); fp32 chunks take twice the shared memory: three
// teams of two slots.  (All measured on GB300; every shape computes the
// same bytes.)  in_bytes is the readable size the caller gives for each
// stream, normally its total size.
template <class T>
cudaError_t launch_reduce_t(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                            void* ws, cudaStream_t stream) {
    uint64_t in_total = 0;
    for (int r = 0; r < R; ++r)
        in_total += (r == 0 && inputs.local != nullptr) ? (uint64_t)T::kElemBytes * n_elems : inputs.in_bytes[r];
    const bool incompressible = 10 * in_total >= 9 * (uint64_t)R * T::kElemBytes * n_elems;
    if constexpr (T::kElemBytes == 4) {
        return launch_reduce_shape<ReduceShape<T, 3, 2>>(inputs, R, n_elems, out, capacity, ws, stream,
                                                          incompressible);
    } else if constexpr (T::kExpBits == 5) {
        return launch_reduce_shape<ReduceShape<T, 3, 6>>(inputs, R, n_elems, out, capacity, ws, stream,
                                                          incompressible);
    } else {
        if (incompressible)
            return launch_reduce_shape<ReduceShape<T, 3, 6>>(inputs, R, n_elems, out, capacity, ws, stream, true);
        if (R >= 6)
            return launch_reduce_shape<ReduceShape<T, 4, 5, 1>>(inputs, R, n_elems, out, capacity, ws, stream, false);
        return launch_reduce_shape<ReduceShape<T, 4, 4>>(inputs, R, n_elems, out, capacity, ws, stream, false);
    }
}

cudaError_t launch_reduce(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                          void* ws, cudaStream_t stream) {
    return launch_reduce_t<Bf16>(inputs, R, n_elems, out, capacity, ws, stream);
}

cudaError_t launch_reduce_typed(uint32_t dtype, const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out,
                                uint64_t capacity, void* ws, cudaStream_t stream) {
    if (dtype == Fp16::kCode) return launch_reduce_t<Fp16>(inputs, R, n_elems, out, capacity, ws, stream);
    if (dtype == Fp32::kCode) return launch_reduce_t<Fp32>(inputs, R, n_elems, out, capacity, ws, stream);
    return launch_reduce_t<Bf16>(inputs, R, n_elems, out, capacity, ws, stream);
}

}  // namespace cccl

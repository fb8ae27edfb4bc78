// cccl_reduce.cu -- the fused reduce kernel: the reduce step of a compressed
// allreduce as one pass, decompress -> binary32 accumulate in rank order ->
// one rounding to the element type -> compress ("CCCL: In-GPU
// Compression-Coupled Collective Communication", section 5, "Integration into
// the NCCL data path" (CopyReducePacks); Figure 2).  Also min and max.
//
// Persistent and pipelined, one CTA per SM with three roles:
//   teams (warps 0..11)  three independent teams of 4 warps.  Per group of
//                        three consecutive output chunks, team t takes chunk
//                        t: it decodes chunk c of every rank, in rank order,
//                        a quarter per warp, keeping 32 binary32 sums per
//                        thread in registers; rounds once to the element type
//                        (bf16, fp16; fp32 needs none) and keeps the chunk in
//                        registers; sizes it (the team meets twice); saves its
//                        state to shared memory and writes its chunk of the
//                        previous group, which the placer has placed meanwhile;
//   loader (warp 12)     checks every rank's stream header once; takes a
//                        ticket per group, one group ahead; locates every
//                        rank's chunks through their offset tables and
//                        streams them to the teams through one ring of staged
//                        rank chunks per team, by bulk (TMA) copies, to
//                        whichever team has a slot free;
//   placer (warp 13)     places each sized group with one decoupled look-back.
// So the look-back of group i overlaps the decode of group i + 1, and the
// copies of later rank chunks are in flight meanwhile.  A team meets once per
// rank chunk (its copy has landed, and every warp is done with the previous
// one, whose slot is then released), and its per-chunk bookkeeping is spread
// over its warps.  The output chunk
// reaches shared memory only as its saved state (a column of words per
// thread), never as staged output.
// Tickets hand out groups in order to CTAs that are already running, and a
// group is sized without waiting on any later group: every look-back ends.
#include <mutex>

#include "cccl_decode.cuh"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kMaxTeams = 4;
constexpr int kTeamThreads = 128;
// decode teams per CTA = output chunks per group: 3, whose 14 warps leave
// 128 registers per thread (a fourth team would leave 96, and the team code
// spills there)
template <class D>
__host__ __device__ constexpr int teams() { return 3; }
template <class D>
__host__ __device__ constexpr int loader_warp() { return 4 * teams<D>(); }
template <class D>
__host__ __device__ constexpr int placer_warp() { return loader_warp<D>() + 1; }
template <class D>
__host__ __device__ constexpr int reduce_threads() { return 32 * (placer_warp<D>() + 1); }
constexpr uint64_t kNoGroup = ~0ull;
// staged rank chunks per team: 4 of 8.2 KB for the 16-bit types, 3 of 16.4 KB
// for fp32
template <class D>
__host__ __device__ constexpr int rslots() { return D::kElemBytes == 4 ? 3 : 4; }
constexpr int kMaxRSlots = 4;
// a team thread's chunk state between sizing and writing: its words, planes[8]
template <class D>
__host__ __device__ constexpr int prev_words() { return thread_words<D>() + 8; }
template <class D>
__host__ __device__ constexpr size_t ring_bytes() { return (size_t)teams<D>() * rslots<D>() * max_chunk_bytes<D>(); }
// sized chunks a team keeps in shared memory while the placer places them:
// a team writes group i - pend_depth at iteration i, so the look-back of a
// group overlaps the decoding of the next group
template <class D>
__host__ __device__ constexpr int pend_depth() { return 1; }
// placement buffers (sizes -> offsets), cycled by group: one more than the depth
template <class D>
__host__ __device__ constexpr int place_bufs() { return pend_depth<D>() + 1; }
constexpr int kMaxPlaceBufs = 3;
// chunk-state slots per team.  The 16-bit types keep one more than the
// pending chunks: the chunk just sized is saved before a pending one is
// written, so their states never share registers.  fp32, short of shared
// memory, writes the pending chunk first and then saves into its slot.
template <class D>
__host__ __device__ constexpr int state_slots() { return D::kElemBytes == 4 ? pend_depth<D>() : pend_depth<D>() + 1; }
template <class D>
__host__ __device__ constexpr size_t reduce_smem() {
    return ring_bytes<D>() + (size_t)teams<D>() * state_slots<D>() * prev_words<D>() * kTeamThreads * 4;
}

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

// What the loader hands the teams for one group.
struct ReduceMeta {
    uint64_t g;                          // group index, or kNoGroup: no more groups
    uint32_t ok;                         // every (chunk, rank) was located
    uint32_t n_out;                      // output chunks in the group
    uint64_t off[kMaxTeams][kMaxRanks];  // rank r's chunk teams * g + t: offset in its stream
    uint32_t bytes[kMaxTeams][kMaxRanks];  //   and size
};

struct ReduceSmem {
    uint64_t meta_ready[2];              // loader -> teams: meta[b] describes the next group (1 arrival)
    uint64_t decoded[2];                 // teams -> loader: meta[b] read (one arrival per team warp)
    uint64_t sized[kMaxPlaceBufs];       // teams -> placer: sizes in size[p] (one arrival per team)
    uint64_t placed[kMaxPlaceBufs];      // placer -> teams: offsets in off[p] (1 arrival)
    uint64_t full[kMaxTeams][kMaxRSlots];   // a rank chunk landed in the slot (transaction count)
    uint64_t free_[kMaxTeams][kMaxRSlots];  // the team is done with the slot (1 arrival)
    unsigned long long tally[kMaxPlaceBufs];  // sized teams (high word) and their bytes (low word)
    uint32_t size[kMaxPlaceBufs][kMaxTeams];
    uint32_t failed[kMaxPlaceBufs][kMaxTeams];   // the team's chunk could not be reduced
    uint64_t gid[kMaxPlaceBufs];         // group sized in buffer p, or kNoGroup
    uint64_t off[kMaxPlaceBufs][kMaxTeams];      // chunk offsets, or kFlagPoison
    TeamPlan pend_pl[kMaxTeams][3][4];   // a pending chunk's plan, per team, slot and warp
    uint64_t pend_c[kMaxTeams][3];       //   its chunk index
    uint32_t pend_bytes[kMaxTeams][3];   //   and size (0: nothing to write)
    uint32_t row_tot[kMaxTeams][4];         // the decoder's per-quarter escape totals
    TeamXch xch[kMaxTeams];                 // the encoder's exchange space
    volatile uint32_t abort;             // a bounded wait ran out: every role stops
    ReduceMeta meta[2];
    uint64_t total[kMaxRanks];           // rank r's stream size from its checked header (0: unusable)
};

__device__ __forceinline__ void set_abort(const StreamOut& so, ReduceSmem& sm) {
    record_error(so.ws, kStatusTimeout);
    sm.abort = 1;
}

// --------------------------------------------------------------------------- loader
template <class D>
__device__ __forceinline__ void reduce_loader(const ReduceInputs& inputs, int R, const StreamOut& so, uint8_t* ring,
                                              ReduceSmem& sm) {
    constexpr int kRSlots = rslots<D>();
    constexpr int kTeams = teams<D>();
    constexpr uint32_t kRawBytes = D::kElemBytes * kChunkElems;
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t n_groups = (so.n_chunks + kTeams - 1) / kTeams;
    // every rank's stream header, checked once
    for (int r = (int)lane; r < R; r += 32)
        sm.total[r] = (r == 0 && inputs.local != nullptr)
                          ? 1u
                          : stream_total<D>(inputs.in[r], inputs.in_bytes[r], so.n_elems, so.n_chunks);
    __syncwarp();
    uint32_t ut[kTeams] = {};  // rank chunks issued to each team
    bool stop = false;
    // lane 0: the ticket for the next group, taken one group ahead so that
    // its latency hides behind this group's work
    uint64_t next = 0;
    if (lane == 0) next = atomicAdd(&so.ws->ticket, 1u);
    for (int i = 0; !stop && !warp_any(sm.abort); ++i) {
        const int b = i & 1;
        // meta[b] was last read by the teams for group i - 2
        if (i >= 2 && !warp_wait(&sm.decoded[b], (uint32_t)((i - 2) >> 1) & 1u)) {
            if (lane == 0) set_abort(so, sm);
            break;
        }
        const uint64_t g = __shfl_sync(0xFFFFFFFFu, next, 0);
        if (lane == 0 && g < n_groups) next = atomicAdd(&so.ws->ticket, 1u);
        ReduceMeta& m = sm.meta[b];
        if (g >= n_groups) {
            if (lane == 0) {
                m.g = kNoGroup;
                mbar_arrive(&sm.meta_ready[b]);
            }
            break;
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
                continue;
            }
            const uint64_t total = sm.total[r];
            ChunkView v{0, 0, 0};
            if (total != 0) v = locate_chunk_at<D>(inputs.in[r], total, so.n_chunks, c0 + t);
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
        if (!ok) continue;  // nothing to stream: the teams poison the group
        // Every team gets its rank chunks in rank order; a team whose next
        // slot is still busy does not hold up the others.
        uint32_t issued[kTeams] = {};  // this group's rank chunks issued to each team
        uint32_t left = n_out * (uint32_t)R;
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
            // every team with chunks left waits for a slot: back off, bounded
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
    }
    // no copy may still be landing when the CTA exits
    for (int t = 0; t < kTeams; ++t)
        for (uint32_t v = ut[t] > (uint32_t)kRSlots ? ut[t] - kRSlots : 0u; v < ut[t]; ++v)
            mbar_wait(&sm.full[t][v % kRSlots], (v / kRSlots) & 1u);
}

// --------------------------------------------------------------------------- placer
template <class D>
__device__ __forceinline__ void reduce_placer(const StreamOut& so, ReduceSmem& sm) {
    constexpr int kPB = place_bufs<D>();
    constexpr int kTeams = teams<D>();
    const uint32_t lane = threadIdx.x & 31;
    for (int i = 0; !warp_any(sm.abort); ++i) {
        const int b = i % kPB;
        if (!warp_wait(&sm.sized[b], (uint32_t)(i / kPB) & 1u)) {
            if (lane == 0) set_abort(so, sm);
            break;
        }
        const uint64_t g = sm.gid[b];
        if (g == kNoGroup) break;
        const uint32_t mine = lane < (uint32_t)kTeams ? sm.size[b][lane] : 0u;
        const bool failed = warp_any(lane < (uint32_t)kTeams && sm.failed[b][lane] != 0);
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
        if (lane < (uint32_t)kTeams) sm.off[b][lane] = go == kFlagPoison ? kFlagPoison : go + (incl - mine);
        if (lane == 0) sm.tally[b] = 0;  // next used for group i + kPB, sized after group i is written
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.placed[b]);
    }
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
template <class D>
__device__ __forceinline__ uint64_t widen(uint32_t v) {
    if constexpr (D::kExpBits == 5)
        return widen_pair_fp16(v);
    else
        return widen_pair(v);
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
            for (int x = 0; x < 16; ++x) acc[x] = widen<D>(V[x]);
        } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = add_f32x2(acc[x], widen<D>(V[x]));
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

// Write this team's pending chunk of group j (sized pend_depth iterations
// earlier) once the placer has placed group j.  `st`: the chunk's state slot.
template <class D>
__device__ __forceinline__ void write_pending(const StreamOut& so, ReduceSmem& sm, int j, uint32_t* st) {
    constexpr int kW = thread_words<D>();
    constexpr int kPB = place_bufs<D>();
    const uint32_t lane = threadIdx.x & 31, team = threadIdx.x >> 7, tt = threadIdx.x & 127, wq = tt >> 5;
    const int slot = j % state_slots<D>();
    const uint32_t bytes = sm.pend_bytes[team][slot];
    if (bytes == 0) return;
    const int pb = j % kPB;
    if (!warp_wait(&sm.placed[pb], (uint32_t)(j / kPB) & 1u)) {
        if (lane == 0) set_abort(so, sm);
        return;
    }
    const uint64_t off = sm.off[pb][team];
    if (off == kFlagPoison) return;
    if (off + bytes > so.capacity) {  // cannot happen for a correct placement
        if (tt == 0) record_error(so.ws, kStatusCorrupt);
        return;
    }
    const uint64_t c = sm.pend_c[team][slot];
    const uint64_t n_full = so.n_elems / kChunkElems;
    uint32_t Pp[kW], Qp[8];
#pragma unroll
    for (int x = 0; x < kW; ++x) Pp[x] = st[kTeamThreads * x];
#pragma unroll
    for (int x = 0; x < 8; ++x) Qp[x] = st[kTeamThreads * (kW + x)];
    uint8_t* dst = so.out + off;
    if (c < n_full)
        write_chunk_team<D>(Pp, Qp, sm.pend_pl[team][slot][wq], dst, st);
    else
        write_tail_chunk_team<D>(Pp, (uint32_t)(so.n_elems - c * kChunkElems), dst);
    if (tt == 64) finish_chunk(so, c, off, bytes);  // warp 0 wrote the chunk header
}

template <class D>
__device__ __forceinline__ void reduce_team(int R, const void* local, uint32_t op, const StreamOut& so,
                                            uint8_t* ring_base, uint32_t* prev_base, ReduceSmem& sm) {
    constexpr int kRSlots = rslots<D>();
    constexpr int kW = thread_words<D>();
    constexpr int kPrevWords = prev_words<D>();
    constexpr int kPend = pend_depth<D>();
    constexpr int kSlots = state_slots<D>();
    constexpr int kPB = place_bufs<D>();
    constexpr uint32_t kSlotBytes = max_chunk_bytes<D>();
    constexpr int kTeams = teams<D>();
    const uint32_t lane = threadIdx.x & 31, team = threadIdx.x >> 7, tt = threadIdx.x & 127, wq = tt >> 5;
    const TeamBarrier bar{1u + team};
    uint8_t* ring = ring_base + (size_t)team * kRSlots * kSlotBytes;
    // pending chunk slot s of this team: word w at st(s)[128 w]
    auto st_of = [&](int s) { return prev_base + ((size_t)team * kSlots + s) * kPrevWords * kTeamThreads + tt; };
    const uint64_t n_full = so.n_elems / kChunkElems;
    if (tt == 0)
        for (int s = 0; s < kSlots; ++s) sm.pend_bytes[team][s] = 0;
    bar.sync();
    uint32_t u = 0;  // rank chunks consumed (the loader's order for this team)
    for (int i = 0;; ++i) {
        const int b = i & 1, pb = i % kPB;
        const bool ready = mbar_wait(&sm.meta_ready[b], (uint32_t)(i >> 1) & 1u);
        if (bar.any(!ready || sm.abort)) {
            if (tt == 0) set_abort(so, sm);
            return;  // the whole team
        }
        const ReduceMeta& m = sm.meta[b];
        const uint64_t g = m.g;
        TeamPlan pl{};
        uint32_t P[kW], planes[8];
        uint32_t bytes = 0, fail = 0;
        uint64_t c = 0;
        uint32_t n_c = 0;
        if (g != kNoGroup) {
            c = g * kTeams + team;
            const bool mine = team < m.n_out;  // uniform over the team
            const uint64_t left = mine ? so.n_elems - c * kChunkElems : 0;
            n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;
            fail = m.ok ? 0u : kStatusCorrupt;
            if (mine && m.ok) {
                uint64_t acc[16];
                bool special = false;
                for (int r = 0; r < R; ++r, ++u) {
                    const uint32_t s = u % kRSlots;
                    uint8_t* buf = ring + (size_t)s * kSlotBytes;
                    const bool landed = !sm.abort && mbar_wait(&sm.full[team][s], (u / kRSlots) & 1u);
                    // one meeting per rank: slot s has landed for every warp,
                    // and every warp is done with the previous rank's slot and
                    // row_tot
                    if (bar.any(!landed)) {
                        if (tt == 0) set_abort(so, sm);
                        return;  // the whole team
                    }
                    if (r > 0 && tt == 32) mbar_arrive(&sm.free_[team][(u - 1) % kRSlots]);
                    uint32_t V[kW];
                    if (fail == 0 && r == 0 && local != nullptr) {
                        // the uncompressed local operand: staged raw, or read in place
                        if (n_c == kChunkElems) {
                            load_raw_full<D>(buf, V);
                        } else {
                            read_raw_partial<D>(static_cast<const uint8_t*>(local) +
                                                    (size_t)D::kElemBytes * c * kChunkElems,
                                                n_c, V);
                        }
                        special = true;
                        accumulate<D>(acc, V, op, true);
                    } else if (fail == 0) {
                        const ChunkHeader h = read_chunk_header(buf);
                        bool good = chunk_header_valid<D>(h, m.bytes[team][r], n_c);  // same for the team
                        if (good) {
                            if (n_c < kChunkElems) {  // partial last chunk: raw values, read those that exist
                                read_raw_partial<D>(buf + kChunkHeaderBytes, n_c, V);
                                special = true;
                            } else {
                                bool sp = false;
                                good = decode_full_chunk<D>(bar, buf, h, V, sm.row_tot[team], sp);
                                special = special || sp;
                            }
                        }
                        if (!good)
                            fail = kStatusCorrupt;
                        else
                            accumulate<D>(acc, V, op, r == 0);
                    }
                }
                // the last rank's slot is released once the team meets again
                const bool any_special = bar.any(special);
                if (tt == 32) mbar_arrive(&sm.free_[team][(u - 1) % kRSlots]);
                if (fail == 0) finish_values<D>(acc, op, any_special, P);
            }
            if (lane == 0) mbar_arrive(&sm.decoded[b]);
            if (mine && fail == 0) {
                if (c < n_full) {
                    pl = plan_chunk_team<D>(bar, P, planes, sm.xch[team]);
                    bytes = pl.bytes;
                } else {
                    bytes = tail_chunk_bytes<D>(n_c);
                }
            }
            if (tt == 96) {  // lane 0 of warp 3: warp 0 writes headers, warp 2 the table
                sm.size[pb][team] = bytes;
                sm.failed[pb][team] = fail;
                if (team == 0) sm.gid[pb] = g;
                if (fail) {
                    record_error(so.ws, fail);
                } else {
                    // the last team to size the group publishes its size at once,
                    // so later groups' look-backs need not wait for the placer
                    const unsigned long long old = atomicAdd(&sm.tally[pb], (1ull << 32) | bytes);
                    if ((old >> 32) == kTeams - 1)
                        publish_unit_size(so.status, g, (uint32_t)old + bytes, data_start(so.n_chunks));
                }
                mbar_arrive(&sm.sized[pb]);
            }
        } else if (tt == 96) {
            if (team == 0) sm.gid[pb] = kNoGroup;
            mbar_arrive(&sm.sized[pb]);
        }
        // this chunk waits in shared memory for its placement; the chunk of
        // group i - kPend is written (at the end, every chunk still pending)
        auto save = [&]() {
            const int slot = i % kSlots;
            uint32_t* st = st_of(slot);
            const uint32_t keep = fail ? 0u : bytes;
            if (keep > 0) {
#pragma unroll
                for (int x = 0; x < kW; ++x) st[kTeamThreads * x] = P[x];
#pragma unroll
                for (int x = 0; x < 8; ++x) st[kTeamThreads * (kW + x)] = planes[x];
            }
            if (lane == 0) sm.pend_pl[team][slot][wq] = pl;
            if (tt == 0) {
                sm.pend_c[team][slot] = c;
                sm.pend_bytes[team][slot] = keep;
            }
        };
        if (kSlots > kPend && g != kNoGroup) save();
        if (i >= kPend) write_pending<D>(so, sm, i - kPend, st_of((i - kPend) % kSlots));
        if (g == kNoGroup) {
            for (int j = i - kPend + 1; j < i; ++j)
                if (j >= 0) write_pending<D>(so, sm, j, st_of(j % kSlots));
            return;
        }
        if (kSlots == kPend) save();
        // (the next iteration's team barrier orders these writes before any read)
    }
}

template <class D>
__global__ void __launch_bounds__(reduce_threads<D>(), 1) reduce_kernel(ReduceInputs inputs, int R, StreamOut so) {
    constexpr int kTeams = teams<D>();
    static_assert(kTeams <= kMaxTeams && rslots<D>() <= kMaxRSlots && state_slots<D>() <= 3 &&
                      place_bufs<D>() <= kMaxPlaceBufs,
                  "the shared-memory bookkeeping arrays are sized for these bounds");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ ReduceSmem sm;
    uint8_t* ring = smem;
    uint32_t* prev = reinterpret_cast<uint32_t*>(smem + ring_bytes<D>());
    const uint32_t w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.meta_ready[b], 1);
            mbar_init(&sm.decoded[b], 4 * kTeams);
        }
        for (int b = 0; b < place_bufs<D>(); ++b) {
            mbar_init(&sm.sized[b], kTeams);
            mbar_init(&sm.placed[b], 1);
            sm.tally[b] = 0;
        }
        for (int t = 0; t < kTeams; ++t)
            for (int s = 0; s < rslots<D>(); ++s) {
                mbar_init(&sm.full[t][s], 1);
                mbar_init(&sm.free_[t][s], 1);
            }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (w == loader_warp<D>())
        reduce_loader<D>(inputs, R, so, ring, sm);
    else if (w == placer_warp<D>())
        reduce_placer<D>(so, sm);
    else
        reduce_team<D>(R, inputs.local, inputs.op, so, ring, prev, sm);
}

template <class D>
cudaError_t launch_reduce_t(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                            void* ws, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(reduce_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)reduce_smem<D>());
    });
    if (attr != cudaSuccess) return attr;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
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
    reduce_kernel<D><<<grid, reduce_threads<D>(), reduce_smem<D>(), stream>>>(inputs, R, so);
    return cudaGetLastError();
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

// cccl_reduce.cu -- the fused reduce kernel: the reduce step of a compressed
// allreduce as one pass, decompress -> binary32 accumulate in rank order ->
// one rounding to bf16 -> compress ("CCCL: In-GPU Compression-Coupled
// Collective Communication", section 5, "Integration into the NCCL data
// path" (CopyReducePacks); Figure 2).
//
// Persistent and pipelined, one CTA per SM with three roles:
//   teams (warps 0..11)  three independent teams of 4 warps.  Per group of
//                        kTeams consecutive output chunks, team t takes chunk
//                        t: it decodes chunk c of every rank, in rank order,
//                        a quarter per warp, keeping 32 binary32 sums per
//                        thread in registers; rounds once to bf16 and keeps
//                        the chunk in registers; sizes it (the team meets
//                        twice); then writes its chunk of the PREVIOUS group,
//                        whose state waited in shared memory while the
//                        placer placed it;
//   loader (warp 12)     takes a ticket per group, locates every rank's
//                        chunks through their offset tables and streams them
//                        to the teams through one ring of staged rank chunks
//                        per team, by bulk (TMA) copies;
//   placer (warp 13)     places each sized group with one decoupled look-back.
// So the look-back of group i overlaps the decode of group i + 1, and the
// copies of later rank chunks are in flight during both.  The output chunk
// never goes through shared memory.
// Tickets hand out groups in order to CTAs that are already running, and a
// group is sized without waiting on any later group: every look-back ends.
#include <mutex>

#include "cccl_decode.cuh"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kTeams = 3;                     // output chunks per group
constexpr int kRSlots = 4;                    // staged rank chunks per team
constexpr int kTeamThreads = 128;
constexpr int kLoaderWarp = 4 * kTeams;
constexpr int kPlacerWarp = kLoaderWarp + 1;
constexpr int kReduceThreads = 32 * (kPlacerWarp + 1);
constexpr int kPrevWords = 24;                // a team thread's chunk state: P[16], planes[8]
constexpr size_t kRingBytes = (size_t)kTeams * kRSlots * kMaxChunkBytes;
constexpr size_t kPrevBytes = (size_t)kTeams * kPrevWords * kTeamThreads * 4;
constexpr size_t kReduceSmemBytes = kRingBytes + kPrevBytes;
constexpr uint64_t kNoGroup = ~0ull;

// binary32 pair -> bf16 pair, round to nearest even (hi lane from the upper word)
__device__ __forceinline__ uint32_t round_pair_bf16(uint64_t v) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "r"((uint32_t)(v >> 32)), "r"((uint32_t)v));
    return d;
}
// every NaN lane -> 0x7FC0
__device__ __forceinline__ uint32_t canonical_nan_pair(uint32_t d) {
    const uint32_t mag = d & 0x7FFF7FFFu;
    const uint32_t nan = (mag + 0x007F007Fu) & 0x80008000u;  // lanes with mag > 0x7F80
    const uint32_t mask = (nan >> 15) * 0xFFFFu;
    return (d & ~mask) | (0x7FC07FC0u & mask);
}

// Element-wise min (op 1) or max (op 2) of two bf16 pairs, exact: a NaN in
// either lane gives a NaN there (made canonical afterwards); otherwise the
// IEEE total order, -0 below +0, through the usual sign-magnitude key
// (negative: all bits flipped; positive: sign bit set), compared as u16.
__device__ __forceinline__ uint32_t order_key_pair(uint32_t x) {
    return x ^ ((((x >> 15) & 0x00010001u) * 0x7FFFu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t from_order_key_pair(uint32_t k) {
    return k ^ ((((~k >> 15) & 0x00010001u) * 0x7FFFu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t nan_lanes_pair(uint32_t x) {  // 0xFFFF where x is a NaN
    return ((((x & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u) >> 15) * 0xFFFFu;
}
__device__ __forceinline__ uint32_t minmax_pair(uint32_t a, uint32_t b, uint32_t op) {
    const uint32_t ka = order_key_pair(a), kb = order_key_pair(b);
    const uint32_t r = from_order_key_pair(op == 1 ? vmin_u16x2(ka, kb) : vmax_u16x2(ka, kb));
    const uint32_t nan = nan_lanes_pair(a) | nan_lanes_pair(b);
    return (r & ~nan) | (0x7FC07FC0u & nan);
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
    uint64_t off[kTeams][kMaxRanks];     // rank r's chunk kTeams g + t: offset in its stream
    uint32_t bytes[kTeams][kMaxRanks];   //   and size
};

struct ReduceSmem {
    uint64_t meta_ready[2];              // loader -> teams: meta[b] describes the next group (1 arrival)
    uint64_t decoded[2];                 // teams -> loader: meta[b] read (one arrival per team warp)
    uint64_t sized[2];                   // teams -> placer: sizes in size[b] (one arrival per team)
    uint64_t placed[2];                  // placer -> teams: offsets in off[b] (1 arrival)
    uint64_t full[kTeams][kRSlots];      // a rank chunk landed in the slot (transaction count)
    uint64_t free_[kTeams][kRSlots];     // the team is done with the slot (1 arrival)
    unsigned long long tally[2];         // sized teams (high word) and their bytes (low word)
    uint32_t size[2][kTeams];
    uint32_t failed[2][kTeams];          // the team's chunk could not be reduced
    uint64_t gid[2];                     // group sized in slot b, or kNoGroup
    uint64_t off[2][kTeams];             // chunk offsets, or kFlagPoison
    uint32_t row_tot[kTeams][4];         // the decoder's per-quarter escape totals
    TeamXch xch[kTeams];                 // the encoder's exchange space
    volatile uint32_t abort;             // a bounded wait ran out: every role stops
    ReduceMeta meta[2];
};

__device__ __forceinline__ void set_abort(const StreamOut& so, ReduceSmem& sm) {
    record_error(so.ws, kStatusTimeout);
    sm.abort = 1;
}

// --------------------------------------------------------------------------- loader
__device__ __forceinline__ void reduce_loader(const ReduceInputs& inputs, int R, const StreamOut& so, uint8_t* ring,
                                              ReduceSmem& sm) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t n_groups = (so.n_chunks + kTeams - 1) / kTeams;
    uint32_t ut[kTeams] = {};  // rank chunks issued to each team
    bool stop = false;
    for (int i = 0; !stop && !warp_any(sm.abort); ++i) {
        const int b = i & 1;
        // meta[b] was last read by the teams for group i - 2
        if (i >= 2 && !warp_wait(&sm.decoded[b], (uint32_t)((i - 2) >> 1) & 1u)) {
            if (lane == 0) set_abort(so, sm);
            break;
        }
        uint64_t g = 0;
        if (lane == 0) g = atomicAdd(&so.ws->ticket, 1u);
        g = __shfl_sync(0xFFFFFFFFu, g, 0);
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
                m.off[t][r] = 2 * kChunkElems * c;
                m.bytes[t][r] = 2 * (uint32_t)(left < kChunkElems ? left : kChunkElems);
                continue;
            }
            const ChunkView v = locate_chunk(inputs.in[r], inputs.in_bytes[r], so.n_elems, so.n_chunks, c0 + t);
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
        // rank-major, so that every team gets its next rank chunk in turn
        for (int r = 0; r < R && !stop; ++r) {
            for (uint32_t t = 0; t < n_out; ++t) {
                const uint32_t s = ut[t] % kRSlots;
                // the slot's previous rank chunk is consumed
                if (ut[t] >= (uint32_t)kRSlots && !warp_wait(&sm.free_[t][s], (ut[t] / kRSlots - 1) & 1u)) {
                    if (lane == 0) set_abort(so, sm);
                    stop = true;
                    break;
                }
                if (warp_any(sm.abort)) {
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    fence_proxy_async_smem();
                    uint8_t* slot = ring + ((size_t)t * kRSlots + s) * kMaxChunkBytes;
                    if (r != 0 || inputs.local == nullptr)
                        bulk_load(slot, inputs.in[r] + m.off[t][r], m.bytes[t][r], &sm.full[t][s]);
                    else if (m.bytes[t][r] == 2 * kChunkElems)  // a full local chunk, staged raw
                        bulk_load(slot, reinterpret_cast<const uint8_t*>(inputs.local) + m.off[t][r],
                                  2 * kChunkElems, &sm.full[t][s]);
                    else  // the partial local chunk is read in place by the team
                        mbar_arrive(&sm.full[t][s]);
                }
                __syncwarp();
                ++ut[t];
            }
        }
    }
    // no copy may still be landing when the CTA exits
    for (int t = 0; t < kTeams; ++t)
        for (uint32_t v = ut[t] > (uint32_t)kRSlots ? ut[t] - kRSlots : 0u; v < ut[t]; ++v)
            mbar_wait(&sm.full[t][v % kRSlots], (v / kRSlots) & 1u);
}

// --------------------------------------------------------------------------- placer
__device__ __forceinline__ void reduce_placer(const StreamOut& so, ReduceSmem& sm) {
    const uint32_t lane = threadIdx.x & 31;
    for (int i = 0; !warp_any(sm.abort); ++i) {
        const int b = i & 1;
        if (!warp_wait(&sm.sized[b], (uint32_t)(i >> 1) & 1u)) {
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
        if (lane == 0) sm.tally[b] = 0;  // next used for group i + 2, after its writers saw placed[b]
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.placed[b]);
    }
}

// --------------------------------------------------------------------------- teams
__device__ __forceinline__ void reduce_team(int R, const uint16_t* local, uint32_t op, const StreamOut& so,
                                            uint8_t* ring_base, uint32_t* prev_base, ReduceSmem& sm) {
    const uint32_t lane = threadIdx.x & 31, team = threadIdx.x >> 7, tt = threadIdx.x & 127;
    const uint32_t wq = tt >> 5;  // warp within the team = quarter of the chunk
    const TeamBarrier bar{1u + team};
    uint8_t* ring = ring_base + (size_t)team * kRSlots * kMaxChunkBytes;
    uint32_t* prev_st = prev_base + (size_t)team * kPrevWords * kTeamThreads + tt;  // word w at prev_st[128 w]
    const uint64_t n_full = so.n_elems / kChunkElems;
    uint32_t u = 0;  // rank chunks consumed (the loader's order for this team)
    TeamPlan prev_pl{};
    uint64_t prev_c = 0;
    uint32_t prev_bytes = 0;  // 0: no previous chunk to write
    for (int i = 0;; ++i) {
        const int b = i & 1;
        const bool ready = mbar_wait(&sm.meta_ready[b], (uint32_t)(i >> 1) & 1u);
        if (bar.any(!ready || sm.abort)) {
            if (tt == 0) set_abort(so, sm);
            return;  // the whole team
        }
        const ReduceMeta& m = sm.meta[b];
        const uint64_t g = m.g;
        TeamPlan pl{};
        uint32_t P[16], planes[8];
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
                    uint8_t* buf = ring + (size_t)s * kMaxChunkBytes;
                    const bool landed = !sm.abort && mbar_wait(&sm.full[team][s], (u / kRSlots) & 1u);
                    if (bar.any(!landed)) {
                        if (tt == 0) set_abort(so, sm);
                        return;  // the whole team
                    }
                    if (fail == 0 && r == 0 && local != nullptr) {
                        // the uncompressed local operand: staged raw, or read in place
                        uint32_t V[16];
                        if (n_c == kChunkElems) {
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                const uint4 v =
                                    *reinterpret_cast<const uint4*>(buf + 512 * (4 * wq + jj) + 16 * lane);
                                V[4 * jj] = v.x;
                                V[4 * jj + 1] = v.y;
                                V[4 * jj + 2] = v.z;
                                V[4 * jj + 3] = v.w;
                            }
                        } else {
                            const uint16_t* vals = local + c * kChunkElems;
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                                for (int x = 0; x < 4; ++x) {
                                    const uint32_t e = 256 * (4 * wq + jj) + 8 * lane + 2 * x;
                                    const uint32_t lo = e < n_c ? vals[e] : 0u, hi = e + 1 < n_c ? vals[e + 1] : 0u;
                                    V[4 * jj + x] = lo | (hi << 16);
                                }
                        }
                        special = true;
#pragma unroll
                        for (int x = 0; x < 16; ++x) acc[x] = op == 0 ? widen_pair(V[x]) : V[x];
                    } else if (fail == 0) {
                        const ChunkHeader h = read_chunk_header(buf);
                        bool good = chunk_header_valid(h, m.bytes[team][r], n_c);  // same for the team
                        uint32_t V[16];
                        if (good) {
                            if (n_c < kChunkElems) {  // partial last chunk: raw values, read those that exist
                                const uint16_t* vals = reinterpret_cast<const uint16_t*>(buf + kChunkHeaderBytes);
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                                    for (int x = 0; x < 4; ++x) {
                                        const uint32_t e = 256 * (4 * wq + jj) + 8 * lane + 2 * x;
                                        const uint32_t lo = e < n_c ? vals[e] : 0u, hi = e + 1 < n_c ? vals[e + 1] : 0u;
                                        V[4 * jj + x] = lo | (hi << 16);
                                    }
                                special = true;
                            } else {
                                bool sp = false;
                                good = decode_full_chunk(bar, buf, h, V, sm.row_tot[team], sp);
                                special = special || sp;
                            }
                        }
                        if (!good) {
                            fail = kStatusCorrupt;
                        } else if (op != 0) {  // min / max: exact, on the bf16 pairs
#pragma unroll
                            for (int x = 0; x < 16; ++x)
                                acc[x] = r == 0 ? V[x] : minmax_pair((uint32_t)acc[x], V[x], op);
                        } else if (r == 0) {
#pragma unroll
                            for (int x = 0; x < 16; ++x) acc[x] = widen_pair(V[x]);
                        } else {
#pragma unroll
                            for (int x = 0; x < 16; ++x) acc[x] = add_f32x2(acc[x], widen_pair(V[x]));
                        }
                    }
                    bar.sync();  // the team is done with slot s and row_tot
                    if (tt == 0) mbar_arrive(&sm.free_[team][s]);
                }
                if (fail == 0) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) P[x] = op == 0 ? round_pair_bf16(acc[x]) : (uint32_t)acc[x];
                    if (bar.any(special)) {
#pragma unroll
                        for (int x = 0; x < 16; ++x) P[x] = canonical_nan_pair(P[x]);
                    }
                }
            }
            if (lane == 0) mbar_arrive(&sm.decoded[b]);
            if (mine && fail == 0) {
                if (c < n_full) {
                    pl = plan_chunk_team(bar, P, planes, sm.xch[team]);
                    bytes = pl.bytes;
                } else {
                    bytes = tail_chunk_bytes(n_c);
                }
            }
            if (tt == 0) {
                sm.size[b][team] = bytes;
                sm.failed[b][team] = fail;
                if (team == 0) sm.gid[b] = g;
                if (fail) {
                    record_error(so.ws, fail);
                } else {
                    // the last team to size the group publishes its size at once,
                    // so later groups' look-backs need not wait for the placer
                    const unsigned long long old = atomicAdd(&sm.tally[b], (1ull << 32) | bytes);
                    if ((old >> 32) == kTeams - 1)
                        publish_unit_size(so.status, g, (uint32_t)old + bytes, data_start(so.n_chunks));
                }
                mbar_arrive(&sm.sized[b]);
            }
        } else if (tt == 0) {
            if (team == 0) sm.gid[b] = kNoGroup;
            mbar_arrive(&sm.sized[b]);
        }
        // write this team's chunk of the previous group
        if (i > 0 && prev_bytes > 0) {
            const int pb = b ^ 1;
            if (warp_wait(&sm.placed[pb], (uint32_t)((i - 1) >> 1) & 1u)) {
                const uint64_t off = sm.off[pb][team];
                if (off != kFlagPoison) {
                    if (off + prev_bytes > so.capacity) {  // cannot happen for a correct placement
                        if (tt == 0) record_error(so.ws, kStatusCorrupt);
                    } else {
                        uint32_t Pp[16], Qp[8];
#pragma unroll
                        for (int x = 0; x < 16; ++x) Pp[x] = prev_st[kTeamThreads * x];
#pragma unroll
                        for (int x = 0; x < 8; ++x) Qp[x] = prev_st[kTeamThreads * (16 + x)];
                        uint8_t* dst = so.out + off;
                        if (prev_c < n_full)
                            write_chunk_team(Pp, Qp, prev_pl, dst, prev_st);
                        else
                            write_tail_chunk_team(Pp, (uint32_t)(so.n_elems - prev_c * kChunkElems), dst);
                        if (tt == 0) finish_chunk(so, prev_c, off, prev_bytes);
                    }
                }
            } else if (lane == 0) {
                set_abort(so, sm);
            }
        }
        if (g == kNoGroup) return;
        // this chunk waits in shared memory for its placement
        prev_bytes = fail ? 0u : bytes;
        if (prev_bytes > 0) {
#pragma unroll
            for (int x = 0; x < 16; ++x) prev_st[kTeamThreads * x] = P[x];
#pragma unroll
            for (int x = 0; x < 8; ++x) prev_st[kTeamThreads * (16 + x)] = planes[x];
            prev_pl = pl;
            prev_c = c;
        }
    }
}

__global__ void __launch_bounds__(kReduceThreads, 1) reduce_kernel(ReduceInputs inputs, int R, StreamOut so) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ ReduceSmem sm;
    uint8_t* ring = smem;
    uint32_t* prev = reinterpret_cast<uint32_t*>(smem + kRingBytes);
    const uint32_t w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.meta_ready[b], 1);
            mbar_init(&sm.decoded[b], 4 * kTeams);
            mbar_init(&sm.sized[b], kTeams);
            mbar_init(&sm.placed[b], 1);
            sm.tally[b] = 0;
        }
        for (int t = 0; t < kTeams; ++t)
            for (int s = 0; s < kRSlots; ++s) {
                mbar_init(&sm.full[t][s], 1);
                mbar_init(&sm.free_[t][s], 1);
            }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (w == kLoaderWarp)
        reduce_loader(inputs, R, so, ring, sm);
    else if (w == kPlacerWarp)
        reduce_placer(so, sm);
    else
        reduce_team(R, inputs.local, inputs.op, so, ring, prev, sm);
}

cudaError_t launch_reduce(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                          void* ws, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kReduceSmemBytes);
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
    const uint64_t n_groups = (so.n_chunks + kTeams - 1) / kTeams;
    const unsigned grid = (unsigned)(n_groups < (uint64_t)sms ? n_groups : (uint64_t)sms);
    reduce_kernel<<<grid, kReduceThreads, kReduceSmemBytes, stream>>>(inputs, R, so);
    return cudaGetLastError();
}

}  // namespace cccl

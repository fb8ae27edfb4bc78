// cccl_reduce.cu -- the fused reduce kernel: the reduce step of a compressed
// allreduce as one pass, decompress -> binary32 accumulate in rank order ->
// one rounding to bf16 -> compress ("CCCL: In-GPU Compression-Coupled
// Collective Communication", section 5, "Integration into the NCCL data
// path" (CopyReducePacks); Figure 2).
//
// Persistent and pipelined, two CTAs per SM.  A CTA has three roles:
//   team (warps 0..3)  per group of 4 consecutive output chunks: decodes
//                      chunk c of every rank, in rank order, the 4 warps
//                      together (a quarter of the chunk each), keeping 32
//                      binary32 sums per thread in registers; rounds once to
//                      bf16 and parks the chunk in shared memory; then each
//                      warp sizes one parked chunk exactly as the compress
//                      kernel does, and writes its chunk of the PREVIOUS
//                      group, which the placer has placed meanwhile;
//   loader (warp 4)    takes a ticket per group, locates every rank's chunks
//                      through their offset tables and streams them through
//                      a ring of staged rank chunks by bulk (TMA) copies;
//   placer (warp 5)    places each sized group with one decoupled look-back.
// So the look-back of group i overlaps the decode of group i + 1, and the
// copies of later rank chunks are in flight during both.
// Tickets hand out groups in order to CTAs that are already running, and a
// group is sized without waiting on any later group: every look-back ends.
#include <mutex>

#include "cccl_decode.cuh"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kRChunks = 4;                         // output chunks per group = team warps
constexpr int kRSlots = 4;                          // staged rank chunks
constexpr int kTeamThreads = 32 * kRChunks;
constexpr int kLoaderWarp = kRChunks;
constexpr int kPlacerWarp = kRChunks + 1;
constexpr int kReduceThreads = 32 * (kRChunks + 2);
constexpr size_t kParkChunkBytes = 2 * kChunkElems;
constexpr size_t kParkBytes = 2 * kRChunks * kParkChunkBytes;  // two groups of parked bf16 chunks
constexpr size_t kReduceSmemBytes = kParkBytes + (size_t)kRSlots * kMaxChunkBytes;
constexpr uint64_t kNoGroup = ~0ull;
using TeamBarrier = NamedBarrier<1, kTeamThreads>;

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

// Warp-uniform reads of the abort flag and of a bounded wait's outcome.
__device__ __forceinline__ bool warp_any(bool p) { return __any_sync(0xFFFFFFFFu, p); }
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity));
}

// What the loader hands the team for one group.
struct ReduceMeta {
    uint64_t g;                           // group index, or kNoGroup: no more groups
    uint32_t ok;                          // every (chunk, rank) was located
    uint32_t n_out;                       // output chunks in the group
    uint64_t off[kRChunks][kMaxRanks];    // rank r's chunk 4 g + j: offset in its stream
    uint32_t bytes[kRChunks][kMaxRanks];  //   and size
};

struct ReduceSmem {
    uint64_t meta_ready[2];       // loader -> team: meta[b] describes the next group (1 arrival)
    uint64_t decoded[2];          // team -> loader: meta[b] read (one arrival per team warp)
    uint64_t sized[2];            // team -> placer: sizes in size[b] (one arrival per team warp)
    uint64_t placed[2];           // placer -> team: offsets in off[b] (1 arrival)
    uint64_t full[kRSlots];       // a rank chunk landed in the slot (transaction count)
    uint64_t free_[kRSlots];      // the team is done with the slot (one arrival per team warp)
    unsigned long long tally[2];  // sized warps (high word) and their bytes (low word)
    uint32_t size[2][kRChunks];
    uint64_t gid[2];              // group sized in slot b, or kNoGroup
    uint32_t failed[2];           // the group could not be reduced: the placer poisons it
    uint64_t off[2][kRChunks];    // chunk offsets, or kFlagPoison
    uint32_t row_tot[4];          // the decoder's per-quarter escape totals
    volatile uint32_t abort;      // a bounded wait ran out: every role stops
    ReduceMeta meta[2];
};

// --------------------------------------------------------------------------- loader
__device__ __forceinline__ void reduce_loader(const ReduceInputs& inputs, int R, const StreamOut& so, uint8_t* ring,
                                              ReduceSmem& sm) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t n_groups = (so.n_chunks + kRChunks - 1) / kRChunks;
    uint32_t u = 0;  // rank chunks issued so far
    for (int i = 0; !warp_any(sm.abort); ++i) {
        const int b = i & 1;
        // meta[b] was last read by the team for group i - 2
        if (i >= 2 && !warp_wait(&sm.decoded[b], (uint32_t)((i - 2) >> 1) & 1u)) {
            if (lane == 0) {
                record_error(so.ws, kStatusTimeout);
                sm.abort = 1;
            }
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
        const uint64_t c0 = g * kRChunks;
        const uint32_t n_out = (uint32_t)min((uint64_t)kRChunks, so.n_chunks - c0);
        bool ok = true;
        for (uint32_t idx = lane; idx < n_out * (uint32_t)R; idx += 32) {
            const uint32_t j = idx / (uint32_t)R, r = idx % (uint32_t)R;
            const ChunkView v = locate_chunk(inputs.in[r], inputs.in_bytes[r], so.n_elems, so.n_chunks, c0 + j);
            m.off[j][r] = v.offset;
            m.bytes[j][r] = v.bytes;
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
        if (!ok) continue;  // nothing to stream: the team poisons the group
        for (uint32_t j = 0; j < n_out && !warp_any(sm.abort); ++j) {
            for (int r = 0; r < R; ++r, ++u) {
                const uint32_t s = u % kRSlots;
                // the slot's previous rank chunk (copy u - kRSlots) is consumed
                if (u >= (uint32_t)kRSlots && !warp_wait(&sm.free_[s], (u / kRSlots - 1) & 1u)) {
                    if (lane == 0) {
                        record_error(so.ws, kStatusTimeout);
                        sm.abort = 1;
                    }
                    break;
                }
                if (warp_any(sm.abort)) break;
                if (lane == 0) {
                    fence_proxy_async_smem();
                    bulk_load(ring + (size_t)s * kMaxChunkBytes, inputs.in[r] + m.off[j][r], m.bytes[j][r],
                              &sm.full[s]);
                }
                __syncwarp();
            }
        }
    }
    // no copy may still be landing when the CTA exits
    for (uint32_t v = u > (uint32_t)kRSlots ? u - kRSlots : 0u; v < u; ++v)
        mbar_wait(&sm.full[v % kRSlots], (v / kRSlots) & 1u);
}

// --------------------------------------------------------------------------- placer
__device__ __forceinline__ void reduce_placer(const StreamOut& so, ReduceSmem& sm) {
    const uint32_t lane = threadIdx.x & 31;
    for (int i = 0; !warp_any(sm.abort); ++i) {
        const int b = i & 1;
        if (!warp_wait(&sm.sized[b], (uint32_t)(i >> 1) & 1u)) {
            if (lane == 0) {
                record_error(so.ws, kStatusTimeout);
                sm.abort = 1;
            }
            break;
        }
        const uint64_t g = sm.gid[b];
        if (g == kNoGroup) break;
        const uint32_t mine = lane < (uint32_t)kRChunks ? sm.size[b][lane] : 0u;
        uint32_t incl = mine;
#pragma unroll
        for (int d = 1; d < kRChunks; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += t;
        }
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, kRChunks - 1);
        uint64_t go;
        if (sm.failed[b]) {
            if (lane == 0) st_relaxed_u64(&so.status[g], kFlagPoison);
            go = kFlagPoison;
        } else {
            go = lookback_offset_wide(so.status, g, total, data_start(so.n_chunks), so.ws, true);
        }
        if (lane < (uint32_t)kRChunks) sm.off[b][lane] = go == kFlagPoison ? kFlagPoison : go + (incl - mine);
        if (lane == 0) sm.tally[b] = 0;  // next used for group i + 2, after its writers saw placed[b]
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.placed[b]);
    }
}

// --------------------------------------------------------------------------- team
struct TeamChunk {  // one warp's output chunk between sizing and writing
    ChunkRegs regs;
    ChunkPlan plan;
    uint32_t bytes;  // 0: nothing to write
    uint64_t c;
};

__device__ __forceinline__ void reduce_team(int R, const StreamOut& so, uint8_t* park_base, const uint8_t* ring,
                                            ReduceSmem& sm) {
    const uint32_t t = threadIdx.x, lane = t & 31, w = t >> 5;
    const uint64_t n_full = so.n_elems / kChunkElems;
    uint32_t u = 0;  // rank chunks consumed so far (the loader's order)
    TeamChunk cur, prev;
    prev.bytes = 0;
    prev.c = 0;
    for (int i = 0;; ++i) {
        const int b = i & 1;
        uint8_t* park = park_base + (size_t)b * kRChunks * kParkChunkBytes;
        const bool ready = mbar_wait(&sm.meta_ready[b], (uint32_t)(i >> 1) & 1u);
        if (TeamBarrier::any(!ready || sm.abort)) {
            if (t == 0) {
                record_error(so.ws, kStatusTimeout);
                sm.abort = 1;
            }
            return;
        }
        const ReduceMeta& m = sm.meta[b];
        const uint64_t g = m.g;
        if (g != kNoGroup) {
            const uint64_t c0 = g * kRChunks;
            const uint32_t n_out = m.n_out;
            // each warp decodes its quarter of every staged rank chunk on its
            // own; the team meets once per group, when the chunks are parked
            uint32_t wfail = m.ok ? 0u : kStatusCorrupt;
            for (uint32_t j = 0; j < n_out && m.ok; ++j) {
                const uint64_t c = c0 + j;
                const uint64_t left = so.n_elems - c * kChunkElems;
                const uint32_t n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;
                uint64_t acc[16];
                bool special = false;
                for (int r = 0; r < R; ++r, ++u) {
                    const uint32_t s = u % kRSlots;
                    const uint8_t* buf = ring + (size_t)s * kMaxChunkBytes;
                    const bool landed = !warp_any(sm.abort) && warp_wait(&sm.full[s], (u / kRSlots) & 1u);
                    if (!landed) {
                        if (lane == 0) {
                            record_error(so.ws, kStatusTimeout);
                            sm.abort = 1;
                        }
                        wfail = kStatusTimeout;
                        continue;  // the slot was not filled: nothing to free
                    }
                    if (wfail == 0) {
                        const ChunkHeader h = read_chunk_header(buf);
                        bool good = chunk_header_valid(h, m.bytes[j][r], n_c);
                        uint32_t P[16];
                        if (good) {
                            if (n_c < kChunkElems) {  // partial last chunk: raw values, read those that exist
                                const uint16_t* vals = reinterpret_cast<const uint16_t*>(buf + kChunkHeaderBytes);
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                                    for (int x = 0; x < 4; ++x) {
                                        const uint32_t e = 256 * (4 * w + jj) + 8 * lane + 2 * x;
                                        const uint32_t lo = e < n_c ? vals[e] : 0u, hi = e + 1 < n_c ? vals[e + 1] : 0u;
                                        P[4 * jj + x] = lo | (hi << 16);
                                    }
                                special = true;
                            } else {
                                bool sp = false;
                                good = decode_quarter_warp(buf, h, w, P, sp);
                                special = special || sp;
                            }
                        }
                        if (!good) {
                            wfail = kStatusCorrupt;
                        } else if (r == 0) {
#pragma unroll
                            for (int x = 0; x < 16; ++x) acc[x] = widen_pair(P[x]);
                        } else {
#pragma unroll
                            for (int x = 0; x < 16; ++x) acc[x] = add_f32x2(acc[x], widen_pair(P[x]));
                        }
                    }
                    __syncwarp();  // the warp is done with slot s
                    if (lane == 0) mbar_arrive(&sm.free_[s]);
                }
                if (wfail == 0) {
                    uint32_t P[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) P[x] = round_pair_bf16(acc[x]);
                    if (special) {
#pragma unroll
                        for (int x = 0; x < 16; ++x) P[x] = canonical_nan_pair(P[x]);
                    }
                    uint8_t* dst = park + (size_t)j * kParkChunkBytes;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        *reinterpret_cast<uint4*>(dst + 512 * (4 * w + jj) + 16 * lane) =
                            make_uint4(P[4 * jj], P[4 * jj + 1], P[4 * jj + 2], P[4 * jj + 3]);
                }
            }
            if (lane == 0) mbar_arrive(&sm.decoded[b]);
            // the parked chunks are complete once the team meets; a raw one
            // leaves by a bulk copy, so order the generic writes for the
            // async proxy first
            fence_proxy_async_smem();
            if (TeamBarrier::any(sm.abort != 0)) return;  // every team warp returns here
            const uint32_t fail = TeamBarrier::any(wfail != 0) ? kStatusCorrupt : 0u;
            cur.c = c0 + w;
            cur.bytes = 0;
            if (fail == 0) {
                if (cur.c < n_full) {
                    cur.plan = plan_chunk_warp(park + (size_t)w * kParkChunkBytes, cur.regs);
                    cur.bytes = cur.plan.bytes;
                } else if (cur.c < so.n_chunks) {
                    cur.bytes = tail_chunk_bytes((uint32_t)(so.n_elems - cur.c * kChunkElems));
                }
            }
            __syncwarp();
            if (lane == 0) {
                sm.size[b][w] = cur.bytes;
                if (w == 0) {
                    sm.gid[b] = g;
                    sm.failed[b] = fail;
                    if (fail) record_error(so.ws, fail);
                }
                if (fail == 0) {
                    // the last warp to size the group publishes its size at once,
                    // so later groups' look-backs need not wait for the placer
                    const unsigned long long old = atomicAdd(&sm.tally[b], (1ull << 32) | cur.bytes);
                    if ((old >> 32) == kRChunks - 1)
                        publish_unit_size(so.status, g, (uint32_t)old + cur.bytes, data_start(so.n_chunks));
                }
                mbar_arrive(&sm.sized[b]);
            }
            if (fail) cur.bytes = 0;
        } else if (lane == 0) {
            if (w == 0) sm.gid[b] = kNoGroup;
            mbar_arrive(&sm.sized[b]);
        }
        // write this warp's chunk of the previous group
        if (i > 0) {
            const int pb = b ^ 1;
            if (warp_wait(&sm.placed[pb], (uint32_t)((i - 1) >> 1) & 1u)) {
                const uint64_t off = sm.off[pb][w];
                if (off != kFlagPoison && prev.bytes > 0) {
                    if (off + prev.bytes > so.capacity) {  // cannot happen for a correct placement
                        if (lane == 0) record_error(so.ws, kStatusCorrupt);
                    } else {
                        const uint8_t* chunk = park_base + ((size_t)pb * kRChunks + w) * kParkChunkBytes;
                        uint8_t* dst = so.out + off;
                        if (prev.c < n_full) {
                            write_chunk_warp(prev.regs, prev.plan, chunk, dst);
                        } else {
                            const uint16_t* vals = reinterpret_cast<const uint16_t*>(chunk);
                            write_tail_chunk_warp([vals](uint32_t e) { return vals[e]; },
                                                  (uint32_t)(so.n_elems - prev.c * kChunkElems), dst);
                        }
                        if (lane == 0) finish_chunk(so, prev.c, off, prev.bytes);
                    }
                }
            } else if (lane == 0) {
                record_error(so.ws, kStatusTimeout);
                sm.abort = 1;
            }
        }
        if (g == kNoGroup) return;
        prev = cur;
    }
}

__global__ void __launch_bounds__(kReduceThreads, 2) reduce_kernel(ReduceInputs inputs, int R, StreamOut so) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ ReduceSmem sm;
    uint8_t* park = smem;
    uint8_t* ring = smem + kParkBytes;
    const uint32_t w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.meta_ready[b], 1);
            mbar_init(&sm.decoded[b], kRChunks);
            mbar_init(&sm.sized[b], kRChunks);
            mbar_init(&sm.placed[b], 1);
            sm.tally[b] = 0;
        }
        for (int s = 0; s < kRSlots; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.free_[s], kRChunks);
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
        reduce_team(R, so, park, ring, sm);
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
    const uint64_t n_groups = (so.n_chunks + kRChunks - 1) / kRChunks;
    const uint64_t slots = 2 * (uint64_t)sms;
    const unsigned grid = (unsigned)(n_groups < slots ? n_groups : slots);
    reduce_kernel<<<grid, kReduceThreads, kReduceSmemBytes, stream>>>(inputs, R, so);
    return cudaGetLastError();
}

}  // namespace cccl

// cccl_compress.cu -- the compress kernel ("CCCL: In-GPU Compression-Coupled
// Collective Communication", sections 4.1, 4.3, 4.4; section 5 for the raw
// partial chunk).
//
// Persistent and pipelined: one CTA per SM, 2 G compute warps (a pair per
// chunk) plus one control warp, and a ring of kRing stages, each holding one
// group of G consecutive chunks staged by bulk (TMA) copies (G = 8 for the
// 16-bit element types, 4 for fp32).  Per group:
//   control warp  takes a ticket (the group index), issues the copies two
//                 groups ahead, and once the pairs have sized the group,
//                 places it with one decoupled look-back;
//   compute pair  sizes its chunk of group i+1 (exponent table, width,
//                 escapes; each warp keeps its half of the offset planes in
//                 registers) while the control warp places group i, then
//                 writes its chunk of group i at the final offset, a half per
//                 warp: the residual section and the escapes read back from
//                 the staged input, the bit-planes from registers, a raw chunk
//                 by one bulk (TMA) store.
// So the look-back's wait for earlier groups overlaps with the sizing of the
// next group, and the next copies are in flight during both.
// Tickets hand out groups in order to CTAs that are already running, so every
// group a look-back waits on belongs to a running CTA: the waits always end.
#include <mutex>

#include "cccl.h"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

// chunks per group: 8 for the 16-bit types, 4 for fp32 (the stage of a group
// is 64 KiB either way); each chunk is encoded by a pair of compute warps
template <class D>
__host__ __device__ constexpr int group_of() { return D::kElemBytes == 4 ? 4 : 8; }
constexpr int kRing = 3;  // groups staged per CTA
template <class D>
__host__ __device__ constexpr size_t raw_chunk_of() { return (size_t)D::kElemBytes * kChunkElems; }
template <class D>
__host__ __device__ constexpr int compress_threads() { return 32 * (2 * group_of<D>() + 1); }
template <class D>
__host__ __device__ constexpr size_t compress_smem() { return (size_t)kRing * group_of<D>() * raw_chunk_of<D>(); }

template <int G>
struct CompressSmem {
    uint64_t load[kRing][G];       // a chunk of the stage landed (one per pair)
    uint64_t sized[kRing];         // every pair sized its chunk of the stage's group
    uint64_t free_[kRing];         // every compute warp wrote its part of the stage's group
    uint64_t placed[2];            // control warp published the offsets
    uint64_t group[kRing];         // group index held by each stage (>= n_groups: none)
    unsigned long long tally[kRing];  // sized pairs (high word) and their bytes (low word)
    uint32_t size[kRing][G];
    uint64_t off[2][G];            // chunk offsets, or kFlagPoison
    PairXch xch[G];                // each pair's exchange record
    uint32_t hist[G][264];         // window-base variant: each pair's exponent histogram
    uint32_t below[2 * G][264];    //   and each warp's prefix counts of it
};

// Control lane: fill stage s with group g (or mark it empty).
template <class D, int G>
__device__ __forceinline__ void issue_group(const uint8_t* in, const Paging& pg, WsHeader* ws, uint64_t g,
                                            uint64_t n_groups, uint64_t n_full, uint8_t* stage, CompressSmem<G>& sm,
                                            int s) {
    constexpr size_t kRaw = raw_chunk_of<D>();
    sm.group[s] = g;
    sm.tally[s] = 0;
    for (int w = 0; w < G; ++w) {
        const uint64_t c = g * G + w;
        const uint64_t e = g < n_groups && c < n_full ? chunk_elem_offset(pg, c) : kBadChunk;
        if (e != kBadChunk) {
            bulk_load(stage + ((size_t)s * G + w) * kRaw, in + e * D::kElemBytes, (uint32_t)kRaw, &sm.load[s][w]);
        } else {
            if (g < n_groups && c < n_full) record_error(ws, kStatusInvalidArg);  // a block outside the pool
            mbar_arrive(&sm.load[s][w]);  // nothing to copy: complete the phase at once
        }
    }
}

// Compute warp, one group: size this warp's half of its pair's chunk of
// group i (into cur) and then write its half of the pair's chunk of group
// i - 1 (from prev).  Returns false once the groups are exhausted (after
// writing group i - 1).  The loop keeps one copy of it: instruction-cache
// space, not register moves, is the scarce resource.
struct WarpChunk {
    HalfRegs regs;
    PairPlan plan;
    uint32_t bytes;
    uint64_t c;
};

template <class D, bool kWindow>
__device__ __forceinline__ bool compute_step(int i, const uint8_t* __restrict__ in, const StreamOut& so,
                                             uint8_t* stage, CompressSmem<group_of<D>()>& sm, WarpChunk& cur,
                                             WarpChunk& prev) {
    constexpr int G = group_of<D>();
    constexpr size_t kRaw = raw_chunk_of<D>();
    using Elem = typename std::conditional<D::kElemBytes == 4, uint32_t, uint16_t>::type;
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5, ci = w >> 1, h = w & 1;
    const PairBarrier bar{1u + ci};
    const uint64_t n_full = so.n_elems / kChunkElems;
    const uint64_t n_groups = (so.n_chunks + G - 1) / G;
    const int s = i % kRing;
    // the pair decides together: a bounded wait that ran out for either warp
    // fails both, so their barriers stay matched
    const bool filled = !bar.any(!mbar_wait(&sm.load[s][ci], (uint32_t)(i / kRing) & 1u));
    const uint64_t g = sm.group[s];
    const bool live = filled && g < n_groups;
    if (live) {
        cur.c = g * G + ci;
        cur.bytes = 0;
        if (cur.c < n_full) {
            const uint8_t* chunk = stage + ((size_t)s * G + ci) * kRaw;
            cur.plan = kWindow ? plan_chunk_pair_window<D>(chunk, cur.regs, h, sm.xch[ci], sm.hist[ci], sm.below[w], bar)
                               : plan_chunk_pair<D>(chunk, cur.regs, h, sm.xch[ci], bar);
            cur.bytes = cur.plan.p.bytes;
        } else if (cur.c < so.n_chunks) {
            cur.bytes = tail_chunk_bytes<D>((uint32_t)(so.n_elems - cur.c * kChunkElems));
        }
        __syncwarp();
        if (h == 0 && lane == 0) {
            sm.size[s][ci] = cur.bytes;
            // the last pair to size the group publishes its size at once, so
            // the look-backs of later groups need not wait for this CTA's
            // control warp
            const unsigned long long old = atomicAdd(&sm.tally[s], (1ull << 32) | cur.bytes);
            if ((old >> 32) == G - 1)
                publish_unit_size(so.status, g, (uint32_t)old + cur.bytes, data_start(so.n_chunks));
            mbar_arrive(&sm.sized[s]);
        }
    } else if (!filled && h == 0 && lane == 0) {
        record_error(so.ws, kStatusTimeout);
    }
    if (i > 0) {  // write group i - 1
        const int ip = i - 1, sp = ip % kRing;
        if (__all_sync(0xFFFFFFFFu, mbar_wait(&sm.placed[ip & 1], (uint32_t)(ip >> 1) & 1u))) {
            const uint64_t off = sm.off[ip & 1][ci];
            if (off != kFlagPoison && prev.bytes > 0) {
                if (off + prev.bytes > so.capacity) {  // cannot happen for a correct placement
                    if (h == 0 && lane == 0) record_error(so.ws, kStatusCorrupt);
                } else {
                    uint8_t* dst = so.out + off;
                    if (prev.c < n_full) {
                        write_chunk_pair<D>(prev.regs, prev.plan, h, stage + ((size_t)sp * G + ci) * kRaw, dst);
                    } else if (h == 0) {
                        // a partial chunk is never paged
                        const Elem* src = reinterpret_cast<const Elem*>(in) + prev.c * kChunkElems;
                        write_tail_chunk_warp<D>([src](uint32_t e) { return src[e]; },
                                                 (uint32_t)(so.n_elems - prev.c * kChunkElems), dst);
                    }
                    if (h == 0 && lane == 0) finish_chunk(so, prev.c, off, prev.bytes);
                }
            }
        } else if (h == 0 && lane == 0) {
            record_error(so.ws, kStatusTimeout);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.free_[sp]);  // this warp is done with stage sp
    }
    return live;
}

template <class D, bool kWindow>
__global__ void __launch_bounds__(compress_threads<D>(), 1)
    compress_kernel(const uint8_t* __restrict__ in, Paging pg, StreamOut so) {
    constexpr int G = group_of<D>();
    constexpr int kCtrl = 2 * G;  // warp index of the control warp
    extern __shared__ __align__(128) uint8_t stage[];
    __shared__ CompressSmem<G> sm;
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint64_t n_full = so.n_elems / kChunkElems;
    const uint64_t n_groups = (so.n_chunks + G - 1) / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            for (int i = 0; i < G; ++i) mbar_init(&sm.load[s][i], 1);
            mbar_init(&sm.sized[s], G);
            mbar_init(&sm.free_[s], 2 * G);
        }
        for (int x = 0; x < 2; ++x) mbar_init(&sm.placed[x], 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (w == kCtrl) {
        // ---------------------------------------------------------------- control warp
        // Tickets fix the placement order, so they are taken in the order the
        // groups will be sized: the second when the first group's data has
        // landed, the third once the first group is sized, later ones as
        // stages free up.  (Taken all at once, every CTA's third ticket would
        // be sized two iterations later than its number says, and every
        // look-back behind it would wait for that.)
        if (lane == 0) issue_group<D>(in, pg, so.ws, atomicAdd(&so.ws->ticket, 1u), n_groups, n_full, stage, sm, 0);
        __syncwarp();
        const bool first_landed = __all_sync(0xFFFFFFFFu, mbar_wait(&sm.load[0][0], 0u));
        if (lane == 0) {
            if (!first_landed) record_error(so.ws, kStatusTimeout);
            issue_group<D>(in, pg, so.ws, atomicAdd(&so.ws->ticket, 1u), n_groups, n_full, stage, sm, 1);
        }
        __syncwarp();
        for (int i = 0;; ++i) {
            const int s = i % kRing;
            const uint64_t g = sm.group[s];
            if (g >= n_groups) break;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sm.sized[s], (uint32_t)(i / kRing) & 1u))) {
                if (lane == 0) record_error(so.ws, kStatusTimeout);
                break;
            }
            if (i == 0) {
                if (lane == 0)
                    issue_group<D>(in, pg, so.ws, atomicAdd(&so.ws->ticket, 1u), n_groups, n_full, stage, sm, 2);
                __syncwarp();
            }
            const uint32_t mine = lane < (uint32_t)G ? sm.size[s][lane] : 0u;
            uint32_t incl = mine;
#pragma unroll
            for (int d = 1; d < G; d <<= 1) {
                const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= (uint32_t)d) incl += t;
            }
            const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, G - 1);
            const uint64_t go = lookback_offset_wide(so.status, g, total, data_start(so.n_chunks), so.ws, true);
            if (lane < (uint32_t)G) sm.off[i & 1][lane] = go == kFlagPoison ? kFlagPoison : go + (incl - mine);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.placed[i & 1]);
            // group i-1 is written out: refill its stage, for group i+2
            if (i >= 1) {
                const int sp = (i - 1) % kRing;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sm.free_[sp], (uint32_t)((i - 1) / kRing) & 1u))) {
                    if (lane == 0) record_error(so.ws, kStatusTimeout);
                    break;
                }
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue_group<D>(in, pg, so.ws, atomicAdd(&so.ws->ticket, 1u), n_groups, n_full, stage, sm, sp);
                }
                __syncwarp();
            }
        }
        return;
    }

    // -------------------------------------------------------------------- compute warps
    WarpChunk cur, prev;  // the chunk being sized and the one being written
    cur.bytes = prev.bytes = 0;
    cur.c = prev.c = 0;
    for (int i = 0;; ++i) {
        if (!compute_step<D, kWindow>(i, in, so, stage, sm, cur, prev)) break;
        prev = cur;
    }
}

// Per-device record of the shared-memory limit set for compress_kernel<D, W>,
// by element type code and table choice (a plain static array, so that each
// copy of this library loaded into a process keeps its own).
static PerDeviceOnce g_compress_smem_limit[4][2];

template <class D, bool kWindow>
cudaError_t launch_compress_t(const uint8_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                              cudaStream_t stream, const Paging& pg) {
    PerDeviceOnce& smem_limit = g_compress_smem_limit[D::kCode][kWindow ? 1 : 0];
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = smem_limit.run(dev, [] {
            return cudaFuncSetAttribute(compress_kernel<D, kWindow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)compress_smem<D>());
        });
    if (e != cudaSuccess) return e;
    StreamOut so;
    so.out = out;
    so.capacity = capacity;
    so.ws = static_cast<WsHeader*>(ws);
    so.status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    so.n_elems = n_elems;
    so.n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    so.version = kWindow ? kVersionWindow : kVersion;
    so.dtype = D::kCode;
    const uint64_t n_groups = (so.n_chunks + group_of<D>() - 1) / group_of<D>();
    const unsigned grid = (unsigned)(n_groups < (uint64_t)sms ? n_groups : (uint64_t)sms);
    compress_kernel<D, kWindow><<<grid, compress_threads<D>(), compress_smem<D>(), stream>>>(in, pg, so);
    return cudaGetLastError();
}

cudaError_t launch_compress(const uint16_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                            cudaStream_t stream, const Paging& pg, bool window) {
    const uint8_t* bytes = reinterpret_cast<const uint8_t*>(in);
    return window ? launch_compress_t<Bf16, true>(bytes, n_elems, out, capacity, ws, stream, pg)
                  : launch_compress_t<Bf16, false>(bytes, n_elems, out, capacity, ws, stream, pg);
}

cudaError_t launch_compress_typed(uint32_t dtype, const void* in, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                                  void* ws, cudaStream_t stream, bool window) {
    const uint8_t* bytes = static_cast<const uint8_t*>(in);
    const Paging pg{nullptr, 1, 0};
    if (dtype == Fp16::kCode)
        return window ? launch_compress_t<Fp16, true>(bytes, n_elems, out, capacity, ws, stream, pg)
                      : launch_compress_t<Fp16, false>(bytes, n_elems, out, capacity, ws, stream, pg);
    if (dtype == Fp32::kCode)
        return window ? launch_compress_t<Fp32, true>(bytes, n_elems, out, capacity, ws, stream, pg)
                      : launch_compress_t<Fp32, false>(bytes, n_elems, out, capacity, ws, stream, pg);
    return window ? launch_compress_t<Bf16, true>(bytes, n_elems, out, capacity, ws, stream, pg)
                  : launch_compress_t<Bf16, false>(bytes, n_elems, out, capacity, ws, stream, pg);
}

// ---------------------------------------------------------------------------
// Compress without any allocation by the caller: the scratch that
// cccl_compress takes as a workspace (status header + one placement word per
// group) lives in this file-scope device array instead.  Every GPU that loads
// the library holds it until the process exits.
// ---------------------------------------------------------------------------
constexpr uint64_t kNoAllocMaxGroups = CCCL_NOALLOC_MAX_ELEMS / kChunkElems / group_of<Bf16>();
constexpr size_t kNoAllocScratchBytes = sizeof(WsHeader) + 8 * kNoAllocMaxGroups;
static_assert(CCCL_NOALLOC_MAX_ELEMS % ((uint64_t)kChunkElems * group_of<Bf16>()) == 0, "whole groups");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so its address is looked up once
// per device (with that device current) and cached.
cudaError_t noalloc_scratch(void** ptr) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_compress_noalloc(const uint16_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                                    cudaStream_t stream) {
    if (n_elems == 0 || n_elems > CCCL_NOALLOC_MAX_ELEMS) return cudaErrorInvalidValue;
    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return e;
    const uint64_t n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    const uint64_t n_groups = (n_chunks + group_of<Bf16>() - 1) / group_of<Bf16>();
    // the scratch keeps the previous call's contents: clear what must start at
    // zero, and the stream header, whose size field then stays 0 unless the
    // whole stream was placed
    e = cudaMemsetAsync(scratch, 0, sizeof(WsHeader) + 8 * n_groups, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(out, 0, kStreamHeaderBytes, stream);
    if (e != cudaSuccess) return e;
    return launch_compress(in, n_elems, out, capacity, scratch, stream, Paging{nullptr, 1, 0}, false);
}

}  // namespace cccl

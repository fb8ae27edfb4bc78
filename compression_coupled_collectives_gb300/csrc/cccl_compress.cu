// cccl_compress.cu -- the compress kernel ("CCCL: In-GPU Compression-Coupled
// Collective Communication", sections 4.1, 4.3, 4.4; section 5 for the raw
// partial chunk).
//
// One CTA of kGroup warps per group of kGroup consecutive chunks: one bulk
// (TMA) copy per chunk stages the input in shared memory, each warp sizes its
// chunk (exponent table, width, escapes), one decoupled look-back places the
// whole group, and each warp writes its chunk straight to its final offset.
#include <mutex>

#include "cccl.h"

#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kGroup = 8;
constexpr size_t kCompressSmemBytes = (size_t)kGroup * 2 * kChunkElems;

// Thread 0: bulk-copy the full chunks of group g into the stage buffers.
__device__ __forceinline__ void load_group(const uint16_t* in, uint64_t g, uint64_t n_full, uint8_t* stage,
                                           uint64_t* bars) {
    for (int i = 0; i < kGroup; ++i) {
        const uint64_t c = g * kGroup + i;
        if (c < n_full) bulk_load(stage + (size_t)i * 2 * kChunkElems, in + c * kChunkElems, 2 * kChunkElems, &bars[i]);
    }
}

__global__ void __launch_bounds__(32 * kGroup, 3) compress_kernel(const uint16_t* __restrict__ in, StreamOut so) {
    extern __shared__ __align__(128) uint8_t stage[];
    __shared__ __align__(8) uint64_t bars[kGroup];
    __shared__ uint32_t s_bytes[kGroup], s_parity[kGroup];
    __shared__ uint64_t s_offset[kGroup];
    __shared__ uint64_t s_group;
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint64_t n_full = so.n_elems / kChunkElems;

    // Groups are placed in ticket order (the look-back's forward-progress
    // guarantee).  Tickets normally follow blockIdx, so the copies of group
    // blockIdx.x start before the ticket arrives and are redone otherwise.
    if (threadIdx.x == 0) {
        for (int i = 0; i < kGroup; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        const uint64_t guess = blockIdx.x;
        load_group(in, guess, n_full, stage, bars);
        const uint64_t g = atomicAdd(&so.ws->ticket, 1u);
        for (int i = 0; i < kGroup; ++i) s_parity[i] = 0;
        if (g != guess) {
            for (int i = 0; i < kGroup; ++i) {
                if (guess * kGroup + i < n_full) {
                    mbar_wait(&bars[i], 0);  // the stage must be idle before it is refilled
                    s_parity[i] = 1;
                }
            }
            load_group(in, g, n_full, stage, bars);
        }
        s_group = g;
    }
    __syncthreads();
    const uint64_t g = s_group;
    const uint64_t c = g * kGroup + w;
    const uint8_t* chunk = stage + (size_t)w * 2 * kChunkElems;

    // phase A: size of this warp's chunk
    ChunkPlan pl{};
    uint32_t bytes = 0;
    bool failed = false;
    if (c < n_full) {
        if (mbar_wait(&bars[w], s_parity[w])) {
            pl = plan_chunk_warp(chunk);
            bytes = pl.bytes;
        } else {
            failed = true;
            if (lane == 0) record_error(so.ws, kStatusTimeout);
        }
    } else if (c < so.n_chunks) {
        bytes = tail_chunk_bytes((uint32_t)(so.n_elems - c * kChunkElems));
    }
    if (lane == 0) s_bytes[w] = bytes;

    // placement of the whole group
    const uint64_t off = place_group<kGroup>(so, g, s_bytes, s_offset, failed);
    if (off == kFlagPoison || bytes == 0) return;
    if (off + bytes > so.capacity) {  // cannot happen for a correct placement; never write past the buffer
        if (lane == 0) record_error(so.ws, kStatusCorrupt);
        return;
    }

    // phase B: write the chunk at its offset
    uint8_t* dst = so.out + off;
    if (c < n_full) {
        write_chunk_warp(chunk, pl, dst);
    } else {
        const uint16_t* src = in + c * kChunkElems;
        write_tail_chunk_warp([src](uint32_t i) { return src[i]; }, (uint32_t)(so.n_elems - c * kChunkElems), dst);
    }
    if (lane == 0) finish_chunk(so, c, off, bytes);
}

cudaError_t launch_compress(const uint16_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                            cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kCompressSmemBytes);
    });
    if (attr != cudaSuccess) return attr;
    StreamOut so;
    so.out = out;
    so.capacity = capacity;
    so.ws = static_cast<WsHeader*>(ws);
    so.status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    so.n_elems = n_elems;
    so.n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    const uint64_t n_groups = (so.n_chunks + kGroup - 1) / kGroup;
    compress_kernel<<<(unsigned)n_groups, 32 * kGroup, kCompressSmemBytes, stream>>>(in, so);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Compress without any allocation by the caller: the scratch that
// cccl_compress takes as a workspace (status header + one placement word per
// group) lives in this file-scope device array instead.  Every GPU that loads
// the library holds it until the process exits.
// ---------------------------------------------------------------------------
constexpr uint64_t kNoAllocMaxGroups = CCCL_NOALLOC_MAX_ELEMS / kChunkElems / kGroup;
constexpr size_t kNoAllocScratchBytes = sizeof(WsHeader) + 8 * kNoAllocMaxGroups;
static_assert(CCCL_NOALLOC_MAX_ELEMS % ((uint64_t)kChunkElems * kGroup) == 0, "whole groups");

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
    const uint64_t n_groups = (n_chunks + kGroup - 1) / kGroup;
    // the scratch keeps the previous call's contents: clear what must start at
    // zero, and the stream header, whose size field then stays 0 unless the
    // whole stream was placed
    e = cudaMemsetAsync(scratch, 0, sizeof(WsHeader) + 8 * n_groups, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(out, 0, kStreamHeaderBytes, stream);
    if (e != cudaSuccess) return e;
    return launch_compress(in, n_elems, out, capacity, scratch, stream);
}

}  // namespace cccl

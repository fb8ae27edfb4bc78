// cccl_api.cu -- the C ABI (include/cccl.h): argument checks, workspace reset
// and kernel launches.  Nothing here allocates memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "cccl.h"
#include "cccl_device.cuh"
#include "cccl_launch.h"

namespace cccl {

// cccl_selftest_timeouts: warp 0 waits on an mbarrier that no thread arrives
// on; warp 1 runs the look-back of unit 1, whose predecessor (unit 0) never
// publishes.  Both waits give up after kWaitLimitNs; each records TIMEOUT.
__global__ void selftest_timeouts_kernel(WsHeader* ws) {
    __shared__ uint64_t never;
    if (threadIdx.x == 0) {
        mbar_init(&never, 1);
        fence_mbar_init();
    }
    __syncthreads();
    uint64_t* status = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + sizeof(WsHeader));
    if (threadIdx.x < 32) {
        const bool done = mbar_wait(&never, 0);
        if (!done && threadIdx.x == 0) record_error(ws, kStatusTimeout);
    } else {
        lookback_offset_wide(status, 1, 16, data_start(2), ws);
    }
}

// cccl_selftest_lookback.  Publication: unit 0 its end offset, the poisoned
// unit (if any) the poison flag, every other unit its size alone.
__global__ void selftest_publish_kernel(const uint32_t* sizes, uint32_t n, uint32_t poison, uint64_t start,
                                        uint64_t* status) {
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < n; g += gridDim.x * blockDim.x)
        status[g] = g == poison ? kFlagPoison : (g == 0 ? (kFlagPrefix | (start + sizes[0])) : (kFlagAggregate | sizes[g]));
}
// Serial order: one warp runs the look-back of units n-1, n-2, ..., 1 in that
// order, so no unit finds a prefix but unit 0's: each walks back over every
// predecessor, many 256-entry windows for the later units.
// The poisoned unit does not look back (a failed unit never does).
__global__ void selftest_lookback_serial_kernel(const uint32_t* sizes, uint32_t n, uint32_t poison, uint64_t start,
                                                WsHeader* ws, uint64_t* status, uint64_t* result) {
    const uint32_t lane = threadIdx.x & 31;
    for (uint32_t g = n - 1; g >= 1; --g) {
        const uint64_t off = g == poison ? kFlagPoison : lookback_offset_wide(status, g, sizes[g], start, ws, true);
        if (lane == 0) result[g] = off;
    }
    if (lane == 0) result[0] = poison == 0 ? kFlagPoison : start;
}
// Concurrent order, as the compress and reduce kernels run it: warps take
// tickets (unit numbers in order, so every predecessor is already being
// worked on), wait a pseudo-random time (up to 20 us; one unit in 64 up to
// 200 us, a late publisher), then publish their size and look back.
__global__ void selftest_lookback_concurrent_kernel(const uint32_t* sizes, uint32_t n, uint32_t poison,
                                                    uint64_t start, WsHeader* ws, uint64_t* status,
                                                    uint64_t* result) {
    const uint32_t lane = threadIdx.x & 31;
    for (;;) {
        uint32_t g = 0;
        if (lane == 0) g = atomicAdd(&ws->ticket, 1u);
        g = __shfl_sync(0xFFFFFFFFu, g, 0);
        if (g >= n) return;
        uint32_t h = g * 2654435761u;
        h ^= h >> 15;
        h *= 2246822519u;
        h ^= h >> 13;
        const uint64_t wait_ns = (h % 64u == 0u) ? 200000u : (h % 20000u);
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < wait_ns) __nanosleep(1000);  // ends: the timer advances
        uint64_t off;
        if (g == poison) {
            if (lane == 0) st_relaxed_u64(&status[g], kFlagPoison);
            off = kFlagPoison;
        } else {
            off = lookback_offset_wide(status, g, sizes[g], start, ws);
        }
        if (lane == 0) result[g] = off;
    }
}

}  // namespace cccl

namespace {

using cccl::kChunkElems;

uint64_t n_chunks_of(size_t n) { return (n + kChunkElems - 1) / kChunkElems; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuMemGetAddressRange, resolved once through the runtime so that the library
// loads (and its pure host functions work) on machines without a driver.
using AddrRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
AddrRangeFn addr_range_fn() {
    static const AddrRangeFn fn = []() -> AddrRangeFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return reinterpret_cast<AddrRangeFn>(p);
    }();
    return fn;
}

// True if [p, p + bytes) lies inside one device (or managed) allocation.
bool device_range(const void* p, size_t bytes) {
    const AddrRangeFn range = addr_range_fn();
    if (p == nullptr || range == nullptr) return false;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return a >= base && bytes <= size && a - base <= size - bytes;
}

cccl_status clear_ws(void* ws, size_t bytes, cudaStream_t s) {
    return cudaMemsetAsync(ws, 0, bytes, s) == cudaSuccess ? CCCL_OK : CCCL_ERR_CUDA;
}

size_t ws_used(size_t n) { return sizeof(cccl::WsHeader) + 8 * n_chunks_of(n); }

// bytes per value of a CCCL_DTYPE_*, 0 for an unknown type
uint64_t elem_bytes(int dtype) {
    if (dtype == CCCL_DTYPE_BF16 || dtype == CCCL_DTYPE_FP16) return 2;
    if (dtype == CCCL_DTYPE_FP32) return 4;
    return 0;
}

}  // namespace

extern "C" {

size_t cccl_compress_bound(size_t n_elems) {
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return 0;
    const uint64_t full = n_elems / kChunkElems, tail = n_elems % kChunkElems;
    uint64_t bytes = cccl::data_start(n_chunks_of(n_elems)) + full * cccl::kMaxChunkBytes;
    if (tail) bytes += 16 + cccl::pad16(2 * tail);
    return (size_t)bytes;
}

size_t cccl_workspace_bytes(size_t n_elems) {
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return 0;
    return (size_t)cccl::pad16(ws_used(n_elems));
}

cccl_status cccl_compress(const uint16_t* d_in, size_t n_elems, void* d_out, size_t out_capacity, void* d_ws,
                          size_t ws_bytes, cccl_stream_t stream) {
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_in) || !aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_in, 2 * n_elems) || !device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_compress(d_in, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws, s,
                              cccl::Paging{nullptr, 1, 0}) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_compress_window(const uint16_t* d_in, size_t n_elems, void* d_out, size_t out_capacity, void* d_ws,
                                 size_t ws_bytes, cccl_stream_t stream) {
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_in) || !aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_in, 2 * n_elems) || !device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_compress(d_in, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws, s,
                              cccl::Paging{nullptr, 1, 0}, true) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_compress_noalloc(const uint16_t* d_in, size_t n_elems, void* d_out, size_t out_capacity,
                                  cccl_stream_t stream) {
    if (n_elems == 0 || n_elems > CCCL_NOALLOC_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_in) || !aligned16(d_out)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_in, 2 * n_elems) || !device_range(d_out, out_capacity)) return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cccl::launch_compress_noalloc(d_in, n_elems, static_cast<uint8_t*>(d_out), out_capacity, s) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_decompress(const void* d_in, size_t in_bytes, uint16_t* d_out, size_t n_elems, void* d_ws,
                            size_t ws_bytes, cccl_stream_t stream) {
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS || in_bytes == 0) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_in) || !aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < sizeof(cccl::WsHeader)) return CCCL_ERR_INVALID_ARG;
    if (!device_range(d_in, in_bytes) || !device_range(d_out, 2 * n_elems) || !device_range(d_ws, ws_bytes))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, sizeof(cccl::WsHeader), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_decompress(static_cast<const uint8_t*>(d_in), in_bytes, d_out, n_elems, d_ws, s,
                                cccl::Paging{nullptr, 1, 0}) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_reduce_compressed(const void* const* h_ins, const size_t* h_in_bytes, int R, size_t n_elems,
                                   void* d_out, size_t out_capacity, void* d_ws, size_t ws_bytes,
                                   cccl_stream_t stream) {
    if (h_ins == nullptr || h_in_bytes == nullptr || R < 1 || R > cccl::kMaxRanks) return CCCL_ERR_INVALID_ARG;
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes)) return CCCL_ERR_INVALID_ARG;
    cccl::ReduceInputs inputs{};
    for (int r = 0; r < R; ++r) {
        if (!aligned16(h_ins[r]) || h_in_bytes[r] == 0 || !device_range(h_ins[r], h_in_bytes[r]))
            return CCCL_ERR_INVALID_ARG;
        inputs.in[r] = static_cast<const uint8_t*>(h_ins[r]);
        inputs.in_bytes[r] = h_in_bytes[r];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_reduce(inputs, R, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws, s) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

// Checks shared by the paged entry points; sets n_elems.
static cccl_status check_paged(const uint16_t* d_pool, size_t pool_blocks, size_t block_elems, const int32_t* d_table,
                               size_t n_blocks, size_t* n_elems) {
    if (block_elems == 0 || block_elems % kChunkElems != 0 || pool_blocks == 0 || n_blocks == 0)
        return CCCL_ERR_INVALID_ARG;
    if (pool_blocks > CCCL_MAX_ELEMS / block_elems || n_blocks > CCCL_MAX_ELEMS / block_elems ||
        pool_blocks > (size_t)INT32_MAX + 1)
        return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_pool) || d_table == nullptr || (reinterpret_cast<uintptr_t>(d_table) & 3) != 0)
        return CCCL_ERR_INVALID_ARG;
    if (!device_range(d_pool, 2 * pool_blocks * block_elems) || !device_range(d_table, 4 * n_blocks))
        return CCCL_ERR_INVALID_ARG;
    *n_elems = n_blocks * block_elems;
    return CCCL_OK;
}

cccl_status cccl_compress_paged(const uint16_t* d_pool, size_t pool_blocks, size_t block_elems, const int32_t* d_table,
                                size_t n_blocks, void* d_out, size_t out_capacity, void* d_ws, size_t ws_bytes,
                                cccl_stream_t stream) {
    size_t n_elems = 0;
    const cccl_status st = check_paged(d_pool, pool_blocks, block_elems, d_table, n_blocks, &n_elems);
    if (st != CCCL_OK) return st;
    if (!aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes)) return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    const cccl::Paging pg{d_table, block_elems / kChunkElems, pool_blocks};
    if (cccl::launch_compress(d_pool, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws, s, pg) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_decompress_paged(const void* d_in, size_t in_bytes, uint16_t* d_pool, size_t pool_blocks,
                                  size_t block_elems, const int32_t* d_table, size_t n_blocks, void* d_ws,
                                  size_t ws_bytes, cccl_stream_t stream) {
    size_t n_elems = 0;
    const cccl_status st = check_paged(d_pool, pool_blocks, block_elems, d_table, n_blocks, &n_elems);
    if (st != CCCL_OK) return st;
    if (in_bytes == 0 || !aligned16(d_in) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < sizeof(cccl::WsHeader)) return CCCL_ERR_INVALID_ARG;
    if (!device_range(d_in, in_bytes) || !device_range(d_ws, ws_bytes)) return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, sizeof(cccl::WsHeader), s) != CCCL_OK) return CCCL_ERR_CUDA;
    const cccl::Paging pg{d_table, block_elems / kChunkElems, pool_blocks};
    if (cccl::launch_decompress(static_cast<const uint8_t*>(d_in), in_bytes, d_pool, n_elems, d_ws, s, pg) !=
        cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_reduce_op(const void* const* h_ins, const size_t* h_in_bytes, int R, size_t n_elems, int op,
                           void* d_out, size_t out_capacity, void* d_ws, size_t ws_bytes, cccl_stream_t stream) {
    if (op != CCCL_OP_SUM && op != CCCL_OP_MIN && op != CCCL_OP_MAX) return CCCL_ERR_INVALID_ARG;
    if (h_ins == nullptr || h_in_bytes == nullptr || R < 1 || R > cccl::kMaxRanks) return CCCL_ERR_INVALID_ARG;
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes)) return CCCL_ERR_INVALID_ARG;
    cccl::ReduceInputs inputs{};
    inputs.op = (uint32_t)op;
    for (int r = 0; r < R; ++r) {
        if (!aligned16(h_ins[r]) || h_in_bytes[r] == 0 || !device_range(h_ins[r], h_in_bytes[r]))
            return CCCL_ERR_INVALID_ARG;
        inputs.in[r] = static_cast<const uint8_t*>(h_ins[r]);
        inputs.in_bytes[r] = h_in_bytes[r];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_reduce(inputs, R, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws, s) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_reduce_mixed(const uint16_t* d_local, const void* const* h_ins, const size_t* h_in_bytes,
                              int n_remote, size_t n_elems, void* d_out, size_t out_capacity, void* d_ws,
                              size_t ws_bytes, cccl_stream_t stream) {
    if (n_remote < 0 || n_remote > cccl::kMaxRanks - 1) return CCCL_ERR_INVALID_ARG;
    if (n_remote > 0 && (h_ins == nullptr || h_in_bytes == nullptr)) return CCCL_ERR_INVALID_ARG;
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_local) || !aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound(n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_local, 2 * n_elems) || !device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes))
        return CCCL_ERR_INVALID_ARG;
    cccl::ReduceInputs inputs{};
    inputs.local = d_local;
    for (int r = 0; r < n_remote; ++r) {
        if (!aligned16(h_ins[r]) || h_in_bytes[r] == 0 || !device_range(h_ins[r], h_in_bytes[r]))
            return CCCL_ERR_INVALID_ARG;
        inputs.in[r + 1] = static_cast<const uint8_t*>(h_ins[r]);
        inputs.in_bytes[r + 1] = h_in_bytes[r];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_reduce(inputs, n_remote + 1, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws, s) !=
        cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

size_t cccl_compress_bound_typed(int dtype, size_t n_elems) {
    const uint64_t b = elem_bytes(dtype);
    if (b == 0 || n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return 0;
    const uint64_t full = n_elems / kChunkElems, tail = n_elems % kChunkElems;
    uint64_t bytes = cccl::data_start(n_chunks_of(n_elems)) + full * (16 + b * kChunkElems);
    if (tail) bytes += 16 + cccl::pad16(b * tail);
    return (size_t)bytes;
}

cccl_status cccl_compress_typed(int dtype, const void* d_in, size_t n_elems, void* d_out, size_t out_capacity,
                                void* d_ws, size_t ws_bytes, int window, cccl_stream_t stream) {
    const uint64_t b = elem_bytes(dtype);
    if (b == 0 || n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_in) || !aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound_typed(dtype, n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_in, b * n_elems) || !device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_compress_typed((uint32_t)dtype, d_in, n_elems, static_cast<uint8_t*>(d_out), out_capacity, d_ws,
                                    s, window != 0) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_decompress_typed(int dtype, const void* d_in, size_t in_bytes, void* d_out, size_t n_elems,
                                  void* d_ws, size_t ws_bytes, cccl_stream_t stream) {
    const uint64_t b = elem_bytes(dtype);
    if (b == 0 || n_elems == 0 || n_elems > CCCL_MAX_ELEMS || in_bytes == 0) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_in) || !aligned16(d_out) || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < sizeof(cccl::WsHeader)) return CCCL_ERR_INVALID_ARG;
    if (!device_range(d_in, in_bytes) || !device_range(d_out, b * n_elems) || !device_range(d_ws, ws_bytes))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, sizeof(cccl::WsHeader), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_decompress_typed((uint32_t)dtype, static_cast<const uint8_t*>(d_in), in_bytes, d_out, n_elems,
                                      d_ws, s) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_reduce_typed(int dtype, int op, const void* d_local, const void* const* h_ins,
                              const size_t* h_in_bytes, int n_streams, size_t n_elems, void* d_out,
                              size_t out_capacity, void* d_ws, size_t ws_bytes, cccl_stream_t stream) {
    const uint64_t b = elem_bytes(dtype);
    if (b == 0 || (op != CCCL_OP_SUM && op != CCCL_OP_MIN && op != CCCL_OP_MAX)) return CCCL_ERR_INVALID_ARG;
    const int first = d_local != nullptr ? 1 : 0;
    const int R = n_streams + first;
    if (n_streams < 0 || R < 1 || R > cccl::kMaxRanks) return CCCL_ERR_INVALID_ARG;
    if (n_streams > 0 && (h_ins == nullptr || h_in_bytes == nullptr)) return CCCL_ERR_INVALID_ARG;
    if (n_elems == 0 || n_elems > CCCL_MAX_ELEMS) return CCCL_ERR_INVALID_ARG;
    if (!aligned16(d_out) || !aligned16(d_ws) || (d_local != nullptr && !aligned16(d_local)))
        return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < cccl_workspace_bytes(n_elems)) return CCCL_ERR_INVALID_ARG;
    if (out_capacity < cccl_compress_bound_typed(dtype, n_elems)) return CCCL_ERR_CAPACITY;
    if (!device_range(d_out, out_capacity) || !device_range(d_ws, ws_bytes)) return CCCL_ERR_INVALID_ARG;
    if (d_local != nullptr && !device_range(d_local, b * n_elems)) return CCCL_ERR_INVALID_ARG;
    cccl::ReduceInputs inputs{};
    inputs.op = (uint32_t)op;
    inputs.local = d_local;
    for (int r = 0; r < n_streams; ++r) {
        if (!aligned16(h_ins[r]) || h_in_bytes[r] == 0 || !device_range(h_ins[r], h_in_bytes[r]))
            return CCCL_ERR_INVALID_ARG;
        inputs.in[r + first] = static_cast<const uint8_t*>(h_ins[r]);
        inputs.in_bytes[r + first] = h_in_bytes[r];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, ws_used(n_elems), s) != CCCL_OK) return CCCL_ERR_CUDA;
    if (cccl::launch_reduce_typed((uint32_t)dtype, inputs, R, n_elems, static_cast<uint8_t*>(d_out), out_capacity,
                                  d_ws, s) != cudaSuccess)
        return CCCL_ERR_CUDA;
    return CCCL_OK;
}

cccl_status cccl_get_result(const void* d_ws, cccl_stream_t stream, uint64_t* out_bytes, cccl_status* dev_status) {
    if (d_ws == nullptr || !aligned16(d_ws)) return CCCL_ERR_INVALID_ARG;
    cccl::WsHeader h{};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, d_ws, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return CCCL_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CCCL_ERR_CUDA;
    if (out_bytes) *out_bytes = h.error ? 0 : h.total_bytes;
    if (dev_status) *dev_status = static_cast<cccl_status>(h.error);
    return CCCL_OK;
}

cccl_status cccl_selftest_timeouts(void* d_ws, size_t ws_bytes, cccl_stream_t stream) {
    const size_t need = cccl_workspace_bytes(8192);
    if (d_ws == nullptr || !aligned16(d_ws) || ws_bytes < need || !device_range(d_ws, need))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, need, s) != CCCL_OK) return CCCL_ERR_CUDA;
    cccl::selftest_timeouts_kernel<<<1, 64, 0, s>>>(static_cast<cccl::WsHeader*>(d_ws));
    return cudaGetLastError() == cudaSuccess ? CCCL_OK : CCCL_ERR_CUDA;
}

cccl_status cccl_selftest_lookback(const uint32_t* d_sizes, uint32_t n_units, uint32_t poison_unit, int concurrent,
                                   uint64_t* d_result, void* d_ws, size_t ws_bytes, cccl_stream_t stream) {
    if (n_units == 0 || n_units > CCCL_SELFTEST_MAX_UNITS) return CCCL_ERR_INVALID_ARG;
    const size_t need = sizeof(cccl::WsHeader) + 8 * (size_t)n_units;
    if (d_sizes == nullptr || d_result == nullptr || d_ws == nullptr || !aligned16(d_ws) ||
        (reinterpret_cast<uintptr_t>(d_sizes) & 3) != 0 || (reinterpret_cast<uintptr_t>(d_result) & 7) != 0)
        return CCCL_ERR_INVALID_ARG;
    if (ws_bytes < need || !device_range(d_ws, need) || !device_range(d_sizes, 4 * (size_t)n_units) ||
        !device_range(d_result, 8 * (size_t)n_units))
        return CCCL_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_ws(d_ws, need, s) != CCCL_OK) return CCCL_ERR_CUDA;
    auto* ws = static_cast<cccl::WsHeader*>(d_ws);
    auto* status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(d_ws) + sizeof(cccl::WsHeader));
    const uint64_t start = 4096;
    if (concurrent) {
        cccl::selftest_lookback_concurrent_kernel<<<4 * 152, 128, 0, s>>>(d_sizes, n_units, poison_unit, start, ws,
                                                                           status, d_result);
    } else {
        cccl::selftest_publish_kernel<<<(n_units + 255) / 256, 256, 0, s>>>(d_sizes, n_units, poison_unit, start,
                                                                            status);
        cccl::selftest_lookback_serial_kernel<<<1, 32, 0, s>>>(d_sizes, n_units, poison_unit, start, ws, status,
                                                               d_result);
    }
    return cudaGetLastError() == cudaSuccess ? CCCL_OK : CCCL_ERR_CUDA;
}

const char* cccl_status_string(cccl_status status) {
    switch (status) {
        case CCCL_OK: return "CCCL_OK";
        case CCCL_ERR_INVALID_ARG: return "CCCL_ERR_INVALID_ARG";
        case CCCL_ERR_CAPACITY: return "CCCL_ERR_CAPACITY";
        case CCCL_ERR_CORRUPT: return "CCCL_ERR_CORRUPT";
        case CCCL_ERR_TIMEOUT: return "CCCL_ERR_TIMEOUT";
        case CCCL_ERR_CUDA: return "CCCL_ERR_CUDA";
        case CCCL_ERR_UNIMPLEMENTED: return "CCCL_ERR_UNIMPLEMENTED";
    }
    return "CCCL_ERR_UNKNOWN";
}

}  // extern "C"

// cccl_launch.h -- launchers of the three kernels (host side, internal).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace cccl {

constexpr int kMaxRanks = 64;

// Rank r's operand: the compressed stream in[r] of in_bytes[r] bytes, except
// that rank 0 is the uncompressed buffer `local` (values of the reduce's
// element type) when it is not null (the selective-compression reduce).
struct ReduceInputs {
    const uint8_t* in[kMaxRanks];
    uint64_t in_bytes[kMaxRanks];
    const void* local;
    uint32_t op;  // 0 sum (binary32, one rounding), 1 min, 2 max (exact)
};

// All pointers are device pointers already validated by the C ABI layer; the
// workspace header and placement words have been cleared on `stream`.
// Paging (cccl_device.cuh): contiguous data when pg.table is null.
struct Paging;
// window: the window-base variant (stream version 2) instead of base = minimum.
cudaError_t launch_compress(const uint16_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                            cudaStream_t stream, const Paging& pg, bool window = false);
// The same compression with its scratch in a static device array (no
// workspace argument); n_elems <= CCCL_NOALLOC_MAX_ELEMS.
cudaError_t launch_compress_noalloc(const uint16_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                                    cudaStream_t stream);
cudaError_t launch_decompress(const uint8_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n_elems, void* ws,
                              cudaStream_t stream, const Paging& pg);
cudaError_t launch_reduce(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                          cudaStream_t stream);

// The same three operations for any element type (dtype: 1 bf16, 2 fp16,
// 3 fp32; values as their bit patterns), contiguous data only.
cudaError_t launch_compress_typed(uint32_t dtype, const void* in, uint64_t n_elems, uint8_t* out, uint64_t capacity,
                                  void* ws, cudaStream_t stream, bool window);
cudaError_t launch_decompress_typed(uint32_t dtype, const uint8_t* in, uint64_t in_bytes, void* out, uint64_t n_elems,
                                    void* ws, cudaStream_t stream);
cudaError_t launch_reduce_typed(uint32_t dtype, const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out,
                                uint64_t capacity, void* ws, cudaStream_t stream);

}  // namespace cccl

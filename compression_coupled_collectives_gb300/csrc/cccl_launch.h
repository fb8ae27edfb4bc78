// cccl_launch.h -- launchers of the three kernels (host side, internal).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace cccl {

// Runs a per-device set-up step (a kernel attribute, which belongs to the
// current device's context) the first time it is asked for on each device:
// run(dev, fn) calls fn() until it has succeeded once for `dev`, then returns
// cudaSuccess without calling it.  Devices 0..63 are remembered; for others
// fn() runs every time.  Concurrent first calls may both run fn(), which is
// harmless for an attribute.
class PerDeviceOnce {
  public:
    template <typename Fn>
    cudaError_t run(int dev, Fn fn) {
        const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
        if (bit != 0 && (done_.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
        const cudaError_t e = fn();
        if (e == cudaSuccess && bit != 0) done_.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }

  private:
    std::atomic<uint64_t> done_{0};
};

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

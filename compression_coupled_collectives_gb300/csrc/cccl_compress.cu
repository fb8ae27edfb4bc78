// cccl_compress.cu -- the compress kernel: one CTA per 4096-element chunk,
// load -> split -> exponent table -> place by decoupled look-back -> write
// ("CCCL: In-GPU Compression-Coupled Collective Communication", sections
// 4.1, 4.3, 4.4; section 5 for the raw partial chunk).
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

__device__ __forceinline__ void load_full_chunk(const uint16_t* in, uint64_t c, uint32_t P[16]) {
    const uint32_t lane = threadIdx.x & 31, q = threadIdx.x >> 5;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(in + c * kChunkElems);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const uint4 v = ld_stream_v4(src + 512 * (4 * q + jj) + 16 * lane);
        P[4 * jj] = v.x;
        P[4 * jj + 1] = v.y;
        P[4 * jj + 2] = v.z;
        P[4 * jj + 3] = v.w;
    }
}

__global__ void __launch_bounds__(kThreads) compress_kernel(const uint16_t* __restrict__ in, StreamOut so) {
    __shared__ EncodeSmem sm;
    __shared__ uint32_t s_ticket;
    const uint64_t n_full = so.n_elems / kChunkElems;

    // Chunks are processed in ticket order (the look-back's forward-progress
    // guarantee).  Tickets normally follow blockIdx, so the load of chunk
    // blockIdx.x starts before the ticket arrives and is redone otherwise.
    uint32_t P[16];
    const uint64_t guess = blockIdx.x;
    if (guess < n_full) load_full_chunk(in, guess, P);
    if (threadIdx.x == 0) s_ticket = atomicAdd(&so.ws->ticket, 1u);
    __syncthreads();
    const uint64_t c = s_ticket;
    if (c < n_full) {
        if (c != guess) load_full_chunk(in, c, P);
        encode_full_chunk(P, c, so, sm);
        return;
    }
    // partial last chunk
    const uint32_t n_c = (uint32_t)(so.n_elems - c * kChunkElems);
    const uint16_t* src = in + c * kChunkElems;
    const uint32_t lane = threadIdx.x & 31, q = threadIdx.x >> 5;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t i = 256 * (4 * q + jj) + 8 * lane + 2 * w;
            const uint32_t lo = i < n_c ? src[i] : 0u, hi = i + 1 < n_c ? src[i + 1] : 0u;
            P[4 * jj + w] = lo | (hi << 16);
        }
    }
    encode_tail_chunk(P, c, n_c, so, sm);
}

cudaError_t launch_compress(const uint16_t* in, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                            cudaStream_t stream) {
    StreamOut so;
    so.out = out;
    so.capacity = capacity;
    so.ws = static_cast<WsHeader*>(ws);
    so.status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    so.n_elems = n_elems;
    so.n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    compress_kernel<<<(unsigned)so.n_chunks, kThreads, 0, stream>>>(in, so);
    return cudaGetLastError();
}

}  // namespace cccl

// cccl_decompress.cu -- the decompress kernel: one CTA per chunk; the chunk
// is staged in shared memory by one bulk (TMA) copy, then each thread
// rebuilds its 32 values ("CCCL: In-GPU Compression-Coupled Collective
// Communication", section 4.1 inverted; the "Decomp." stage of Figure 2).
#include "cccl_decode.cuh"
#include "cccl_launch.h"

namespace cccl {

__global__ void __launch_bounds__(kThreads)
    decompress_kernel(const uint8_t* __restrict__ s, uint64_t in_bytes, uint16_t* __restrict__ out, uint64_t n_elems,
                      uint64_t n_chunks, WsHeader* ws) {
    __shared__ __align__(128) uint8_t buf[kMaxChunkBytes];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_bytes, s_ok;
    __shared__ uint32_t row_tot[16];
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;
    const uint64_t c = blockIdx.x;
    const uint64_t left = n_elems - c * kChunkElems;
    const uint32_t n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;

    if (t == 0) {
        const ChunkView v = locate_chunk(s, in_bytes, n_elems, n_chunks, c);
        s_ok = v.ok;
        s_bytes = v.bytes;
        if (v.ok) {
            mbar_init(&bar, 1);
            fence_mbar_init();
            bulk_load(buf, s + v.offset, v.bytes, &bar);
        }
    }
    __syncthreads();
    if (!s_ok) {
        if (t == 0) record_error(ws, kStatusCorrupt);
        return;
    }
    const bool arrived = mbar_wait(&bar, 0);
    if (__syncthreads_or(!arrived)) {
        if (t == 0) record_error(ws, kStatusTimeout);
        return;
    }
    const ChunkHeader h = read_chunk_header(buf);
    if (!chunk_header_valid(h, s_bytes, n_c)) {
        if (t == 0) record_error(ws, kStatusCorrupt);
        return;
    }
    uint16_t* dst = out + c * kChunkElems;
    if (n_c < kChunkElems) {  // partial last chunk: raw by construction
        const uint16_t* vals = reinterpret_cast<const uint16_t*>(buf + kChunkHeaderBytes);
        for (uint32_t i = t; i < n_c; i += kThreads) dst[i] = vals[i];
        return;
    }
    uint32_t P[16];
    bool special = false;
    if (!decode_full_chunk(CtaBarrier{}, buf, h, P, row_tot, special)) {
        if (t == 0) record_error(ws, kStatusCorrupt);
        return;
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
        *reinterpret_cast<uint4*>(dst + 256 * (4 * q + jj) + 8 * lane) =
            make_uint4(P[4 * jj], P[4 * jj + 1], P[4 * jj + 2], P[4 * jj + 3]);
}

cudaError_t launch_decompress(const uint8_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n_elems, void* ws,
                              cudaStream_t stream) {
    const uint64_t n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    decompress_kernel<<<(unsigned)n_chunks, kThreads, 0, stream>>>(in, in_bytes, out, n_elems, n_chunks,
                                                                   static_cast<WsHeader*>(ws));
    return cudaGetLastError();
}

}  // namespace cccl

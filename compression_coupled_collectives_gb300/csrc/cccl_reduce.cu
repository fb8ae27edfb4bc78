// cccl_reduce.cu -- the fused reduce kernel: the reduce step of a compressed
// allreduce as one pass, decompress -> binary32 accumulate in rank order ->
// one rounding to bf16 -> compress ("CCCL: In-GPU Compression-Coupled
// Collective Communication", section 5, CopyReducePacks; Figure 2).
//
// One CTA per output chunk.  Chunk c of every rank is staged in shared
// memory by bulk (TMA) copies through a ring of kStages buffers, so the next
// ranks' chunks are in flight while the current one is decoded; the 32
// running sums of each thread stay in registers as binary32 pairs.
#include "cccl_decode.cuh"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kStages = 4;
constexpr size_t kReduceSmemBytes = (size_t)kStages * kMaxChunkBytes;

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
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
// bf16 pair -> binary32 pair (exact)
__device__ __forceinline__ uint64_t widen_pair(uint32_t p) {
    return (uint64_t)(p << 16) | ((uint64_t)(p & 0xFFFF0000u) << 32);
}

__global__ void __launch_bounds__(kThreads) reduce_kernel(ReduceInputs inputs, int R, StreamOut so) {
    extern __shared__ __align__(128) uint8_t stage[];
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ uint64_t s_off[kMaxRanks];
    __shared__ uint32_t s_bytes[kMaxRanks];
    __shared__ EncodeSmem sm;
    __shared__ uint32_t s_ticket;
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;

    if (t == 0) s_ticket = atomicAdd(&so.ws->ticket, 1u);
    bool ok = true;
    __syncthreads();
    const uint64_t c = s_ticket;
    const uint64_t left = so.n_elems - c * kChunkElems;
    const uint32_t n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;
    if ((int)t < R) {
        const ChunkView v = locate_chunk(inputs.in[t], inputs.in_bytes[t], so.n_elems, so.n_chunks, c);
        s_off[t] = v.offset;
        s_bytes[t] = v.bytes;
        ok = v.ok != 0;
    }
    if (t == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    if (!__syncthreads_and(ok)) {
        if (t == 0) {
            record_error(so.ws, kStatusCorrupt);
            st_relaxed_u64(&so.status[c], kFlagPoison);
        }
        return;
    }
    if (t == 0)
        for (int r = 0; r < min(R, kStages); ++r)
            bulk_load(stage + (size_t)r * kMaxChunkBytes, inputs.in[r] + s_off[r], s_bytes[r], &bars[r]);

    uint64_t acc[16];
    bool special = false;
    uint32_t fail = 0;  // 0, or the device status that stops this CTA
    int r = 0;
    for (; r < R; ++r) {
        const int st = r % kStages;
        uint8_t* buf = stage + (size_t)st * kMaxChunkBytes;
        const bool arrived = mbar_wait(&bars[st], (uint32_t)(r / kStages) & 1u);
        if (__syncthreads_or(!arrived)) {
            fail = kStatusTimeout;
            break;
        }
        const ChunkHeader h = read_chunk_header(buf);
        bool good = chunk_header_valid(h, s_bytes[r], n_c);
        uint32_t P[16];
        if (good) {
            if (n_c < kChunkElems) {  // partial last chunk: raw values, read those that exist
                const uint16_t* vals = reinterpret_cast<const uint16_t*>(buf + kChunkHeaderBytes);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t i = 256 * (4 * q + jj) + 8 * lane + 2 * w;
                        const uint32_t lo = i < n_c ? vals[i] : 0u, hi = i + 1 < n_c ? vals[i + 1] : 0u;
                        P[4 * jj + w] = lo | (hi << 16);
                    }
                special = true;
            } else {
                bool sp = false;
                good = decode_full_chunk(buf, h, P, sm.row_tot, sp);
                special = special || sp;
            }
        }
        if (!good) {  // CTA-uniform
            fail = kStatusCorrupt;
            break;
        }
        if (r == 0) {
#pragma unroll
            for (int w = 0; w < 16; ++w) acc[w] = widen_pair(P[w]);
        } else {
#pragma unroll
            for (int w = 0; w < 16; ++w) acc[w] = add_f32x2(acc[w], widen_pair(P[w]));
        }
        __syncthreads();  // every thread is done with this stage
        if (t == 0 && r + kStages < R) {
            fence_proxy_async_smem();
            bulk_load(buf, inputs.in[r + kStages] + s_off[r + kStages], s_bytes[r + kStages], &bars[st]);
        }
    }
    if (fail) {
        if (t == 0) {
            record_error(so.ws, fail);
            // copies for the next ranks (and rank r itself after a timeout) may
            // still be landing in the ring: wait for them (bounded) before the
            // CTA gives its shared memory back
            for (int rr = (fail == kStatusTimeout ? r : r + 1); rr < min(R, r + kStages); ++rr)
                mbar_wait(&bars[rr % kStages], (uint32_t)(rr / kStages) & 1u);
            st_relaxed_u64(&so.status[c], kFlagPoison);
        }
        return;
    }

    uint32_t P[16];
#pragma unroll
    for (int w = 0; w < 16; ++w) P[w] = round_pair_bf16(acc[w]);
    if (__syncthreads_or(special)) {
#pragma unroll
        for (int w = 0; w < 16; ++w) P[w] = canonical_nan_pair(P[w]);
    }
    if (n_c < kChunkElems)
        encode_tail_chunk(P, c, n_c, so, sm);
    else
        encode_full_chunk(P, c, so, sm);
}

cudaError_t launch_reduce(const ReduceInputs& inputs, int R, uint64_t n_elems, uint8_t* out, uint64_t capacity, void* ws,
                          cudaStream_t stream) {
    static_assert(kReduceSmemBytes <= 48 * 1024, "stage ring must fit the default dynamic shared memory");
    StreamOut so;
    so.out = out;
    so.capacity = capacity;
    so.ws = static_cast<WsHeader*>(ws);
    so.status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    so.n_elems = n_elems;
    so.n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    reduce_kernel<<<(unsigned)so.n_chunks, kThreads, kReduceSmemBytes, stream>>>(inputs, R, so);
    return cudaGetLastError();
}

}  // namespace cccl

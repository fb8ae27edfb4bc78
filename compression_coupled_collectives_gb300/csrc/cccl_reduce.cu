// cccl_reduce.cu -- the fused reduce kernel: the reduce step of a compressed
// allreduce as one pass, decompress -> binary32 accumulate in rank order ->
// one rounding to bf16 -> compress ("CCCL: In-GPU Compression-Coupled
// Collective Communication", section 5, CopyReducePacks; Figure 2).
//
// One CTA of kRGroup warps per group of kRGroup consecutive output chunks.
// For each output chunk, chunk c of every rank streams through a ring of
// kStages shared-memory buffers filled by bulk (TMA) copies, so later ranks'
// (and later chunks') data are in flight while the current one is decoded;
// the 4 warps decode it together (32 values per thread) and keep 32 running
// binary32 sums per thread in registers.  The rounded bf16 chunk is parked in
// shared memory; once the group is reduced, each warp sizes and writes one
// chunk exactly as the compress kernel does, after one look-back per group.
#include <mutex>

#include "cccl_decode.cuh"
#include "cccl_encode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kRGroup = 4;
constexpr int kStages = 4;
constexpr size_t kParkBytes = (size_t)kRGroup * 2 * kChunkElems;
constexpr size_t kReduceSmemBytes = kParkBytes + (size_t)kStages * kMaxChunkBytes;

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
__global__ void __launch_bounds__(32 * kRGroup, 3) reduce_kernel(ReduceInputs inputs, int R, StreamOut so) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* park = smem;                // kRGroup rounded bf16 chunks
    uint8_t* ring = smem + kParkBytes;   // kStages staged rank chunks
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ uint64_t s_in_off[kRGroup][kMaxRanks];
    __shared__ uint32_t s_in_bytes[kRGroup][kMaxRanks];
    __shared__ uint32_t s_row_tot[16];
    __shared__ uint32_t s_bytes[kRGroup];
    __shared__ uint64_t s_offset[kRGroup];
    __shared__ uint64_t s_group;
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;

    if (t == 0) s_group = atomicAdd(&so.ws->ticket, 1u);
    __syncthreads();
    const uint64_t g = s_group;
    const uint64_t c0 = g * kRGroup;
    const int n_out = (int)min((uint64_t)kRGroup, so.n_chunks - c0);  // output chunks of this group

    // locate chunk c0 + i of every rank through its offset table
    bool ok = true;
    for (int idx = (int)t; idx < n_out * R; idx += 32 * kRGroup) {
        const int i = idx / R, r = idx % R;
        const ChunkView v = locate_chunk(inputs.in[r], inputs.in_bytes[r], so.n_elems, so.n_chunks, c0 + i);
        s_in_off[i][r] = v.offset;
        s_in_bytes[i][r] = v.bytes;
        ok = ok && v.ok;
    }
    if (t == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    if (!__syncthreads_and(ok)) {
        if (t == 0) {
            record_error(so.ws, kStatusCorrupt);
            st_relaxed_u64(&so.status[g], kFlagPoison);
        }
        return;
    }
    // the copy sequence: u = i * R + r for output chunk i, rank r
    const int U = n_out * R;
    if (t == 0)
        for (int u = 0; u < min(U, kStages); ++u)
            bulk_load(ring + (size_t)u * kMaxChunkBytes, inputs.in[u % R] + s_in_off[u / R][u % R],
                      s_in_bytes[u / R][u % R], &bars[u]);

    uint32_t fail = 0;  // 0, or the device status that stops this CTA
    int u = 0;
    for (int i = 0; i < n_out && !fail; ++i) {
        const uint64_t c = c0 + i;
        const uint64_t left = so.n_elems - c * kChunkElems;
        const uint32_t n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;
        uint64_t acc[16];
        bool special = false;
        for (int r = 0; r < R; ++r, ++u) {
            const int st = u % kStages;
            uint8_t* buf = ring + (size_t)st * kMaxChunkBytes;
            const bool arrived = mbar_wait(&bars[st], (uint32_t)(u / kStages) & 1u);
            if (__syncthreads_or(!arrived)) {
                fail = kStatusTimeout;
                break;
            }
            const ChunkHeader h = read_chunk_header(buf);
            bool good = chunk_header_valid(h, s_in_bytes[i][r], n_c);
            uint32_t P[16];
            if (good) {
                if (n_c < kChunkElems) {  // partial last chunk: raw values, read those that exist
                    const uint16_t* vals = reinterpret_cast<const uint16_t*>(buf + kChunkHeaderBytes);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const uint32_t e = 256 * (4 * q + jj) + 8 * lane + 2 * w;
                            const uint32_t lo = e < n_c ? vals[e] : 0u, hi = e + 1 < n_c ? vals[e + 1] : 0u;
                            P[4 * jj + w] = lo | (hi << 16);
                        }
                    special = true;
                } else {
                    bool sp = false;
                    good = decode_full_chunk(buf, h, P, s_row_tot, sp);
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
            if (t == 0 && u + kStages < U) {
                const int un = u + kStages;
                fence_proxy_async_smem();
                bulk_load(buf, inputs.in[un % R] + s_in_off[un / R][un % R], s_in_bytes[un / R][un % R], &bars[st]);
            }
        }
        if (fail) break;
        uint32_t P[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) P[w] = round_pair_bf16(acc[w]);
        if (__syncthreads_or(special)) {
#pragma unroll
            for (int w = 0; w < 16; ++w) P[w] = canonical_nan_pair(P[w]);
        }
        uint8_t* dst = park + (size_t)i * 2 * kChunkElems;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<uint4*>(dst + 512 * (4 * q + jj) + 16 * lane) =
                make_uint4(P[4 * jj], P[4 * jj + 1], P[4 * jj + 2], P[4 * jj + 3]);
    }
    if (fail) {
        if (t == 0) {
            record_error(so.ws, fail);
            // copies still landing in the ring (and copy u itself after a
            // timeout): wait for them, bounded, before the CTA gives its
            // shared memory back
            for (int uu = (fail == kStatusTimeout ? u : u + 1); uu < min(U, u + kStages); ++uu)
                mbar_wait(&bars[uu % kStages], (uint32_t)(uu / kStages) & 1u);
            st_relaxed_u64(&so.status[g], kFlagPoison);
        }
        return;
    }
    // the parked chunks were written by generic stores and a raw chunk leaves
    // by a bulk copy: order them for the async proxy, then for every warp
    fence_proxy_async_smem();
    __syncthreads();

    // encode: warp w sizes and writes output chunk c0 + w
    const uint64_t c = c0 + q;
    uint8_t* chunk = park + (size_t)q * 2 * kChunkElems;
    const uint64_t n_full = so.n_elems / kChunkElems;
    ChunkPlan pl{};
    ChunkRegs regs;
    uint32_t bytes = 0;
    if (c < n_full) {
        pl = plan_chunk_warp(chunk, regs);
        bytes = pl.bytes;
    } else if (c < so.n_chunks) {
        bytes = tail_chunk_bytes((uint32_t)(so.n_elems - c * kChunkElems));
    }
    if (lane == 0) s_bytes[q] = bytes;
    const uint64_t off = place_group<kRGroup>(so, g, s_bytes, s_offset, false);
    if (off == kFlagPoison || bytes == 0) return;
    if (off + bytes > so.capacity) {
        if (lane == 0) record_error(so.ws, kStatusCorrupt);
        return;
    }
    uint8_t* dst = so.out + off;
    if (c < n_full) {
        write_chunk_warp(regs, pl, chunk, dst);
    } else {
        const uint16_t* vals = reinterpret_cast<const uint16_t*>(chunk);
        write_tail_chunk_warp([vals](uint32_t e) { return vals[e]; }, (uint32_t)(so.n_elems - c * kChunkElems), dst);
    }
    if (lane == 0) finish_chunk(so, c, off, bytes);
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
    StreamOut so;
    so.out = out;
    so.capacity = capacity;
    so.ws = static_cast<WsHeader*>(ws);
    so.status = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    so.n_elems = n_elems;
    so.n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    const uint64_t n_groups = (so.n_chunks + kRGroup - 1) / kRGroup;
    reduce_kernel<<<(unsigned)n_groups, 32 * kRGroup, kReduceSmemBytes, stream>>>(inputs, R, so);
    return cudaGetLastError();
}

}  // namespace cccl

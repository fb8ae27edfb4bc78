// cccl_decompress.cu -- the decompress kernel ("CCCL: In-GPU
// Compression-Coupled Collective Communication", section 4.1 inverted; the
// "Decomp." stage of Figure 2).
//
// Persistent: several CTAs per SM, each taking every gridDim-th chunk.  A CTA
// has a producer warp, which locates its chunks through the offset table (32
// at a time, one per lane) and stages them by bulk (TMA) copies in a small
// ring of buffers, and a team of 4 decode warps, which rebuild 32 values per
// thread from each staged chunk and store them with 16-byte writes.  So the
// location and the copy of later chunks overlap the decoding of the current
// one.  One kernel per element type.
#include "cccl_decode.cuh"
#include "cccl_launch.h"

namespace cccl {

constexpr int kDTeamThreads = 128;
constexpr int kDProducerWarp = 4;
constexpr int kDThreads = kDTeamThreads + 32;
// staged chunks per CTA and CTAs per SM: three 8.2 KB slots for the 16-bit
// types, two 16.4 KB slots for fp32; 8 CTAs per SM for bf16, 7 for fp16 (its
// decode holds 8 more words), 6 for fp32 (registers and shared memory)
template <class D>
__host__ __device__ constexpr int dslots() { return D::kElemBytes == 4 ? 2 : 3; }
template <class D>
__host__ __device__ constexpr int dctas_per_sm() { return D::kElemBytes == 4 ? 6 : (D::kExpBits == 5 ? 7 : 8); }

constexpr int kMaxDSlots = 3;
struct DecompressSmem {
    uint64_t full[kMaxDSlots];   // the slot's chunk landed, or its meta says there is none
    uint64_t free_[kMaxDSlots];  // the team is done with the slot (1 arrival)
    uint32_t bytes[kMaxDSlots];  // staged chunk size
    uint32_t ok[kMaxDSlots];     // the chunk was located
    uint32_t row_tot[4];
    volatile uint32_t abort;
};

template <class D>
__global__ void __launch_bounds__(kDThreads, dctas_per_sm<D>())
    decompress_kernel(const uint8_t* __restrict__ s, uint64_t in_bytes, uint8_t* __restrict__ out, Paging pg,
                      uint64_t n_elems, uint64_t n_chunks, WsHeader* ws) {
    constexpr int kDSlots = dslots<D>();
    static_assert(kDSlots <= kMaxDSlots, "DecompressSmem holds kMaxDSlots slots");
    using Elem = typename std::conditional<D::kElemBytes == 4, uint32_t, uint16_t>::type;
    __shared__ __align__(128) uint8_t ring[kDSlots][max_chunk_bytes<D>()];
    __shared__ DecompressSmem sm;
    const uint32_t t = threadIdx.x, lane = t & 31, q = t >> 5;
    if (t == 0) {
        for (int i = 0; i < kDSlots; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.free_[i], 1);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t stride = gridDim.x;

    if (q == kDProducerWarp) {
        // ------------------------------------------------------------ producer
        // The stream header is checked once; this CTA's chunks are located 32
        // at a time, one per lane, so a copy waits only for its slot.
        const uint64_t total = stream_total<D>(s, in_bytes, n_elems, n_chunks);
        uint32_t i = 0;
        bool stop = false;
        for (uint64_t c0 = blockIdx.x; c0 < n_chunks && !stop; c0 += 32 * stride) {
            const uint64_t mine = c0 + lane * stride;
            ChunkView v{0, 0, 0};
            if (mine < n_chunks && total != 0) v = locate_chunk_at<D>(s, total, n_chunks, mine);
            const uint64_t here = (n_chunks - c0 + stride - 1) / stride;
            const uint32_t n_here = here < 32 ? (uint32_t)here : 32u;
            for (uint32_t j = 0; j < n_here; ++j, ++i) {
                const uint32_t slot = i % kDSlots;
                if (i >= (uint32_t)kDSlots &&
                    !__all_sync(0xFFFFFFFFu, mbar_wait(&sm.free_[slot], (i / kDSlots - 1) & 1u))) {
                    if (lane == 0) {
                        record_error(ws, kStatusTimeout);
                        sm.abort = 1;
                    }
                    stop = true;
                    break;
                }
                if (__any_sync(0xFFFFFFFFu, sm.abort != 0)) {
                    stop = true;
                    break;
                }
                const uint64_t off = __shfl_sync(0xFFFFFFFFu, v.offset, j);
                const uint32_t bytes = __shfl_sync(0xFFFFFFFFu, v.bytes, j);
                const uint32_t ok = __shfl_sync(0xFFFFFFFFu, v.ok, j);
                if (lane == 0) {
                    sm.ok[slot] = ok;
                    sm.bytes[slot] = bytes;
                    if (ok) {
                        fence_proxy_async_smem();
                        bulk_load(ring[slot], s + off, bytes, &sm.full[slot]);
                    } else {
                        mbar_arrive(&sm.full[slot]);  // nothing to stage; the team reports it
                    }
                }
                __syncwarp();
            }
        }
        // no copy may still be landing when the CTA exits
        for (uint32_t v = i > (uint32_t)kDSlots ? i - kDSlots : 0u; v < i; ++v)
            mbar_wait(&sm.full[v % kDSlots], (v / kDSlots) & 1u);
        return;
    }

    // ---------------------------------------------------------------- decode team
    const TeamBarrier bar{1u};
    uint32_t i = 0;
    for (uint64_t c = blockIdx.x; c < n_chunks; c += stride, ++i) {
        const uint32_t slot = i % kDSlots;
        uint8_t* buf = ring[slot];
        const bool landed = !sm.abort && mbar_wait(&sm.full[slot], (i / kDSlots) & 1u);
        // one meeting per chunk: it has landed for every warp, and every warp
        // is done with the previous chunk's slot and row_tot
        if (bar.any(!landed)) {
            if (t == 0) {
                record_error(ws, kStatusTimeout);
                sm.abort = 1;
            }
            return;  // the whole team
        }
        if (i > 0 && t == 32) mbar_arrive(&sm.free_[(i - 1) % kDSlots]);
        const uint64_t left = n_elems - c * kChunkElems;
        const uint32_t n_c = left < kChunkElems ? (uint32_t)left : kChunkElems;
        const uint64_t e = chunk_elem_offset(pg, c);
        Elem* dst = reinterpret_cast<Elem*>(out) + e;
        if (e == kBadChunk && t == 0) record_error(ws, kStatusInvalidArg);  // a block outside the pool
        bool good = sm.ok[slot] != 0 && e != kBadChunk;
        ChunkHeader h{};
        if (good) {
            h = read_chunk_header(buf);
            good = chunk_header_valid<D>(h, sm.bytes[slot], n_c);  // the same verdict for every thread
        }
        if (good) {
            if (n_c < kChunkElems) {  // partial last chunk: raw by construction
                const Elem* vals = reinterpret_cast<const Elem*>(buf + kChunkHeaderBytes);
                for (uint32_t x = t; x < n_c; x += kDTeamThreads) dst[x] = vals[x];
            } else {
                uint32_t P[thread_words<D>()];
                bool special = false;
                good = decode_full_chunk<D>(bar, buf, h, P, sm.row_tot, special);
                if (good) {
                    if constexpr (D::kElemBytes == 4) {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            uint4* row = reinterpret_cast<uint4*>(dst + 256 * (4 * q + jj) + 8 * lane);
                            row[0] = make_uint4(P[8 * jj], P[8 * jj + 1], P[8 * jj + 2], P[8 * jj + 3]);
                            row[1] = make_uint4(P[8 * jj + 4], P[8 * jj + 5], P[8 * jj + 6], P[8 * jj + 7]);
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            *reinterpret_cast<uint4*>(dst + 256 * (4 * q + jj) + 8 * lane) =
                                make_uint4(P[4 * jj], P[4 * jj + 1], P[4 * jj + 2], P[4 * jj + 3]);
                    }
                }
            }
        }
        if (!good && e != kBadChunk && t == 0) record_error(ws, kStatusCorrupt);
    }
}

template <class D>
cudaError_t launch_decompress_t(const uint8_t* in, uint64_t in_bytes, void* out, uint64_t n_elems, void* ws,
                                cudaStream_t stream, const Paging& pg) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const uint64_t n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
    const uint64_t slots = (uint64_t)sms * dctas_per_sm<D>();
    const unsigned grid = (unsigned)(n_chunks < slots ? n_chunks : slots);
    decompress_kernel<D><<<grid, kDThreads, 0, stream>>>(in, in_bytes, static_cast<uint8_t*>(out), pg, n_elems,
                                                         n_chunks, static_cast<WsHeader*>(ws));
    return cudaGetLastError();
}

cudaError_t launch_decompress(const uint8_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n_elems, void* ws,
                              cudaStream_t stream, const Paging& pg) {
    return launch_decompress_t<Bf16>(in, in_bytes, out, n_elems, ws, stream, pg);
}

cudaError_t launch_decompress_typed(uint32_t dtype, const uint8_t* in, uint64_t in_bytes, void* out, uint64_t n_elems,
                                    void* ws, cudaStream_t stream) {
    const Paging pg{nullptr, 1, 0};
    if (dtype == Fp16::kCode) return launch_decompress_t<Fp16>(in, in_bytes, out, n_elems, ws, stream, pg);
    if (dtype == Fp32::kCode) return launch_decompress_t<Fp32>(in, in_bytes, out, n_elems, ws, stream, pg);
    return launch_decompress_t<Bf16>(in, in_bytes, out, n_elems, ws, stream, pg);
}

}  // namespace cccl

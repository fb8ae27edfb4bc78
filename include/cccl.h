/*
 * cccl.h -- C ABI of libcccl: lossless compression of bf16 (and fp16, fp32)
 * communication buffers and the compressed reduce step of an allreduce, on
 * one GPU.
 *
 * Method: "CCCL: In-GPU Compression-Coupled Collective Communication"
 * (arXiv 2604.17172).
 *   - section 4.1, "Compression Principle": a bf16 value splits into sign,
 *     exponent and fraction; sign and fraction travel raw and only the
 *     skewed 8-bit exponent is re-encoded;
 *   - section 4.3, "Localized Frequency Tables": each block builds its own
 *     exponent table from its own data and gives every exponent symbol a
 *     fixed-length bit code;
 *   - section 4.4, "Reducing Global Memory Access": each block writes its
 *     compressed output straight into its final place in one preallocated
 *     buffer (one global-memory round, no coalescing pass);
 *   - section 5, "Handling data alignment": data that does not fill a
 *     whole chunk travels uncompressed;
 *   - section 5 (CopyReducePacks) and Figure 2: the reduce step of an
 *     allreduce is receive -> decompress -> reduce -> compress -> send.
 *
 * The pages fix no bitstream; this library's stream (little endian):
 *   64-byte header  magic "CCB1" (u32 0x31424343), version u16 = 1,
 *                   dtype u16 = 1 (bf16), chunk_elems u32 = 4096, u32 0,
 *                   n_elems u64, n_chunks u64, total_bytes u64, 24 zero bytes
 *   offset table    n_chunks x u64 absolute byte offsets, zero-padded to 16
 *   chunks          contiguous in chunk order, each a multiple of 16 bytes:
 *     16-byte header  mode u8 (0 packed, 1 raw), k u8, base u8, u8 0,
 *                     n_c u16, n_esc u16, chunk_bytes u32, u32 0
 *     packed body     4096 sign+fraction bytes, k bit-planes of 512 bytes,
 *                     n_esc escape bytes, zero padding to 16
 *     raw body        n_c bf16 values, zero padding to 16
 *   Bit-plane p (p = 0 the code's least significant bit) is 128 u32 words;
 *   element i = 256 j + 8 l + s (j < 16, l < 32, s < 8) keeps its bit in
 *   word 32 (j / 4) + l, bit 8 (s % 4) + 2 (j % 4) + s / 4.  The escape bytes
 *   follow bit-plane order: by word, then by bit.
 *   A full chunk is packed with width k (offsets e - base below 2^k - 1 are
 *   codes, the rest escape with their raw exponent) when that is smaller
 *   than its raw form; the last chunk, when shorter than 4096 elements, is
 *   raw.  Exactly one stream is valid for each input.
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer.  The library allocates nothing per call.
 *     Between calls it keeps only cccl_compress_noalloc's static scratch and,
 *     per device, a record that each kernel's shared-memory limit was set.
 *     Calls with distinct workspaces may run concurrently.
 *   - d_* pointers are device pointers (cudaMalloc'd or managed), 16-byte
 *     aligned.  h_* pointers are host pointers.  Each device buffer, with the
 *     size passed for it, must lie inside one device allocation; a range that
 *     does not is refused with CCCL_ERR_INVALID_ARG before anything is
 *     enqueued.  (The check sees allocations, not sub-allocations: a size
 *     that overruns a tensor but stays inside its allocator's segment is the
 *     caller's error and is not detected.)
 *   - Work is enqueued on `stream` (NULL: the legacy default stream) and
 *     runs asynchronously.  Argument errors are detected on the host before
 *     anything is enqueued and return immediately.  Errors found on the
 *     device (corrupt input, a wait that ran out) and the compressed size
 *     land in the workspace; read them with cccl_get_result.
 *   - n_elems counts values: bf16 values (passed as their uint16 bit
 *     patterns), except in the typed entry points below.
 */
#ifndef CCCL_H
#define CCCL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream).  NULL: the legacy default stream. */
typedef struct CUstream_st *cccl_stream_t;

typedef enum {
    CCCL_OK = 0,
    CCCL_ERR_INVALID_ARG = 1,   /* bad pointer, alignment, size or count */
    CCCL_ERR_CAPACITY = 2,      /* output capacity below cccl_compress_bound */
    CCCL_ERR_CORRUPT = 3,       /* input stream malformed or not for n_elems */
    CCCL_ERR_TIMEOUT = 4,       /* a bounded device wait ran out */
    CCCL_ERR_CUDA = 5,          /* a CUDA call failed (launch, memset, copy) */
    CCCL_ERR_UNIMPLEMENTED = 6
} cccl_status;

/* Largest number of elements one call accepts (2^40). */
#define CCCL_MAX_ELEMS ((size_t)1 << 40)

/* Worst-case stream size for n_elems values (every chunk raw):
 * 64 + pad16(8 * n_chunks) + sum over chunks of 16 + pad16(2 * n_c).
 * Returns 0 when n_elems is 0 or above CCCL_MAX_ELEMS. */
size_t cccl_compress_bound(size_t n_elems);

/* Workspace bytes for a call on n_elems values: a 16-byte status header
 * (chunk ticket u32, device error u32, stream size u64) plus one u64
 * placement word per chunk.  Returns 0 when n_elems is 0 or too large. */
size_t cccl_workspace_bytes(size_t n_elems);

/* Compress n_elems bf16 values (sections 4.1, 4.3, 4.4; section 5 for the
 * partial last chunk).
 *   d_in          n_elems uint16 bf16 bit patterns, read only.
 *   d_out         receives the stream; out_capacity must be at least
 *                 cccl_compress_bound(n_elems).  Bytes past the stream's
 *                 total size are left untouched.
 *   d_ws          ws_bytes >= cccl_workspace_bytes(n_elems); overwritten.
 * The stream size (the header's total_bytes) is readable with
 * cccl_get_result once the work is done.
 * Returns INVALID_ARG (null or misaligned pointer, n_elems 0 or above the
 * limit, small workspace), CAPACITY, CUDA, or OK. */
cccl_status cccl_compress(const uint16_t *d_in, size_t n_elems, void *d_out, size_t out_capacity, void *d_ws,
                          size_t ws_bytes, cccl_stream_t stream);

/* The window-base variant of cccl_compress: the same stream layout with
 * version 2 in its header.  For every code width k the chunk's base is the
 * start of the window of 2^k - 1 exponents that leaves the fewest escapes
 * (every exponent outside the window, below it included, is an escape; ties
 * to the smaller base), instead of the minimum exponent; then the smallest
 * size wins as in cccl_compress (ties to the smaller k, raw when not smaller
 * than 4096 bytes of exponents).  Section 4.3's per-block frequency table
 * taken at its word: the codes go to the most frequent run of exponent
 * symbols, so rare low outliers (zeros, subnormals) become escapes instead
 * of stretching the range.  Never larger than cccl_compress's stream, chunk
 * by chunk.  Arguments and errors as for cccl_compress; cccl_decompress,
 * cccl_reduce_compressed and cccl_reduce_mixed read both versions. */
cccl_status cccl_compress_window(const uint16_t *d_in, size_t n_elems, void *d_out, size_t out_capacity, void *d_ws,
                                 size_t ws_bytes, cccl_stream_t stream);

/* Largest n_elems cccl_compress_noalloc accepts (2^30 values, 2 GiB). */
#define CCCL_NOALLOC_MAX_ELEMS ((size_t)1 << 30)

/* cccl_compress for callers that cannot allocate device memory: code that
 * runs while another component owns the memory pool and forbids side
 * allocations, paths that must not call cudaMalloc because it can
 * synchronise the device or is not allowed at that point, and embeddings
 * without an allocator at all.  It has no counterpart in the paper.
 * It produces exactly the stream cccl_compress produces, without a workspace
 * argument: its scratch (about 256 KiB: the status header and one placement
 * word per group of 8 chunks for CCCL_NOALLOC_MAX_ELEMS values) is a static
 * device array that every GPU which loads this library keeps until the
 * process exits.  Nothing is allocated per call.
 *   d_in, n_elems, d_out, out_capacity, stream: as for cccl_compress.
 *   n_elems must be 1..CCCL_NOALLOC_MAX_ELEMS, else CCCL_ERR_INVALID_ARG.
 * The first call on a device looks up the scratch's device address (with
 * that device current) and caches it.  Each call clears the scratch it uses
 * and the 64-byte stream header on `stream` before compressing.
 * The compressed size is the stream header's total_bytes (bytes 32..39 of
 * d_out) once the work is done: the header is cleared first, and the size is
 * written when the last chunk has been placed.  There is no workspace to
 * report a device-side error in: a wait that ran out (TIMEOUT, which only a
 * fault inside the kernel could cause) goes unreported, and the stream can
 * then lack chunks even though total_bytes is set.  A caller that needs the
 * device status uses cccl_compress with a workspace and cccl_get_result.
 * All calls on a device share the one scratch array: calls that may overlap
 * on the GPU (different streams without ordering between them) race and must
 * not be issued; calls on one stream are ordered and safe.
 * Returns INVALID_ARG, CAPACITY, CUDA or OK synchronously. */
cccl_status cccl_compress_noalloc(const uint16_t *d_in, size_t n_elems, void *d_out, size_t out_capacity,
                                  cccl_stream_t stream);

/* Decompress a stream made for n_elems values (the inverse of section 4.1's
 * split; the "Decomp." stage of Figure 2).
 *   d_in          the stream; in_bytes is the size of the readable buffer
 *                 (at least the stream's total_bytes).  Nothing past
 *                 in_bytes is read.
 *   d_out         receives n_elems uint16 bf16 bit patterns.
 *   d_ws          ws_bytes >= 16 (cccl_workspace_bytes(n_elems) is enough).
 * A stream that is malformed or was made for another n_elems is reported
 * as CORRUPT by cccl_get_result; the contents of d_out are then undefined.
 * Returns INVALID_ARG, CUDA or OK synchronously. */
cccl_status cccl_decompress(const void *d_in, size_t in_bytes, uint16_t *d_out, size_t n_elems, void *d_ws,
                            size_t ws_bytes, cccl_stream_t stream);

/* The reduce step of a compressed allreduce over R ranks whose buffers are
 * resident in this GPU's memory (section 5, CopyReducePacks; Figure 2:
 * decompress -> reduce -> compress, fused in one kernel).
 *   h_ins         host array of R device pointers to compressed streams,
 *                 each made for n_elems values; h_in_bytes their readable
 *                 sizes.  1 <= R <= 64.
 *   d_out         receives the compressed element-wise sum; out_capacity
 *                 must be at least cccl_compress_bound(n_elems).
 *   d_ws          ws_bytes >= cccl_workspace_bytes(n_elems).
 * The sum of element i is acc = x_0[i] in binary32, then acc = acc + x_r[i]
 * for r = 1..R-1 in that order (round to nearest even, subnormals kept),
 * rounded once to bf16 (nearest even; every NaN becomes 0x7FC0), and the
 * result is compressed exactly as cccl_compress would.
 * Input errors are reported as CORRUPT by cccl_get_result.
 * Returns INVALID_ARG, CAPACITY, CUDA or OK synchronously. */
cccl_status cccl_reduce_compressed(const void *const *h_ins, const size_t *h_in_bytes, int R, size_t n_elems,
                                   void *d_out, size_t out_capacity, void *d_ws, size_t ws_bytes,
                                   cccl_stream_t stream);

/* Reduce operators of cccl_reduce_op ("CCCL: In-GPU Compression-Coupled
 * Collective Communication", section 5: CopyReducePacks performs "the
 * required collective operation (e.g., sum, min, max)"). */
#define CCCL_OP_SUM 0 /* binary32 sum in rank order, one rounding: cccl_reduce_compressed */
#define CCCL_OP_MIN 1 /* exact element-wise minimum: any NaN gives 0x7FC0; -0 below +0 */
#define CCCL_OP_MAX 2 /* exact element-wise maximum: any NaN gives 0x7FC0; +0 above -0 */

/* cccl_reduce_compressed with the operator `op` (CCCL_OP_*).  The result is
 * compressed exactly as cccl_compress would.  An unknown op is INVALID_ARG;
 * the other arguments and errors are those of cccl_reduce_compressed. */
cccl_status cccl_reduce_op(const void *const *h_ins, const size_t *h_in_bytes, int R, size_t n_elems, int op,
                           void *d_out, size_t out_capacity, void *d_ws, size_t ws_bytes, cccl_stream_t stream);

/* Paged payload: the KV-cache blocks that prefill sends to decode ("CCCL:
 * In-GPU Compression-Coupled Collective Communication", section 6.2 and
 * Figure 3: PD disaggregation), compressed from where they lie in a paged
 * cache and decompressed into the receiver's blocks; no transport here.
 *   d_pool        pool_blocks blocks of block_elems bf16 values each,
 *                 contiguous; block_elems is a multiple of 4096, so no chunk
 *                 straddles two blocks.
 *   d_table       device array of n_blocks int32 block indices: the logical
 *                 buffer is blocks d_table[0], d_table[1], ... in that order
 *                 (n_elems = n_blocks * block_elems).
 * cccl_compress_paged produces exactly the stream cccl_compress produces for
 * the gathered buffer (d_out, out_capacity, d_ws, ws_bytes as there).
 * cccl_decompress_paged decompresses a stream made for n_elems values into the
 * named blocks; the table's entries must then be distinct.
 * A table entry outside 0..pool_blocks-1 is reported by cccl_get_result as
 * CCCL_ERR_INVALID_ARG (its chunks are skipped; the output is unspecified).
 * Returns INVALID_ARG, CAPACITY (compress), CUDA or OK synchronously. */
cccl_status cccl_compress_paged(const uint16_t *d_pool, size_t pool_blocks, size_t block_elems, const int32_t *d_table,
                                size_t n_blocks, void *d_out, size_t out_capacity, void *d_ws, size_t ws_bytes,
                                cccl_stream_t stream);
cccl_status cccl_decompress_paged(const void *d_in, size_t in_bytes, uint16_t *d_pool, size_t pool_blocks,
                                  size_t block_elems, const int32_t *d_table, size_t n_blocks, void *d_ws,
                                  size_t ws_bytes, cccl_stream_t stream);

/* The selective-compression reduce step (section 5, "Selective compression
 * across collective stages": an intermediate reduction merges the locally
 * available, uncompressed data with received compressed partial results, and
 * only the remote data are decompressed).
 *   d_local       n_elems uint16 bf16 bit patterns, uncompressed: rank 0.
 *   h_ins         host array of n_remote device pointers to compressed
 *                 streams made for n_elems values (ranks 1..n_remote);
 *                 h_in_bytes their readable sizes.  0 <= n_remote <= 63
 *                 (both arrays may be NULL when n_remote is 0).
 *   d_out, d_ws   as for cccl_reduce_compressed.
 * The result is that of cccl_reduce_compressed on the R = n_remote + 1 ranks
 * with rank 0's operand given uncompressed: acc = local[i] in binary32, then
 * the remote ranks added in order, one rounding to bf16 (every NaN becomes
 * 0x7FC0), compressed as cccl_compress would.
 * Returns INVALID_ARG, CAPACITY, CUDA or OK synchronously. */
cccl_status cccl_reduce_mixed(const uint16_t *d_local, const void *const *h_ins, const size_t *h_in_bytes,
                              int n_remote, size_t n_elems, void *d_out, size_t out_capacity, void *d_ws,
                              size_t ws_bytes, cccl_stream_t stream);

/* Element types of the typed entry points: the stream header's dtype field.
 * Section 4.1's split is stated for floating-point values and worked out for
 * bf16; fp16 and fp32 take the same split with their own exponent field
 * (this library's reading: the same scheme, other widths).  Values are
 * passed as their bit patterns: uint16 for bf16 and fp16, uint32 for fp32.
 *   bf16  exponent bits 7..14 (8 bits); packed body: 4096 bytes of
 *         sign << 7 | fraction bits 0..6, then the exponent planes.
 *   fp16  exponent bits 10..14 (5 bits); packed body: 4096 bytes of fraction
 *         bits 0..7, three bit-planes (fraction bit 8, fraction bit 9, sign),
 *         then the exponent planes; widths 1..4.
 *   fp32  exponent bits 23..30 (8 bits); the upper 16 bits are coded as a
 *         bf16 value: packed body: 4096 bytes of sign << 7 | fraction bits
 *         16..22, the 4096 lower halves (fraction bits 0..15) as u16, then
 *         the exponent planes.
 * The other layers (header, offset table, chunk header, plane layout, escape
 * bytes, raw chunks of n_c values) are as described at the top.  A full
 * chunk is packed only when 512 k + pad16(n_esc) is below 512 * (exponent
 * bits), else raw. */
#define CCCL_DTYPE_BF16 1
#define CCCL_DTYPE_FP16 2
#define CCCL_DTYPE_FP32 3

/* Worst-case stream size of n_elems values of `dtype` (every chunk raw):
 * 64 + pad16(8 * n_chunks) + sum over chunks of 16 + pad16(bytes * n_c).
 * 0 for n_elems 0 or above CCCL_MAX_ELEMS, or an unknown dtype.
 * cccl_workspace_bytes(n_elems) serves every dtype. */
size_t cccl_compress_bound_typed(int dtype, size_t n_elems);

/* cccl_compress (window = 0) or cccl_compress_window (window != 0) for any
 * element type.  d_in holds n_elems bit patterns of `dtype`;
 * out_capacity >= cccl_compress_bound_typed(dtype, n_elems).  With
 * CCCL_DTYPE_BF16 the stream is exactly cccl_compress's (or
 * cccl_compress_window's).  Returns INVALID_ARG (also for an unknown dtype),
 * CAPACITY, CUDA or OK. */
cccl_status cccl_compress_typed(int dtype, const void *d_in, size_t n_elems, void *d_out, size_t out_capacity,
                                void *d_ws, size_t ws_bytes, int window, cccl_stream_t stream);

/* cccl_decompress for any element type: d_out receives n_elems bit patterns
 * of `dtype`.  A stream whose header names another element type is CORRUPT
 * (reported by cccl_get_result).  Returns INVALID_ARG, CUDA or OK. */
cccl_status cccl_decompress_typed(int dtype, const void *d_in, size_t in_bytes, void *d_out, size_t n_elems,
                                  void *d_ws, size_t ws_bytes, cccl_stream_t stream);

/* The reduce step for any element type and operator (section 5,
 * CopyReducePacks: sum, min, max), with an optional uncompressed local
 * operand (section 5, selective compression).
 *   d_local       NULL, or n_elems bit patterns of `dtype`: rank 0.
 *   h_ins         host array of n_streams device pointers to compressed
 *                 streams of `dtype` made for n_elems values, the next ranks
 *                 in order; h_in_bytes their readable sizes.  The ranks
 *                 R = n_streams + (d_local != NULL) must be 1..64.
 *   op            CCCL_OP_SUM: acc = x_0[i] in binary32, acc = acc + x_r[i]
 *                 in rank order (round to nearest even, subnormals kept),
 *                 then one rounding to the type (bf16 and fp16: nearest
 *                 even, with subnormals and overflow to Inf; fp32: none);
 *                 CCCL_OP_MIN / CCCL_OP_MAX: exact, -0 below +0.  Any NaN
 *                 becomes the type's NaN: 0x7FC0, 0x7E00, 0x7FC00000.
 *   d_out, d_ws   out_capacity >= cccl_compress_bound_typed(dtype, n_elems),
 *                 ws_bytes >= cccl_workspace_bytes(n_elems).
 * The result is compressed exactly as cccl_compress_typed (window 0) would.
 * Input errors are reported as CORRUPT by cccl_get_result.
 * Returns INVALID_ARG, CAPACITY, CUDA or OK synchronously. */
cccl_status cccl_reduce_typed(int dtype, int op, const void *d_local, const void *const *h_ins,
                              const size_t *h_in_bytes, int n_streams, size_t n_elems, void *d_out,
                              size_t out_capacity, void *d_ws, size_t ws_bytes, cccl_stream_t stream);

/* Wait for the work enqueued on `stream` and read the outcome stored in the
 * workspace of the last call that used it.
 *   out_bytes     (may be NULL) the compressed stream size of a compress or
 *                 reduce call; 0 after a decompress.
 *   dev_status    (may be NULL) OK, CORRUPT or TIMEOUT.
 * Synchronises `stream`.  Returns INVALID_ARG for a null or misaligned
 * workspace, CUDA if the copy or the synchronisation failed, else OK. */
cccl_status cccl_get_result(const void *d_ws, cccl_stream_t stream, uint64_t *out_bytes, cccl_status *dev_status);

/* Failure-detection self test of the library's bounded waits ("CCCL: In-GPU
 * Compression-Coupled Collective Communication" gives no failure model; every
 * device wait here gives up after 2 s of GPU time rather than spin forever).
 * One small kernel runs both kinds of wait against a condition that never
 * completes: an mbarrier no thread arrives on, and a decoupled look-back
 * whose predecessor never publishes its size.  Each gives up after the
 * library's wait limit (2 s) and records TIMEOUT in the workspace, as a
 * stalled compress, decompress or reduce would; nothing faults, and the
 * context stays usable.
 *   d_ws          device workspace of at least cccl_workspace_bytes(8192)
 *                 bytes, 16-byte aligned; cleared here first.
 *   stream        the stream to run on.
 * Returns INVALID_ARG for a null, misaligned, too small or non-device
 * workspace, CUDA if the clear or the launch failed, else OK; then
 * cccl_get_result reports TIMEOUT (after about 2 s). */
cccl_status cccl_selftest_timeouts(void *d_ws, size_t ws_bytes, cccl_stream_t stream);

/* Largest n_units cccl_selftest_lookback accepts. */
#define CCCL_SELFTEST_MAX_UNITS ((uint32_t)1 << 20)

/* Self test of the decoupled look-back that places variable-size units of
 * chunks densely in a stream (section 4.4 of "CCCL: In-GPU Compression-
 * Coupled Collective Communication" writes each block straight into its
 * final place; here every unit's place is the exclusive prefix sum of the
 * sizes before it, found by looking back over its predecessors' published
 * sizes).  It runs the library's own look-back over n_units units of the
 * given sizes and writes each unit's offset (the prefix sum plus 4096).
 *   d_sizes       n_units device uint32 sizes, each below 2^17 (a unit of the
 *                 compress and reduce kernels is at most 8 chunks of 16,400
 *                 bytes); read only.
 *   poison_unit   a unit that publishes the poison flag instead of its size
 *                 (as a failed unit would); every later unit then reports
 *                 poison; n_units or more for none.
 *   concurrent    0: every unit's size is published first (unit 0 as its end
 *                 offset), then one warp looks back for units n_units-1 down
 *                 to 1, so each walks over all its predecessors (many 256-unit
 *                 windows).  1: warps take units in ticket order, wait a
 *                 pseudo-random time (up to 20 us, one unit in 64 up to
 *                 200 us), publish and look back concurrently, as the
 *                 kernels do.
 *   d_result      n_units device uint64: the offset of each unit, or
 *                 0xC000000000000000 (poison) for the poisoned unit and every
 *                 unit after it.
 *   d_ws          workspace of at least 16 + 8 * n_units bytes, 16-byte
 *                 aligned; cleared here first.
 * Every wait is the library's bounded one: a wait that runs out records
 * TIMEOUT, which cccl_get_result reports.
 * Returns INVALID_ARG for an argument outside these rules, CUDA if the clear
 * or a launch failed, else OK. */
cccl_status cccl_selftest_lookback(const uint32_t *d_sizes, uint32_t n_units, uint32_t poison_unit, int concurrent,
                                   uint64_t *d_result, void *d_ws, size_t ws_bytes, cccl_stream_t stream);

/* Static, human-readable name of a status code. */
const char *cccl_status_string(cccl_status status);

#ifdef __cplusplus
}
#endif

#endif /* CCCL_H */

/*
 * zccl.h -- C ABI of libzccl, a GB300 (sm_103a) library for the lossless BF16
 * exponent codec of "ZipCCL: Efficient Lossless Data Compression of
 * Communication Collectives for Accelerating LLM Training" (technical
 * summary sections 2.A-2.D of the page of that title).
 *
 * What the codec does (ZipCCL 2.A, 2.B): each BF16 value is split into a
 * sign-mantissa byte and its 8-bit exponent; an exponent that is one of the
 * 7 entries of a LUT becomes a 3-bit code 001..111, any other exponent gets
 * the zero-point code 000 and is stored whole, in element order, in a
 * separate zero-point array.  The LUT is derived from the standard deviation
 * sigma of the tensor, so compression needs no statistics pass.
 *
 * Stream format (little-endian; every region a multiple of 128 bytes,
 * ZipCCL 2.C).  Elements are cut into chunks of 4096; the last chunk keeps
 * roundup(count, 1024) slots.
 *   [0,128)    header: u32 magic 0x4C43435A ("ZCCL"), u16 version 1,
 *              u16 log2(chunk) = 12, u64 n, u64 n_esc, u8 lut[7], u8 0,
 *              u64 zp_offset, zeros
 *   blocks     per chunk of L slots: L sign-mantissa bytes (sign in bit 7,
 *              mantissa in bits 0..6), then 3 code planes of L/8 bytes; plane
 *              p holds bit p of each code, slot s is bit (s mod 32) of the
 *              little-endian 32-bit word s/32; padding slots are all zero
 *   zp_offset  = 128 + 11 * (total slots) / 8: n_esc raw exponent bytes,
 *              zero-padded to a multiple of 128
 * Total size = zp_offset + roundup(n_esc, 128) bytes: 11 bits per element
 * slot plus 8 bits per escape plus header and padding (ZipCCL 2.B: 16 -> 11
 * bits).  No per-chunk offset table is stored: the decoder recounts escapes
 * from the code planes and rescans.
 *
 * Conventions for every call:
 *   - all calls are stateless and thread-safe, never throw, and never
 *     allocate: the caller owns every buffer, including the workspace;
 *   - device pointers refer to memory of the current CUDA device; data
 *     buffers (inputs, outputs, streams, workspace) must be 16-byte aligned,
 *     else ZCCL_ERR_INVALID_ARG; d_out_bytes must be 8-byte aligned;
 *   - all device work is queued asynchronously on `stream`; errors the host
 *     can see are returned at once and then nothing is launched;
 *   - data-dependent errors (corrupt stream, bad segment, timeout) are
 *     written to the optional device word *d_status (first error wins, by
 *     compare-and-swap from 0).  The library never clears it: set it to 0
 *     before the call and read it after the stream has synchronised;
 *   - n is limited to 2^40 elements per stream.
 *
 * Workspace: a device buffer of zccl_workspace_bytes() bytes that holds a
 * call's intermediate results: per-chunk escape counts and the per-range
 * look-back words and bases of the device-wide scan (compression also stages each
 * chunk's escapes there, up to 4096 bytes per chunk, so its workspace is
 * about n bytes).  It must be zeroed once before its first use
 * (zccl_workspace_init or any memset to 0).  A call that ends with
 * *d_status 0, ZCCL_ERR_CORRUPT_STREAM or ZCCL_ERR_INVALID_ARG leaves it
 * ready for the next call.  A call that ends with ZCCL_ERR_TIMEOUT (a
 * device wait ran out, so some CTAs stopped mid-call), or whose launch
 * failed, may leave its control words mid-call: zero the workspace again
 * (zccl_workspace_init) before its next use.  A workspace must not be used
 * by two calls that may run at the same time (different streams): they
 * would race.
 */
#ifndef ZCCL_H
#define ZCCL_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZCCL_OK = 0,
    ZCCL_ERR_INVALID_ARG = 1,      /* bad pointer, alignment, size or LUT   */
    ZCCL_ERR_BUFFER_TOO_SMALL = 2, /* output or workspace below the bound   */
    ZCCL_ERR_CORRUPT_STREAM = 3,   /* header / escape count inconsistent    */
    ZCCL_ERR_CUDA = 4,             /* a CUDA runtime call failed            */
    ZCCL_ERR_TIMEOUT = 5           /* a bounded device wait ran out (~1 s)  */
} zccl_status_t;

/* exp[r] is the biased BF16 exponent coded as r+1 (codes 001..111). The 7
 * bytes must be pairwise distinct. */
typedef struct {
    uint8_t exp[7];
} zccl_lut_t;

/* One segment of a batched compression: `n` BF16 values at device address
 * `in` compressed into its own stream at device address `out`, which has
 * room for `out_capacity` bytes (at least zccl_max_compressed_bytes(n)). */
typedef struct {
    const uint16_t* in;
    uint64_t n;
    void* out;
    uint64_t out_capacity;
} zccl_segment_t;

/* Operation selector for zccl_workspace_bytes. */
typedef enum {
    ZCCL_OP_COMPRESS = 0,
    ZCCL_OP_DECOMPRESS = 1,
    ZCCL_OP_COMPRESS_BATCHED = 2,
    ZCCL_OP_DECOMPRESS_REDUCE = 3
} zccl_op_t;

#define ZCCL_MAX_SEGMENTS 4096u /* segments per zccl_compress_batched call   */
#define ZCCL_MAX_SHARDS 1024u   /* shards per zccl_decompress_reduce call    */

/* LUT from sigma (ZipCCL 2.A): the 7 biased exponents E in 1..254 with the
 * largest Gaussian binade mass 2(Phi(2^(k+1)/sigma) - Phi(2^k/sigma)),
 * k = E - 127, computed in double; most probable first (exp[0] -> code 001);
 * equal masses order by smaller E.  Host only.  Returns INVALID_ARG unless
 * sigma is finite and > 0 and lut is non-NULL. */
zccl_status_t zccl_lut_from_sigma(double sigma, zccl_lut_t* lut);

/* Stream size when every element escapes: an upper bound for any input of
 * n elements (ZipCCL 2.B sizes, 2.C padding).  Host only. */
uint64_t zccl_max_compressed_bytes(uint64_t n);

/* Byte offset of the zero-point array in a stream of n elements; it depends
 * on n only, so header + chunk blocks of a stream (its frame) have a size
 * known before compression, and only the zero-point tail varies with the
 * data (see zccl_decompress_split).  Host only. */
uint64_t zccl_zero_point_offset(uint64_t n);

/* Workspace bytes for one call of `op`.  n: elements (compress, decompress,
 * decompress_reduce) or an upper bound of the segments' total elements
 * (batched); k: segment count (batched) or shard count (reduce), else
 * ignored.  Host only. */
zccl_status_t zccl_workspace_bytes(int op, uint64_t n, uint32_t k, uint64_t* bytes);

/* Zero a workspace on `stream` (one cudaMemsetAsync). */
zccl_status_t zccl_workspace_init(void* d_ws, uint64_t ws_bytes, cudaStream_t stream);

/* Compress (ZipCCL 2.B, 2.C): n BF16 values at d_in -> one stream at d_out.
 * out_capacity must be >= zccl_max_compressed_bytes(n) (else
 * BUFFER_TOO_SMALL).  The stream's byte size is written to *d_out_bytes
 * (device).  Bytes of d_out past that size are not written. */
zccl_status_t zccl_compress(const uint16_t* d_in, uint64_t n, const zccl_lut_t* lut,
                            void* d_out, uint64_t out_capacity, uint64_t* d_out_bytes,
                            void* d_ws, uint64_t ws_bytes, uint32_t* d_status,
                            cudaStream_t stream);

/* Decompress (inverse of ZipCCL 2.B): the stream of in_bytes bytes at d_in
 * -> n BF16 values at d_out.  The host checks in_bytes >=
 * zccl_zero_point_offset(n) (header and blocks present); the device checks
 * magic, version, chunk size, n, zp_offset, that the zero-point array fits
 * in in_bytes and that the escapes recounted from the code planes equal the
 * header's n_esc, and reports CORRUPT_STREAM in *d_status otherwise (the
 * output is then unspecified).  The header's LUT is used as stored. */
zccl_status_t zccl_decompress(const void* d_in, uint64_t in_bytes, uint16_t* d_out, uint64_t n,
                              void* d_ws, uint64_t ws_bytes, uint32_t* d_status,
                              cudaStream_t stream);

/* Decompress a stream held in two pieces (ZipCCL 2.D: the static part of a
 * two-phase all-to-all is sent first, and with the framing of 2.C its size is
 * fixed): d_frame = the stream's first zccl_zero_point_offset(n) bytes (header
 * and chunk blocks; their size depends on n only, so a receive of exactly
 * that size can be posted before compression), d_tail = the rest, the
 * zero-point array, tail_bytes long (the header's escape count rounded up to
 * 128; d_tail may be NULL when tail_bytes == 0).  Both 16-byte aligned.  The
 * result, checks and status are those of zccl_decompress on the two pieces
 * joined; nothing is copied to join them.  The paper sends the parts; this
 * receiving side is this library's. */
zccl_status_t zccl_decompress_split(const void* d_frame, const void* d_tail, uint64_t tail_bytes, uint16_t* d_out,
                                    uint64_t n, void* d_ws, uint64_t ws_bytes, uint32_t* d_status,
                                    cudaStream_t stream);

/* Batched compress of ragged segments in one launch (ZipCCL 2.D: the
 * static and dynamic parts of an MoE all-to-all payload).  d_segs is a
 * DEVICE array of n_segs descriptors (routing sizes never visit the host);
 * total_n must be >= the sum of their n (it sizes the grid and the
 * workspace; an undercount is reported as INVALID_ARG in *d_status and
 * nothing is written).  Every segment becomes an independent stream, exactly
 * what zccl_compress writes for it; its size goes to d_out_bytes[s]
 * (device array of n_segs).  A segment with a misaligned pointer, n >= 2^40
 * or too small a capacity is skipped: d_out_bytes[s] = 0 and *d_status
 * gets INVALID_ARG or BUFFER_TOO_SMALL.  n_segs <= ZCCL_MAX_SEGMENTS. */
zccl_status_t zccl_compress_batched(const zccl_segment_t* d_segs, uint32_t n_segs,
                                    uint64_t total_n, const zccl_lut_t* lut,
                                    uint64_t* d_out_bytes, void* d_ws, uint64_t ws_bytes,
                                    uint32_t* d_status, cudaStream_t stream);

/* Local reduction of the zipped all-to-all path of reduce-scatter (ZipCCL
 * 2.D): decode S streams of n elements each and write
 *   d_out[i] = RNE_bf16( (((x_0[i] + x_1[i]) + x_2[i]) + ... ) + x_{S-1}[i] )
 * with every add in fp32 round-to-nearest (no FMA, no flush to zero), in
 * shard order, rounded to nearest-even BF16; any NaN result becomes 0x7FC0.
 * d_streams and d_in_bytes are DEVICE arrays of S entries; each stream keeps
 * its own LUT.  Every stream must hold exactly n elements, else
 * CORRUPT_STREAM.  1 <= S <= ZCCL_MAX_SHARDS. */
zccl_status_t zccl_decompress_reduce(const void* const* d_streams, const uint64_t* d_in_bytes,
                                     uint32_t S, uint16_t* d_out, uint64_t n, void* d_ws,
                                     uint64_t ws_bytes, uint32_t* d_status,
                                     cudaStream_t stream);

/* The same local reduction as one rank of a zipped reduce-scatter runs it
 * (ZipCCL 2.D): the S inputs in rank order are the other ranks' compressed
 * streams plus the rank's own shard, which it holds uncompressed.
 *   d_local:    that shard, n plain BF16 values in device memory (16-byte
 *               aligned), at position local_pos (< S) of the fold; the entries
 *               of d_streams and d_in_bytes at local_pos are not read.  NULL:
 *               all S inputs are streams, as in zccl_decompress_reduce.
 *   accumulate: nonzero: the fold starts from the BF16 values already in
 *               d_out, so d_out[i] = RNE_bf16(((d_out[i] + x_0[i]) + ...) +
 *               x_{S-1}[i]); zero: as zccl_decompress_reduce.
 * Adds, rounding, NaN rule, errors and workspace as zccl_decompress_reduce
 * (workspace: zccl_workspace_bytes(ZCCL_OP_DECOMPRESS_REDUCE, n, S)). */
zccl_status_t zccl_decompress_reduce_local(const void* const* d_streams, const uint64_t* d_in_bytes,
                                           uint32_t S, const uint16_t* d_local, uint32_t local_pos,
                                           int accumulate, uint16_t* d_out, uint64_t n, void* d_ws,
                                           uint64_t ws_bytes, uint32_t* d_status, cudaStream_t stream);

/* Exponent histogram of n BF16 values: d_hist[e] (device, 256 uint64_t,
 * 8-byte aligned) = how many of them have biased exponent e.  accumulate = 0
 * overwrites d_hist; accumulate != 0 adds the counts to those already there
 * (one histogram over several tensors, e.g. a bucket sharing one LUT).  For a
 * LUT measured from the data rather than derived from sigma (ZipCCL 2.A
 * derives it from sigma precisely to avoid this statistics pass; the measured
 * LUT covers at least as many values on any payload).  d_in 16-byte aligned
 * unless n == 0; n < 2^40.  Asynchronous on `stream`; no workspace. */
zccl_status_t zccl_exponent_histogram(const uint16_t* d_in, uint64_t n, uint64_t* d_hist, int accumulate,
                                      cudaStream_t stream);

/* Host: the LUT of the 7 most frequent exponents of a histogram (256 host
 * uint64_t, e.g. copied back from zccl_exponent_histogram), in rank order
 * (code 1 = most frequent), ties to the smaller exponent.  Any exponent may
 * enter, including 0 (zeros and subnormals) and 255. */
zccl_status_t zccl_lut_from_histogram(const uint64_t* hist, zccl_lut_t* lut);

/* The measured LUT of n BF16 values in one call: zccl_exponent_histogram into
 * d_hist (device scratch, 256 uint64_t, 8-byte aligned; holds the histogram
 * on return), a copy back and zccl_lut_from_histogram.  Synchronises
 * `stream`; *lut (host) is written on ZCCL_OK only.  Same argument rules as
 * zccl_exponent_histogram. */
zccl_status_t zccl_lut_from_data(const uint16_t* d_in, uint64_t n, uint64_t* d_hist, zccl_lut_t* lut,
                                 cudaStream_t stream);

/* Diagnostics of the bounded device waits.  The kernels wait on two kinds
 * of things: mbarriers that their own TMA copies complete (every kernel that
 * stages through shared memory), and -- inside the cooperative compress and
 * decompress launches and the escape scan of decompress-reduce -- the
 * call's done counter and the flag words (run totals, per-chunk entries,
 * per-range look-back words) that other CTAs of the launch write.  Every
 * such wait gives up after 1 s and reports ZCCL_ERR_TIMEOUT rather than
 * hang.  These calls run the same waits, with a limit of limit_us
 * microseconds (1..1,000,000), on something that never completes, so
 * *d_status must become ZCCL_ERR_TIMEOUT.  The paper has no counterpart;
 * they exist to test the failure path.
 *
 * zccl_check_bounded_wait: an mbarrier phase nothing completes.
 * zccl_check_bounded_poll: kind ZCCL_POLL_COUNTER waits, as the done-counter
 * wait does, for the uint32_t at d_word to reach 1; kind ZCCL_POLL_FLAG
 * polls, as the flag-word waits do, for bit 63 of the uint64_t at d_word.
 * d_word: device memory, 8-byte aligned, that the caller keeps at zero. */
zccl_status_t zccl_check_bounded_wait(uint32_t limit_us, uint32_t* d_status, cudaStream_t stream);
enum { ZCCL_POLL_COUNTER = 1, ZCCL_POLL_FLAG = 2 };
zccl_status_t zccl_check_bounded_poll(int kind, uint32_t limit_us, const void* d_word, uint32_t* d_status,
                                      cudaStream_t stream);

/* Size of the static device scratch used by zccl_decompress_noalloc, and the
 * largest stream it can decode (the workspace of zccl_decompress for that n
 * fits in the scratch). */
#define ZCCL_NOALLOC_SCRATCH_BYTES (1u << 20)
#define ZCCL_NOALLOC_MAX_ELEMS 502267904ull /* 122,624 chunks of 4096 */

/* zccl_decompress for callers that cannot allocate device memory -- such as
 * a communication library's progress thread or transport plugin, or a
 * framework hook that must stay inside the framework's own memory pool,
 * where a cudaMalloc could block on device-wide synchronisation, fail under
 * a fixed memory budget or fragment the pool in the middle of a collective.
 * The paper has no counterpart to this entry point.
 * Same arguments and results as zccl_decompress, minus the workspace: the
 * library uses a static device array of ZCCL_NOALLOC_SCRATCH_BYTES (1 MiB)
 * that every GPU loading the library holds until the process exits.  n above
 * ZCCL_NOALLOC_MAX_ELEMS returns ZCCL_ERR_INVALID_ARG and queues nothing.
 * The array's device address is looked up by the first call made with a
 * given device current; make that first call before any stream capture.  A
 * lookup that fails returns ZCCL_ERR_CUDA and is tried again by the next
 * call.
 * Every call shares the array (the part the call uses is cleared at the
 * start of each call), so calls that overlap on the GPU -- e.g. issued on two
 * streams -- race: serialise them. */
zccl_status_t zccl_decompress_noalloc(const void* d_in, uint64_t in_bytes, uint16_t* d_out, uint64_t n,
                                      uint32_t* d_status, cudaStream_t stream);

/* Reduce-scatter switcher (ZipCCL 2.D: profile the link's bandwidth and
 * latency and the compression ratio, then run either the native
 * reduce-scatter or a zipped all-to-all plus a local decompress-and-reduce,
 * whichever is faster).  The pages give the inputs but no formula; this is
 * a time model of the two paths, host only, with no collective:
 *   ranks P, each holding `bytes` of BF16 (P shards of s = bytes / P);
 *   native ring:  (P-1) * (latency + s / link)
 *   zipped:       compress (P-1)*s  + (P-1) * (latency + ratio*s / link)
 *                 + decompress-reduce P*s (the own shard uncompressed)
 * where a codec step on x bytes of BF16 input takes fixed_us + x / gbs.
 * Rates are GB/s (1e9 bytes/s) of BF16 input, e.g. measured with this
 * library on the payload; ratio = compressed bytes / BF16 bytes. */
typedef struct {
    uint32_t ranks;           /* P >= 1                                      */
    uint64_t bytes;           /* BF16 bytes per rank (all P shards)          */
    double ratio;             /* finite, > 0                                 */
    double link_gbs;          /* per-rank link bandwidth, finite, > 0       */
    double link_latency_us;   /* per message, finite, >= 0                  */
    double compress_gbs;      /* finite, > 0                                 */
    double compress_fixed_us; /* per call, finite, >= 0                      */
    double reduce_gbs;        /* decompress-reduce, finite, > 0             */
    double reduce_fixed_us;   /* per call, finite, >= 0                      */
} zccl_rs_model_t;

typedef struct {
    int zipped;                 /* 1: zipped all-to-all + local reduce is faster */
    double native_us;           /* modelled time of each path                    */
    double zipped_us;
    double breakeven_link_gbs;  /* zipped wins below this link bandwidth; 0 if
                                   ratio >= 1 (never), independent of latency */
} zccl_rs_plan_t;

/* Fill *plan from *model (ties go to the native path; P == 1 exchanges
 * nothing: native, all times 0).  INVALID_ARG on a null pointer or a field
 * outside its range.  Host only. */
zccl_status_t zccl_rs_plan(const zccl_rs_model_t* model, zccl_rs_plan_t* plan);

/* Static text for a status code. */
const char* zccl_status_string(zccl_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* ZCCL_H */

// zccl_decompress.cu -- decompression: inverse scan of the escape counts
// (recounted from the code planes) and gather from the zero-point array.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B (a code
// 001..111 names a LUT exponent; code 000 takes the next entry of the
// zero-point array) and 2.C (128-byte aligned blocks, three 1-bit code
// arrays, asynchronous global->shared copies with double buffering).
//
// GB300 design.
//
//  escape_scan_kernel (used by the fused reduction, zccl_reduce.cu)  reads only the code planes (3/8 byte per element).
//    One CTA per range of 32 chunks, taken by ticket (an atomic counter, so
//    every range below a CTA's own was taken by a CTA already running, in
//    whatever order the hardware starts CTAs): each warp counts the escapes
//    of 8 chunks with 16-byte loads (the next two chunks' loads in flight
//    while one is counted) and popc of ~(p0|p1|p2), and the CTA records each
//    chunk's count, the escapes before
//    each of its quarters (1024 slots: the share of one reducing warp) and
//    its prefix within the range.  The range's offset in its stream -- the
//    inverse of the encoder's device-wide scan -- comes from a decoupled
//    look-back: the CTA publishes the range total at once, then warp 0 reads
//    the words of the ranges before it, nearest first, 32 at a time, and adds
//    totals until it meets a published inclusive prefix; it then publishes
//    its own.  The CTA of a stream's last range checks the stream's total
//    against its header.  It serves S streams at once for the fused
//    reduction.  It is launched as a programmatic dependent of the preceding
//    work and waits for it first, so its launch overlaps that work's tail.
//  decompress_kernel  one cooperative kernel with no grid barrier: each CTA
//    counts the escapes of its own run of chunks from their planes and
//    publishes the run total as a flag word, sums the earlier runs' totals
//    itself, and publishes each of its chunks' zero-point offset and count as
//    a flag word; then CTAs stream chunks taken by ticket (in a large call a
//    ticket is 4 or 2 consecutive chunks until its last part): per chunk, one TMA
//    bulk copy brings the block and a second brings the chunk's run of the
//    zero-point array, both completing on one mbarrier, double-buffered.
//    Escaped exponents are scattered to their element slots in shared
//    memory; each thread rebuilds 8 consecutive elements: plane bytes spread
//    to nibble codes, one byte permute per 4 elements looks the codes up in
//    the LUT (two registers), another makes the escape mask, and byte
//    permutes interleave sign-mantissa and exponent bytes into BF16, stored
//    with one 16-byte write.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_decode.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;

// ============================================================================
// Kernel 1: escape offsets from the code planes
// ============================================================================
struct __align__(16) ScanSmem {
    uint64_t qinfo[kRangeChunks];
    uint32_t scan[kThreads / 32];
    uint64_t range;  // the range being counted (thread 0's ticket)
    uint32_t hdr_ok;
};

// The scan's header check: a 16-byte aligned stream whose header and blocks
// fit in in_bytes, and a header that passes header_valid.
__device__ __forceinline__ bool stream_header_ok(const uint8_t* base, uint64_t in_bytes, uint64_t n,
                                                 uint64_t* n_esc_out)
{
    *n_esc_out = 0;
    if (base == nullptr || ((uintptr_t)base & 15) != 0 || in_bytes < zp_offset_of(n)) return false;
    return header_valid(reinterpret_cast<const uint32_t*>(base), in_bytes, n, n_esc_out);
}

__device__ __forceinline__ const uint8_t* scan_stream(const ScanArgs& a, uint32_t s)
{
    return a.streams == nullptr ? a.single : reinterpret_cast<const uint8_t*>(a.streams[s]);
}
__device__ __forceinline__ uint64_t scan_in_bytes(const ScanArgs& a, uint32_t s)
{
    return a.in_bytes_dev == nullptr ? a.in_bytes : a.in_bytes_dev[s];
}

// Escape count of one chunk, by one warp (valid elements only).
__device__ __forceinline__ uint32_t warp_chunk_escapes(const uint8_t* blk, uint32_t valid)
{
    const int lane = threadIdx.x & 31;
    const uint32_t L = slots_of(valid);
    uint32_t c = 0;
    if (valid == kChunk) {
        const uint4 p0 = reinterpret_cast<const uint4*>(blk + kChunk)[lane];
        const uint4 p1 = reinterpret_cast<const uint4*>(blk + kChunk + kChunk / 8)[lane];
        const uint4 p2 = reinterpret_cast<const uint4*>(blk + kChunk + kChunk / 4)[lane];
        c = __popc(~(p0.x | p1.x | p2.x)) + __popc(~(p0.y | p1.y | p2.y)) + __popc(~(p0.z | p1.z | p2.z)) +
            __popc(~(p0.w | p1.w | p2.w));
    } else {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(blk + L);
        for (uint32_t w = lane; w < L / 32; w += 32) {
            const uint32_t w0 = 32u * w;
            const uint32_t vmask = w0 + 32 <= valid ? 0xFFFFFFFFu
                                   : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
            c += __popc(~(pw[w] | pw[L / 32 + w] | pw[L / 16 + w]) & vmask);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
}

// Escapes of one chunk, by one warp: lane l counts slots [128 l, 128 l + 128)
// (16 bytes of each plane), so lanes 8q .. 8q + 7 cover quarter q.  Returns
// the chunk's quarter word: escapes before quarters 1, 2, 3 and the chunk
// total, 16 bits each (quarter_before / quarter_end).  p holds the lane's plane words
// for a whole chunk (valid == 4096); otherwise they are loaded here, masked
// to the valid slots.
__device__ __forceinline__ uint64_t warp_chunk_quarters(const uint4 (&p)[3], const uint8_t* blk, uint32_t valid)
{
    const int lane = threadIdx.x & 31;
    uint32_t e = 0;
    if (valid == kChunk) {
        e = __popc(~(p[0].x | p[1].x | p[2].x)) + __popc(~(p[0].y | p[1].y | p[2].y)) +
            __popc(~(p[0].z | p[1].z | p[2].z)) + __popc(~(p[0].w | p[1].w | p[2].w));
    } else {
        const uint32_t L = slots_of(valid);
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(blk + L);
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) {
            const uint32_t w = 4u * lane + k;
            if (w < L / 32) {
                const uint32_t w0 = 32u * w;
                const uint32_t vmask = w0 + 32 <= valid ? 0xFFFFFFFFu
                                       : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
                e += __popc(~(pw[w] | pw[L / 32 + w] | pw[L / 16 + w]) & vmask);
            }
        }
    }
    e += __shfl_xor_sync(0xffffffffu, e, 1);
    e += __shfl_xor_sync(0xffffffffu, e, 2);
    e += __shfl_xor_sync(0xffffffffu, e, 4);
    const uint64_t q0 = __shfl_sync(0xffffffffu, e, 0), q1 = __shfl_sync(0xffffffffu, e, 8);
    const uint64_t q2 = __shfl_sync(0xffffffffu, e, 16), q3 = __shfl_sync(0xffffffffu, e, 24);
    return q0 | ((q0 + q1) << 16) | ((q0 + q1 + q2) << 32) | ((q0 + q1 + q2 + q3) << 48);
}

// Warp 0 of the CTA scanning range r, whose stream's ranges start at r0 < r:
// the escapes of ranges r0 .. r - 1.  Lane i reads the look-back word of
// range j - i (j = r - 1, r - 33, ...), waiting (bounded) until it is
// published; the window's words up to the nearest inclusive prefix are
// summed, and the walk stops there.  *ok is false if a wait timed out.
__device__ uint64_t look_back(const uint64_t* lb, uint64_t r, uint64_t r0, bool* ok)
{
    const int lane = threadIdx.x & 31;
    uint64_t sum = 0;
    for (int64_t j = (int64_t)r - 1; j >= (int64_t)r0; j -= 32) {
        const int64_t i = j - lane;
        uint64_t w = kLbInclusive;  // before the stream's first range: an inclusive prefix of 0
        bool mine = true;
        if (i >= (int64_t)r0) w = poll_u64(lb + i, [](uint64_t v) { return (v & kLbState) != 0; }, &mine);
        if (!__all_sync(0xffffffffu, mine)) {
            *ok = false;
            return 0;
        }
        const uint32_t inc = __ballot_sync(0xffffffffu, (w & kLbState) == kLbInclusive);
        const int stop = inc ? __ffs(inc) - 1 : 31;
        uint64_t v = lane <= stop ? (w & kLbValue) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        sum += v;
        if (inc) break;
    }
    return sum;
}

// Checks stream s's header and that its escape count is `total` (the
// recount from its planes); reports a mismatch.
__device__ __forceinline__ void check_stream_total(const ScanArgs& a, uint32_t s, uint64_t total)
{
    uint64_t n_esc = 0;
    if (!stream_header_ok(scan_stream(a, s), scan_in_bytes(a, s), a.n, &n_esc) || n_esc != total)
        report(a.status, ZCCL_ERR_CORRUPT_STREAM);
}

// Thread 0: a range ticket of the running call.  Every CTA draws the same
// number of tickets, ceil(nr / gridDim.x), so a call makes exactly that many
// times gridDim.x draws (tickets past the last range are skipped); the CTA
// that draws the last ticket resets the counter.
__device__ __forceinline__ uint64_t draw_range(WsCtrl* ctrl, uint64_t last)
{
    const uint64_t t = atomicAdd(&ctrl->sticket, 1ull);
    if (t == last) st_relaxed_u64(reinterpret_cast<uint64_t*>(&ctrl->sticket), 0ull);
    return t;
}

__global__ void __launch_bounds__(kThreads, 7) escape_scan_kernel(const ScanArgs a)
{
    __shared__ ScanSmem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t units = (uint32_t)units_of(a.n);
    // launched as a programmatic dependent of whatever precedes it in the
    // stream: nothing is read before that work is complete and visible
    pdl_wait();
    const uint32_t rps = (units + kRangeChunks - 1) / kRangeChunks;  // ranges per stream
    const uint64_t nr = (uint64_t)rps * a.S;
    if (nr == 0) {  // no chunks: every stream must hold no escapes
        if (blockIdx.x == 0)
            for (uint32_t s = tid; s < a.S; s += kThreads)
                if (s != a.skip) check_stream_total(a, s, 0);
        pdl_launch_dependents();
        return;
    }

    // Ranges are taken by ticket: every range below a CTA's own was taken by
    // a CTA that is already running, in whatever order the hardware starts
    // CTAs, so the look-back never waits for a CTA that has not started.
    // With more than one draw per CTA, the next is drawn while the current
    // range is counted.
    const uint64_t draws = (nr + gridDim.x - 1) / gridDim.x;
    const uint64_t last = draws * gridDim.x - 1;
    uint64_t next = 0;
    if (tid == 0) sm.range = draw_range(a.ctrl, last);
    __syncthreads();
    for (uint64_t d = 0; d < draws; ++d) {
        const uint64_t r = sm.range;
        if (tid == 0 && d + 1 < draws) next = draw_range(a.ctrl, last);
        if (r >= nr) {  // a ticket past the last range (the same for the whole CTA)
            __syncthreads();
            if (tid == 0) sm.range = next;
            __syncthreads();
            continue;
        }
        const uint32_t s = (uint32_t)(r / rps), q = (uint32_t)(r % rps);
        // Counting needs only that the stream's blocks are there; the header
        // itself is checked by the CTA of the stream's last range (and again
        // by the reduce kernel before it uses it).  (The plain BF16
        // position, if any, has no stream: zero counts.)
        if (tid == 0) {
            const uint8_t* base = scan_stream(a, s);
            sm.hdr_ok = s != a.skip && base != nullptr && ((uintptr_t)base & 15) == 0 &&
                        scan_in_bytes(a, s) >= zp_offset_of(a.n);
        }
        __syncthreads();
        const uint32_t c0 = q * kRangeChunks;
        const uint32_t nch = min(kRangeChunks, units - c0);
        const bool ok = sm.hdr_ok != 0;
        if (ok) {
            // each warp counts 8 chunks, one at a time, the planes of the
            // next two chunks in flight while one is counted
            const uint8_t* base = scan_stream(a, s);
            auto load = [&](uint32_t i, uint4 (&p)[3]) {
                const uint64_t c = c0 + i;
                if (i < nch && (c + 1) * kChunk <= a.n) {
                    const uint4* pw = reinterpret_cast<const uint4*>(base + kHeaderBytes + c * kBlockBytes + kChunk);
#pragma unroll
                    for (int qq = 0; qq < 3; ++qq) p[qq] = __ldg(pw + qq * 32 + lane);
                }
            };
            uint4 pa[3], pb[3], pc[3];
            load(warp, pa);
            load(warp + 4, pb);
#pragma unroll
            for (int b = 0; b < kRangeChunks / (kThreads / 32); ++b) {
                const uint32_t i = warp + 4 * b;
                if (b + 2 < kRangeChunks / (kThreads / 32)) load(i + 8, pc);
                if (i < nch) {
                    const uint64_t c = c0 + i;
                    const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - c * kChunk);
                    const uint64_t qi = warp_chunk_quarters(pa, base + kHeaderBytes + c * kBlockBytes, valid);
                    if (lane == 0) sm.qinfo[i] = qi;
                }
#pragma unroll
                for (int qq = 0; qq < 3; ++qq) {
                    pa[qq] = pb[qq];
                    pb[qq] = pc[qq];
                }
            }
        }
        __syncthreads();
        const uint64_t qi = (ok && tid < (int)nch) ? sm.qinfo[tid] : 0ull;
        const uint32_t cnt = chunk_escapes(qi);
        uint32_t agg;
        const uint32_t ex = block_exclusive_scan<kThreads>(cnt, sm.scan, &agg);
        if (tid < (int)nch) {
            a.local[(uint64_t)s * units + c0 + tid] = ex;
            a.qinfo[(uint64_t)s * units + c0 + tid] = qi;
        }
        if (warp == 0) {
            // publish the range's total at once (the stream's first range:
            // its inclusive prefix), then look back for its offset
            if (lane == 0) st_relaxed_u64(a.lookback + r, (q == 0 ? kLbInclusive : kLbAggregate) | agg);
            bool waited = true;
            const uint64_t base = q == 0 ? 0 : look_back(a.lookback, r, r - q, &waited);
            if (lane == 0) {
                if (!waited) report(a.status, ZCCL_ERR_TIMEOUT);
                if (q != 0) st_relaxed_u64(a.lookback + r, kLbInclusive | (base + agg));
                a.bases[r] = base;
                if (q == rps - 1 && s != a.skip) check_stream_total(a, s, base + agg);
            }
        }
        if (tid == 0) sm.range = next;
        __syncthreads();
    }
    // The reduction may launch only now: launched while ranges are still
    // looking back, its CTAs (which wait for this grid before reading
    // anything) were measured to slow the look-back down more than their
    // early start saves.
    pdl_launch_dependents();
}

// ============================================================================
// Decompression: one cooperative kernel, no grid barrier
// ============================================================================
// Phase 1: CTA b counts the escapes of run b (a contiguous run of chunks, one
// per CTA) from their code planes -- TMA bulk copies of up to 15 chunks'
// planes at once into the still unused stream buffers, popc there -- and
// publishes the run's total as a flag word.  It then sums the totals of the
// runs before it (each CTA reads them itself: no CTA waits for the whole
// grid) and publishes, per chunk of its run, one entry word: flag | zero-point
// offset << 13 | escape count.  Phase 2 streams chunks taken by atomic ticket
// (SMs that get their data faster take more): per chunk one bulk copy of the
// block and one of its run of the zero-point array, completing on one
// mbarrier, double-buffered; the chunk's entry is read (and cleared) one
// iteration ahead, and the next ticket is drawn one iteration ahead, so
// neither round trip stalls the CTA.
constexpr uint32_t kPlaneBytes = kChunk * 3 / 8;  // the three planes of a full chunk: 1536 bytes
constexpr uint32_t kPlaneSlots = 15;               // chunks whose planes fit the stream buffers at once
constexpr uint32_t kCountBits = 13;                // entry word: escapes (<= 4096) in the low 13 bits

struct __align__(16) DecodeSmem {  // blk, zpb and expo must stay contiguous (phase-1 slots)
    uint8_t blk[2][kBlockBytes];   // double-buffered chunk blocks
    uint8_t zpb[2][kZpBufBytes];   // the chunk's zero-point run (16-byte aligned cover)
    uint8_t expo[kChunk];          // escaped exponents at their element slot
    uint32_t hdr[kHeaderBytes / 4];  // the stream header
    uint64_t rloc[kThreads];       // last batch of my run: chunk offset within the run
    uint32_t rcnt[kThreads];       //                      escapes per chunk
    uint64_t bar[2];
    uint64_t pbar;                 // plane copies of phase 1
    uint64_t hbar;                 // header copy
    uint64_t scan64[kThreads / 32];
    uint32_t chunk[2];             // chunk held by each buffer
    uint32_t zdelta[2];            // offset of the run's first byte inside zpb
    uint32_t zcount[2];            // escapes of the chunk
    uint32_t scan[kThreads / 32];
    uint32_t abort;
    uint32_t hdr_ok;
    uint32_t par;
    uint32_t lut_lo, lut_hi;
    uint64_t n_esc;
};

__device__ __forceinline__ uint32_t run_lo(uint32_t r, uint32_t T, uint32_t G)
{
    return (uint32_t)(((uint64_t)r * T + G - 1) / G);
}

__device__ __forceinline__ bool entry_ready(uint64_t e) { return (e & kValid) != 0; }

// Thread 0: start the block copy of chunk c into buffer buf (no arrival).
__device__ __forceinline__ void start_block(const DecompressArgs& a, DecodeSmem& sm, uint32_t c, int buf)
{
    const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - (uint64_t)c * kChunk);
    const uint32_t bytes = slots_of(valid) * 11 / 8;
    mbar_expect_tx(&sm.bar[buf], bytes);
    bulk_g2s(sm.blk[buf], a.in + kHeaderBytes + (uint64_t)c * kBlockBytes, bytes, &sm.bar[buf]);
}

// Thread 0: clear chunk c's entry (its one reader is done with it), start
// the copy of its zero-point run into buffer buf and arrive.
__device__ __forceinline__ void start_zp(const DecompressArgs& a, DecodeSmem& sm, int buf, uint32_t c, uint64_t e)
{
    a.entry[c] = 0;
    const uint64_t o0 = (e & ~kValid) >> kCountBits;
    const uint32_t cnt = (uint32_t)(e & ((1u << kCountBits) - 1));
    const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - (uint64_t)c * kChunk);
    uint32_t zbytes = 0, delta = 0, zc = 0;
    if (o0 + cnt <= sm.n_esc && cnt <= valid) {
        zc = cnt;
        if (cnt) {  // a.zp is 16-byte aligned: align the run's offsets within it
            const uint64_t lo16 = o0 & ~15ull, hi16 = round_up(o0 + cnt, 16);
            zbytes = (uint32_t)(hi16 - lo16);
            delta = (uint32_t)(o0 - lo16);
        }
    } else {
        report(a.status, ZCCL_ERR_CORRUPT_STREAM);
    }
    sm.zdelta[buf] = delta;
    sm.zcount[buf] = zc;
    mbar_arrive_expect_tx(&sm.bar[buf], zbytes);
    if (zbytes) bulk_g2s(sm.zpb[buf], a.zp + (o0 & ~15ull), zbytes, &sm.bar[buf]);
}

// Phase 2 of one chunk whose block and zero-point run are in buffer buf:
// escaped exponents to their slots, then 8 elements a thread rebuilt and
// stored.  kFull: a whole 4096-element chunk (every chunk but the last), so
// the plane offsets are constants and no store is partial.
template <bool kFull>
__device__ __forceinline__ void decode_chunk(const DecompressArgs& a, DecodeSmem& sm, int buf, uint64_t first,
                                             uint32_t valid_arg, uint32_t lut_lo, uint32_t lut_hi)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t valid = kFull ? kChunk : valid_arg;
    const uint32_t L = kFull ? kChunk : slots_of(valid);
    const uint8_t* blk = sm.blk[buf];
    uint32_t esc = 0;
    if (kFull || tid < (int)(L / 32)) {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(blk + L);
        const uint32_t w0 = 32u * tid;
        const uint32_t vmask =
            kFull || w0 + 32 <= valid ? 0xFFFFFFFFu : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
        esc = ~(pw[tid] | pw[L / 32 + tid] | pw[L / 16 + tid]) & vmask;
    }
    uint32_t agg;
    const uint32_t excl = block_exclusive_scan<kThreads, uint32_t, false>((uint32_t)__popc(esc), sm.scan, &agg);
    const bool good = agg == sm.zcount[buf];
    if (good) {
        const uint8_t* src = sm.zpb[buf] + sm.zdelta[buf] + excl;
        uint32_t m = esc, j = 0;
        while (m) {
            const uint32_t bb = __ffs(m) - 1;
            m &= m - 1;
            sm.expo[32u * tid + bb] = src[j++];
        }
    } else if (tid == 0) {
        report(a.status, ZCCL_ERR_CORRUPT_STREAM);
    }
    // warp w decodes elements [1024w, 1024w + 1024): the escape words of its
    // own lanes, so its exponents in sm.expo were placed by the warp itself
    __syncwarp();
    if (good) {
        uint16_t* dst = a.out + first;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
            if (!kFull && e0 >= valid) continue;
            const uint4 o = decode8(*reinterpret_cast<const uint2*>(blk + e0), blk[L + (e0 >> 3)],
                                    blk[L + L / 8 + (e0 >> 3)], blk[L + L / 4 + (e0 >> 3)], lut_lo, lut_hi,
                                    *reinterpret_cast<const uint2*>(sm.expo + e0));
            if (kFull || e0 + 8 <= valid) {
                *reinterpret_cast<uint4*>(dst + e0) = o;
            } else {
                store_partial(dst + e0, o, valid - e0);
            }
        }
    }
}

// Thread 0's chunk tickets in the streaming phase.  A chunk is taken from
// the ticket in hand when it has one; otherwise a ticket is drawn now and
// read one iteration later, where the chunk is first needed, so a CTA holds
// no more chunks ahead than the double buffer needs (a deeper reserve would
// lengthen the call's tail).
constexpr uint32_t kDrawn = 0xFFFFFFFFu;
// Chunks per ticket: 4 while at least 32 x gridDim.x chunks remain after it,
// 2 while at least 16 x gridDim.x do, then 1.  Decompression keeps
// one-chunk tickets longer than compression: taking consecutive chunks per
// ticket measured 1-3% slower here whenever the counter's slice keeps up,
// and only calls this large had a counter that could fall behind.
__device__ __forceinline__ uint32_t stream_ticket_chunks(uint32_t remaining)
{
    const uint32_t G = gridDim.x;
    return remaining >= 32u * G ? 4u : (remaining >= 16u * G ? 2u : 1u);
}
// Takes ticket [t, t + m) in hand, its first `used` chunks already started,
// and sizes the next draw.
__device__ __forceinline__ void hand_ticket(uint32_t t, uint32_t m, uint32_t used, uint32_t T, uint32_t& nx,
                                            uint32_t& nx_end, uint32_t& mq)
{
    const uint32_t end = t + m;
    nx = t + used;
    nx_end = end < T ? end : T;
    mq = stream_ticket_chunks(end < T ? T - end : 0u);
}
// The next chunk from the ticket in hand, else kDrawn with a draw started.
__device__ __forceinline__ uint32_t next_or_draw(uint32_t* counter, uint32_t& nx, uint32_t nx_end, uint32_t& tq,
                                                 uint32_t mq)
{
    if (nx < nx_end) return nx++;
    tq = atomicAdd(counter, mq);
    return kDrawn;
}

// kMulti: tickets of several chunks (calls of at least 16 x grid chunks); the
// other instantiation keeps one-chunk tickets with no ticket-in-hand state.
template <bool kMulti>
__global__ void __launch_bounds__(kThreads, 8) decompress_kernel(const DecompressArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t b = blockIdx.x, G = gridDim.x;
    const uint32_t T = (uint32_t)units_of(a.n);
    const uint32_t lo = run_lo(b, T, G), hi = run_lo(b + 1, T, G);

    uint32_t calls = 0;
    uint32_t published = 0;  // thread 0: run totals published before mine (compared only at exit)
    // thread 0: chunks of the ticket in hand not started yet [nx, nx_end);
    // the draw in flight (tq, of mq chunks), read where it is first needed
    uint32_t nx = 0, nx_end = 0, tq = 0, mq = 0;
    if (tid == 0) {
        calls = call_read(a.ctrl);  // used after phase 1
        sm.abort = 0;
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        mbar_init(&sm.pbar, 1);
        mbar_init(&sm.hbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&sm.hbar, kHeaderBytes);  // the header, read while phase 1 runs
        bulk_g2s(sm.hdr, a.in, kHeaderBytes, &sm.hbar);
    }
    __syncthreads();

    // ---- phase 1: escape counts of run b from the planes ----
    // The planes of up to kPlaneSlots chunks come in at once by TMA bulk
    // copies into the (not yet used) block / zero-point / exponent buffers.
    uint8_t* slots = sm.blk[0];
    uint64_t run_total = 0;
    uint32_t pphase = 0;
    for (uint32_t base = lo; base < hi; base += kThreads) {
        const uint32_t nb = min((uint32_t)kThreads, hi - base);
        for (uint32_t s0 = 0; s0 < nb; s0 += kPlaneSlots) {
            const uint32_t ns = min(kPlaneSlots, nb - s0);
            if (tid == 0) {
                uint32_t bytes = 0;
                for (uint32_t i = 0; i < ns; ++i)
                    if ((uint64_t)(base + s0 + i + 1) * kChunk <= a.n) bytes += kPlaneBytes;
                mbar_arrive_expect_tx(&sm.pbar, bytes);
                for (uint32_t i = 0; i < ns; ++i) {
                    const uint64_t c = base + s0 + i;
                    if ((c + 1) * kChunk <= a.n)
                        bulk_g2s(slots + i * kPlaneBytes, a.in + kHeaderBytes + c * kBlockBytes + kChunk, kPlaneBytes,
                                 &sm.pbar);
                }
            }
            if (!mbar_wait(&sm.pbar, pphase)) atomicExch(&sm.abort, 1u);
            pphase ^= 1;
            for (uint32_t i = warp; i < ns; i += kThreads / 32) {
                const uint64_t c = base + s0 + i;
                uint32_t e;
                if ((c + 1) * kChunk <= a.n) {
                    const uint4* pw = reinterpret_cast<const uint4*>(slots + i * kPlaneBytes);
                    const uint4 p0 = pw[lane], p1 = pw[32 + lane], p2 = pw[64 + lane];
                    e = __popc(~(p0.x | p1.x | p2.x)) + __popc(~(p0.y | p1.y | p2.y)) + __popc(~(p0.z | p1.z | p2.z)) +
                        __popc(~(p0.w | p1.w | p2.w));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
                } else {  // the stream's tail chunk, straight from global memory
                    e = warp_chunk_escapes(a.in + kHeaderBytes + c * kBlockBytes, (uint32_t)(a.n - c * kChunk));
                }
                if (lane == 0) sm.rcnt[s0 + i] = e;
            }
            __syncthreads();  // the slots are free for the next batch
        }
        const uint32_t cnt = tid < (int)nb ? sm.rcnt[tid] : 0u;
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan<kThreads>(cnt, sm.scan, &tot);
        if (tid < (int)nb) {
            const uint64_t loc = run_total + ex;
            if (base + kThreads < hi) {  // an earlier batch: park it in the entry (no flag yet)
                a.entry[base + tid] = (loc << kCountBits) | cnt;
            } else {
                sm.rloc[tid] = loc;
                sm.rcnt[tid] = cnt;
            }
        }
        run_total += tot;
        __syncthreads();
    }
    if (tid == 0) {
        bool ok = mbar_wait(&sm.hbar, 0);
        uint64_t n_esc = 0;
        ok = ok && header_valid(sm.hdr, a.in_bytes, a.n, &n_esc);
        sm.hdr_ok = ok && !sm.abort;
        sm.n_esc = n_esc;
        sm.lut_lo = sm.hdr[6] << 8;
        sm.lut_hi = (sm.hdr[6] >> 24) | (sm.hdr[7] << 8);
        const uint32_t par = calls & 1;
        sm.par = par;
        if (sm.hdr_ok) {
            st_relaxed_u64(a.flags + (uint64_t)par * kFlagWords + b, kValid | run_total);
            // a hint for the pollers (the flag bit decides), and the call's
            // completion count: the last to publish advances `calls`
            published = atomicAdd(&a.ctrl->done[par], 1u);
            // the first two chunks (by ticket): their blocks need no offsets,
            // so start them now; the arrival comes with their zero-point copy
            const uint32_t m0 = kMulti ? max(stream_ticket_chunks(T), 2u) : 2u;
            const uint32_t t = atomicAdd(&a.ctrl->dticket[par], m0);
            for (int i = 0; i < 2; ++i) {
                sm.chunk[i] = t + i;
                if (t + i < T) start_block(a, sm, t + i, i);
            }
            if constexpr (kMulti) hand_ticket(t, m0, 2u, T, nx, nx_end, mq);
        } else {
            if (sm.abort) report(a.status, ZCCL_ERR_TIMEOUT);
            else if (b == 0) report(a.status, ZCCL_ERR_CORRUPT_STREAM);
        }
    }
    __syncthreads();
    const uint32_t par = sm.par;
    uint64_t* flags = a.flags + (uint64_t)par * kFlagWords;
    clear_other_parity(a.ctrl, a.flags, par);
    if (!sm.hdr_ok) {
        if (tid == 0) call_end(a.ctrl, calls, sm.hdr_ok && published == G - 1);
        return;
    }

    // ---- the zero-point offset of run b: the sum of the earlier runs' totals ----
    // Thread 0 waits until every run has published (one poller per CTA), then
    // the CTA reads the totals it needs once; a flag not yet visible is polled.
    bool waited = true;
    if (tid == 0 && !wait_count(&a.ctrl->done[par], G)) sm.abort = 1;
    __syncthreads();
    uint64_t part = 0;
    for (uint32_t r0 = tid; r0 < b && !sm.abort; r0 += 8 * kThreads) {
        uint64_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t r = r0 + j * kThreads;
            v[j] = r < b ? ld_relaxed_u64(flags + r) : kValid;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (!entry_ready(v[j]) && waited) v[j] = poll_u64(flags + r0 + j * kThreads, entry_ready, &waited);
            part += v[j] & ~kValid;
        }
    }
    if (!waited) atomicExch(&sm.abort, 1u);
    const uint64_t run_base = block_sum_u64<kThreads>(part, sm.scan64);
    if (tid == 0 && b == G - 1 && run_base + run_total != sm.n_esc) report(a.status, ZCCL_ERR_CORRUPT_STREAM);
    // publish my run's entries: flag | offset << 13 | count
    for (uint32_t c = lo + tid; c < hi; c += kThreads) {
        const uint32_t last0 = hi - 1 - (hi - 1 - lo) % kThreads;  // first chunk of the last batch
        const uint64_t e = c >= last0 ? (sm.rloc[c - last0] << kCountBits) | sm.rcnt[c - last0]
                                      : __ldcg(a.entry + c);
        st_relaxed_u64(a.entry + c, kValid | (e + (run_base << kCountBits)));
    }
    __syncthreads();
    if (sm.abort) {  // an earlier run's total never came (bounded wait ran out)
        if (tid == 0) {
            report(a.status, ZCCL_ERR_TIMEOUT);
            for (int i = 0; i < 2; ++i) {  // let the started copies land
                if (sm.chunk[i] >= T) continue;
                mbar_arrive(&sm.bar[i]);
                mbar_wait(&sm.bar[i], 0);
            }
            call_end(a.ctrl, calls, sm.hdr_ok && published == G - 1);
        }
        return;
    }
    const uint32_t lut_lo = sm.lut_lo, lut_hi = sm.lut_hi;

    // ---- phase 2: stream chunks taken by ticket ----
    uint32_t tn = T;  // thread 0: the next chunk (kDrawn: a draw in flight), one iteration ahead
    uint64_t en = 0;  // thread 0: its entry, read one iteration ahead
    if (tid == 0) {
        bool ok = true;
        uint64_t e[2] = {0, 0};
        for (int i = 0; i < 2; ++i)
            if (sm.chunk[i] < T) e[i] = poll_u64(a.entry + sm.chunk[i], entry_ready, &ok);
        if (!ok) {  // cannot happen unless a run never published: let the started copies land
            report(a.status, ZCCL_ERR_TIMEOUT);
            for (int i = 0; i < 2; ++i) {
                if (sm.chunk[i] >= T) continue;
                mbar_arrive(&sm.bar[i]);
                mbar_wait(&sm.bar[i], 0);
            }
            sm.abort = 1;
        } else {
            for (int i = 0; i < 2; ++i)
                if (sm.chunk[i] < T) start_zp(a, sm, i, sm.chunk[i], e[i]);
            if (sm.chunk[1] < T)
                tn = kMulti ? next_or_draw(&a.ctrl->dticket[par], nx, nx_end, tq, mq)
                            : atomicAdd(&a.ctrl->dticket[par], 1u);
        }
    }
    __syncthreads();
    if (sm.abort) {
        if (tid == 0) call_end(a.ctrl, calls, sm.hdr_ok && published == G - 1);
        return;
    }
    for (uint32_t k = 0;; ++k) {
        const int buf = k & 1;
        const uint32_t c = sm.chunk[buf];
        if (c >= T) break;
        const uint64_t first = (uint64_t)c * kChunk;
        const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - first);
        if (!mbar_wait(&sm.bar[buf], (k >> 1) & 1)) atomicExch(&sm.abort, 1u);
        __syncthreads();
        if (sm.abort) {
            if (tid == 0) {
                report(a.status, ZCCL_ERR_TIMEOUT);
                if (sm.chunk[buf ^ 1] < T) mbar_wait(&sm.bar[buf ^ 1], ((k + 1) >> 1) & 1);
            }
            break;
        }
        if (tid == 0) {
            if (kMulti && tn == kDrawn) {  // the draw made at the last refill
                const uint32_t t = tq;
                tn = t < T ? t : T;
                if (t < T) hand_ticket(t, mq, 1u, T, nx, nx_end, mq);
            }
            if (tn < T) en = ld_relaxed_u64(a.entry + tn);  // used at the refill below
        }
        if (valid == kChunk)
            decode_chunk<true>(a, sm, buf, first, valid, lut_lo, lut_hi);
        else
            decode_chunk<false>(a, sm, buf, first, valid, lut_lo, lut_hi);
        __syncthreads();  // buffer buf (block, zero-point run, expo) is free again
        if (tid == 0) {
            uint32_t t = tn;
            if (t < T && !entry_ready(en)) {  // its run had not published yet
                bool ok = true;
                en = poll_u64(a.entry + t, entry_ready, &ok);
                if (!ok) {
                    report(a.status, ZCCL_ERR_TIMEOUT);
                    t = T;
                }
            }
            sm.chunk[buf] = t;
            if (t < T) {
                start_block(a, sm, t, buf);
                start_zp(a, sm, buf, t, en);
                tn = kMulti ? next_or_draw(&a.ctrl->dticket[par], nx, nx_end, tq, mq)
                            : atomicAdd(&a.ctrl->dticket[par], 1u);
            } else {
                tn = T;
            }
        }
        // (no barrier: what thread 0 just wrote for buffer buf is read two
        // iterations on, after the next iteration's barriers)
    }
    if (tid == 0) call_end(a.ctrl, calls, sm.hdr_ok && published == G - 1);
}

template <typename K>
int occupancy(K kernel, size_t smem)
{
    int blocks = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kThreads, smem) != cudaSuccess) return 1;
    return blocks > 0 ? blocks : 1;
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, uint32_t grid, cudaStream_t stream)
{
    return launch_dependent(escape_scan_kernel, grid, kThreads, 0, stream, a);
}

cudaError_t launch_decompress(const DecompressArgs& a, uint32_t grid, cudaStream_t stream)
{
    const size_t smem = sizeof(DecodeSmem);
    const bool multi = units_of(a.n) >= 16ull * grid;  // (the kernel's first ticket is then 2 or 4 chunks)
    auto kernel = multi ? decompress_kernel<true> : decompress_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_cooperative(kernel, grid, kThreads, smem, stream, a);
}

int scan_ctas_per_sm() { return occupancy(escape_scan_kernel, 0); }
int decompress_ctas_per_sm()
{
    const int one = occupancy(decompress_kernel<false>, sizeof(DecodeSmem));
    const int multi = occupancy(decompress_kernel<true>, sizeof(DecodeSmem));
    return one < multi ? one : multi;
}

}  // namespace zccl

// zccl_compress.cu -- compression: split, remap, code planes, escape counts,
// device-wide exclusive scan and zero-point compaction, for one stream or
// for a batch of ragged segments, in one cooperative kernel.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B (split
// into sign-mantissa and exponent bits; exponents in the top-7 LUT -> 3-bit
// codes 001..111, others -> zero-point code 000 + raw exponent in the
// zero-point array), 2.C (128-byte aligned chunk blocks; the 3-bit codes as
// three independent 1-bit arrays; asynchronous global->shared copies with
// double buffering) and 2.D (static/dynamic MoE parts -> batched segments).
//
// GB300 design.  One persistent, cooperatively launched grid of 128-thread
// CTAs; all segments' 4096-element chunks form one index space, cut into one
// contiguous run per CTA for the scan.  No CTA ever waits for the whole grid.
//
//  Phase 1 streams the input once.  CTAs take chunks by atomic ticket (SMs
//    that get their data faster take more chunks; a ticket is 4, 2 or 1
//    consecutive chunks, smaller as the call nears its end, and each is drawn
//    while the one before is being coded).  Each chunk's 8 KB arrives
//    in shared memory by a TMA bulk copy, double-buffered so the next chunk
//    lands while this one is coded.  A thread codes 8 consecutive elements
//    from one 16-byte shared load: byte permutes give the sign-mantissa
//    bytes, a 256-entry shared table gives each exponent's three code bits
//    pre-spread one byte apart, accumulated into one word whose bytes are the
//    three plane bytes (whole 4096-element chunks take a coder specialised
//    for them).  The coded block leaves by one bulk store.  popc over
//    ~(p0|p1|p2) counts the chunk's escapes; they are compacted within the
//    chunk into a staging slot of the workspace, the count is recorded (plus
//    one, so that 0 means not yet), and the chunk is added to its run's flag
//    word (one coded chunk, plus its escapes unless a segment starts after it
//    within its run).  When the CTA runs out of tickets, one thread counts
//    the CTA's chunks (and the CTA) on the call's done counter with one
//    release add.
//  Phase 2: CTA b takes run b.  The flag words of the runs back to its
//    segment's start (their escapes are its carry: the device-wide exclusive
//    scan done O(grid) per CTA) and its run's chunk counts are loaded at
//    once; both show whether they are final.  Thread 0 then polls the done
//    counter until every chunk is coded, and what was not final is loaded
//    again.  The CTA scans its run's chunk counts from the carry, copies each
//    chunk's staged escapes to their place in the zero-point array (clearing
//    the staging words; these are read only after the wait's acquire), and
//    finishes the streams that end in the run (header, zero padding, size).
//  The run flag words and the counter come in two sets picked by the parity
//  of the call count of the workspace; each call clears the set the next
//  one will use.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kInBytes = kChunk * 2;  // 8192
constexpr uint32_t kBatch = kThreads;       // chunks placed per round in phase 2
constexpr uint32_t kAborted = 0xFFFFFFFFu;  // code_chunk: the chunk's load never landed

__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Why a batched segment descriptor cannot be compressed (0 = it can).
__device__ __forceinline__ uint32_t segment_error(const zccl_segment_t& d)
{
    if (d.n >= kMaxElems || ((uintptr_t)d.out & 15) || (d.n && ((uintptr_t)d.in & 15)))
        return ZCCL_ERR_INVALID_ARG;
    if (d.out_capacity < stream_bytes_of(d.n, d.n)) return ZCCL_ERR_BUFFER_TOO_SMALL;
    return 0;
}

__device__ __forceinline__ zccl_segment_t seg_get(const CompressArgs& a, uint32_t s)
{
    return a.segs == nullptr ? a.single : a.segs[s];
}

// Largest s with start[s] <= x (start has n_segs + 1 non-decreasing entries).
__device__ __forceinline__ uint32_t find_segment(const uint32_t* start, uint32_t n_segs, uint32_t x)
{
    uint32_t lo = 0, hi = n_segs;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (start[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

struct __align__(16) CompressSmem {
    uint8_t in[2][kInBytes];   // double-buffered BF16 input chunk
    uint8_t blk[kBlockBytes];  // coded block being assembled
    uint32_t code_bits[256];   // exponent -> b0 | b1 << 8 | b2 << 16
    uint64_t bar[2];
    uint64_t scan64[kThreads / 32];
    int64_t smax[kThreads / 32];
    uint32_t scan[kThreads / 32];
    uint32_t scan_f[kThreads / 32];
    uint32_t cnt[kBatch];
    uint64_t off[kBatch];
    uint32_t abort;
    uint32_t par;
    uint32_t calls;
    uint32_t next[2];  // the chunk of iteration k + 1, in next[(k + 1) & 1]: slow threads
                       // still read one slot while thread 0 fills the other
    uint32_t nseg[2];  // ... and its segment
};
// followed by ustart[n_segs + 1]: first global chunk of each segment, and
// (up to kSegCache segments) each segment's input address and length, so
// that the per-chunk lookups stay in shared memory
constexpr uint32_t kSegCache = 128;
__device__ __forceinline__ uint64_t* seg_cache(uint32_t* ustart, uint32_t n_segs)
{
    return reinterpret_cast<uint64_t*>(ustart + ((n_segs + 2) & ~1u));  // 8-byte aligned: in[n_segs], n[n_segs]
}
// A segment's input address and length.
struct SegIn {
    const uint16_t* in;
    uint64_t n;
};
__device__ __forceinline__ SegIn seg_in(const CompressArgs& a, const uint32_t* ustart, uint32_t s)
{
    if (a.n_segs <= kSegCache) {
        const uint64_t* sc = seg_cache(const_cast<uint32_t*>(ustart), a.n_segs);
        return SegIn{reinterpret_cast<const uint16_t*>(sc[s]), sc[a.n_segs + s]};
    }
    const zccl_segment_t d = seg_get(a, s);
    return SegIn{d.in, d.n};
}

// Per-segment first chunk in shared memory (invalid segments get no chunks);
// returns the total chunk count.  All threads; contains barriers.
__device__ uint64_t segment_table(const CompressArgs& a, uint32_t* ustart, uint64_t* scan64)
{
    uint64_t run = 0;
    for (uint32_t base = 0; base < a.n_segs; base += kThreads) {
        const uint32_t s = base + threadIdx.x;
        uint64_t u = 0;
        if (s < a.n_segs) {
            const zccl_segment_t d = seg_get(a, s);
            if (a.segs == nullptr || segment_error(d) == 0) u = units_of(d.n);
            if (a.n_segs <= kSegCache) {
                uint64_t* sc = seg_cache(ustart, a.n_segs);
                sc[s] = reinterpret_cast<uint64_t>(d.in);
                sc[a.n_segs + s] = d.n;
            }
        }
        uint64_t tot;
        const uint64_t ex = block_exclusive_scan<kThreads, uint64_t>(u, scan64, &tot);
        if (s < a.n_segs) ustart[s] = (uint32_t)(run + ex);  // used only when the total fits
        run += tot;
    }
    if (threadIdx.x == 0) ustart[a.n_segs] = (uint32_t)run;
    __syncthreads();
    return run;
}

// Thread 0: starts the load of chunk c into buffer buf; returns its segment.
__device__ __forceinline__ uint32_t issue_chunk_load(const CompressArgs& a, const uint32_t* ustart, CompressSmem& sm,
                                                     uint32_t c, int buf)
{
    const uint32_t s = find_segment(ustart, a.n_segs, c);
    const SegIn d = seg_in(a, ustart, s);
    const uint64_t first = (uint64_t)(c - ustart[s]) * kChunk;
    const uint32_t valid = (uint32_t)umin64(kChunk, d.n - first);
    const uint32_t bytes = (valid * 2) & ~15u;  // whole 16-byte pieces; the rest by plain loads
    if (bytes) {
        mbar_arrive_expect_tx(&sm.bar[buf], bytes);
        bulk_g2s(sm.in[buf], d.in + first, bytes, &sm.bar[buf]);
    } else {
        mbar_arrive(&sm.bar[buf]);
    }
    return s;
}

// Header of a finished stream (the 32 lanes of one warp write 4 bytes each).
__device__ __forceinline__ void write_header(uint8_t* out, uint64_t n, uint64_t n_esc, const uint8_t* lut,
                                             int lane)
{
    uint32_t w = 0;
    const uint64_t zp = zp_offset_of(n);
    switch (lane) {
        case 0: w = kMagic; break;
        case 1: w = kVersion | (kLog2Chunk << 16); break;
        case 2: w = (uint32_t)n; break;
        case 3: w = (uint32_t)(n >> 32); break;
        case 4: w = (uint32_t)n_esc; break;
        case 5: w = (uint32_t)(n_esc >> 32); break;
        case 6: w = lut[0] | (lut[1] << 8) | (lut[2] << 16) | ((uint32_t)lut[3] << 24); break;
        case 7: w = lut[4] | (lut[5] << 8) | (lut[6] << 16); break;
        case 8: w = (uint32_t)zp; break;
        case 9: w = (uint32_t)(zp >> 32); break;
        default: w = 0;
    }
    reinterpret_cast<uint32_t*>(out)[lane] = w;
}

// Codes one chunk (already in sm.in[buf]) into sm.blk, stores the block and
// stages the escapes; returns the chunk's escape count (all threads).
// kFull: a whole 4096-element chunk (every chunk but a segment's last), so
// the block and plane offsets are constants and no lane masks its tail.
template <bool kFull>
__device__ __forceinline__ uint32_t code_chunk(const CompressArgs& a, CompressSmem& sm, int buf, uint32_t c,
                                               uint8_t* out, uint32_t cl, uint32_t valid_arg,
                                               bool timed_out)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t valid = kFull ? kChunk : valid_arg;
    const uint32_t L = kFull ? kChunk : slots_of(valid);
    const uint8_t* src = sm.in[buf];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
        if (!kFull && e0 >= L) continue;
        uint4 v = *reinterpret_cast<const uint4*>(src + 2 * e0);
        uint32_t keep = 0xFFu;
        if (!kFull && e0 + 8 > valid) {
            const uint32_t nv = valid > e0 ? valid - e0 : 0;  // 0..7
            keep = (1u << nv) - 1u;
            const uint32_t m0 = (keep & 1 ? 0x0000FFFFu : 0u) | (keep & 2 ? 0xFFFF0000u : 0u);
            const uint32_t m1 = (keep & 4 ? 0x0000FFFFu : 0u) | (keep & 8 ? 0xFFFF0000u : 0u);
            const uint32_t m2 = (keep & 16 ? 0x0000FFFFu : 0u) | (keep & 32 ? 0xFFFF0000u : 0u);
            const uint32_t m3 = (keep & 64 ? 0x0000FFFFu : 0u) | (keep & 128 ? 0xFFFF0000u : 0u);
            v = make_uint4(v.x & m0, v.y & m1, v.z & m2, v.w & m3);
        }
        // sign-mantissa bytes: (hi & 0x80) | (lo & 0x7F) for 4 elements at once
        const uint32_t lo01 = __byte_perm(v.x, v.y, 0x6420), hi01 = __byte_perm(v.x, v.y, 0x7531);
        const uint32_t lo23 = __byte_perm(v.z, v.w, 0x6420), hi23 = __byte_perm(v.z, v.w, 0x7531);
        const uint32_t smA = (hi01 & 0x80808080u) | (lo01 & 0x7F7F7F7Fu);
        const uint32_t smB = (hi23 & 0x80808080u) | (lo23 & 0x7F7F7F7Fu);
        *reinterpret_cast<uint2*>(sm.blk + e0) = make_uint2(smA, smB);
        // code bits: byte p of acc = plane p bits of the 8 elements (the
        // shifted table words share no bit, so adding them is OR'ing them)
        uint32_t acc = sm.code_bits[(v.x >> 7) & 0xFF];
        acc += sm.code_bits[(v.x >> 23) & 0xFF] << 1;
        acc += sm.code_bits[(v.y >> 7) & 0xFF] << 2;
        acc += sm.code_bits[(v.y >> 23) & 0xFF] << 3;
        acc += sm.code_bits[(v.z >> 7) & 0xFF] << 4;
        acc += sm.code_bits[(v.z >> 23) & 0xFF] << 5;
        acc += sm.code_bits[(v.w >> 7) & 0xFF] << 6;
        acc += sm.code_bits[(v.w >> 23) & 0xFF] << 7;
        if (!kFull) acc &= keep * 0x010101u;
        uint8_t* planes = sm.blk + L + (e0 >> 3);
        planes[0] = (uint8_t)acc;
        planes[L / 8] = (uint8_t)(acc >> 8);
        planes[L / 4] = (uint8_t)(acc >> 16);
    }
    fence_proxy_async_smem();
    // (also the CTA's verdict on the chunk's load: if it never landed in
    // some thread's bounded wait, nothing is stored)
    if (__syncthreads_or(timed_out)) return kAborted;
    if (tid == 0) {
        bulk_s2g(out + kHeaderBytes + (uint64_t)cl * kBlockBytes, sm.blk, L * 11 / 8);
        bulk_commit();
    }
    // escapes: words from the planes, chunk-local compaction into the stage
    uint32_t esc = 0;
    if (kFull || tid < (int)(L / 32)) {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(sm.blk + L);
        const uint32_t w0 = 32u * tid;
        const uint32_t vmask =
            kFull || w0 + 32 <= valid ? 0xFFFFFFFFu : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
        esc = ~(pw[tid] | pw[L / 32 + tid] | pw[L / 16 + tid]) & vmask;
    }
    uint32_t agg;
    const uint32_t excl = block_exclusive_scan<kThreads, uint32_t, false>((uint32_t)__popc(esc), sm.scan, &agg);
    uint8_t* dst = a.stage + (uint64_t)c * kChunk + excl;
    const uint16_t* x16 = reinterpret_cast<const uint16_t*>(src);
    uint32_t m = esc, j = 0;
    while (m) {
        const uint32_t b = __ffs(m) - 1;
        m &= m - 1;
        dst[j++] = (uint8_t)(x16[32u * tid + b] >> 7);
    }
    return agg;
}

// Runs: the T chunks cut into runs of 2^shift consecutive chunks, the
// smallest power of two that leaves at most one run per CTA, so that a
// chunk's run is a shift (no division on the per-chunk path).  CTA b takes
// run b in phase 2; run r = [run_lo(r), run_lo(r + 1)).
__device__ __forceinline__ uint32_t run_shift(uint32_t T, uint32_t G)
{
    uint32_t sh = 0;
    while (((uint64_t)T + (1ull << sh) - 1) >> sh > G) ++sh;
    return sh;
}
__device__ __forceinline__ uint32_t run_lo(uint32_t r, uint32_t T, uint32_t sh)
{
    return (uint32_t)min((uint64_t)r << sh, (uint64_t)T);
}
__device__ __forceinline__ uint32_t run_of(uint32_t c, uint32_t sh) { return c >> sh; }

// A run's flag word: chunks of the run coded so far << 40 | the escapes of
// those chunks that carry into the next run.
constexpr int kBookkeeper = 32;  // lane 0 of warp 1: per-chunk counts and flag words
constexpr uint32_t kDoneShift = 40;
constexpr uint64_t kDoneOne = 1ull << kDoneShift;

__global__ void __launch_bounds__(kThreads) compress_kernel(const CompressArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    CompressSmem& sm = *reinterpret_cast<CompressSmem*>(smem_raw);
    uint32_t* ustart = reinterpret_cast<uint32_t*>(smem_raw + sizeof(CompressSmem));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t b = blockIdx.x, G = gridDim.x;

    uint32_t calls = 0;    // thread 0: read now, used once the first chunk is coded
    uint32_t coded = 0;    // bookkeeper: chunks this CTA coded
    bool last = false;     // bookkeeper: this CTA completed the call's done count
    if (tid == 0) calls = call_read(a.ctrl);
    uint32_t nx = 0, nx_end = 0, tq = 0, mq = 0;  // thread 0: tickets (take_chunk)
    for (int e = tid; e < 256; e += kThreads) {
        uint32_t c = 0;
#pragma unroll
        for (int r = 0; r < 7; ++r)
            if (a.lut[r] == e) c = r + 1;
        sm.code_bits[e] = (c & 1) | (((c >> 1) & 1) << 8) | (((c >> 2) & 1) << 16);
    }
    const uint64_t total64 = segment_table(a, ustart, sm.scan64);  // (contains barriers)
    const bool fits = total64 <= a.max_units;
    const uint32_t T = fits ? (uint32_t)total64 : 0u;
    const uint32_t sh = run_shift(T, G);

    // ---- phase 1: code chunks taken by ticket, stage escapes, count ----
    if (tid == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
        sm.abort = 0;
        first_ticket(&a.ctrl->ticket, T, 1u, tq, mq);
        const uint32_t t = take_chunk(&a.ctrl->ticket, T, nx, nx_end, tq, mq);
        sm.next[0] = t;
        if (t < T) sm.nseg[0] = issue_chunk_load(a, ustart, sm, t, 0);
    }
    __syncthreads();
    uint32_t c = sm.next[0], k = 0;
    while (c < T) {
        const int buf = k & 1;
        if (tid == 0) {  // the next chunk (the load of this one is in flight)
            const uint32_t tn = take_chunk(&a.ctrl->ticket, T, nx, nx_end, tq, mq);
            sm.next[(k + 1) & 1] = tn;
            if (tn < T) sm.nseg[(k + 1) & 1] = issue_chunk_load(a, ustart, sm, tn, buf ^ 1);
            if (k == 0) sm.calls = calls;  // for the bookkeeper, after the first chunk
        }
        const uint32_t s = sm.nseg[k & 1];  // (found by thread 0 when it started the load)
        const SegIn d = seg_in(a, ustart, s);
        // the output address only for thread 0's block store (read now,
        // used after the coding)
        uint8_t* out = tid == 0 ? (uint8_t*)seg_get(a, s).out : nullptr;
        const uint32_t cl = c - ustart[s];
        const uint64_t first = (uint64_t)cl * kChunk;
        const uint32_t valid = (uint32_t)umin64(kChunk, d.n - first);
        const bool timed_out = !mbar_wait(&sm.bar[buf], (k >> 1) & 1);
        if (valid < kChunk) {  // tail: the last < 8 elements come by plain loads
            const uint32_t done = valid & ~7u;
            if (tid < (int)(valid - done) && !timed_out)
                reinterpret_cast<uint16_t*>(sm.in[buf])[done + tid] = d.in[first + done + tid];
            __syncthreads();
        }
        const uint32_t agg = valid == kChunk ? code_chunk<true>(a, sm, buf, c, out, cl, valid, timed_out)
                                             : code_chunk<false>(a, sm, buf, c, out, cl, valid, timed_out);
        if (agg == kAborted) {  // a bulk load never landed (bounded wait ran out)
            if (tid == 0) {
                sm.abort = 1;
                report(a.status, ZCCL_ERR_TIMEOUT);
            }
            __syncthreads();
            break;
        }
        if (tid == kBookkeeper) {  // (thread 0 is busy with the tickets and the bulk copies)
            a.counts[c] = agg + 1;  // (0: not written yet)
            // the chunk's escapes carry into the next run unless its segment
            // ends inside this run
            const uint32_t r = run_of(c, sh);
            const uint32_t carry = ustart[s + 1] >= run_lo(r + 1, T, sh) ? agg : 0u;
            uint64_t* acc = a.flags + (uint64_t)(sm.calls & 1) * kFlagWords;
            atomicAdd((unsigned long long*)&acc[r], kDoneOne | carry);
            ++coded;
        }
        if (tid == 0) bulk_wait_read0();  // the block's store has read the block buffer
        __syncthreads();
        c = sm.next[(k + 1) & 1];
        ++k;
    }
    if (tid == 0 && sm.abort && sm.next[(k + 1) & 1] < T)
        mbar_wait(&sm.bar[(k & 1) ^ 1], ((k + 1) >> 1) & 1);  // a load still in flight
    // Count this CTA's chunks (and the CTA itself) done: thread 0's release
    // add, after a barrier, orders everything the CTA wrote before it (its
    // counts, staged escapes and flag-word adds) ahead of the count.
    if (tid == 0) {
        sm.calls = calls;
        sm.par = calls & 1;
    }
    __syncthreads();
    const uint32_t par = sm.par;
    if (tid == kBookkeeper) {
        last = atom_add_release_u32(&a.ctrl->done[par], coded + 1) + coded + 1 == T + G;
        if (last) st_relaxed_u32(&a.ctrl->ticket, 0u);  // every draw of the call has returned
    }
    clear_other_parity(a.ctrl, a.flags, par);
    const uint64_t* acc = a.flags + (uint64_t)par * kFlagWords;

    if (b == 0 && a.segs != nullptr) {
        for (uint32_t s = tid; s < a.n_segs; s += kThreads) {
            const uint32_t bad = segment_error(a.segs[s]);
            if (bad) {
                report(a.status, bad);
                a.out_bytes[s] = 0;
            }
        }
    }
    if (!fits) {
        if (b == 0 && tid == 0) report(a.status, ZCCL_ERR_INVALID_ARG);
        if (tid == 0) bulk_wait0();
        if (tid == kBookkeeper) call_end(a.ctrl, sm.calls, last);
        return;
    }
    // empty, valid segments: header only (CTA 0)
    if (b == 0) {
        for (uint32_t s = warp; s < a.n_segs; s += kThreads / 32) {
            const zccl_segment_t d = seg_get(a, s);
            if (d.n != 0 || (a.segs != nullptr && segment_error(d))) continue;
            write_header((uint8_t*)d.out, 0, 0, a.lut, lane);
            if (lane == 0) a.out_bytes[s] = kHeaderBytes;
        }
    }
    const uint32_t lo = run_lo(b, T, sh), hi = run_lo(b + 1, T, sh);
    if (lo >= hi || sm.abort) {
        if (tid == 0) bulk_wait0();
        if (tid == kBookkeeper) call_end(a.ctrl, sm.calls, last);
        return;
    }

    // ---- phase 2: run b.  carry = escapes from the start of lo's segment ----
    // Once every chunk is coded (thread 0 polls the call's counter), the
    // escapes on the flag words of runs [h0, b) are the carry.  A run word is
    // final once its count says the run is complete, and a chunk count once
    // it is nonzero, so both are loaded before the wait; only what was not
    // final yet is loaded again after it.  (The staged escape bytes are read
    // only after the wait and its acquire load.)
    const uint32_t st = ustart[find_segment(ustart, a.n_segs, lo)];
    const uint32_t h0 = st < lo ? run_of(st, sh) : b;  // flag words [h0, b) make the carry
    uint64_t part = 0;
    bool reload = false;  // some run word of mine was not final yet
    for (uint32_t q0 = h0 + tid; q0 < b; q0 += 8 * kThreads) {  // all loads of a round in flight at once
        uint64_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = q0 + j * kThreads < b ? __ldcg(acc + q0 + j * kThreads) : 0ull;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t q = q0 + j * kThreads;
            if (q >= b) continue;
            const uint64_t size = run_lo(q + 1, T, sh) - run_lo(q, T, sh);
            if ((v[j] >> kDoneShift) == size) part += v[j] & (kDoneOne - 1);
            else reload = true;
        }
    }
    const uint32_t nb0 = min(kBatch, hi - lo);
    uint32_t cnt0 = tid < (int)nb0 ? __ldcg(a.counts + lo + tid) : 1u;  // my chunk count + 1 (first batch)
    if (tid == 0) {
        const bool ok = wait_count(&a.ctrl->done[par], T + G);
        // acquire the count that the poll saw complete: it was made by a chain
        // of release adds, one per CTA, so every coder's writes are ordered
        // before what follows (cheaper than a full fence, which also waits for
        // this thread's own stores)
        (void)ld_acquire_u32(&a.ctrl->done[par]);
        if (!ok) sm.abort = 1;
    }
    __syncthreads();
    if (sm.abort) {
        if (tid == 0) {
            report(a.status, ZCCL_ERR_TIMEOUT);
            bulk_wait0();
        }
        if (tid == kBookkeeper) call_end(a.ctrl, sm.calls, last);
        return;
    }
    if (reload) {  // every run is complete now: load my words again
        part = 0;
        for (uint32_t q0 = h0 + tid; q0 < b; q0 += 8 * kThreads) {
            uint64_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = q0 + j * kThreads < b ? __ldcg(acc + q0 + j * kThreads) : 0ull;
#pragma unroll
            for (int j = 0; j < 8; ++j) part += v[j] & (kDoneOne - 1);
        }
    }
    uint64_t carry = block_sum_u64<kThreads>(part, sm.scan64);
    uint32_t* stage32 = reinterpret_cast<uint32_t*>(a.stage);
    for (uint32_t base = lo; base < hi; base += kBatch) {
        const uint32_t nb = min(kBatch, hi - base);
        // issue every load of the batch before using any: my chunk count and
        // the first staged word of each of my warp's first 8 chunks
        const uint32_t cc = base + tid;
        uint32_t cnt1 = base == lo ? cnt0 : (tid < (int)nb ? __ldcg(a.counts + cc) : 1u);
        if (cnt1 == 0) cnt1 = __ldcg(a.counts + cc);  // written before the wait ended
        const uint32_t cnt = tid < (int)nb ? cnt1 - 1 : 0u;
        uint32_t v[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
            const uint32_t i = warp + 4 * ii;
            v[ii] = i < nb ? __ldcg(stage32 + (uint64_t)(base + i) * (kChunk / 4) + lane) : 0u;
        }
        const bool head = tid < (int)nb && ustart[find_segment(ustart, a.n_segs, cc)] == cc;
        uint64_t carry_out;
        const uint64_t off = seg_block_excl_scan<kThreads>(head, cnt, carry, sm.scan64, sm.scan_f, &carry_out);
        sm.cnt[tid] = cnt;
        sm.off[tid] = off;
        if (tid < (int)nb) a.counts[cc] = 0;  // its one reader is done with it
        __syncthreads();
        // each warp moves its chunks' staged escapes, 8 chunks at a time, and
        // clears the staging words it read
        for (uint32_t i0 = warp; i0 < nb; i0 += 32) {
            if (i0 != (uint32_t)warp) {
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) {
                    const uint32_t i = i0 + 4 * ii;
                    v[ii] = i < nb ? __ldcg(stage32 + (uint64_t)(base + i) * (kChunk / 4) + lane) : 0u;
                }
            }
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const uint32_t i = i0 + 4 * ii;
                if (i >= nb) continue;
                const uint32_t ci = base + i;
                const uint32_t s = find_segment(ustart, a.n_segs, ci);
                const zccl_segment_t d = seg_get(a, s);
                const uint32_t cnt_i = sm.cnt[i];
                const uint64_t zp = zp_offset_of(d.n);
                uint8_t* out = (uint8_t*)d.out;
                uint8_t* to = out + zp + sm.off[i];
                uint32_t* from = stage32 + (uint64_t)ci * (kChunk / 4);
                if (4 * lane < cnt_i) {
#pragma unroll
                    for (uint32_t q = 0; q < 4; ++q)
                        if (4 * lane + q < cnt_i) to[4 * lane + q] = (uint8_t)(v[ii] >> (8 * q));
                    from[lane] = 0;
                }
                for (uint32_t w = 32 + lane; 4 * w < cnt_i; w += 32) {  // escape-heavy chunks
                    const uint32_t x = __ldcg(from + w);
#pragma unroll
                    for (uint32_t q = 0; q < 4; ++q)
                        if (4 * w + q < cnt_i) to[4 * w + q] = (uint8_t)(x >> (8 * q));
                    from[w] = 0;
                }
                if (ci + 1 == ustart[s + 1]) {  // the segment's last chunk: finish its stream
                    const uint64_t n_esc = sm.off[i] + cnt_i;
                    const uint64_t pad_end = round_up(n_esc, 128);
                    for (uint64_t p = n_esc + lane; p < pad_end; p += 32) out[zp + p] = 0;
                    write_header(out, d.n, n_esc, a.lut, lane);
                    if (lane == 0) a.out_bytes[s] = zp + pad_end;
                }
            }
        }
        carry = carry_out;
        __syncthreads();
    }
    if (tid == 0) bulk_wait0();  // the chunk blocks' bulk stores are written
    if (tid == kBookkeeper) call_end(a.ctrl, sm.calls, last);
}

}  // namespace

size_t compress_smem_bytes(uint32_t n_segs)
{
    return sizeof(CompressSmem) + 4ull * ((n_segs + 2) & ~1u) + (n_segs <= kSegCache ? 16ull * n_segs : 0ull);
}

cudaError_t launch_compress(const CompressArgs& a, uint32_t grid, cudaStream_t stream)
{
    const size_t smem = compress_smem_bytes(a.n_segs);
    cudaError_t e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_cooperative(compress_kernel, grid, kThreads, smem, stream, a);
}

int compress_ctas_per_sm(uint32_t n_segs)
{
    int blocks = 0;
    const size_t smem = compress_smem_bytes(n_segs);
    if (cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, compress_kernel, kThreads, smem) != cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

}  // namespace zccl

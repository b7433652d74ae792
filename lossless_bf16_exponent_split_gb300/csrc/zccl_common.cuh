// zccl_common.cuh -- device-side building blocks shared by the codec kernels:
// stream geometry, the workspace control block and its per-call parity,
// sm_90+/sm_103a PTX wrappers (1-D bulk copies through the TMA engine,
// mbarriers, relaxed and acquire flags, %globaltimer), flag polling with a
// bounded wait, and block scans.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B
// (zero-point array) and 2.C (128-byte aligned chunk blocks, three 1-bit
// code arrays, asynchronous global->shared staging with double buffering).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/zccl.h"

namespace zccl {

// ---- stream geometry --------------------------------------------------------
constexpr uint32_t kChunk = 4096;               // element slots per full chunk
constexpr uint32_t kLog2Chunk = 12;
constexpr uint32_t kTailGrain = 1024;           // tail slots rounded up to this
constexpr uint32_t kHeaderBytes = 128;
constexpr uint32_t kBlockBytes = kChunk * 11 / 8;  // 5632 = 44 * 128
constexpr uint32_t kMagic = 0x4C43435Au;
constexpr uint32_t kVersion = 1;
constexpr uint64_t kMaxElems = 1ull << 40;

__host__ __device__ inline uint64_t round_up(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }
__host__ __device__ inline uint64_t units_of(uint64_t n) { return (n + kChunk - 1) / kChunk; }

// Slots of the chunk that holds `valid` elements (valid in 1..4096).
__host__ __device__ inline uint32_t slots_of(uint32_t valid)
{
    return valid == kChunk ? kChunk : (uint32_t)round_up(valid, kTailGrain);
}

// Header + all chunk blocks: full chunks of 5632 bytes plus the tail chunk.
__host__ __device__ inline uint64_t zp_offset_of(uint64_t n)
{
    uint64_t full = n / kChunk, tail = n % kChunk;
    return kHeaderBytes + full * kBlockBytes + round_up(tail, kTailGrain) * 11 / 8;
}

__host__ __device__ inline uint64_t stream_bytes_of(uint64_t n, uint64_t n_esc)
{
    return zp_offset_of(n) + round_up(n_esc, 128);
}

// ---- stream header -----------------------------------------------------------
// The 128-byte header, as 32 little-endian words h[0..31], against the
// format and the caller's n and in_bytes: magic, version and log2 chunk;
// n; a LUT of 7 distinct exponents (bytes 24..30) and byte 31 zero;
// zp_offset equal to its formula; n_esc <= n with the zero-point array
// inside in_bytes; bytes 40..127 zero.  *n_esc_out = the header's n_esc.
__device__ __forceinline__ bool header_valid(const uint32_t* h, uint64_t in_bytes, uint64_t n, uint64_t* n_esc_out)
{
    const uint64_t hn = h[2] | ((uint64_t)h[3] << 32);
    const uint64_t n_esc = h[4] | ((uint64_t)h[5] << 32);
    const uint64_t zp = h[8] | ((uint64_t)h[9] << 32);
    *n_esc_out = n_esc;
    bool ok = h[0] == kMagic && h[1] == (kVersion | (kLog2Chunk << 16)) && hn == n && zp == zp_offset_of(n) &&
              n_esc <= n && zp + round_up(n_esc, 128) <= in_bytes && (h[7] >> 24) == 0;
    uint32_t reserved = 0;
#pragma unroll
    for (int w = 10; w < 32; ++w) reserved |= h[w];
    const uint64_t lut = h[6] | ((uint64_t)(h[7] & 0xFFFFFFu) << 32);
#pragma unroll
    for (int i = 0; i < 7; ++i)
#pragma unroll
        for (int j = i + 1; j < 7; ++j) ok = ok && ((lut >> (8 * i)) & 0xFF) != ((lut >> (8 * j)) & 0xFF);
    return ok && reserved == 0;
}

// ---- workspace --------------------------------------------------------------
// [0, kCtrlBytes): control words, then the flag area (two sets of kMaxGrid
// 64-bit words, one per call parity); the rest of the workspace is laid out
// per call by the host layer.
//
// Calls of the compress and decompress kernels on one workspace alternate
// between the two flag sets by the parity of `calls`: a call reads `calls`
// as it starts (without waiting for the value), and once it has the value
// uses flag set (calls & 1) and done[calls & 1], and clears the other set
// and the other done counter for the next call.  Every CTA adds to
// done[calls & 1] after it has used the value; the CTA whose add completes
// the call's count (all CTAs have read `calls` by then) advances `calls`.
// Decompression draws chunk tickets from dticket[calls & 1] (it knows the
// parity by then) and clears the other one; compression draws them from one
// counter before it knows the parity, and the CTA whose add completes the
// call's done count (every draw has returned by then) resets it.  Calls
// on one workspace run in stream order, so a call never sees another call's
// state.
constexpr uint32_t kArrivalGroups = 32;
struct WsCtrl {
    uint32_t calls;         // compress/decompress calls made on this workspace
    uint32_t pad0[31];
    uint32_t ticket;        // compress: chunk tickets of the running call
    uint32_t pad2[31];
    uint32_t dticket[2];    // decompress: chunk tickets, by call parity
    uint32_t pad5[30];
    uint32_t done[2];       // progress count of the running call, by call parity
    uint32_t pad4[30];
    unsigned long long sticket;  // escape scan: range tickets of the running call
    uint32_t pad6[30];
    uint32_t top;           // arrivals of the group leaders (own 32-byte sector)
    uint32_t pad3[7];
    struct {
        uint32_t count;     // arrivals in group g (each in its own 32-byte sector)
        uint32_t pad[7];
    } group[kArrivalGroups];
};
constexpr uint64_t kCtrlBytes = 2048;
static_assert(sizeof(WsCtrl) <= kCtrlBytes, "control block fits");
constexpr uint32_t kFlagWords = 4096;  // per parity; one per CTA of the largest grid
constexpr uint64_t kFlagBytes = 2ull * 8 * kFlagWords;
constexpr uint64_t kPrefixBytes = kCtrlBytes + kFlagBytes;

// A published 64-bit flag word: bit 63 set, the value in the low bits.
constexpr uint64_t kValid = 1ull << 63;

// Chunks per range: the unit of the escape scan's per-range totals.
constexpr uint32_t kRangeChunks = 32;

// Look-back word of one range of the escape scan: the state in bits 62..63
// (0: not yet published; kLbAggregate: the value is the range's own escape
// total; kLbInclusive: the value is the escapes of its stream up to and
// including the range) and the value in bits 0..61.
constexpr uint64_t kLbState = 3ull << 62;
constexpr uint64_t kLbAggregate = 1ull << 62;
constexpr uint64_t kLbInclusive = 2ull << 62;
constexpr uint64_t kLbValue = (1ull << 62) - 1;

// A chunk's quarter word, written by the escape scan for the fused
// reduction: the escapes before quarter q (q = 1, 2, 3; a quarter is 1024
// slots) in bits 16(q-1) .. 16q-1, and the chunk's total in bits 48..63.
// Quarter q's escapes are those from quarter_before(q) up to quarter_end(q).
__host__ __device__ inline uint32_t quarter_before(uint64_t qi, uint32_t q)
{
    return q == 0 ? 0u : (uint32_t)(qi >> (16 * (q - 1))) & 0xFFFFu;
}
__host__ __device__ inline uint32_t quarter_end(uint64_t qi, uint32_t q)
{
    return (uint32_t)(qi >> (16 * q)) & 0xFFFFu;
}
__host__ __device__ inline uint32_t chunk_escapes(uint64_t qi) { return (uint32_t)(qi >> 48); }

// A bounded wait gives up after this long (then reports ZCCL_ERR_TIMEOUT).
constexpr uint64_t kSpinTimeoutNs = 1000000000ull;

// ---- status -----------------------------------------------------------------
__device__ __forceinline__ void report(uint32_t* status, uint32_t code)
{
    if (status != nullptr) atomicCAS(status, 0u, code);
}

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Polls *p until `ready(value)` holds, with back-off; gives up after
// kSpinTimeoutNs.  Returns the last value read; *ok is false on timeout.
template <class Ready>
__device__ __forceinline__ uint64_t poll_u64(const uint64_t* p, Ready ready, bool* ok,
                                             uint64_t limit_ns = kSpinTimeoutNs)
{
    uint64_t v = ld_relaxed_u64(p);
    if (ready(v)) return v;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        __nanosleep(32);
        v = ld_relaxed_u64(p);
        if (ready(v)) return v;
        if ((it & 15) == 15 && globaltimer() - t0 > limit_ns) {
            *ok = false;
            return v;
        }
    }
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Expect `bytes` more transaction bytes in the current phase, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`; false if it did not complete
// within `limit_ns` (the copies it waits for are then reported lost).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kSpinTimeoutNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0 && globaltimer() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> shared through the TMA engine, completing on `bar`
// (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy shared -> global (bulk-group completion).
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the bulk stores issued by this thread have finished reading smem.
__device__ __forceinline__ void bulk_wait_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... all but the most recent bulk-store group.
__device__ __forceinline__ void bulk_wait_read1()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until the bulk stores issued by this thread are complete.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic-proxy smem writes before later bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory accesses by 32-bit shared address.  They are volatile so
// that they stay where they are written relative to the waits (also
// volatile) that make their data valid.
__device__ __forceinline__ uint32_t lds_u32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds_u128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_u8(uint32_t a, uint32_t v)
{
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v));
}
__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v));
}
__device__ __forceinline__ uint64_t lds_u64w(uint32_t a)
{
    uint64_t v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_u64(uint32_t a, uint64_t v)
{
    asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(v));
}

// 16-byte asynchronous copy global -> shared by one thread (cp.async, L2
// only): src_bytes of 16 are read, the rest of the 16 bytes zero-filled.
// Both addresses 16-byte aligned.  Completion: cp_async_commit() closes the
// thread's current group; cp_async_wait<N>() waits until at most N of its
// groups are pending.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes = 16)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- warp / block helpers ---------------------------------------------------
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive scan of `v` over a block of kThreads threads; returns the
// exclusive prefix and writes the block total to *total.  `scratch` holds at
// least kThreads/32 words.  Contains __syncthreads (call from all threads).
// kTrailingBarrier = false skips the final barrier: only for callers that
// pass another barrier before the scratch is written again.
template <int kThreads, typename T = uint32_t, bool kTrailingBarrier = true>
__device__ __forceinline__ T block_exclusive_scan(T v, T* scratch, T* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    T before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        T t = scratch[w];
        before += (w < warp) ? t : 0;
        all += t;
    }
    *total = all;
    if (kTrailingBarrier) __syncthreads();  // scratch may be reused right after
    return before + incl - v;
}

// ---- programmatic dependent launch -------------------------------------------
// The first kernel of a pair lets the second launch once its CTAs are done
// with their main work; the second waits for the first's completion (and its
// memory) before reading what the first wrote.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- arrival counters --------------------------------------------------------
__device__ __forceinline__ uint32_t atom_inc_acq_rel(uint32_t* p, uint32_t wrap)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap) : "memory");
    return old;
}

// Thread 0 of every CTA calls this once per pass.  CTAs arrive in up to 32
// groups, each on its own counter, and the last of each group on the top
// counter, so no address takes more than ~gridDim/32 atomics.  Returns true
// in the one CTA that arrives last overall.  The counters wrap back to 0
// (atom.inc) for the next pass; acquire-release order makes everything the
// others wrote before arriving visible to the last CTA.
__device__ __forceinline__ bool arrive_counters(WsCtrl* ctrl)
{
    const uint32_t G = gridDim.x;
    const uint32_t groups = G < kArrivalGroups ? G : kArrivalGroups;
    const uint32_t g = blockIdx.x % groups;
    const uint32_t members = (G - g + groups - 1) / groups;  // CTAs b < G with b % groups == g
    if (atom_inc_acq_rel(&ctrl->group[g].count, members - 1) != members - 1) return false;
    return atom_inc_acq_rel(&ctrl->top, groups - 1) == groups - 1;
}

// Every CTA calls this exactly once, with all its threads, after its last
// global write of the pass; returns true in the one CTA that arrives last,
// which may then read everything the others wrote.
__device__ inline bool arrive_last(WsCtrl* ctrl, uint32_t* s_flag)
{
    __syncthreads();
    if (threadIdx.x == 0) *s_flag = arrive_counters(ctrl) ? 1u : 0u;
    __syncthreads();
    return *s_flag != 0;
}

// ---- call parity (compress / decompress) -------------------------------------
// Thread 0 of every CTA, first thing: starts reading `calls` (the value is
// used only later, so the load does not hold the CTA up).
__device__ __forceinline__ uint32_t call_read(const WsCtrl* ctrl)
{
    return ld_relaxed_u32(&ctrl->calls);
}

// Thread 0 of the CTA whose add completed the call's done count: advances
// `calls` for the next call on the workspace.
__device__ __forceinline__ void call_end(WsCtrl* ctrl, uint32_t calls, bool last)
{
    if (last) st_relaxed_u32(&ctrl->calls, calls + 1);
}

// Thread 0 of compression: chunk tickets from one counter (decompression
// sizes its own, in its kernel).  A ticket is a run of
// consecutive chunks: 4 while at least 16 x gridDim.x chunks remain after it,
// 2 while at least 4 x gridDim.x do, then 1, so the counter sees a quarter of
// the draws for most of a large call and the tail still balances chunk by
// chunk.  (With one draw per chunk, the counter's L2 slice could not keep up
// under the call's own streaming traffic on some placements of the counter.)
__device__ __forceinline__ uint32_t ticket_chunks(uint32_t remaining)
{
    const uint32_t G = gridDim.x;
    return remaining >= 16u * G ? 4u : (remaining >= 4u * G ? 2u : 1u);
}
// The first draw of a CTA: at least min_chunks chunks.
__device__ __forceinline__ void first_ticket(uint32_t* counter, uint32_t T, uint32_t min_chunks, uint32_t& tq,
                                             uint32_t& mq)
{
    mq = max(ticket_chunks(T), min_chunks);
    tq = atomicAdd(counter, mq);
}
// Compression's next chunk (T: none left).  [nx, nx_end) are the chunks of
// the ticket in hand not started yet; (tq, mq) is the ticket drawn ahead.
// Taking a ticket in hand draws the next one at once, so the atomic's round
// trip overlaps the work on the ticket's chunks; a CTA draws no more once a
// draw comes back at or past T.
__device__ __forceinline__ uint32_t take_chunk(uint32_t* counter, uint32_t T, uint32_t& nx, uint32_t& nx_end,
                                               uint32_t& tq, uint32_t& mq)
{
    if (nx < nx_end) return nx++;
    const uint32_t t = tq;
    if (t >= T) return T;
    const uint32_t end = t + mq;
    nx = t + 1;
    nx_end = end < T ? end : T;
    mq = ticket_chunks(end < T ? T - end : 0u);
    tq = atomicAdd(counter, mq);
    return t;
}

// All threads: clear this CTA's share of the other parity's flag set (and,
// in CTA 0, the other parity's done counter) for the next call.
__device__ __forceinline__ void clear_other_parity(WsCtrl* ctrl, uint64_t* flags, uint32_t par)
{
    const uint32_t b = blockIdx.x, G = gridDim.x;
    uint64_t* other = flags + (uint64_t)(par ^ 1) * kFlagWords;
    for (uint32_t i = b * kFlagWords / G + threadIdx.x; i < (b + 1) * kFlagWords / G; i += blockDim.x) other[i] = 0;
    if (b == 0 && threadIdx.x == 0) {
        ctrl->done[par ^ 1] = 0;
        ctrl->dticket[par ^ 1] = 0;
    }
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint32_t atom_add_release_u32(uint32_t* p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Thread 0 only: waits (with back-off, bounded) until *p >= target; false
// on timeout.  One poller per CTA keeps the polled line from flooding L2.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t target, uint64_t limit_ns = kSpinTimeoutNs)
{
    uint32_t ns = 64;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (ld_relaxed_u32(p) >= target) return true;
        if ((it & 7) == 7 && globaltimer() - t0 > limit_ns) return false;
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;
    }
}

// ---- warp scans --------------------------------------------------------------------
// Exclusive prefix sum over the 32 lanes; *total = the warp's sum.
__device__ __forceinline__ uint32_t warp_exclusive_scan(uint32_t v, uint32_t* total)
{
    const int lane = threadIdx.x & 31;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    *total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - v;
}

// ---- block reductions ------------------------------------------------------------
template <int kThreads>
__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, uint64_t* scratch)
{
    v = warp_sum_u64(v);
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    uint64_t t = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t += scratch[w];
    __syncthreads();
    return t;
}

template <int kThreads>
__device__ __forceinline__ int64_t block_max_i64(int64_t v, int64_t* scratch)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int64_t y = __shfl_xor_sync(0xffffffffu, v, o);
        v = y > v ? y : v;
    }
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    int64_t t = scratch[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) t = scratch[w] > t ? scratch[w] : t;
    __syncthreads();
    return t;
}

// ---- segmented exclusive scan of one value per thread -------------------------
// Thread t holds (head_t, v_t) in order t = 0..kThreads-1, after a carry-in
// state `carry` (the sum since the last segment start before thread 0).
// Returns sum(v) over earlier threads of t's segment (+ carry if no segment
// start lies between thread 0 and t; 0 if head_t); *carry_out = the state
// after the last thread.  Contains barriers.
template <int kThreads>
__device__ __forceinline__ uint64_t seg_block_excl_scan(bool head, uint64_t v, uint64_t carry, uint64_t* sv,
                                                        uint32_t* sf, uint64_t* carry_out)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t f = head;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t fu = __shfl_up_sync(0xffffffffu, f, o);
        const uint64_t xu = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) {
            if (!f) x += xu;
            f |= fu;
        }
    }
    if (lane == 31) {
        sf[warp] = f;
        sv[warp] = x;
    }
    uint32_t fe = __shfl_up_sync(0xffffffffu, f, 1);
    uint64_t xe = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) {
        fe = 0;
        xe = 0;
    }
    __syncthreads();
    uint64_t px = carry;
    for (int w = 0; w < warp; ++w) px = sf[w] ? sv[w] : px + sv[w];
    px = fe ? xe : px + xe;
    uint64_t tx = carry;
    for (int w = 0; w < kThreads / 32; ++w) tx = sf[w] ? sv[w] : tx + sv[w];
    __syncthreads();
    *carry_out = tx;
    return head ? 0 : px;
}

}  // namespace zccl

// zccl_common.cuh -- device-side building blocks shared by the codec kernels:
// stream geometry, sm_90+/sm_103a PTX wrappers (1-D bulk copies through the
// TMA engine, mbarriers, acquire/release flags, %globaltimer), block scans and
// the single-pass decoupled look-back that turns per-chunk escape counts into
// zero-point offsets (the device-wide exclusive scan of the codec).
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

// ---- workspace --------------------------------------------------------------
// [0,128): control words; then one 64-bit look-back flag per chunk (per shard
// and chunk for the reduction).
struct WsCtrl {
    uint32_t ticket;  // next chunk ticket of the running call; 0 between calls
    uint32_t done;    // CTAs finished (wraps to 0 at gridDim.x via atomicInc)
    uint32_t gen;     // calls completed on this workspace; tags the flags
    uint32_t pad[29];
};
static_assert(sizeof(WsCtrl) == 128, "control block is 128 bytes");
constexpr uint64_t kCtrlBytes = 128;

// flag word: [63:62] state, [61:40] call tag, [39:0] value
constexpr uint64_t kFlagAgg = 1, kFlagPrefix = 2, kFlagPoison = 3;
constexpr uint32_t kTagMod = (1u << 22) - 1;  // tags run 1..kTagMod
constexpr uint64_t kValueMask = (1ull << 40) - 1;

__device__ __forceinline__ uint32_t tag_of_gen(uint32_t gen) { return gen % kTagMod + 1; }
__device__ __forceinline__ uint64_t make_flag(uint64_t state, uint32_t tag, uint64_t v)
{
    return (state << 62) | ((uint64_t)tag << 40) | (v & kValueMask);
}

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

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
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
// within kSpinTimeoutNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0 && globaltimer() - t0 > kSpinTimeoutNs) return false;
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
// Wait until the bulk stores issued by this thread are complete.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic-proxy smem writes before later bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
template <int kThreads, typename T = uint32_t>
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
    __syncthreads();  // scratch may be reused right after
    return before + incl - v;
}

// ---- decoupled look-back ----------------------------------------------------
// Called by one full warp for work unit `unit` whose scan segment starts at
// `seg_first`.  Publishes `agg` (the unit's escape count), reads predecessors'
// flags 32*kPerLane at a time (each lane kPerLane of them, bounded waits) and
// returns the exclusive prefix in *exclusive.  Units are taken by ticket, so
// every predecessor is held by a CTA that is running or done and every wait
// ends; a wait that still runs out (or a poisoned predecessor) marks this
// unit poisoned and returns ZCCL_ERR_TIMEOUT.
template <int kPerLane>
__device__ inline uint32_t lookback(uint64_t* flags, uint32_t unit, uint32_t seg_first, uint64_t agg,
                                    uint32_t tag, uint64_t* exclusive)
{
    const int lane = threadIdx.x & 31;
    if (unit == seg_first) {
        if (lane == 0) st_release(&flags[unit], make_flag(kFlagPrefix, tag, agg));
        *exclusive = 0;
        return ZCCL_OK;
    }
    if (lane == 0) st_release(&flags[unit], make_flag(kFlagAgg, tag, agg));
    uint64_t excl = 0;
    int64_t base = (int64_t)unit - 1;
    const uint64_t t0 = globaltimer();
    for (;;) {
        uint64_t state[kPerLane], val[kPerLane];
        bool timed_out = false;
#pragma unroll
        for (int q = 0; q < kPerLane; ++q) {
            const int64_t idx = base - lane - 32 * q;  // distance lane + 32 q
            state[q] = kFlagPrefix;
            val[q] = 0;
            if (idx >= (int64_t)seg_first && !timed_out) {
                for (uint32_t it = 0;; ++it) {
                    const uint64_t f = ld_acquire(&flags[idx]);
                    if ((uint32_t)((f >> 40) & 0x3FFFFF) == tag && (f >> 62) != 0) {
                        state[q] = f >> 62;
                        val[q] = f & kValueMask;
                        break;
                    }
                    if ((it & 31) == 31) {
                        if (globaltimer() - t0 > kSpinTimeoutNs) {
                            timed_out = true;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
            }
        }
        bool bad_lane = timed_out;
#pragma unroll
        for (int q = 0; q < kPerLane; ++q) bad_lane = bad_lane || state[q] == kFlagPoison;
        if (__ballot_sync(0xffffffffu, bad_lane)) {
            if (lane == 0) st_release(&flags[unit], make_flag(kFlagPoison, tag, 0));
            *exclusive = 0;
            return ZCCL_ERR_TIMEOUT;
        }
        // nearest PREFIX: smallest distance lane + 32 q
        bool found = false;
        uint64_t part = 0;
#pragma unroll
        for (int q = 0; q < kPerLane; ++q) {
            if (found) break;
            const uint32_t pm = __ballot_sync(0xffffffffu, state[q] == kFlagPrefix);
            if (pm) {
                const int first = __ffs(pm) - 1;
                part += lane <= first ? val[q] : 0;
                found = true;
            } else {
                part += val[q];
            }
        }
        excl += warp_sum_u64(part);
        if (found) break;
        base -= 32 * kPerLane;
    }
    if (lane == 0) st_release(&flags[unit], make_flag(kFlagPrefix, tag, excl + agg));
    *exclusive = excl;
    return ZCCL_OK;
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

// Chunks per scan range of the small look-back kernels.
constexpr uint32_t kRangeChunks = 32;

// ---- end of a call ----------------------------------------------------------
// Every CTA calls this once, last, with all its threads.  The CTA that
// finishes last resets the ticket, advances the generation (so the next
// call's flags carry a new tag) and, once every kTagMod calls, clears the
// flags so a tag can never meet a stale flag of its own value.
__device__ inline void finish_call(WsCtrl* ctrl, uint64_t* flags, uint64_t n_flag_words, uint32_t gen,
                                   uint32_t* s_flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t old = atomicInc(&ctrl->done, gridDim.x - 1);
        *s_flag = (old == gridDim.x - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (*s_flag) {
        const uint32_t next = gen + 1;
        if (next % kTagMod == 0) {
            for (uint64_t i = threadIdx.x; i < n_flag_words; i += blockDim.x) flags[i] = 0;
            __threadfence();
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            atomicExch(&ctrl->ticket, 0u);
            __threadfence();
            atomicExch(&ctrl->gen, next);
        }
    }
}

}  // namespace zccl

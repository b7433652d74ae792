// zccl_hist.cu -- exponent histogram of a BF16 tensor, for a LUT measured
// from the data instead of derived from sigma.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.A: the
// method picks the top-7 exponents from a theoretical bound on sigma so that
// it needs no online statistics; this is that statistics pass, for payloads
// the Gaussian model fits badly.
//
// GB300 design.  The pass reads 2n bytes once, so it is HBM-bound provided
// the counting costs only a few instructions a value.  Each CTA keeps its
// counters in shared memory as cnt[256 exponents][32 lanes] of 32-bit words,
// each word holding two 16-bit counters: one for the values in the low half
// of a 32-bit load word, one for the high half.  Lane L of every warp adds to
// column L only, so the 32 lanes of a `red.shared` always fall in 32
// different banks whatever their exponents are, and the byte offset of a
// value's counter word is its own exponent field masked in place
// (e * 128 == bits & 0x7F80): one mask, one add and one fire-and-forget
// reduction per value.  Before a 16-bit counter can overflow, and at the
// end, the CTA folds its columns into per-bin totals; the totals go to the
// global histogram with one 64-bit atomic add per non-empty bin.
//
// Overwrite mode zeroes the histogram in a one-CTA kernel that the counting
// kernel follows by programmatic dependent launch: counting starts at once
// and only the final global adds wait for the zeroing.  The first kernel is
// itself launched as a programmatic dependent of the preceding work in the
// stream and waits for it before anything else, so its launch overlaps that
// work's tail.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kHistThreads = 1024;
constexpr int kHistWarps = kHistThreads / 32;
constexpr int kHistBatch = 2;  // 16-byte vectors a lane loads per round
constexpr int kHistCtasPerSm = 2;
constexpr uint32_t kHistSmemBytes = 256 * 32 * sizeof(uint32_t);  // under the 48 KB that needs no opt-in
constexpr uint64_t kVectorsPerRound = (uint64_t)kHistWarps * 32 * kHistBatch;
// a counter gains at most 4 per vector (four values per half-word position),
// from each warp's lane of its column: fold before 65535 could be passed
constexpr int kRoundsPerFold = 65535 / (kHistWarps * kHistBatch * 4);
static_assert(kRoundsPerFold >= 1, "16-bit counters would overflow within one round");

__device__ __forceinline__ void red_shared_add(uint32_t addr, uint32_t v)
{
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// one value's exponent field sits at bits 7..14 of `bits`; its counter word
// is at column + exponent * 128 bytes
__device__ __forceinline__ void count_low(uint32_t column, uint32_t bits)
{
    red_shared_add(column + (bits & 0x7F80u), 1u);
}

__device__ __forceinline__ void count_high(uint32_t column, uint32_t bits)
{
    red_shared_add(column + ((bits >> 16) & 0x7F80u), 0x10000u);
}

__global__ void __launch_bounds__(256) hist_zero_kernel(uint64_t* hist)
{
    // the preceding work (which may write the input or the histogram) first
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    hist[threadIdx.x] = 0;
}

__global__ void __launch_bounds__(kHistThreads, kHistCtasPerSm)
    hist_kernel(const uint16_t* in, uint64_t n, unsigned long long* hist, bool wait_first)
{
    // accumulate mode: launched right behind the preceding work, which may
    // write the input; overwrite mode: behind the zeroing kernel, which
    // starts it only once that work is complete
    if (wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ uint32_t cnt[];  // [256][32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 256 * 32; i += kHistThreads) cnt[i] = 0;
    __syncthreads();
    const uint32_t column = (uint32_t)__cvta_generic_to_shared(cnt) + lane * 4;
    const uint64_t nv = n / 8;
    const uint4* v = reinterpret_cast<const uint4*>(in);
    uint64_t total = 0;  // thread tid < 256 owns exponent tid

    // the CTA's columns into per-bin totals; called by every thread
    auto fold = [&]() {
        __syncthreads();
        if (tid < 256) {
            uint32_t lo = 0, hi = 0;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) {
                const int L = (j + tid) & 31;  // rotated: the warp's 32 reads hit 32 banks
                const uint32_t w = cnt[tid * 32 + L];
                cnt[tid * 32 + L] = 0;
                lo += w & 0xFFFFu;
                hi += w >> 16;
            }
            total += (uint64_t)lo + hi;
        }
        __syncthreads();
    };

    // rounds are CTA-uniform (every warp runs each one, guarding its own
    // vectors), so the folds' barriers are reached by all threads
    int rounds = 0;
    for (uint64_t cbase = (uint64_t)blockIdx.x * kVectorsPerRound; cbase < nv;
         cbase += (uint64_t)gridDim.x * kVectorsPerRound) {
        const uint64_t base = cbase + (uint64_t)warp * 32 * kHistBatch + lane;
        uint4 x[kHistBatch];
#pragma unroll
        for (int b = 0; b < kHistBatch; ++b) {
            const uint64_t i = base + (uint64_t)b * 32;
            x[b] = i < nv ? __ldg(v + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int b = 0; b < kHistBatch; ++b) {
            if (base + (uint64_t)b * 32 < nv) {
                const uint32_t w[4] = {x[b].x, x[b].y, x[b].z, x[b].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    count_low(column, w[q]);
                    count_high(column, w[q]);
                }
            }
        }
        if (++rounds == kRoundsPerFold) {
            fold();
            rounds = 0;
        }
    }
    if (blockIdx.x == 0 && warp == 0 && lane < (int)(n % 8)) count_low(column, in[nv * 8 + lane]);
    fold();
    // the zeroing kernel (overwrite mode) must be complete before adding
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid < 256 && total) atomicAdd(&hist[tid], (unsigned long long)total);
}

}  // namespace

cudaError_t launch_histogram(const uint16_t* in, uint64_t n, uint64_t* hist, bool accumulate, int sms,
                             cudaStream_t stream)
{
    uint64_t grid = (n / 8 + kVectorsPerRound - 1) / kVectorsPerRound;
    const uint64_t full = (uint64_t)sms * kHistCtasPerSm;
    if (grid > full) grid = full;
    if (grid < 1) grid = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((uint32_t)grid);
    cfg.blockDim = dim3(kHistThreads);
    cfg.dynamicSmemBytes = kHistSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (!accumulate) {
        cudaLaunchConfig_t zc = {};
        zc.gridDim = dim3(1);
        zc.blockDim = dim3(256);
        zc.stream = stream;
        zc.attrs = attr;
        zc.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&zc, hist_zero_kernel, hist);
        if (e != cudaSuccess) return e;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hist_kernel, in, n, reinterpret_cast<unsigned long long*>(hist), accumulate);
}

}  // namespace zccl

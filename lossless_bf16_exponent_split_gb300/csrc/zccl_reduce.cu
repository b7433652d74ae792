// zccl_reduce.cu -- fused decompress + reduce: the local-reduction step of
// the zipped all-to-all path of reduce-scatter.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.D (the
// reduce-scatter switcher picks native reduce-scatter or zipped all-to-all +
// local reduction) and 2.B (decoding).
//
// out[i] = RNE_bf16( (((x_0[i] + x_1[i]) + x_2[i]) + ...) + x_{S-1}[i] ), each
// add an IEEE fp32 add (no FMA, no flush to zero) in shard order, x_s decoded
// from stream s; a NaN sum becomes 0x7FC0.
//
// GB300 design: the escape scan kernel (zccl_decompress.cu) first computes
// every shard's per-chunk zero-point offsets (range base + prefix within the
// range) from the code planes; then,
// started by programmatic dependent launch, reduce_kernel walks the chunks
// (persistent grid, static stride) and, for each chunk, the S shard blocks
// in order through a 3-stage ring of shared buffers: each step is one TMA
// bulk copy of the shard's block plus one of its zero-point run, so two
// steps are in flight while one decodes.  Each thread decodes 32 elements of
// the step straight into fp32 accumulators held in registers; after the
// last shard it rounds and stores 16-byte vectors.  Every compressed byte is
// read once and the BF16 result written once.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_decode.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;
// Shared memory (three stages, about 35 KB) admits 6 CTAs per SM; registers
// are capped to match, so neither instance falls below it.
constexpr int kCtasPerSm = 6;

// One stage of the ring: a shard's block and its zero-point run, or a chunk
// of plain BF16 (the rank's own shard, or the output being accumulated into).
struct __align__(16) Stage {
    uint8_t blk[kBlockBytes];
    uint8_t zpb[kZpBufBytes];
};
static_assert(sizeof(Stage) >= 2 * kChunk, "a chunk of plain BF16 fits a stage");

struct __align__(16) ReduceSmem {
    Stage stage[kStages];
    uint8_t expo[kChunk];
    uint64_t bar[kStages];
    uint32_t zdelta[kStages];
    uint32_t zcount[kStages];
    uint32_t scan[2][kThreads / 32];  // the warps' escape totals, by step parity
    uint32_t abort;
    uint32_t last;
    uint32_t spread[256];  // spread_nibbles of every byte
};
// followed by per-shard tables: const uint8_t* base[S]; uint64_t n_esc[S]; uint32_t lut[S][2]

struct ShardTables {
    const uint8_t** base;
    uint64_t* n_esc;
    uint32_t* lut;
};

__device__ __forceinline__ ShardTables shard_tables(uint8_t* smem_raw, uint32_t S)
{
    ShardTables t;
    uint8_t* p = smem_raw + sizeof(ReduceSmem);
    t.base = reinterpret_cast<const uint8_t**>(p);
    t.n_esc = reinterpret_cast<uint64_t*>(p + 8ull * S);
    t.lut = reinterpret_cast<uint32_t*>(p + 16ull * S);
    return t;
}

// The steps of an output chunk: (accumulating) the output's current values,
// then the S inputs in rank order -- each a shard's compressed stream, or
// the plain BF16 of the rank's own shard at local_pos.
enum : uint32_t { kStepStream = 0, kStepLocal = 1, kStepOut = 2 };

// kPlain: some steps read plain BF16 (the rank's own shard, or the output
// being accumulated into); without them every step is a stream, in order.
template <bool kPlain>
__device__ __forceinline__ uint32_t steps_per_chunk(const ReduceArgs& a)
{
    return kPlain ? a.S + (a.accumulate ? 1u : 0u) : a.S;
}

// Kind of step q of a chunk; *shard gets the input position of a stream step.
template <bool kPlain>
__device__ __forceinline__ uint32_t step_kind(const ReduceArgs& a, uint32_t q, uint32_t* shard)
{
    if (!kPlain) {
        *shard = q;
        return kStepStream;
    }
    if (a.accumulate) {
        if (q == 0) return kStepOut;
        --q;
    }
    *shard = q;
    return (a.local != nullptr && q == a.local_pos) ? kStepLocal : kStepStream;
}

// Offsets of one stream step's zero-point run: the range base plus the
// chunk's prefix within its range, and its escape count (loaded one
// iteration ahead of their use by issue_step, so thread 0 never waits on
// them).
struct StepOffsets {
    uint64_t base;
    uint32_t local, count;
};

template <bool kPlain>
__device__ __forceinline__ StepOffsets load_offsets(const ReduceArgs& a, uint32_t c, uint32_t q, uint32_t total)
{
    StepOffsets o{0, 0, 0};
    uint32_t s = 0;
    if (c >= total || step_kind<kPlain>(a, q, &s) != kStepStream) return o;
    const uint32_t rps = (total + kRangeChunks - 1) / kRangeChunks;
    const uint64_t idx = (uint64_t)s * total + c;
    o.base = __ldcg(a.bases + (uint64_t)s * rps + c / kRangeChunks);
    o.local = __ldcg(a.local_off + idx);
    o.count = __ldcg(a.count + idx);
    return o;
}

// Thread 0: queue step q of chunk c into stage st.
template <bool kPlain>
__device__ __forceinline__ void issue_step(const ReduceArgs& a, ReduceSmem& sm, const ShardTables& t, uint32_t c,
                                           uint32_t q, int st, uint32_t total, const StepOffsets& off)
{
    if (c >= total) return;
    uint32_t s = 0;
    const uint32_t kind = step_kind<kPlain>(a, q, &s);
    const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - (uint64_t)c * kChunk);
    if (kind != kStepStream) {  // plain BF16: whole 16-byte pieces by bulk copy, the rest by plain loads
        const uint16_t* src = (kind == kStepLocal ? a.local : a.out) + (uint64_t)c * kChunk;
        const uint32_t bytes = (valid * 2) & ~15u;
        mbar_arrive_expect_tx(&sm.bar[st], bytes);
        if (bytes) bulk_g2s(sm.stage[st].blk, src, bytes, &sm.bar[st]);
        return;
    }
    const uint32_t bytes = slots_of(valid) * 11 / 8;
    const uint64_t o0 = off.base + off.local;
    const uint64_t o1 = o0 + off.count;
    uint32_t zbytes = 0, delta = 0, cnt = 0;
    const uint64_t zp = zp_offset_of(a.n);
    if (o1 <= t.n_esc[s] && o1 - o0 <= kChunk) {
        cnt = (uint32_t)(o1 - o0);
        if (cnt) {
            const uint64_t lo = zp + o0, lo16 = lo & ~15ull, hi16 = round_up(zp + o1, 16);
            zbytes = (uint32_t)(hi16 - lo16);
            delta = (uint32_t)(lo - lo16);
        }
    } else {
        report(a.status, ZCCL_ERR_CORRUPT_STREAM);
    }
    sm.zdelta[st] = delta;
    sm.zcount[st] = cnt;
    mbar_arrive_expect_tx(&sm.bar[st], bytes + zbytes);
    bulk_g2s(sm.stage[st].blk, t.base[s] + kHeaderBytes + (uint64_t)c * kBlockBytes, bytes, &sm.bar[st]);
    if (zbytes) bulk_g2s(sm.stage[st].zpb, t.base[s] + ((zp + o0) & ~15ull), zbytes, &sm.bar[st]);
}

// One step's share of a thread: decode (or read) its 32 elements of the
// stage and add them to its accumulators.  kFull: the chunk is whole, so
// no element needs a bound check and the four groups interleave freely.
template <bool kFull>
__device__ __forceinline__ void fold_step(const uint8_t* blk, uint32_t L, uint32_t kind, uint32_t lut_lo,
                                          uint32_t lut_hi, const ReduceSmem& sm, float2 (&acc)[16], bool first_step)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (kFull) L = kChunk;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
        if (kFull || e0 < L) {
            const uint4 o = kind == kStepStream
                                ? decode8(*reinterpret_cast<const uint2*>(blk + e0), blk[L + (e0 >> 3)],
                                          blk[L + L / 8 + (e0 >> 3)], blk[L + L / 4 + (e0 >> 3)], lut_lo, lut_hi,
                                          *reinterpret_cast<const uint2*>(sm.expo + e0), sm.spread)
                                : *reinterpret_cast<const uint4*>(blk + 2 * e0);
            const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
                acc[4 * i + k] = first_step ? f : __fadd2_rn(acc[4 * i + k], f);
            }
        }
    }
}

// All threads of the CTA: the CTA's chunks (static stride), each over its
// steps in order.  The fp32 sums are kept as pairs and added with the
// two-lane add (each lane rounds to nearest even exactly as a scalar add).
template <bool kPlain>
__device__ __forceinline__ void reduce_chunks(const ReduceArgs& a, ReduceSmem& sm, const ShardTables& t)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t total = (uint32_t)units_of(a.n);
    const uint32_t Q = steps_per_chunk<kPlain>(a);
    // thread 0: `ahead` holds the offsets of the next step to queue, at
    // (ic, iq); (pc, pq) is the step after it
    StepOffsets ahead{0, 0, 0};
    uint32_t pc = blockIdx.x, pq = 0, ic = 0, iq = 0;
    auto advance = [&]() {
        if (++pq == Q) {
            pq = 0;
            pc += gridDim.x;
        }
    };
    if (tid == 0) {
        for (int j = 0; j + 1 < kStages; ++j) {
            issue_step<kPlain>(a, sm, t, pc, pq, j, total, load_offsets<kPlain>(a, pc, pq, total));
            advance();
        }
        ic = pc;
        iq = pq;
        ahead = load_offsets<kPlain>(a, pc, pq, total);
        advance();
    }

    float2 acc[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = make_float2(0.0f, 0.0f);

    uint32_t j = 0, q = 0, c = blockIdx.x;  // step, its place in the chunk's steps, its chunk
    for (;; ++j) {
        if (c >= total) break;
        const int st = j % kStages;
        uint32_t s = 0;
        const uint32_t kind = step_kind<kPlain>(a, q, &s);
        const uint64_t first = (uint64_t)c * kChunk;
        const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - first);
        const uint32_t L = slots_of(valid);
        if (!mbar_wait(&sm.bar[st], (j / kStages) & 1)) atomicExch(&sm.abort, 1u);
        uint8_t* blk = sm.stage[st].blk;
        uint32_t esc = 0, incl = 0;
        if (kind != kStepStream) {  // plain BF16: the last < 8 values by plain loads
            const uint32_t done = valid & ~7u;
            if (tid < (int)(valid - done)) {
                const uint16_t* src = kind == kStepLocal ? a.local : a.out;
                reinterpret_cast<uint16_t*>(blk)[done + tid] = src[first + done + tid];
            }
        } else {
            if (tid < (int)(L / 32)) {
                const uint32_t* pw = reinterpret_cast<const uint32_t*>(blk + L);
                const uint32_t w0 = 32u * tid;
                const uint32_t vmask = w0 + 32 <= valid ? 0xFFFFFFFFu
                                       : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
                esc = ~(pw[tid] | pw[L / 32 + tid] | pw[L / 16 + tid]) & vmask;
            }
            incl = __popc(esc);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sm.scan[j & 1][warp] = incl;
        }
        // the step's one barrier: stage st has landed for every thread, the
        // warps' escape totals are posted, and every thread is past step
        // j - 1, so its stage is free (a warp reaches the next step's
        // totals, in the other parity's slots, only through this barrier)
        __syncthreads();
        if (sm.abort) {
            if (tid == 0) report(a.status, ZCCL_ERR_TIMEOUT);
            break;
        }
        // refill the freed stage with step j + kStages - 1
        if (tid == 0) {
            issue_step<kPlain>(a, sm, t, ic, iq, (j + kStages - 1) % kStages, total, ahead);
            ic = pc;
            iq = pq;
            ahead = load_offsets<kPlain>(a, pc, pq, total);
            advance();
        }
        if (kind == kStepStream) {
            uint32_t before = 0, agg = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                const uint32_t v = sm.scan[j & 1][w];
                before += w < warp ? v : 0u;
                agg += v;
            }
            if (agg == sm.zcount[st]) {
                const uint8_t* src = sm.stage[st].zpb + sm.zdelta[st] + before + incl - __popc(esc);
                uint32_t m = esc, jj = 0;
                while (m) {
                    const uint32_t b = __ffs(m) - 1;
                    m &= m - 1;
                    sm.expo[32u * tid + b] = src[jj++];
                }
            } else if (tid == 0) {
                report(a.status, ZCCL_ERR_CORRUPT_STREAM);
            }
            // warp w folds elements [1024w, 1024w + 1024): its own lanes'
            // escape words, so the warp placed its exponents itself
            __syncwarp();
        }
        const uint32_t lut_lo = t.lut[2 * s], lut_hi = t.lut[2 * s + 1];
        if (L == kChunk) {
            fold_step<true>(blk, L, kind, lut_lo, lut_hi, sm, acc, q == 0);
        } else {
            fold_step<false>(blk, L, kind, lut_lo, lut_hi, sm, acc, q == 0);
        }
        if (q + 1 == Q) {
            // the chunk's offset words have had their one reader (loaded
            // steps ago): clear them
            for (uint32_t r = tid; r < a.S; r += kThreads) {
                a.local_off[(uint64_t)r * total + c] = 0;
                a.count[(uint64_t)r * total + c] = 0;
            }
            uint16_t* dst = a.out + first;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
                if (e0 >= valid) continue;
                uint4 o;
                o.x = rne_bf16(acc[4 * i + 0].x) | (rne_bf16(acc[4 * i + 0].y) << 16);
                o.y = rne_bf16(acc[4 * i + 1].x) | (rne_bf16(acc[4 * i + 1].y) << 16);
                o.z = rne_bf16(acc[4 * i + 2].x) | (rne_bf16(acc[4 * i + 2].y) << 16);
                o.w = rne_bf16(acc[4 * i + 3].x) | (rne_bf16(acc[4 * i + 3].y) << 16);
                if (e0 + 8 <= valid) {
                    *reinterpret_cast<uint4*>(dst + e0) = o;
                } else {
                    store_partial(dst + e0, o, valid - e0);
                }
            }
        }
        if (++q == Q) {  // the next chunk's first step
            q = 0;
            c += gridDim.x;
        }
    }
    // steps still in flight after an early stop at step j: j + 1 .. j + kStages - 2
    // (step j + kStages - 1 is issued only after step j's barrier); wait for
    // them (bounded)
    if (tid == 0 && sm.abort) {
        for (uint32_t jj = j + 1; jj + 1 < j + kStages; ++jj) {
            if (blockIdx.x + (jj / Q) * gridDim.x < total) mbar_wait(&sm.bar[jj % kStages], (jj / kStages) & 1);
        }
    }
}

template <bool kPlain>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) reduce_kernel(const ReduceArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    ReduceSmem& sm = *reinterpret_cast<ReduceSmem*>(smem_raw);
    const ShardTables t = shard_tables(smem_raw, a.S);
    const int tid = threadIdx.x;
    const uint32_t total = (uint32_t)units_of(a.n);

    // every shard's header (the scan kernel reports a bad one; here it only
    // stops this kernel from reading out of bounds)
    bool ok = true;
    for (uint32_t s = tid; s < a.S; s += kThreads) {
        if (a.local != nullptr && s == a.local_pos) {  // the plain BF16 input: no stream
            t.base[s] = nullptr;
            t.n_esc[s] = 0;
            t.lut[2 * s] = t.lut[2 * s + 1] = 0;
            continue;
        }
        const uint8_t* base = reinterpret_cast<const uint8_t*>(a.streams[s]);
        const uint64_t in_bytes = a.in_bytes[s];
        bool good = base != nullptr && ((uintptr_t)base & 15) == 0 && in_bytes >= zp_offset_of(a.n);
        if (good) {
            const uint32_t* h = reinterpret_cast<const uint32_t*>(base);
            const uint64_t hn = h[2] | ((uint64_t)h[3] << 32);
            const uint64_t n_esc = h[4] | ((uint64_t)h[5] << 32);
            const uint64_t zp = h[8] | ((uint64_t)h[9] << 32);
            good = h[0] == kMagic && h[1] == (kVersion | (kLog2Chunk << 16)) && hn == a.n &&
                   zp == zp_offset_of(a.n) && n_esc <= a.n && zp + round_up(n_esc, 128) <= in_bytes;
            t.n_esc[s] = n_esc;
            t.lut[2 * s] = h[6] << 8;
            t.lut[2 * s + 1] = (h[6] >> 24) | (h[7] << 8);
        }
        t.base[s] = base;
        ok = ok && good;
    }
    for (uint32_t b = tid; b < 256; b += kThreads) sm.spread[b] = spread_nibbles(b);
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&sm.bar[i], 1);
        fence_mbar_init();
        sm.abort = 0;
    }
    pdl_wait();  // offsets of the scan kernel
    if (__syncthreads_and(ok)) {
        reduce_chunks<kPlain>(a, sm, t);
    } else {  // a bad header: nothing to decode, but leave the scratch clear
        for (uint32_t c = blockIdx.x; c < total; c += gridDim.x)
            for (uint32_t s = tid; s < a.S; s += kThreads) {
                a.local_off[(uint64_t)s * total + c] = 0;
                a.count[(uint64_t)s * total + c] = 0;
            }
    }
    // the last CTA to finish clears the range bases: the workspace is left
    // all zero past its control block and flag area
    if (arrive_last(a.ctrl, &sm.last)) {
        const uint64_t nb = (uint64_t)a.S * ((total + kRangeChunks - 1) / kRangeChunks);
        for (uint64_t i = tid; i < nb; i += kThreads) a.bases[i] = 0;
    }
}

}  // namespace

static size_t reduce_smem_bytes(uint32_t S) { return sizeof(ReduceSmem) + 24ull * S; }

cudaError_t launch_reduce(const ScanArgs& s, const ReduceArgs& a, uint32_t grid_scan, uint32_t grid,
                          cudaStream_t stream)
{
    const size_t smem = reduce_smem_bytes(a.S);
    const bool plain = a.local != nullptr || a.accumulate;
    cudaError_t e = plain ? cudaFuncSetAttribute(reduce_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem)
                          : cudaFuncSetAttribute(reduce_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_scan(s, grid_scan, stream);
    if (e != cudaSuccess) return e;
    return plain ? launch_dependent(reduce_kernel<true>, grid, kThreads, smem, stream, a)
                 : launch_dependent(reduce_kernel<false>, grid, kThreads, smem, stream, a);
}

template <bool kPlain>
static int reduce_occupancy(size_t smem)
{
    int blocks = 0;
    if (cudaFuncSetAttribute(reduce_kernel<kPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, reduce_kernel<kPlain>, kThreads, smem) !=
        cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

// CTAs per SM for either instance (the grid is sized once for both)
int reduce_ctas_per_sm(uint32_t S)
{
    const size_t smem = reduce_smem_bytes(S);
    const int a = reduce_occupancy<true>(smem), b = reduce_occupancy<false>(smem);
    return a < b ? a : b;
}

}  // namespace zccl

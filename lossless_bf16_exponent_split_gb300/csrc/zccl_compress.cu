// zccl_compress.cu -- compression: split, remap, code planes, escape counts,
// device-wide exclusive scan and zero-point compaction, for one stream or
// for a batch of ragged segments.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B (split
// into sign-mantissa and exponent bits; exponents in the top-7 LUT -> 3-bit
// codes 001..111, others -> zero-point code 000 + raw exponent in the
// zero-point array), 2.C (128-byte aligned chunk blocks; the 3-bit codes as
// three independent 1-bit arrays; asynchronous global->shared copies with
// double buffering) and 2.D (static/dynamic MoE parts -> batched segments).
//
// GB300 design: two kernels back to back on the caller's stream, the second
// started by programmatic dependent launch so its launch overlaps the
// first's tail.
//
//  compress_blocks_kernel  streams the input once.  A persistent grid of
//    128-thread CTAs walks the 4096-element chunks; each chunk's 8 KB arrives
//    in shared memory by a TMA bulk copy, double-buffered so the next chunk
//    lands while this one is coded.  A thread codes 8 consecutive elements
//    from one 16-byte shared load: byte permutes give the sign-mantissa
//    bytes, a 256-entry shared table gives each exponent's three code bits
//    pre-spread one byte apart, accumulated into one word whose bytes are the
//    three plane bytes.  The coded block leaves by one bulk store.  popc over
//    ~(p0|p1|p2) counts the chunk's escapes; they are compacted within the
//    chunk into a staging slot of the workspace, the count is recorded and
//    added (one atomic) to its 32-chunk range's total.  No CTA waits for
//    another: the CTA that finishes last (an atomic arrival counter) runs one
//    segmented exclusive scan over the few hundred range totals -- the
//    device-wide scan of the escape counts -- giving each range's base.
//  compress_place_kernel  one CTA per range: scans its 32 counts, copies
//    each chunk's staged escapes to base + prefix in the zero-point array,
//    and finishes each stream (header, padding, size).
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kInBytes = kChunk * 2;  // 8192

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

// Per-segment chunk (and range) starts in shared memory: ustart[s] = first
// global chunk of segment s, rstart[s] = first global range.  Invalid
// segments get no chunks.  Returns the totals through *units, *ranges.
// All threads; contains barriers.
__device__ void segment_table(const CompressArgs& a, uint32_t* ustart, uint32_t* rstart, uint64_t* scan64,
                              uint64_t* units_total, uint64_t* ranges_total)
{
    uint64_t run_u = 0, run_r = 0;
    for (uint32_t base = 0; base < a.n_segs; base += kThreads) {
        const uint32_t s = base + threadIdx.x;
        uint64_t u = 0;
        if (s < a.n_segs) {
            const zccl_segment_t d = seg_get(a, s);
            if (a.segs == nullptr || segment_error(d) == 0) u = units_of(d.n);
        }
        const uint64_t r = (u + kRangeChunks - 1) / kRangeChunks;
        uint64_t tot_u, tot_r;
        const uint64_t ex_u = block_exclusive_scan<kThreads, uint64_t>(u, scan64, &tot_u);
        const uint64_t ex_r = block_exclusive_scan<kThreads, uint64_t>(r, scan64, &tot_r);
        if (s < a.n_segs) {
            ustart[s] = (uint32_t)(run_u + ex_u);  // used only when the totals are in range
            rstart[s] = (uint32_t)(run_r + ex_r);
        }
        run_u += tot_u;
        run_r += tot_r;
    }
    if (threadIdx.x == 0) {
        ustart[a.n_segs] = (uint32_t)run_u;
        rstart[a.n_segs] = (uint32_t)run_r;
    }
    *units_total = run_u;
    *ranges_total = run_r;
    __syncthreads();
}

// ============================================================================
// Kernel 1: code blocks, count and stage escapes
// ============================================================================
struct __align__(16) BlocksSmem {
    uint8_t in[2][kInBytes];   // double-buffered BF16 input chunk
    uint8_t blk[kBlockBytes];  // coded block being assembled
    uint32_t code_bits[256];   // exponent -> b0 | b1 << 8 | b2 << 16
    uint64_t bar[2];
    uint64_t scan64[kThreads / 32];
    uint32_t scan[kThreads / 32];
    uint32_t scan_f[kThreads / 32];
    uint32_t abort;
    uint32_t last;
};

__device__ __forceinline__ void issue_chunk_load(const CompressArgs& a, const uint32_t* ustart, BlocksSmem& sm,
                                                 uint32_t c, int buf)
{
    const uint32_t s = find_segment(ustart, a.n_segs, c);
    const zccl_segment_t d = seg_get(a, s);
    const uint64_t first = (uint64_t)(c - ustart[s]) * kChunk;
    const uint32_t valid = (uint32_t)umin64(kChunk, d.n - first);
    const uint32_t bytes = (valid * 2) & ~15u;  // whole 16-byte pieces; the rest by plain loads
    if (bytes) {
        mbar_arrive_expect_tx(&sm.bar[buf], bytes);
        bulk_g2s(sm.in[buf], d.in + first, bytes, &sm.bar[buf]);
    } else {
        mbar_arrive(&sm.bar[buf]);
    }
}

__global__ void __launch_bounds__(kThreads) compress_blocks_kernel(const CompressArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    BlocksSmem& sm = *reinterpret_cast<BlocksSmem*>(smem_raw);
    uint32_t* ustart = reinterpret_cast<uint32_t*>(smem_raw + sizeof(BlocksSmem));
    uint32_t* rstart = ustart + a.n_segs + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < 256; e += kThreads) {
        uint32_t c = 0;
#pragma unroll
        for (int r = 0; r < 7; ++r)
            if (a.lut[r] == e) c = r + 1;
        sm.code_bits[e] = (c & 1) | (((c >> 1) & 1) << 8) | (((c >> 2) & 1) << 16);
    }
    uint64_t total64, ranges64;
    segment_table(a, ustart, rstart, sm.scan64, &total64, &ranges64);
    const bool fits = total64 <= a.max_units && ranges64 <= a.max_ranges;  // else reported by the placement kernel
    const uint32_t total = fits ? (uint32_t)total64 : 0u;
    if (tid == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
        sm.abort = 0;
        if (blockIdx.x < total) issue_chunk_load(a, ustart, sm, blockIdx.x, 0);
    }
    __syncthreads();

    uint32_t k = 0;
    for (uint32_t c = blockIdx.x; c < total; c += gridDim.x, ++k) {
        const int buf = k & 1;
        if (tid == 0 && c + gridDim.x < total) issue_chunk_load(a, ustart, sm, c + gridDim.x, buf ^ 1);
        const uint32_t s = find_segment(ustart, a.n_segs, c);
        const zccl_segment_t d = seg_get(a, s);
        const uint32_t cl = c - ustart[s];
        const uint64_t first = (uint64_t)cl * kChunk;
        const uint32_t valid = (uint32_t)umin64(kChunk, d.n - first);
        const uint32_t L = slots_of(valid);

        if (!mbar_wait(&sm.bar[buf], (k >> 1) & 1)) atomicExch(&sm.abort, 1u);
        if (valid < kChunk) {  // tail: the last < 8 elements come by plain loads
            const uint32_t done = valid & ~7u;
            if (tid < (int)(valid - done))
                reinterpret_cast<uint16_t*>(sm.in[buf])[done + tid] = d.in[first + done + tid];
        }
        __syncthreads();
        if (sm.abort) {  // a bulk load never landed (bounded wait ran out)
            if (tid == 0) report(a.status, ZCCL_ERR_TIMEOUT);
            break;
        }

        // ---- split + remap + plane bytes: 8 elements per thread per step ----
        const uint8_t* src = sm.in[buf];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
            if (e0 >= L) continue;
            uint4 v = *reinterpret_cast<const uint4*>(src + 2 * e0);
            uint32_t keep = 0xFFu;
            if (e0 + 8 > valid) {
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
            // code bits: byte p of acc = plane p bits of the 8 elements
            uint32_t acc = sm.code_bits[(v.x >> 7) & 0xFF];
            acc |= sm.code_bits[(v.x >> 23) & 0xFF] << 1;
            acc |= sm.code_bits[(v.y >> 7) & 0xFF] << 2;
            acc |= sm.code_bits[(v.y >> 23) & 0xFF] << 3;
            acc |= sm.code_bits[(v.z >> 7) & 0xFF] << 4;
            acc |= sm.code_bits[(v.z >> 23) & 0xFF] << 5;
            acc |= sm.code_bits[(v.w >> 7) & 0xFF] << 6;
            acc |= sm.code_bits[(v.w >> 23) & 0xFF] << 7;
            acc &= keep * 0x010101u;
            uint8_t* planes = sm.blk + L + (e0 >> 3);
            planes[0] = (uint8_t)acc;
            planes[L / 8] = (uint8_t)(acc >> 8);
            planes[L / 4] = (uint8_t)(acc >> 16);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g((uint8_t*)d.out + kHeaderBytes + (uint64_t)cl * kBlockBytes, sm.blk, L * 11 / 8);
            bulk_commit();
        }

        // ---- escapes: words from the planes, chunk-local compaction ----
        uint32_t esc = 0;
        if (tid < (int)(L / 32)) {
            const uint32_t* pw = reinterpret_cast<const uint32_t*>(sm.blk + L);
            const uint32_t p0 = pw[tid], p1 = pw[L / 32 + tid], p2 = pw[L / 16 + tid];
            const uint32_t w0 = 32u * tid;
            const uint32_t vmask = w0 + 32 <= valid ? 0xFFFFFFFFu
                                   : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
            esc = ~(p0 | p1 | p2) & vmask;
        }
        uint32_t agg;
        const uint32_t excl = block_exclusive_scan<kThreads>((uint32_t)__popc(esc), sm.scan, &agg);
        uint8_t* dst = a.stage + (uint64_t)c * kChunk + excl;
        const uint16_t* x16 = reinterpret_cast<const uint16_t*>(src);
        uint32_t m = esc, j = 0;
        while (m) {
            const uint32_t b = __ffs(m) - 1;
            m &= m - 1;
            dst[j++] = (uint8_t)(x16[32u * tid + b] >> 7);
        }
        if (tid == 0) {
            a.counts[c] = agg;
            if (agg) atomicAdd(&a.totals[rstart[s] + cl / kRangeChunks], agg);
            bulk_wait_read0();
        }
        __syncthreads();
    }
    if (tid == 0) bulk_wait0();
    pdl_launch_dependents();
    // the last CTA: exclusive scan of the range totals within each segment
    if (arrive_last(a.ctrl, &sm.last) && fits) {
        const uint32_t R = (uint32_t)ranges64;
        cta_segmented_exclusive_scan<kThreads, 2>(
            a.totals, a.bases, R,
            [&](uint32_t r) { return rstart[find_segment(rstart, a.n_segs, r)] == r; }, sm.scan64, sm.scan_f);
        // leave the totals at zero for the next call
        for (uint32_t r = tid; r < R; r += kThreads) a.totals[r] = 0;
    }
}

// ============================================================================
// Kernel 2: scan counts, place escapes, finish streams
// ============================================================================
struct __align__(16) PlaceSmem {
    uint64_t scan64[kThreads / 32];
    uint32_t scan[kThreads / 32];
    uint32_t cnt[kRangeChunks];
    uint32_t excl[kRangeChunks];
};

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

__global__ void __launch_bounds__(kThreads) compress_place_kernel(const CompressArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    PlaceSmem& sm = *reinterpret_cast<PlaceSmem*>(smem_raw);
    uint32_t* ustart = reinterpret_cast<uint32_t*>(smem_raw + sizeof(PlaceSmem));
    uint32_t* rstart = ustart + a.n_segs + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_wait();  // counts, range bases and staged escapes of the blocks kernel
    uint64_t total_units, total_ranges;
    segment_table(a, ustart, rstart, sm.scan64, &total_units, &total_ranges);
    if (blockIdx.x == 0 && a.segs != nullptr) {
        for (uint32_t s = tid; s < a.n_segs; s += kThreads) {
            const uint32_t bad = segment_error(a.segs[s]);
            if (bad) {
                report(a.status, bad);
                a.out_bytes[s] = 0;
            }
        }
    }
    if (total_units > a.max_units || total_ranges > a.max_ranges) {
        if (blockIdx.x == 0 && tid == 0) report(a.status, ZCCL_ERR_INVALID_ARG);
        return;
    }
    // empty, valid segments: header only (CTA 0)
    if (blockIdx.x == 0) {
        for (uint32_t s = warp; s < a.n_segs; s += kThreads / 32) {
            const zccl_segment_t d = seg_get(a, s);
            if (d.n != 0 || (a.segs != nullptr && segment_error(d))) continue;
            write_header((uint8_t*)d.out, 0, 0, a.lut, lane);
            if (lane == 0) a.out_bytes[s] = kHeaderBytes;
        }
    }

    const uint32_t nr = (uint32_t)total_ranges;
    for (uint32_t r = blockIdx.x; r < nr; r += gridDim.x) {
        const uint32_t s = find_segment(rstart, a.n_segs, r);
        const zccl_segment_t d = seg_get(a, s);
        const uint32_t q = r - rstart[s];
        const uint32_t seg_units = (uint32_t)units_of(d.n);
        const uint32_t c0 = q * kRangeChunks;                       // first chunk, segment-local
        const uint32_t nch = min(kRangeChunks, seg_units - c0);
        const uint32_t g0 = ustart[s] + c0;                          // first chunk, global
        const uint32_t cnt = tid < (int)nch ? __ldcg(a.counts + g0 + tid) : 0u;
        uint32_t agg;
        const uint32_t ex = block_exclusive_scan<kThreads>(cnt, sm.scan, &agg);
        if (tid < (int)kRangeChunks) {
            sm.cnt[tid] = cnt;
            sm.excl[tid] = ex;
        }
        __syncthreads();
        const uint64_t P = __ldcg(a.bases + r);
        const uint64_t zp = zp_offset_of(d.n);
        uint8_t* out = (uint8_t*)d.out;
        // each warp moves 8 chunks' staged escapes: all word loads first
        // (one memory latency), then byte stores to the unaligned target
        constexpr int kPerWarp = kRangeChunks / (kThreads / 32);
        const uint32_t* stage32 = reinterpret_cast<const uint32_t*>(a.stage);
        uint32_t v[kPerWarp];
#pragma unroll
        for (int ii = 0; ii < kPerWarp; ++ii) {
            const uint32_t i = warp + 4 * ii;
            v[ii] = (i < nch && 4 * lane < sm.cnt[i]) ? __ldcg(stage32 + (uint64_t)(g0 + i) * (kChunk / 4) + lane)
                                                       : 0u;
        }
#pragma unroll
        for (int ii = 0; ii < kPerWarp; ++ii) {
            const uint32_t i = warp + 4 * ii;
            if (i >= nch) continue;
            const uint32_t cnt_i = sm.cnt[i];
            uint8_t* to = out + zp + P + sm.excl[i];
#pragma unroll
            for (uint32_t b = 0; b < 4; ++b)
                if (4 * lane + b < cnt_i) to[4 * lane + b] = (uint8_t)(v[ii] >> (8 * b));
            // escape-heavy chunks: the rest, 128 bytes per round
            for (uint32_t w = 32 + lane; 4 * w < cnt_i; w += 32) {
                const uint32_t x = __ldcg(stage32 + (uint64_t)(g0 + i) * (kChunk / 4) + w);
#pragma unroll
                for (uint32_t b = 0; b < 4; ++b)
                    if (4 * w + b < cnt_i) to[4 * w + b] = (uint8_t)(x >> (8 * b));
            }
        }
        if (c0 + nch == seg_units) {  // last range: header, zero padding, size
            const uint64_t n_esc = P + agg;
            const uint64_t pad_end = round_up(n_esc, 128);
            for (uint64_t b = n_esc + tid; b < pad_end; b += kThreads) out[zp + b] = 0;
            if (warp == 1) write_header(out, d.n, n_esc, a.lut, lane);
            if (tid == 0) a.out_bytes[s] = zp + pad_end;
        }
        __syncthreads();
    }
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

size_t compress_smem_bytes(uint32_t n_segs) { return sizeof(BlocksSmem) + 8ull * (n_segs + 1); }
static size_t place_smem_bytes(uint32_t n_segs) { return sizeof(PlaceSmem) + 8ull * (n_segs + 1); }

cudaError_t launch_compress(const CompressArgs& a, uint32_t grid_blocks, uint32_t grid_place, cudaStream_t stream)
{
    const size_t smem1 = compress_smem_bytes(a.n_segs), smem2 = place_smem_bytes(a.n_segs);
    cudaError_t e = cudaFuncSetAttribute(compress_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(compress_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
    if (e != cudaSuccess) return e;
    compress_blocks_kernel<<<grid_blocks, kThreads, smem1, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dependent(compress_place_kernel, grid_place, kThreads, smem2, stream, a);
}

int compress_ctas_per_sm(uint32_t n_segs) { return occupancy(compress_blocks_kernel, compress_smem_bytes(n_segs)); }
int place_ctas_per_sm(uint32_t n_segs) { return occupancy(compress_place_kernel, place_smem_bytes(n_segs)); }

}  // namespace zccl

// zccl_compress.cu -- compress kernel: split, remap, code planes, escape
// counts, single-pass scan and zero-point compaction, for one stream or for a
// batch of ragged segments in a single launch.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B (split
// into sign-mantissa and exponent bits; exponents in the top-7 LUT -> 3-bit
// codes 001..111, others -> zero-point code 000 + raw exponent in the
// zero-point array), 2.C (128-byte aligned chunk blocks; the 3-bit codes as
// three independent 1-bit arrays; asynchronous global->shared copies with
// double buffering) and 2.D (static/dynamic MoE parts -> batched segments).
//
// GB300 design.  A persistent grid of 128-thread CTAs takes 4096-element
// chunks by ticket.  Each chunk's 8 KB of BF16 arrives in shared memory by a
// TMA bulk copy (cp.async.bulk + mbarrier), double-buffered so the next
// chunk streams in while this one is coded.  Each thread codes 8 consecutive
// elements per step from one 16-byte shared load: byte permutes give the
// sign-mantissa bytes; a 256-entry shared table gives each exponent's three
// code bits pre-spread one byte apart, accumulated into one word whose bytes
// are the three plane bytes.  The coded block (sign-mantissa bytes + planes)
// is assembled in shared memory and leaves by one bulk store.  Escape counts
// come from popc over the plane words; a decoupled look-back (bounded waits)
// gives the chunk's zero-point offset, and the escapes are written straight
// to their compacted place: one pass over HBM, no escape scratch.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kInBytes = kChunk * 2;  // 8192

struct __align__(16) CompressSmem {
    uint8_t in[2][kInBytes];       // double-buffered BF16 input chunk
    uint8_t blk[kBlockBytes];      // coded block being assembled
    uint32_t code_bits[256];       // exponent -> b0 | b1 << 8 | b2 << 16
    uint64_t bar[2];               // one mbarrier per input buffer
    uint32_t scan[kThreads / 32];
    uint64_t scan64[kThreads / 32];
    uint64_t total_units;
    uint32_t ticket_next;
    uint32_t gen;
    uint32_t flag;
    uint32_t lb_status;
    uint64_t lb_prefix;
    uint32_t abort;
};

__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Why a batched segment descriptor cannot be compressed (0 = it can).
__device__ __forceinline__ uint32_t segment_error(const zccl_segment_t& d)
{
    if (d.n >= kMaxElems || ((uintptr_t)d.out & 15) || (d.n && ((uintptr_t)d.in & 15)))
        return ZCCL_ERR_INVALID_ARG;
    if (d.out_capacity < stream_bytes_of(d.n, d.n)) return ZCCL_ERR_BUFFER_TOO_SMALL;
    return 0;
}

// Segment of `unit`: largest s with seg_start[s] <= unit (seg_start has
// n_segs + 1 entries, non-decreasing).
__device__ __forceinline__ uint32_t find_segment(const uint32_t* seg_start, uint32_t n_segs, uint32_t unit)
{
    uint32_t lo = 0, hi = n_segs;  // answer in [lo, hi)
    while (hi - lo > 1) {
        uint32_t mid = (lo + hi) >> 1;
        if (seg_start[mid] <= unit) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void seg_get(const CompressArgs& a, uint32_t s, const uint16_t*& in, uint64_t& n,
                                        uint8_t*& out)
{
    if (a.segs == nullptr) {
        in = a.single.in;
        n = a.single.n;
        out = (uint8_t*)a.single.out;
    } else {
        zccl_segment_t d = a.segs[s];
        in = d.in;
        n = d.n;
        out = (uint8_t*)d.out;
    }
}

// Queue the bulk load of `unit` into buffer `buf` (thread 0 only).
__device__ __forceinline__ void issue_load(const CompressArgs& a, const uint32_t* seg_start, CompressSmem& sm,
                                           uint32_t unit, int buf)
{
    const uint32_t s = find_segment(seg_start, a.n_segs, unit);
    const uint16_t* in;
    uint64_t n;
    uint8_t* out;
    seg_get(a, s, in, n, out);
    const uint64_t c = unit - seg_start[s];
    const uint64_t first = c * kChunk;
    const uint32_t valid = (uint32_t)umin64(kChunk, n - first);
    const uint32_t bytes = (valid * 2) & ~15u;  // whole 16-byte pieces
    if (bytes) {
        mbar_arrive_expect_tx(&sm.bar[buf], bytes);
        bulk_g2s(sm.in[buf], in + first, bytes, &sm.bar[buf]);
    } else {
        mbar_arrive(&sm.bar[buf]);
    }
}

// Header of a finished stream (32 threads of one warp write 4 bytes each).
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

__global__ void __launch_bounds__(kThreads) compress_kernel(const CompressArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    CompressSmem& sm = *reinterpret_cast<CompressSmem*>(smem_raw);
    uint32_t* seg_start = reinterpret_cast<uint32_t*>(smem_raw + sizeof(CompressSmem));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- prologue: code table, segment table, barriers, generation ----
    for (int e = tid; e < 256; e += kThreads) {
        uint32_t c = 0;
#pragma unroll
        for (int r = 0; r < 7; ++r)
            if (a.lut[r] == e) c = r + 1;
        sm.code_bits[e] = (c & 1) | (((c >> 1) & 1) << 8) | (((c >> 2) & 1) << 16);
    }
    // units per segment (invalid segments get none), then an exclusive scan
    uint64_t running = 0;
    for (uint32_t base = 0; base < a.n_segs; base += kThreads) {
        const uint32_t s = base + tid;
        uint64_t units = 0;
        if (s < a.n_segs) {
            if (a.segs == nullptr) {
                units = units_of(a.single.n);
            } else {
                const zccl_segment_t d = a.segs[s];
                const uint32_t bad = segment_error(d);
                if (bad) {
                    if (blockIdx.x == 0) {
                        report(a.status, bad);
                        a.out_bytes[s] = 0;
                    }
                } else {
                    units = units_of(d.n);
                }
            }
        }
        uint64_t total;
        const uint64_t ex = block_exclusive_scan<kThreads, uint64_t>(units, sm.scan64, &total);
        if (s < a.n_segs) seg_start[s] = (uint32_t)(running + ex);  // used only if in range
        running += total;
    }
    if (tid == 0) {
        seg_start[a.n_segs] = (uint32_t)running;
        sm.total_units = running;
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
        sm.gen = *(volatile uint32_t*)&a.ctrl->gen;
        sm.abort = 0;
    }
    __syncthreads();
    const uint32_t tag = tag_of_gen(sm.gen);
    if (sm.total_units > a.max_units) {
        if (blockIdx.x == 0 && tid == 0) report(a.status, ZCCL_ERR_INVALID_ARG);
        finish_call(a.ctrl, a.flags, a.n_flag_words, sm.gen, &sm.flag);
        return;
    }
    const uint32_t total_units = (uint32_t)sm.total_units;
    // empty, valid segments: header only (CTA 0)
    if (blockIdx.x == 0) {
        for (uint32_t s = warp; s < a.n_segs; s += kThreads / 32) {
            if (seg_start[s + 1] != seg_start[s]) continue;
            const uint16_t* in;
            uint64_t n;
            uint8_t* out;
            seg_get(a, s, in, n, out);
            if (n != 0) continue;                                     // skipped: invalid
            if (a.segs != nullptr && segment_error(a.segs[s])) continue;  // skipped: invalid
            write_header(out, 0, 0, a.lut, lane);
            if (lane == 0) a.out_bytes[s] = kHeaderBytes;
        }
    }

    // ---- main loop over chunk tickets ----
    if (tid == 0) {
        const uint32_t t = atomicAdd(&a.ctrl->ticket, 1u);
        sm.ticket_next = t;
        if (t < total_units) issue_load(a, seg_start, sm, t, 0);
    }
    __syncthreads();
    uint32_t cur = sm.ticket_next;
    uint32_t k = 0;
    while (cur < total_units) {
        const int buf = k & 1;
        if (tid == 0) {
            const uint32_t t = atomicAdd(&a.ctrl->ticket, 1u);
            sm.ticket_next = t;
            if (t < total_units) issue_load(a, seg_start, sm, t, buf ^ 1);
        }
        const uint32_t s = find_segment(seg_start, a.n_segs, cur);
        const uint16_t* in;
        uint64_t n;
        uint8_t* out;
        seg_get(a, s, in, n, out);
        const uint32_t c = cur - seg_start[s];
        const uint64_t first = (uint64_t)c * kChunk;
        const uint32_t valid = (uint32_t)umin64(kChunk, n - first);
        const uint32_t L = slots_of(valid);

        if (!mbar_wait(&sm.bar[buf], (k >> 1) & 1)) atomicExch(&sm.abort, 1u);
        if (valid < kChunk) {  // tail: the last < 8 elements come by plain loads
            const uint32_t done = ((valid * 2) & ~15u) / 2;
            if (tid < (int)(valid - done))
                reinterpret_cast<uint16_t*>(sm.in[buf])[done + tid] = in[first + done + tid];
        }
        __syncthreads();
        if (sm.abort) {  // a bulk load never landed: poison this chunk and the prefetched one
            if (tid == 0) {
                report(a.status, ZCCL_ERR_TIMEOUT);
                st_release(&a.flags[cur], make_flag(kFlagPoison, tag, 0));
                if (sm.ticket_next < total_units)
                    st_release(&a.flags[sm.ticket_next], make_flag(kFlagPoison, tag, 0));
            }
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
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t m = ((keep >> (2 * q)) & 1 ? 0x0000FFFFu : 0u) |
                                       ((keep >> (2 * q + 1)) & 1 ? 0xFFFF0000u : 0u);
                    w[q] &= m;
                }
                v = make_uint4(w[0], w[1], w[2], w[3]);
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
            bulk_s2g(out + kHeaderBytes + (uint64_t)c * kBlockBytes, sm.blk, L * 11 / 8);
            bulk_commit();
        }

        // ---- escape words, counts, block scan ----
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

        // ---- zero-point offset of this chunk: decoupled look-back ----
        if (warp == 0) {
            uint64_t pre;
            const uint32_t st = lookback(a.flags, cur, seg_start[s], agg, tag, &pre);
            if (lane == 0) {
                sm.lb_status = st;
                sm.lb_prefix = pre;
            }
        }
        __syncthreads();
        if (sm.lb_status != ZCCL_OK) {
            if (tid == 0) report(a.status, sm.lb_status);
        } else {
            const uint64_t P = sm.lb_prefix;
            const uint64_t zp = zp_offset_of(n);
            // compacted escapes, element order
            uint8_t* dst = out + zp + P + excl;
            const uint16_t* x16 = reinterpret_cast<const uint16_t*>(src);
            uint32_t m = esc, j = 0;
            while (m) {
                const uint32_t b = __ffs(m) - 1;
                m &= m - 1;
                dst[j++] = (uint8_t)(x16[32u * tid + b] >> 7);
            }
            // last chunk of the segment: header, zero padding, size
            if (c + 1 == seg_start[s + 1] - seg_start[s]) {
                const uint64_t n_esc = P + agg;
                const uint64_t pad_end = round_up(n_esc, 128);
                for (uint64_t b = n_esc + tid; b < pad_end; b += kThreads) out[zp + b] = 0;
                if (warp == 1) write_header(out, n, n_esc, a.lut, lane);
                if (tid == 0) a.out_bytes[s] = zp + pad_end;
            }
        }
        if (tid == 0) bulk_wait_read0();
        __syncthreads();
        cur = sm.ticket_next;
        ++k;
    }
    if (tid == 0) bulk_wait0();
    // a buffer may still have a load in flight if the loop stopped early
    // (abort): wait for it, bounded, before the CTA's smem is released
    if (tid == 0 && cur < total_units && sm.ticket_next < total_units) {
        mbar_wait(&sm.bar[(k & 1) ^ 1], ((k + 1) >> 1) & 1);
    }
    finish_call(a.ctrl, a.flags, a.n_flag_words, sm.gen, &sm.flag);
}

}  // namespace

size_t compress_smem_bytes(uint32_t n_segs) { return sizeof(CompressSmem) + 4ull * (n_segs + 1); }

cudaError_t launch_compress(const CompressArgs& a, uint32_t grid, cudaStream_t stream)
{
    const size_t smem = compress_smem_bytes(a.n_segs);
    cudaError_t e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    compress_kernel<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
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

// zccl_decompress.cu -- decompress kernel: recount escapes from the code
// planes, single-pass scan (inverse of the encoder's), gather from the
// zero-point array, rebuild BF16.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B (a code
// 001..111 names a LUT exponent; code 000 takes the next entry of the
// zero-point array) and 2.C (128-byte aligned blocks, three 1-bit code
// arrays, asynchronous global->shared copies with double buffering).
//
// GB300 design.  Persistent 128-thread CTAs take 4096-element chunks by
// ticket; each chunk block (5632 bytes) arrives by a TMA bulk copy into one
// of two shared buffers.  popc over ~(p0|p1|p2) gives the chunk's escape
// count; a decoupled look-back gives its offset into the zero-point array;
// escaped exponents are scattered into a per-element shared array.  Each
// thread then rebuilds 8 consecutive elements: the three plane bytes are
// spread to nibble codes, one byte-permute per 4 elements looks the codes up
// in the LUT (held in two registers), a second permute makes the escape
// mask, and byte permutes interleave sign-mantissa and exponent bytes into
// BF16, stored with one 16-byte write.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;

struct __align__(16) DecompressSmem {
    uint8_t blk[2][kBlockBytes];  // double-buffered chunk blocks
    uint8_t expo[kChunk];         // escaped exponents at their element slot
    uint64_t bar[2];
    uint32_t scan[kThreads / 32];
    uint32_t ticket_next;
    uint32_t gen;
    uint32_t flag;
    uint32_t lb_status;
    uint32_t abort;
    uint32_t hdr_ok;
    uint32_t lut_lo, lut_hi;  // byte r+1 = exponent of code r+1; byte 0 = 0
    uint64_t lb_prefix;
    uint64_t n_esc;
};

__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// bit k of an 8-bit value -> bit 4k
__device__ __forceinline__ uint32_t spread_nibbles(uint32_t x)
{
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    return x;
}

__device__ __forceinline__ void issue_load(const DecompressArgs& a, DecompressSmem& sm, uint32_t unit, int buf)
{
    const uint32_t valid = (uint32_t)umin64(kChunk, a.n - (uint64_t)unit * kChunk);
    const uint32_t bytes = slots_of(valid) * 11 / 8;
    mbar_arrive_expect_tx(&sm.bar[buf], bytes);
    bulk_g2s(sm.blk[buf], a.in + kHeaderBytes + (uint64_t)unit * kBlockBytes, bytes, &sm.bar[buf]);
}

// Rebuilds 8 consecutive elements from a chunk block: sign-mantissa bytes,
// plane bytes pb0..pb2, LUT in two registers, escaped exponents `xe`.
__device__ __forceinline__ uint4 decode8(uint2 smb, uint32_t pb0, uint32_t pb1, uint32_t pb2, uint32_t lut_lo,
                                         uint32_t lut_hi, uint2 xe)
{
    const uint32_t N = spread_nibbles(pb0) | (spread_nibbles(pb1) << 1) | (spread_nibbles(pb2) << 2);
    uint32_t e_lo = __byte_perm(lut_lo, lut_hi, N);
    uint32_t e_hi = __byte_perm(lut_lo, lut_hi, N >> 16);
    const uint32_t m_lo = __byte_perm(0xFFu, 0u, N);  // 0xFF where code == 0
    const uint32_t m_hi = __byte_perm(0xFFu, 0u, N >> 16);
    e_lo = (e_lo & ~m_lo) | (xe.x & m_lo);
    e_hi = (e_hi & ~m_hi) | (xe.y & m_hi);
    const uint32_t lo_a = (smb.x & 0x7F7F7F7Fu) | ((e_lo << 7) & 0x80808080u);
    const uint32_t hi_a = (smb.x & 0x80808080u) | ((e_lo >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo_b = (smb.y & 0x7F7F7F7Fu) | ((e_hi << 7) & 0x80808080u);
    const uint32_t hi_b = (smb.y & 0x80808080u) | ((e_hi >> 1) & 0x7F7F7F7Fu);
    return make_uint4(__byte_perm(lo_a, hi_a, 0x5140), __byte_perm(lo_a, hi_a, 0x7362),
                      __byte_perm(lo_b, hi_b, 0x5140), __byte_perm(lo_b, hi_b, 0x7362));
}

__global__ void __launch_bounds__(kThreads) decompress_kernel(const DecompressArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    DecompressSmem& sm = *reinterpret_cast<DecompressSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t total_units = (uint32_t)units_of(a.n);

    if (tid == 0) {
        // header checks: magic, version, chunk size, n, zp_offset, sizes
        const uint32_t* h = reinterpret_cast<const uint32_t*>(a.in);
        const uint64_t hn = h[2] | ((uint64_t)h[3] << 32);
        const uint64_t n_esc = h[4] | ((uint64_t)h[5] << 32);
        const uint64_t zp = h[8] | ((uint64_t)h[9] << 32);
        bool ok = h[0] == kMagic && h[1] == (kVersion | (kLog2Chunk << 16)) && hn == a.n &&
                  zp == zp_offset_of(a.n) && n_esc <= a.n && zp + round_up(n_esc, 128) <= a.in_bytes;
        sm.hdr_ok = ok ? 1u : 0u;
        sm.n_esc = n_esc;
        sm.lut_lo = h[6] << 8;                     // codes 1..3 in bytes 1..3, byte 0 = 0
        sm.lut_hi = (h[6] >> 24) | (h[7] << 8);    // codes 4..7
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
        sm.gen = *(volatile uint32_t*)&a.ctrl->gen;
        sm.abort = 0;
    }
    __syncthreads();
    const uint32_t tag = tag_of_gen(sm.gen);
    if (!sm.hdr_ok) {
        if (blockIdx.x == 0 && tid == 0) report(a.status, ZCCL_ERR_CORRUPT_STREAM);
        finish_call(a.ctrl, a.flags, a.n_flag_words, sm.gen, &sm.flag);
        return;
    }
    const uint32_t lut_lo = sm.lut_lo, lut_hi = sm.lut_hi;
    const uint64_t n_esc = sm.n_esc;
    const uint8_t* zp_base = a.in + zp_offset_of(a.n);

    if (tid == 0) {
        const uint32_t t = atomicAdd(&a.ctrl->ticket, 1u);
        sm.ticket_next = t;
        if (t < total_units) issue_load(a, sm, t, 0);
    }
    __syncthreads();
    uint32_t cur = sm.ticket_next;
    uint32_t k = 0;
    while (cur < total_units) {
        const int buf = k & 1;
        if (tid == 0) {
            const uint32_t t = atomicAdd(&a.ctrl->ticket, 1u);
            sm.ticket_next = t;
            if (t < total_units) issue_load(a, sm, t, buf ^ 1);
        }
        const uint64_t first = (uint64_t)cur * kChunk;
        const uint32_t valid = (uint32_t)umin64(kChunk, a.n - first);
        const uint32_t L = slots_of(valid);
        if (!mbar_wait(&sm.bar[buf], (k >> 1) & 1)) atomicExch(&sm.abort, 1u);
        __syncthreads();
        if (sm.abort) {
            if (tid == 0) {
                report(a.status, ZCCL_ERR_TIMEOUT);
                st_release(&a.flags[cur], make_flag(kFlagPoison, tag, 0));
                if (sm.ticket_next < total_units)
                    st_release(&a.flags[sm.ticket_next], make_flag(kFlagPoison, tag, 0));
            }
            break;
        }
        const uint8_t* blk = sm.blk[buf];

        // ---- escape words from the planes, counts, block scan ----
        uint32_t esc = 0;
        if (tid < (int)(L / 32)) {
            const uint32_t* pw = reinterpret_cast<const uint32_t*>(blk + L);
            const uint32_t p0 = pw[tid], p1 = pw[L / 32 + tid], p2 = pw[L / 16 + tid];
            const uint32_t w0 = 32u * tid;
            const uint32_t vmask = w0 + 32 <= valid ? 0xFFFFFFFFu
                                   : (w0 >= valid ? 0u : ((1u << (valid - w0)) - 1u));
            esc = ~(p0 | p1 | p2) & vmask;
        }
        uint32_t agg;
        const uint32_t excl = block_exclusive_scan<kThreads>((uint32_t)__popc(esc), sm.scan, &agg);
        if (warp == 0) {
            uint64_t pre;
            const uint32_t st = lookback(a.flags, cur, 0, agg, tag, &pre);
            if (lane == 0) {
                sm.lb_status = st;
                sm.lb_prefix = pre;
            }
        }
        __syncthreads();
        bool ok = sm.lb_status == ZCCL_OK;
        if (!ok) {
            if (tid == 0) report(a.status, sm.lb_status);
        } else {
            const uint64_t P = sm.lb_prefix;
            const bool last = cur + 1 == total_units;
            if (P + agg > n_esc || (last && P + agg != n_esc)) {
                if (tid == 0) report(a.status, ZCCL_ERR_CORRUPT_STREAM);
                ok = false;
            } else {
                const uint8_t* src = zp_base + P + excl;
                uint32_t m = esc, j = 0;
                while (m) {
                    const uint32_t b = __ffs(m) - 1;
                    m &= m - 1;
                    sm.expo[32u * tid + b] = src[j++];
                }
            }
        }
        __syncthreads();
        if (ok) {
            uint16_t* dst = a.out + first;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
                if (e0 >= valid) continue;
                const uint2 smb = *reinterpret_cast<const uint2*>(blk + e0);
                const uint32_t pb0 = blk[L + (e0 >> 3)];
                const uint32_t pb1 = blk[L + L / 8 + (e0 >> 3)];
                const uint32_t pb2 = blk[L + L / 4 + (e0 >> 3)];
                const uint2 xe = *reinterpret_cast<const uint2*>(sm.expo + e0);
                const uint4 o = decode8(smb, pb0, pb1, pb2, lut_lo, lut_hi, xe);
                if (e0 + 8 <= valid) {
                    *reinterpret_cast<uint4*>(dst + e0) = o;
                } else {
                    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
                    for (uint32_t q = 0; q < valid - e0; ++q)
                        dst[e0 + q] = (uint16_t)(w[q >> 1] >> (16 * (q & 1)));
                }
            }
        }
        __syncthreads();
        cur = sm.ticket_next;
        ++k;
    }
    if (tid == 0 && cur < total_units && sm.ticket_next < total_units) {
        mbar_wait(&sm.bar[(k & 1) ^ 1], ((k + 1) >> 1) & 1);
    }
    finish_call(a.ctrl, a.flags, a.n_flag_words, sm.gen, &sm.flag);
}

}  // namespace

cudaError_t launch_decompress(const DecompressArgs& a, uint32_t grid, cudaStream_t stream)
{
    const size_t smem = sizeof(DecompressSmem);
    cudaError_t e = cudaFuncSetAttribute(decompress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    decompress_kernel<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

int decompress_ctas_per_sm()
{
    int blocks = 0;
    const size_t smem = sizeof(DecompressSmem);
    if (cudaFuncSetAttribute(decompress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, decompress_kernel, kThreads, smem) != cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

}  // namespace zccl

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
// GB300 design.  A CTA takes a 4096-element chunk by ticket and walks its S
// shard blocks in order through a 3-stage ring of shared buffers filled by
// TMA bulk copies (two steps in flight while one decodes).  For each shard
// block it counts escapes from the planes, runs that shard's decoupled
// look-back (one flag array per shard), gathers the shard's escapes and
// decodes 32 elements per thread straight into fp32 accumulators held in
// registers; after the last shard it rounds and stores 16-byte vectors.  The
// compressed shards are read once and the BF16 result written once.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;

struct __align__(16) ReduceSmem {
    uint8_t blk[kStages][kBlockBytes];
    uint8_t expo[kChunk];
    uint64_t bar[kStages];
    uint32_t stage_unit[kStages];
    uint32_t stage_shard[kStages];
    uint32_t scan[kThreads / 32];
    uint32_t gen;
    uint32_t flag;
    uint32_t lb_status;
    uint32_t abort;
    uint32_t load_unit;
    uint32_t ended;
    uint64_t lb_prefix;
};
// followed by per-shard tables: const uint8_t* base[S]; uint64_t n_esc[S]; uint32_t lut[S][2]

__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint32_t spread_nibbles(uint32_t x)
{
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    return x;
}

__device__ __forceinline__ uint4 decode8(uint2 smb, uint32_t pb0, uint32_t pb1, uint32_t pb2, uint32_t lut_lo,
                                         uint32_t lut_hi, uint2 xe)
{
    const uint32_t N = spread_nibbles(pb0) | (spread_nibbles(pb1) << 1) | (spread_nibbles(pb2) << 2);
    uint32_t e_lo = __byte_perm(lut_lo, lut_hi, N);
    uint32_t e_hi = __byte_perm(lut_lo, lut_hi, N >> 16);
    const uint32_t m_lo = __byte_perm(0xFFu, 0u, N);
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

// fp32 -> BF16, round to nearest, ties to even; NaN -> 0x7FC0.
__device__ __forceinline__ uint32_t rne_bf16(float f)
{
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

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

// Thread 0: queue the load of step j (unit = j / S-th ticket, shard j % S).
__device__ __forceinline__ void issue_step(const ReduceArgs& a, ReduceSmem& sm, const ShardTables& t,
                                           uint32_t j, uint32_t total_units)
{
    const int stage = j % kStages;
    const uint32_t s = j % a.S;
    if (s == 0 && !sm.ended) {
        sm.load_unit = atomicAdd(&a.ctrl->ticket, 1u);
        if (sm.load_unit >= total_units) sm.ended = 1;
    }
    if (sm.ended) {
        sm.stage_unit[stage] = 0xFFFFFFFFu;
        return;
    }
    const uint32_t unit = sm.load_unit;
    sm.stage_unit[stage] = unit;
    sm.stage_shard[stage] = s;
    const uint32_t valid = (uint32_t)umin64(kChunk, a.n - (uint64_t)unit * kChunk);
    const uint32_t bytes = slots_of(valid) * 11 / 8;
    mbar_arrive_expect_tx(&sm.bar[stage], bytes);
    bulk_g2s(sm.blk[stage], t.base[s] + kHeaderBytes + (uint64_t)unit * kBlockBytes, bytes, &sm.bar[stage]);
}

__global__ void __launch_bounds__(kThreads) reduce_kernel(const ReduceArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    ReduceSmem& sm = *reinterpret_cast<ReduceSmem*>(smem_raw);
    const ShardTables t = shard_tables(smem_raw, a.S);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t total_units = (uint32_t)units_of(a.n);

    // ---- prologue: validate every shard's header, keep what decoding needs ----
    bool ok = true;
    for (uint32_t s = tid; s < a.S; s += kThreads) {
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
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&sm.bar[i], 1);
        fence_mbar_init();
        sm.gen = *(volatile uint32_t*)&a.ctrl->gen;
        sm.abort = 0;
        sm.ended = 0;
    }
    const bool all_ok = __syncthreads_and(ok) != 0;
    const uint32_t tag = tag_of_gen(sm.gen);
    if (!all_ok) {
        if (blockIdx.x == 0 && tid == 0) report(a.status, ZCCL_ERR_CORRUPT_STREAM);
        finish_call(a.ctrl, a.flags, a.n_flag_words, sm.gen, &sm.flag);
        return;
    }

    if (tid == 0)
        for (uint32_t j = 0; j + 1 < kStages; ++j) issue_step(a, sm, t, j, total_units);
    __syncthreads();

    float acc[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) acc[q] = 0.0f;

    uint32_t k = 0;
    for (;; ++k) {
        const int stage = k % kStages;
        if (tid == 0) issue_step(a, sm, t, k + kStages - 1, total_units);
        const uint32_t unit = sm.stage_unit[stage];
        if (unit >= total_units) break;
        const uint32_t s = sm.stage_shard[stage];
        const uint64_t first = (uint64_t)unit * kChunk;
        const uint32_t valid = (uint32_t)umin64(kChunk, a.n - first);
        const uint32_t L = slots_of(valid);
        if (!mbar_wait(&sm.bar[stage], (k / kStages) & 1)) atomicExch(&sm.abort, 1u);
        __syncthreads();
        if (sm.abort) {
            if (tid == 0) {
                report(a.status, ZCCL_ERR_TIMEOUT);
                st_release(&a.flags[(uint64_t)s * total_units + unit], make_flag(kFlagPoison, tag, 0));
            }
            break;
        }
        const uint8_t* blk = sm.blk[stage];

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
            const uint32_t st = lookback(a.flags + (uint64_t)s * total_units, unit, 0, agg, tag, &pre);
            if (lane == 0) {
                sm.lb_status = st;
                sm.lb_prefix = pre;
            }
        }
        __syncthreads();
        bool good = sm.lb_status == ZCCL_OK;
        if (!good) {
            if (tid == 0) report(a.status, sm.lb_status);
        } else {
            const uint64_t P = sm.lb_prefix;
            const uint64_t n_esc = t.n_esc[s];
            if (P + agg > n_esc || (unit + 1 == total_units && P + agg != n_esc)) {
                if (tid == 0) report(a.status, ZCCL_ERR_CORRUPT_STREAM);
                good = false;
            } else {
                const uint8_t* src = t.base[s] + zp_offset_of(a.n) + P + excl;
                uint32_t m = esc, j = 0;
                while (m) {
                    const uint32_t b = __ffs(m) - 1;
                    m &= m - 1;
                    sm.expo[32u * tid + b] = src[j++];
                }
            }
        }
        __syncthreads();
        const uint32_t lut_lo = t.lut[2 * s], lut_hi = t.lut[2 * s + 1];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
            if (e0 < L) {
                const uint2 smb = *reinterpret_cast<const uint2*>(blk + e0);
                const uint32_t pb0 = blk[L + (e0 >> 3)];
                const uint32_t pb1 = blk[L + L / 8 + (e0 >> 3)];
                const uint32_t pb2 = blk[L + L / 4 + (e0 >> 3)];
                const uint2 xe = *reinterpret_cast<const uint2*>(sm.expo + e0);
                const uint4 o = decode8(smb, pb0, pb1, pb2, lut_lo, lut_hi, xe);
                const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float f0 = __uint_as_float(w[q] << 16);
                    const float f1 = __uint_as_float(w[q] & 0xFFFF0000u);
                    if (s == 0) {
                        acc[8 * i + 2 * q] = f0;
                        acc[8 * i + 2 * q + 1] = f1;
                    } else {
                        acc[8 * i + 2 * q] = __fadd_rn(acc[8 * i + 2 * q], f0);
                        acc[8 * i + 2 * q + 1] = __fadd_rn(acc[8 * i + 2 * q + 1], f1);
                    }
                }
            }
        }
        if (s + 1 == a.S) {
            uint16_t* dst = a.out + first;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t e0 = 1024u * warp + 256u * i + 8u * lane;
                if (e0 >= valid) continue;
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = rne_bf16(acc[8 * i + 2 * q]) | (rne_bf16(acc[8 * i + 2 * q + 1]) << 16);
                if (e0 + 8 <= valid) {
                    *reinterpret_cast<uint4*>(dst + e0) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    for (uint32_t q = 0; q < valid - e0; ++q)
                        dst[e0 + q] = (uint16_t)(w[q >> 1] >> (16 * (q & 1)));
                }
            }
        }
        __syncthreads();
    }
    // loads still in flight (steps issued but not consumed): wait, bounded
    if (tid == 0) {
        for (uint32_t j = k + 1; j < k + kStages; ++j) {
            if (sm.stage_unit[j % kStages] < total_units) mbar_wait(&sm.bar[j % kStages], (j / kStages) & 1);
        }
    }
    finish_call(a.ctrl, a.flags, a.n_flag_words, sm.gen, &sm.flag);
}

}  // namespace

static size_t reduce_smem_bytes(uint32_t S) { return sizeof(ReduceSmem) + 24ull * S; }

cudaError_t launch_reduce(const ReduceArgs& a, uint32_t grid, cudaStream_t stream)
{
    const size_t smem = reduce_smem_bytes(a.S);
    cudaError_t e = cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    reduce_kernel<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

int reduce_ctas_per_sm(uint32_t S)
{
    int blocks = 0;
    const size_t smem = reduce_smem_bytes(S);
    if (cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, reduce_kernel, kThreads, smem) != cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

}  // namespace zccl

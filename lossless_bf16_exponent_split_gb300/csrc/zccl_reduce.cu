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
// GB300 design: the escape scan kernel (zccl_decompress.cu) first computes,
// for every shard and chunk, the chunk's zero-point offset (range base +
// prefix within the range) and the escapes before each quarter of the chunk
// (1024 slots).  Then, started by programmatic dependent launch,
// reduce_kernel hands each warp one chunk quarter at a time: the four warps
// of a CTA take the four quarters of the CTA's chunks (static stride over
// the chunks).  A warp walks the S shards of its quarter in order through
// its own 3-stage ring of shared buffers, which its lanes fill themselves
// with 16-byte asynchronous copies (cp.async): each lane the 32
// sign-mantissa bytes it decodes, 24 lanes the quarter's 128 bytes of each
// code plane, and as many lanes as needed the 16-byte aligned cover of the
// quarter's run of the zero-point array.  A step waits for its own copies
// (cp.async.wait_group) and then for the warp's (a warp barrier).  No warp
// ever waits for another, and no single thread issues copies for others.
// Every per-step address and check (the step's shard and chunk, its source
// bytes, its zero-point offset, count and cover, the bounds checks) is
// computed ahead by the warp's lanes, one step each, 16 steps at a time,
// into a 32-step ring in shared memory: a step's copy issue is two shared
// loads and per-lane constant offsets.
// Lane l owns slots [32 l, 32 l + 32) of the quarter, i.e. one word of each
// code plane: after a warp scan of the escape counts it places its own
// escaped exponents, then decodes its 32 elements straight into fp32 sums
// held in registers.  After the last shard it rounds and stores them.
// Every compressed byte is read once and the BF16 result written once.
//
// Shared-memory accesses are laid out so that no bank is hit twice by one
// instruction: a lane's 32 sign-mantissa bytes are read as two 16-byte
// halves in an order that alternates with bit 2 of the lane, and its
// escaped exponents are stored in 8-byte groups whose order is XOR-swizzled
// with bits 2..3 of the lane.  The code-plane words are read one per lane.
//
// The fold starts every chunk from -0.0: -0.0 + x == x exactly for every
// fp32 x (including +0, -0, subnormals, infinities and NaN), so every shard,
// the first included, is one add and no step needs a separate first form.
// The adds widen BF16 to fp32 inside the add instruction (exact), so a
// packed pair of BF16 values feeds two adds directly.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_decode.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr uint32_t kQuarter = kChunk / 4;          // slots of one warp's share of a chunk
constexpr uint32_t kStageBytes = 2 * kQuarter;     // a quarter of plain BF16, or its block part + zero points
constexpr uint32_t kPlaneOff = kQuarter;           // after the sign-mantissa bytes: 3 planes of 128 bytes
constexpr uint32_t kPlaneBytes = kQuarter / 8;
constexpr uint32_t kZpOff = kQuarter + 3 * kPlaneBytes;
constexpr uint32_t kZpCap = 512;                   // one 16-byte copy per lane: the cover of up to 482 escapes
// Shared memory (about 35 KB) admits 6 CTAs per SM; registers are capped
// to match.
constexpr int kCtasPerSm = 6;
static_assert(kZpOff % 16 == 0 && kZpOff + kZpCap <= kStageBytes, "the zero-point cover fits the stage");
// The step window: a ring of kWin steps per warp, refilled kWinLoad at a time.
constexpr uint32_t kWin = 32, kWinLoad = 16;
// A step's info word: the escape count of the quarter (bits 0..12), the
// bytes of its 16-byte aligned zero-point cover when that fits the stage
// (bits 16..26; else 0), whether it does (bit 30), whether the offsets
// passed the bounds checks (bit 31); bit 29 marks a plain BF16 step.
constexpr uint32_t kInfoCount = 0x1FFFu, kInfoInStage = 1u << 30, kInfoOk = 1u << 31, kInfoPlain = 1u << 29;
__device__ __forceinline__ uint32_t info_cover(uint32_t info) { return (info >> 16) & 0x7FFu; }

struct __align__(128) ReduceSmem {
    uint8_t stage[kWarps][kStages][kStageBytes];
    uint8_t xe[kWarps][kQuarter];  // each lane's escaped exponents (rotated), 32 bytes
    uint32_t spread[3][256];       // spread_nibbles(b) << p, p = plane
    // Per warp, a ring of kWin steps (two halves of kWinLoad): each step's
    // copy sources and checks, computed ahead by the warp's lanes, one step
    // each (load_window).  wptr: the quarter's first source byte (a stream
    // step: its sign-mantissa bytes; a plain step: its BF16) and the first
    // byte of its zero-point run; winfo: a stream step's plane size L / 8
    // (a plain step: its valid slots) and the info word (kInfo*).
    uint64_t wptr[kWarps][kWin][2];
    uint32_t winfo[kWarps][kWin][2];
    uint32_t last;
};
// followed by per-shard tables: blk[S], zpa[S], n_esc[S] (8 bytes each), lut[S] (uint2)

// Per shard: where its chunk blocks and its zero-point array start, its
// escape count, and its LUT with every exponent rotated right by one bit
// (entry c <-> code c; entry 0, code 000, unused).
struct ShardTables {
    const uint8_t** blk;
    const uint8_t** zpa;
    uint64_t* n_esc;
    uint2* lut;
};

__device__ __forceinline__ ShardTables shard_tables(uint8_t* smem_raw, uint32_t S)
{
    ShardTables t;
    uint8_t* p = smem_raw + sizeof(ReduceSmem);
    t.blk = reinterpret_cast<const uint8_t**>(p);
    t.zpa = reinterpret_cast<const uint8_t**>(p + 8ull * S);
    t.n_esc = reinterpret_cast<uint64_t*>(p + 16ull * S);
    t.lut = reinterpret_cast<uint2*>(p + 24ull * S);
    return t;
}

// Exponent bytes are held rotated right by one bit: bit 7 = exponent bit 0,
// bits 0..6 = exponent >> 1 -- the low and high byte of a BF16 value then
// each take one masked merge with the sign-mantissa byte.
//
// One exponent byte e rotated, in the low byte only (bits above it are
// garbage), for a byte store: e * 257 = e | e << 8 for e < 256, and a shift
// right by one brings bit 0 of the low copy under bit 7.  One multiply-add
// and one shift.
__device__ __forceinline__ uint32_t rot_exp_lo8(uint32_t e) { return (e * 257u) >> 1; }
__device__ __forceinline__ uint32_t rot_exp4(uint32_t w) { return ((w >> 1) & 0x7F7F7F7Fu) | ((w << 7) & 0x80808080u); }

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

// acc += the two BF16 values packed in w (low half to .x, high half to
// .y): each an fp32 add of the exactly widened BF16 value, rounded to
// nearest even, no flush to zero.
__device__ __forceinline__ void add_bf16x2(float2& acc, uint32_t w)
{
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n add.rn.f32.bf16 %0, lo, %0;\n add.rn.f32.bf16 %1, hi, %1;\n}"
        : "+f"(acc.x), "+f"(acc.y)
        : "r"(w));
}

// Adds 8 BF16 values (packed in pairs) to four fp32 pairs.
__device__ __forceinline__ void add8(float2* acc, uint4 o)
{
    add_bf16x2(acc[0], o.x);
    add_bf16x2(acc[1], o.y);
    add_bf16x2(acc[2], o.z);
    add_bf16x2(acc[3], o.w);
}

// Two fp32 sums -> a packed pair of BF16 values (lo in the low half), each
// rounded to nearest, ties to even, by the conversion instruction.  A NaN
// comes out as some NaN; canonical_nan makes it 0x7FC0.
__device__ __forceinline__ uint32_t pack_rne(float lo, float hi)
{
    uint32_t w;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
    return w;
}
// Bit 15 (31) set where the low (high) half of a BF16 pair is a NaN:
// |v| > 0x7F80 in each half, by one add that cannot carry across halves.
__device__ __forceinline__ uint32_t nan_halves(uint32_t w) { return ((w & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u; }
__device__ __forceinline__ uint32_t canonical_nan(uint32_t w)
{
    const uint32_t m = ((nan_halves(w) >> 15) & 0x00010001u) * 0xFFFFu;
    return (w & ~m) | (0x7FC07FC0u & m);
}

// Decodes 8 elements and adds them to four fp32 pairs: N their code
// nibbles, smb their sign-mantissa bytes, xe their escaped exponents
// (rotated; bytes of other elements are ignored), lut the rotated LUT.
__device__ __forceinline__ void decode_add8(float2* acc, uint32_t N, uint2 smb, uint2 lut, uint2 xe)
{
    uint32_t e_lo = __byte_perm(lut.x, lut.y, N);      // nibble k of N selects byte k
    uint32_t e_hi = __byte_perm(lut.x, lut.y, N >> 16);
    const uint32_t m_lo = __byte_perm(0xFFu, 0u, N);   // 0xFF where the code is 000
    const uint32_t m_hi = __byte_perm(0xFFu, 0u, N >> 16);
    e_lo = (e_lo & ~m_lo) | (xe.x & m_lo);
    e_hi = (e_hi & ~m_hi) | (xe.y & m_hi);
    // low byte = exponent bit 0 << 7 | mantissa; high byte = sign << 7 | exponent >> 1
    const uint32_t lo_a = (e_lo & 0x80808080u) | (smb.x & 0x7F7F7F7Fu);
    const uint32_t hi_a = (smb.x & 0x80808080u) | (e_lo & 0x7F7F7F7Fu);
    const uint32_t lo_b = (e_hi & 0x80808080u) | (smb.y & 0x7F7F7F7Fu);
    const uint32_t hi_b = (smb.y & 0x80808080u) | (e_hi & 0x7F7F7F7Fu);
    add_bf16x2(acc[0], __byte_perm(lo_a, hi_a, 0x5140));
    add_bf16x2(acc[1], __byte_perm(lo_a, hi_a, 0x7362));
    add_bf16x2(acc[2], __byte_perm(lo_b, hi_b, 0x5140));
    add_bf16x2(acc[3], __byte_perm(lo_b, hi_b, 0x7362));
}

// One warp: the window entries of its steps w .. w + kWinLoad - 1 (lane i:
// step w + i), into half (w / kWinLoad) & 1 of its ring.  All the per-step
// address arithmetic and bounds checks happen here, a step per lane; the
// loads are waited for here, once per kWinLoad steps.
template <bool kPlain>
__device__ __forceinline__ void load_window(const ReduceArgs& a, ReduceSmem& sm, const ShardTables& t, uint32_t w,
                                            uint32_t steps)
{
    const uint32_t lane = threadIdx.x & 31, q = threadIdx.x >> 5, step = w + lane;
    if (lane >= kWinLoad) return;
    const uint32_t total = (uint32_t)units_of(a.n);
    const uint32_t Q = steps_per_chunk<kPlain>(a);
    uint64_t src = 0, zsrc = 0;
    uint32_t l8 = 0, info = 0;
    if (step < steps) {
        const uint32_t k = step / Q, sq = step - k * Q;
        const uint64_t c = blockIdx.x + (uint64_t)k * gridDim.x;
        const uint32_t valid = (uint32_t)min((uint64_t)kChunk, a.n - c * kChunk);
        uint32_t s = 0;
        const uint32_t kind = step_kind<kPlain>(a, sq, &s);
        if (kind == kStepStream) {
            const uint32_t L = slots_of(valid);
            const uint32_t rps = (total + kRangeChunks - 1) / kRangeChunks;
            const uint64_t qi = __ldcg(a.qinfo + (uint64_t)s * total + c);
            const uint32_t before = quarter_before(qi, q);
            const uint64_t zq = __ldcg(a.bases + (uint64_t)s * rps + c / kRangeChunks) +
                                __ldcg(a.local_off + (uint64_t)s * total + c) + before;
            const uint32_t cnt = quarter_end(qi, q) - before;
            src = reinterpret_cast<uint64_t>(t.blk[s] + c * kBlockBytes + q * kQuarter);
            l8 = L / 8;
            if (cnt <= kQuarter && zq + cnt <= t.n_esc[s]) {
                zsrc = reinterpret_cast<uint64_t>(t.zpa[s] + zq);
                const uint32_t cover = (((uint32_t)zsrc & 15u) + cnt + 15u) & ~15u;
                info = cnt | kInfoOk | (cover <= kZpCap ? (cover << 16) | kInfoInStage : 0u);
            }
        } else {
            const uint16_t* base = kind == kStepLocal ? a.local : a.out;
            src = reinterpret_cast<uint64_t>(base + c * kChunk + q * kQuarter);
            l8 = min(kQuarter, valid - q * kQuarter);
            info = kInfoPlain;
        }
    }
    const uint32_t e = ((w / kWinLoad) & 1) * kWinLoad + lane;
    sts_u64(smem_addr(&sm.wptr[q][e][0]), src);
    sts_u64(smem_addr(&sm.wptr[q][e][1]), zsrc);
    sts_u32(smem_addr(&sm.winfo[q][e][0]), l8);
    sts_u32(smem_addr(&sm.winfo[q][e][1]), info);
}

// One warp: its quarter q of the CTA's chunks blockIdx.x + k * gridDim.x,
// each over its steps in order.  The fp32 sums are kept as pairs.
template <bool kPlain>
__device__ __forceinline__ void reduce_quarters(const ReduceArgs& a, ReduceSmem& sm, const ShardTables& t)
{
    const uint32_t lane = threadIdx.x & 31, q = threadIdx.x >> 5;
    const uint32_t total = (uint32_t)units_of(a.n);
    const uint32_t Q = steps_per_chunk<kPlain>(a);
    const uint32_t G = gridDim.x;
    const uint32_t tab = smem_addr(t.blk);
    const uint32_t S = a.S;
    auto unit_valid = [&](uint32_t k) -> uint32_t {
        return (uint32_t)min((uint64_t)kChunk, a.n - (blockIdx.x + (uint64_t)k * G) * kChunk);
    };
    // this warp's chunks; the tail chunk may have no slots in quarter q
    uint32_t units = 0;
    if (blockIdx.x < total) {
        units = (total - 1 - blockIdx.x) / G + 1;
        if (q * kQuarter >= slots_of(unit_valid(units - 1))) --units;
    }
    const uint32_t steps = units * Q;
    const uint32_t stage0 = smem_addr(sm.stage[q][0]);

    load_window<kPlain>(a, sm, t, 0, steps);
    load_window<kPlain>(a, sm, t, kWinLoad, steps);
    __syncwarp();

    // lane constants of the copies: this lane's piece of the planes (lanes
    // 0..23: 16 bytes of plane lane / 8), at src + (8 + lane / 8) * L / 8 +
    // 16 (lane % 8) - 896 q from the quarter's first sign-mantissa byte
    const uint32_t pmul = 8 + (lane >> 3);
    const uint32_t pconst = 16 * (lane & 7) - (kQuarter - kPlaneBytes) * q;
    const uint32_t wp0 = smem_addr(&sm.wptr[q][0][0]), wi0 = smem_addr(&sm.winfo[q][0][0]);

    // Issue cursor: step ij into stage ist.  Every lane copies; each step is
    // one cp.async group of every lane (empty past the last step, so that
    // the group count stays uniform).
    uint32_t ij = 0, ist = 0;
    auto issue = [&]() {
        if (ij < steps) {
            // the next half of the window: it held steps all consumed by now
            if ((ij & (kWinLoad - 1)) == kWinLoad / 2 && ij >= kWinLoad) {
                load_window<kPlain>(a, sm, t, (ij & ~(kWinLoad - 1)) + kWinLoad, steps);
                __syncwarp();
            }
            const uint32_t e = ij & (kWin - 1);
            const uint4 wp = lds_u128(wp0 + 16 * e);
            const uint2 wi = lds_u64(wi0 + 8 * e);
            const uint8_t* src = reinterpret_cast<const uint8_t*>(((uint64_t)wp.y << 32) | wp.x);
            const uint32_t dst = stage0 + ist * kStageBytes;
            if (kPlain && (wi.y & kInfoPlain)) {  // plain BF16: the lane's whole 16-byte pieces, the rest by plain loads
#pragma unroll
                for (uint32_t k = 0; k < 4; ++k) {
                    const uint32_t e0 = 32 * lane + 8 * k;  // the piece's first element
                    if (e0 + 8 <= wi.x) cp_async16(dst + 2 * e0, src + 2 * e0);
                }
            } else {
                // the lane's sign-mantissa bytes
                cp_async16(dst + 32 * lane, src + 32 * lane);
                cp_async16(dst + 32 * lane + 16, src + 32 * lane + 16);
                if (lane < 24) cp_async16(dst + kPlaneOff + 16 * lane, src + (pmul * wi.x + pconst));
                // the quarter's zero points: its 16-byte aligned cover, one piece per lane
                const uint64_t z = ((uint64_t)wp.w << 32) | wp.z;
                if (16 * lane < info_cover(wi.y))
                    cp_async16(dst + kZpOff + 16 * lane, reinterpret_cast<const uint8_t*>((z & ~15ull) + 16 * lane));
            }
            ++ij;
            if (++ist == kStages) ist = 0;
        }
        cp_async_commit();
    };
    for (int i = 0; i + 1 < kStages; ++i) issue();

    // lane constants of the conflict-free layouts
    const uint32_t h = (lane >> 2) & 1;            // which 16-byte half of its bytes the lane reads first
    const uint32_t x = (2 * h) ^ (lane >> 2 & 3);  // processing group i <-> swizzled escape group i ^ x
    const uint32_t xa = smem_addr(sm.xe[q] + 32 * lane);  // the lane's escaped exponents
    const uint32_t xsw = 8 * (lane >> 2 & 3);      // escape byte of element b sits at xa + (b ^ xsw)
    const uint32_t sp = smem_addr(sm.spread[0]);
    const uint32_t lut0 = tab + 24 * S;

    float2 acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = make_float2(-0.0f, -0.0f);

    uint32_t cst = 0, j = 0;  // consume cursor: stage, step
    for (uint32_t k = 0; k < units; ++k) {
        const uint64_t c = blockIdx.x + (uint64_t)k * G;
        const uint32_t valid = unit_valid(k);
        const uint32_t vq = min(kQuarter, valid - q * kQuarter);
        const uint32_t e0 = 32 * lane;
        const uint32_t vmask = e0 + 32 <= vq ? 0xFFFFFFFFu : (e0 >= vq ? 0u : ((1u << (vq - e0)) - 1u));
        for (uint32_t sq = 0; sq < Q; ++sq, ++j) {
            // every lane is past step j - 1: refill its stage with step j + kStages - 1
            __syncwarp();
            issue();
            cp_async_wait<kStages - 1>();  // this lane's copies of step j
            __syncwarp();                  // ... and every lane's
            const uint32_t stg = stage0 + cst * kStageBytes;
            uint32_t s = 0;
            const uint32_t kind = step_kind<kPlain>(a, sq, &s);
            if (kind == kStepStream) {
                const uint32_t P0 = lds_u32(stg + kPlaneOff + 4 * lane);
                const uint32_t P1 = lds_u32(stg + kPlaneOff + kPlaneBytes + 4 * lane);
                const uint32_t P2 = lds_u32(stg + kPlaneOff + 2 * kPlaneBytes + 4 * lane);
                const uint4 A = lds_u128(stg + 32 * lane + 16 * h);
                const uint4 B = lds_u128(stg + 32 * lane + 16 * (h ^ 1));
                const uint32_t esc = ~(P0 | P1 | P2) & vmask;
                const uint32_t ne = __popc(esc);
                uint32_t incl = ne;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= (uint32_t)o) incl += y;
                }
                const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
                const uint32_t e = j & (kWin - 1);
                const uint32_t info = lds_u32(wi0 + 8 * e + 4);
                if ((info & kInfoOk) && tot == (info & kInfoCount)) {
                    if (esc) {
                        const uint8_t* zsrc = reinterpret_cast<const uint8_t*>(lds_u64w(wp0 + 16 * e + 8));
                        const uint32_t zmis = (uint32_t)(uintptr_t)zsrc & 15u;
                        uint32_t m = esc;
                        if (info & kInfoInStage) {  // the run is in the stage
                            const uint32_t src = stg + kZpOff + zmis + (incl - ne);
                            for (uint32_t r = 0; m; ++r) {
                                const uint32_t b = __ffs(m) - 1;
                                m &= m - 1;
                                sts_u8(xa + (b ^ xsw), rot_exp_lo8(lds_u8(src + r)));
                            }
                        } else {  // a run too long for the stage: read in place
                            const uint8_t* src = zsrc + (incl - ne);
                            for (uint32_t r = 0; m; ++r) {
                                const uint32_t b = __ffs(m) - 1;
                                m &= m - 1;
                                sts_u8(xa + (b ^ xsw), rot_exp_lo8(__ldg(src + r)));
                            }
                        }
                    }
                } else if (lane == 0) {
                    report(a.status, ZCCL_ERR_CORRUPT_STREAM);
                }
                const uint2 lut = lds_u64(lut0 + 8 * s);
                // planes rotated so that processing group i is byte i of each word
                const uint32_t R0 = __funnelshift_r(P0, P0, 16 * h);
                const uint32_t R1 = __funnelshift_r(P1, P1, 16 * h);
                const uint32_t R2 = __funnelshift_r(P2, P2, 16 * h);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t N = lds_u32(sp + 4 * ((R0 >> (8 * i)) & 0xFF)) |
                                       lds_u32(sp + 1024 + 4 * ((R1 >> (8 * i)) & 0xFF)) |
                                       lds_u32(sp + 2048 + 4 * ((R2 >> (8 * i)) & 0xFF));
                    const uint2 xe = lds_u64(xa + 8 * (i ^ x));
                    const uint2 smb = i == 0 ? make_uint2(A.x, A.y)
                                      : i == 1 ? make_uint2(A.z, A.w)
                                      : i == 2 ? make_uint2(B.x, B.y)
                                               : make_uint2(B.z, B.w);
                    decode_add8(&acc[4 * i], N, smb, lut, xe);
                }
            } else {  // plain BF16: the last vq % 8 values by plain loads
                const uint32_t done = vq & ~7u;
                if (lane < vq - done) {
                    const uint16_t* src = kind == kStepLocal ? a.local : a.out;
                    reinterpret_cast<uint16_t*>(sm.stage[q][cst])[done + lane] = src[c * kChunk + q * kQuarter + done + lane];
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) add8(&acc[4 * i], lds_u128(stg + 64 * lane + 16 * (i ^ (2 * h))));
            }
            if (++cst == kStages) cst = 0;
        }
        // the quarter is complete: round, store, start the next one
        uint32_t w[16];
        uint32_t nan = 0;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            w[kk] = pack_rne(acc[kk].x, acc[kk].y);
            nan |= nan_halves(w[kk]);
            acc[kk] = make_float2(-0.0f, -0.0f);
        }
        if (__any_sync(0xffffffffu, nan != 0)) {
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) w[kk] = canonical_nan(w[kk]);
        }
        uint16_t* dst = a.out + c * kChunk + q * kQuarter;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t e = 32 * lane + 8 * (i ^ (2 * h));
            const uint4 o = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            if (e + 8 <= vq) {
                *reinterpret_cast<uint4*>(dst + e) = o;
            } else if (e < vq) {
                store_partial(dst + e, o, vq - e);
            }
        }
    }
    cp_async_wait<0>();  // nothing in flight when the warp leaves
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
            t.blk[s] = nullptr;
            t.zpa[s] = nullptr;
            t.n_esc[s] = 0;
            t.lut[s] = make_uint2(0, 0);
            continue;
        }
        const uint8_t* base = reinterpret_cast<const uint8_t*>(a.streams[s]);
        const uint64_t in_bytes = a.in_bytes[s];
        bool good = base != nullptr && ((uintptr_t)base & 15) == 0 && in_bytes >= zp_offset_of(a.n);
        if (good) {
            const uint32_t* h = reinterpret_cast<const uint32_t*>(base);
            uint64_t n_esc = 0;
            good = header_valid(h, in_bytes, a.n, &n_esc);
            t.n_esc[s] = n_esc;
            // LUT bytes, rotated: entry 0 (code 000) unused, entry c = exponent of code c
            t.lut[s] = make_uint2(rot_exp4(h[6] << 8), rot_exp4((h[6] >> 24) | (h[7] << 8)));
        }
        t.blk[s] = base + kHeaderBytes;
        t.zpa[s] = base + zp_offset_of(a.n);
        ok = ok && good;
    }
    for (uint32_t b = tid; b < 256; b += kThreads) {
        const uint32_t v = spread_nibbles(b);
        sm.spread[0][b] = v;
        sm.spread[1][b] = v << 1;
        sm.spread[2][b] = v << 2;
    }
    pdl_wait();  // offsets of the scan kernel
    if (__syncthreads_and(ok)) reduce_quarters<kPlain>(a, sm, t);
    // every warp of the CTA is past its last read of the offset words: clear
    // those of the CTA's chunks (no other CTA reads them)
    __syncthreads();
    for (uint32_t c = blockIdx.x; c < total; c += gridDim.x)
        for (uint32_t s = tid; s < a.S; s += kThreads) {
            a.local_off[(uint64_t)s * total + c] = 0;
            a.qinfo[(uint64_t)s * total + c] = 0;
        }
    // the last CTA to finish clears the range bases and the scan's look-back
    // words: the workspace is left all zero past its control block and flag
    // area
    if (arrive_last(a.ctrl, &sm.last)) {
        const uint64_t nb = (uint64_t)a.S * ((total + kRangeChunks - 1) / kRangeChunks);
        for (uint64_t i = tid; i < nb; i += kThreads) {
            a.bases[i] = 0;
            a.lookback[i] = 0;
        }
    }
}

}  // namespace

template <bool kPlain>
static size_t reduce_smem_bytes(uint32_t S) { return sizeof(ReduceSmem) + 32ull * S; }

cudaError_t launch_reduce(const ScanArgs& s, const ReduceArgs& a, uint32_t grid_scan, uint32_t grid,
                          cudaStream_t stream)
{
    const bool plain = a.local != nullptr || a.accumulate;
    const size_t smem = plain ? reduce_smem_bytes<true>(a.S) : reduce_smem_bytes<false>(a.S);
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
static int reduce_occupancy(uint32_t S)
{
    const size_t smem = reduce_smem_bytes<kPlain>(S);
    int blocks = 0;
    if (cudaFuncSetAttribute(reduce_kernel<kPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, reduce_kernel<kPlain>, kThreads, smem) !=
        cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

// CTAs per SM of the instance with plain BF16 steps (plain) or without
int reduce_ctas_per_sm(uint32_t S, bool plain)
{
    return plain ? reduce_occupancy<true>(S) : reduce_occupancy<false>(S);
}

}  // namespace zccl

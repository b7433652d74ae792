// zccl_decode.cuh -- rebuilding BF16 values from a chunk block: code planes
// -> LUT exponents (or escaped exponents) + sign-mantissa bytes.  Used by
// the decompress kernel; the fused decompress-reduce kernel shares the
// nibble spreading and the partial store.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.B
// (codes 001..111 name the LUT's exponents, 000 the next zero-point entry).
#pragma once

#include <cstdint>

namespace zccl {

// Shared buffer for a chunk's run of the zero-point array: up to 4096 bytes,
// copied as a 16-byte aligned cover (up to 15 extra bytes on each side).
constexpr uint32_t kZpBufBytes = 4096 + 32;

// bit k of an 8-bit value -> bit 4k
__device__ __forceinline__ uint32_t spread_nibbles(uint32_t x)
{
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    return x;
}

// Rebuilds 8 consecutive elements: `smb` their sign-mantissa bytes, pb0..pb2
// their plane bytes (bit k = element k), lut_lo/lut_hi the 8-entry byte
// table (entry 0 unused, entry c = exponent of code c), `xe` the escaped
// exponents at the elements' slots.  Returns the 8 BF16 values.
// 8 elements from their code nibbles N (nibble k = element k's 3-bit code),
// sign-mantissa bytes and escaped exponents.
__device__ __forceinline__ uint4 decode8_nibbles(uint32_t N, uint2 smb, uint32_t lut_lo, uint32_t lut_hi, uint2 xe)
{
    uint32_t e_lo = __byte_perm(lut_lo, lut_hi, N);        // nibble k of N selects byte k
    uint32_t e_hi = __byte_perm(lut_lo, lut_hi, N >> 16);
    const uint32_t m_lo = __byte_perm(0xFFu, 0u, N);       // 0xFF where the code is 000
    const uint32_t m_hi = __byte_perm(0xFFu, 0u, N >> 16);
    e_lo = (e_lo & ~m_lo) | (xe.x & m_lo);
    e_hi = (e_hi & ~m_hi) | (xe.y & m_hi);
    // low byte = exponent bit 0 << 7 | mantissa; high byte = sign << 7 | exponent >> 1
    const uint32_t lo_a = (smb.x & 0x7F7F7F7Fu) | ((e_lo << 7) & 0x80808080u);
    const uint32_t hi_a = (smb.x & 0x80808080u) | ((e_lo >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo_b = (smb.y & 0x7F7F7F7Fu) | ((e_hi << 7) & 0x80808080u);
    const uint32_t hi_b = (smb.y & 0x80808080u) | ((e_hi >> 1) & 0x7F7F7F7Fu);
    return make_uint4(__byte_perm(lo_a, hi_a, 0x5140), __byte_perm(lo_a, hi_a, 0x7362),
                      __byte_perm(lo_b, hi_b, 0x5140), __byte_perm(lo_b, hi_b, 0x7362));
}

__device__ __forceinline__ uint4 decode8(uint2 smb, uint32_t pb0, uint32_t pb1, uint32_t pb2, uint32_t lut_lo,
                                         uint32_t lut_hi, uint2 xe)
{
    const uint32_t N = spread_nibbles(pb0) | (spread_nibbles(pb1) << 1) | (spread_nibbles(pb2) << 2);
    return decode8_nibbles(N, smb, lut_lo, lut_hi, xe);
}

__device__ __forceinline__ void store_partial(uint16_t* dst, uint4 o, uint32_t count)
{
#pragma unroll
    for (uint32_t q = 0; q < 8; ++q) {
        if (q < count) {
            const uint32_t w = q < 2 ? o.x : q < 4 ? o.y : q < 6 ? o.z : o.w;
            dst[q] = (uint16_t)(w >> (16 * (q & 1)));
        }
    }
}

}  // namespace zccl

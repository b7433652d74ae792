/*
 * zccl_oracle.c -- the ORACLE for the lossless BF16 exponent codec.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct CPU
 * statement of what the codec computes.  Only the tests, the package's smoke
 * check and the CPU-baseline leg of bench.py may build, load or call it.  It
 * shares no source, header, table or helper with the CUDA library; the two
 * meet only in the stream bytes they must agree on.
 *
 * Source of the method: the page "ZipCCL: Efficient Lossless Data Compression
 * of Communication Collectives for Accelerating LLM Training" (gist.science
 * summary, three language editions).  Citations below name its technical
 * summary sections: "ZipCCL 2.A" = theoretical insight (Gaussian tensors,
 * top-7 exponents, LUT from sigma), "ZipCCL 2.B" = exponent coding
 * (split, remap to 001..111, zero-point code 000 + zero-point array,
 * 16 -> 11 bits), "ZipCCL 2.C" = GPU layout (128-byte padded blocks,
 * three 1-bit code arrays), "ZipCCL 2.D" = adaptive strategies (MoE
 * static/dynamic parts, zipped all-to-all + local reduction).
 *
 * Where the page leaves a choice open, the reading taken here is marked
 * [R<k>]; the same readings are listed in the design notes.
 *
 * Parity pins (checked by the CPU tests, not by this file):
 *   LUT           - ranks recomputed with 40-digit mpmath erfc; sigma sweep.
 *   encode/decode - brute force over all 65,536 BF16 patterns, several LUTs;
 *                   hand-built 64-element stream fixture (format bytes).
 *   size          - 11 bits per slot + 8 bits per escape + header/padding,
 *                   escapes counted independently with numpy.
 *   coverage      - measured top-7 fraction vs the closed form.
 *   rounding      - nearest-even by distance vs torch's fp32->bf16 cast on
 *                   random patterns, plus hand-worked midpoints.
 *   reduce        - numpy float32 in-order sums; a case where (a+b)+c
 *                   differs from a+(b+c).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float arithmetic evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

/* status codes (same numbering as the library's, written out separately) */
enum { ZO_OK = 0, ZO_INVALID_ARG = 1, ZO_TOO_SMALL = 2, ZO_CORRUPT = 3 };

/* ---- stream format constants [R5..R12] ---------------------------------- */
#define ZO_MAGIC 0x4C43435Au /* bytes 'Z','C','C','L' */
#define ZO_VERSION 1u
#define ZO_LOG2_CHUNK 12u
#define ZO_CHUNK 4096u       /* element slots per full chunk                  */
#define ZO_TAIL_GRAIN 1024u  /* tail chunk slots rounded up to this [R7]      */
#define ZO_HEADER 128u       /* header bytes; every region 128-byte aligned  */

static uint64_t round_up(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }

/* Slots of chunk c for a stream of n elements [R7]. */
static uint64_t chunk_slots(uint64_t n, uint64_t c)
{
    uint64_t first = c * ZO_CHUNK;
    uint64_t cnt = n - first < ZO_CHUNK ? n - first : ZO_CHUNK;
    return cnt == ZO_CHUNK ? ZO_CHUNK : round_up(cnt, ZO_TAIL_GRAIN);
}

static uint64_t chunk_count(uint64_t n) { return (n + ZO_CHUNK - 1) / ZO_CHUNK; }

/* Offset of the zero-point array: header + all chunk blocks (11 bits per
 * slot: one sign-mantissa byte + three code bits) [R10]. */
uint64_t zo_zero_point_offset(uint64_t n)
{
    uint64_t off = ZO_HEADER;
    for (uint64_t c = 0; c < chunk_count(n); c++) off += chunk_slots(n, c) * 11 / 8;
    return off;
}

/* Total stream bytes for n elements with n_esc escapes [R10]. */
uint64_t zo_stream_bytes(uint64_t n, uint64_t n_esc)
{
    return zo_zero_point_offset(n) + round_up(n_esc, 128);
}

/* Bound for any input: every element escaped. */
uint64_t zo_max_bytes(uint64_t n) { return zo_stream_bytes(n, n); }

/* ---- a1: LUT from sigma (ZipCCL 2.A) ------------------------------------- */

/* Probability that |X| lies in the binade [2^k, 2^(k+1)) for X ~ N(0, sigma^2),
 * k = E - 127:  2 (Phi(2^(k+1)/sigma) - Phi(2^k/sigma)), written with erfc so
 * the tail is not lost to cancellation. */
double zo_binade_mass(double sigma, int E)
{
    int k = E - 127;
    double lo = ldexp(1.0, k) / sigma;
    double hi = ldexp(1.0, k + 1) / sigma;
    return erfc(lo / sqrt(2.0)) - erfc(hi / sqrt(2.0));
}

/* The 7 exponents of largest binade mass, most probable first (code 1 = rank 0)
 * [R1].  Candidates are the normal binades E = 1..254 only [R2]; equal masses
 * order by smaller E [R3]; sigma must be finite and > 0 [R4]. */
int zo_lut_from_sigma(double sigma, uint8_t lut[7])
{
    if (lut == NULL || !(sigma > 0.0) || !isfinite(sigma)) return ZO_INVALID_ARG;
    int taken[256] = {0};
    for (int r = 0; r < 7; r++) {
        int best = -1;
        double best_mass = -1.0;
        for (int E = 1; E <= 254; E++) {
            if (taken[E]) continue;
            double m = zo_binade_mass(sigma, E);
            if (m > best_mass) { /* strict: the first (smallest) E wins ties */
                best_mass = m;
                best = E;
            }
        }
        taken[best] = 1;
        lut[r] = (uint8_t)best;
    }
    return ZO_OK;
}

static int lut_is_valid(const uint8_t lut[7])
{
    for (int a = 0; a < 7; a++)
        for (int b = a + 1; b < 7; b++)
            if (lut[a] == lut[b]) return 0;
    return 1;
}

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put_u32(uint8_t* p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put_u64(uint8_t* p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get_u32(const uint8_t* p)
{
    uint32_t v = 0;
    for (int i = 3; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}
static uint64_t get_u64(const uint8_t* p)
{
    uint64_t v = 0;
    for (int i = 7; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}

/* ---- a2..a7: compress (ZipCCL 2.B, 2.C) ---------------------------------- */
int zo_compress(const uint16_t* x, uint64_t n, const uint8_t lut[7], uint8_t* out,
                uint64_t out_capacity, uint64_t* out_bytes)
{
    if ((n > 0 && x == NULL) || lut == NULL || out == NULL || !lut_is_valid(lut))
        return ZO_INVALID_ARG;
    if (out_capacity < zo_max_bytes(n)) return ZO_TOO_SMALL;

    uint8_t* sm = malloc(n ? n : 1);    /* sign-mantissa byte per element */
    uint8_t* code = malloc(n ? n : 1);  /* 3-bit code per element         */
    uint8_t* zp = malloc(n ? n : 1);    /* zero-point array (raw exps)    */
    if (!sm || !code || !zp) { free(sm); free(code); free(zp); return ZO_INVALID_ARG; }
    uint64_t n_esc = 0;

    for (uint64_t i = 0; i < n; i++) {
        uint16_t v = x[i];
        /* Split: sign bit + 7 mantissa bits -> one byte (sign in bit 7) [R5];
         * the 8 exponent bits separately (ZipCCL 2.B). */
        uint8_t s = (uint8_t)(v >> 15);
        uint8_t e = (uint8_t)((v >> 7) & 0xFF);
        uint8_t m = (uint8_t)(v & 0x7F);
        sm[i] = (uint8_t)((s << 7) | m);
        /* Remap: an exponent among the top 7 gets code r+1 (001..111); any
         * other gets the zero-point code 000 and goes, whole, to the
         * zero-point array, in element order (ZipCCL 2.B). */
        uint8_t c = 0;
        for (int r = 0; r < 7; r++)
            if (lut[r] == e) c = (uint8_t)(r + 1);
        code[i] = c;
        if (c == 0) zp[n_esc++] = e;
    }

    uint64_t zp_offset = zo_zero_point_offset(n);
    uint64_t total = zp_offset + round_up(n_esc, 128);
    memset(out, 0, total);

    /* Header [R12]. */
    put_u32(out + 0, ZO_MAGIC);
    put_u16(out + 4, ZO_VERSION);
    put_u16(out + 6, ZO_LOG2_CHUNK);
    put_u64(out + 8, n);
    put_u64(out + 16, n_esc);
    memcpy(out + 24, lut, 7);
    put_u64(out + 32, zp_offset);

    /* Chunk blocks, 128-byte multiples (ZipCCL 2.C): the chunk's sign-mantissa
     * bytes, then its three 1-bit code planes (ZipCCL 2.C); plane p holds bit p
     * of each code [R6]; slot s of the chunk is bit (s mod 32) of 32-bit
     * little-endian word s/32 [R8]; padding slots stay 0 [R9]. */
    uint64_t pos = ZO_HEADER;
    for (uint64_t c = 0; c < chunk_count(n); c++) {
        uint64_t first = c * ZO_CHUNK;
        uint64_t cnt = n - first < ZO_CHUNK ? n - first : ZO_CHUNK;
        uint64_t L = chunk_slots(n, c);
        for (uint64_t s = 0; s < cnt; s++) out[pos + s] = sm[first + s];
        for (int p = 0; p < 3; p++) {
            uint8_t* plane = out + pos + L + (uint64_t)p * (L / 8);
            for (uint64_t s = 0; s < cnt; s++) {
                if ((code[first + s] >> p) & 1) {
                    uint64_t word = s / 32, bit = s % 32;
                    plane[4 * word + bit / 8] |= (uint8_t)(1u << (bit % 8));
                }
            }
        }
        pos += L * 11 / 8;
    }

    /* Zero-point array after the blocks, zero-padded to 128 bytes [R10]. */
    memcpy(out + zp_offset, zp, n_esc);
    *out_bytes = total;
    free(sm);
    free(code);
    free(zp);
    return ZO_OK;
}

/* ---- a8: decompress (inverse of ZipCCL 2.B) ------------------------------ */

/* Checks every header field, every padding byte and the escape total [R13]. */
int zo_decompress(const uint8_t* in, uint64_t in_bytes, uint16_t* x, uint64_t n)
{
    if (in == NULL || (n > 0 && x == NULL)) return ZO_INVALID_ARG;
    if (in_bytes < ZO_HEADER) return ZO_CORRUPT;
    if (get_u32(in + 0) != ZO_MAGIC || get_u16(in + 4) != ZO_VERSION ||
        get_u16(in + 6) != ZO_LOG2_CHUNK || get_u64(in + 8) != n)
        return ZO_CORRUPT;
    uint64_t n_esc = get_u64(in + 16);
    uint8_t lut[7];
    memcpy(lut, in + 24, 7);
    if (!lut_is_valid(lut) || in[31] != 0) return ZO_CORRUPT;
    uint64_t zp_offset = get_u64(in + 32);
    if (zp_offset != zo_zero_point_offset(n) || n_esc > n) return ZO_CORRUPT;
    for (int b = 40; b < (int)ZO_HEADER; b++)
        if (in[b] != 0) return ZO_CORRUPT;
    uint64_t total = zp_offset + round_up(n_esc, 128);
    if (in_bytes < total) return ZO_CORRUPT;

    uint64_t k = 0; /* next zero-point entry */
    uint64_t pos = ZO_HEADER;
    for (uint64_t c = 0; c < chunk_count(n); c++) {
        uint64_t first = c * ZO_CHUNK;
        uint64_t cnt = n - first < ZO_CHUNK ? n - first : ZO_CHUNK;
        uint64_t L = chunk_slots(n, c);
        for (uint64_t s = 0; s < L; s++) {
            uint8_t sm = in[pos + s];
            uint8_t code = 0;
            for (int p = 0; p < 3; p++) {
                const uint8_t* plane = in + pos + L + (uint64_t)p * (L / 8);
                uint64_t word = s / 32, bit = s % 32;
                if ((plane[4 * word + bit / 8] >> (bit % 8)) & 1) code |= (uint8_t)(1u << p);
            }
            if (s >= cnt) { /* padding slot: must be all zero [R9] */
                if (sm != 0 || code != 0) return ZO_CORRUPT;
                continue;
            }
            uint8_t e;
            if (code != 0) {
                e = lut[code - 1];
            } else {
                if (k >= n_esc) return ZO_CORRUPT;
                e = in[zp_offset + k];
                k++;
            }
            x[first + s] = (uint16_t)(((uint16_t)(sm >> 7) << 15) | ((uint16_t)e << 7) | (sm & 0x7F));
        }
        pos += L * 11 / 8;
    }
    if (k != n_esc) return ZO_CORRUPT;
    for (uint64_t b = zp_offset + n_esc; b < total; b++)
        if (in[b] != 0) return ZO_CORRUPT;
    return ZO_OK;
}

/* ---- a10: local reduction of the zipped all-to-all (ZipCCL 2.D) ---------- */

/* BF16 bit pattern (magnitude only) as a real number; the pattern 0x7F80 is
 * given the value 2^128, the next power of two past the largest finite BF16,
 * which is what round-to-nearest compares against at the overflow edge. */
static double bf16_magnitude_value(uint32_t b)
{
    if (b == 0x7F80u) return ldexp(1.0, 128);
    uint32_t u = b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* fp32 -> BF16 by the definition of round-to-nearest, ties-to-even: of the two
 * BF16 neighbours of f, the nearer one; on a tie the one whose last mantissa
 * bit is 0.  Any NaN becomes the canonical quiet NaN 0x7FC0 [R14].  Distances
 * are exact in double (both neighbours lie within a factor of 2 of |f|). */
uint16_t zo_round_bf16(float f)
{
    if (isnan(f)) return 0x7FC0;
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag == 0x7F800000u) return (uint16_t)(sign | 0x7F80u); /* infinity */
    uint32_t lo = mag >> 16; /* magnitude truncated toward zero */
    uint32_t hi = lo + 1;    /* next BF16 magnitude up           */
    double a = fabs((double)f);
    double d_lo = a - bf16_magnitude_value(lo);
    double d_hi = bf16_magnitude_value(hi) - a;
    uint32_t pick;
    if (d_lo < d_hi) pick = lo;
    else if (d_hi < d_lo) pick = hi;
    else pick = (lo & 1u) == 0 ? lo : hi;
    return (uint16_t)(sign | pick);
}

/* zo_round_bf16 over an array (lets the tests pin it on millions of values). */
void zo_round_bf16_n(const float* f, uint16_t* out, uint64_t n)
{
    for (uint64_t i = 0; i < n; i++) out[i] = zo_round_bf16(f[i]);
}

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* out[i] = RNE_bf16( ((x_0[i] + x_1[i]) + x_2[i]) + ... + x_{S-1}[i] ), every
 * add in fp32, in shard order, x_s decoded from stream s [R14]. */
int zo_decompress_reduce(const uint8_t* const* in, const uint64_t* in_bytes, uint32_t S,
                         uint16_t* out, uint64_t n)
{
    if (in == NULL || in_bytes == NULL || S == 0 || (n > 0 && out == NULL)) return ZO_INVALID_ARG;
    uint16_t** dec = calloc(S, sizeof(uint16_t*));
    if (!dec) return ZO_INVALID_ARG;
    int st = ZO_OK;
    for (uint32_t s = 0; s < S && st == ZO_OK; s++) {
        dec[s] = malloc((n ? n : 1) * sizeof(uint16_t));
        if (!dec[s]) { st = ZO_INVALID_ARG; break; }
        st = zo_decompress(in[s], in_bytes[s], dec[s], n);
    }
    if (st == ZO_OK) {
        for (uint64_t i = 0; i < n; i++) {
            float acc = bf16_to_float(dec[0][i]);
            for (uint32_t s = 1; s < S; s++) acc = acc + bf16_to_float(dec[s][i]);
            out[i] = zo_round_bf16(acc);
        }
    }
    for (uint32_t s = 0; s < S; s++) free(dec[s]);
    free(dec);
    return st;
}

/* The local-reduction step as a rank of a zipped reduce-scatter sees it
 * (ZipCCL 2.D): S inputs in rank order, every one a compressed stream except
 * the rank's own shard at position local_pos, which is plain BF16 (local may
 * be NULL: then all S are streams and local_pos is ignored).  With
 * accumulate != 0 the fold starts from the BF16 values already in out:
 *   acc = accumulate ? out[i] : x_0;  acc += x_s for the remaining inputs in
 *   order;  out[i] = round_bf16(acc)
 * in float, one IEEE add at a time [R14].  in[local_pos] is not read. */
int zo_decompress_reduce_local(const uint8_t* const* in, const uint64_t* in_bytes, uint32_t S,
                               const uint16_t* local, uint32_t local_pos, int accumulate,
                               uint16_t* out, uint64_t n)
{
    if (in == NULL || in_bytes == NULL || S == 0 || (n > 0 && out == NULL)) return ZO_INVALID_ARG;
    if (local != NULL && local_pos >= S) return ZO_INVALID_ARG;
    uint16_t** dec = calloc(S, sizeof(uint16_t*));
    if (!dec) return ZO_INVALID_ARG;
    int st = ZO_OK;
    for (uint32_t s = 0; s < S && st == ZO_OK; s++) {
        if (local != NULL && s == local_pos) continue;
        dec[s] = malloc((n ? n : 1) * sizeof(uint16_t));
        if (!dec[s]) { st = ZO_INVALID_ARG; break; }
        st = zo_decompress(in[s], in_bytes[s], dec[s], n);
    }
    if (st == ZO_OK) {
        for (uint64_t i = 0; i < n; i++) {
            float acc = 0.0f;
            int have = 0;
            if (accumulate) {
                acc = bf16_to_float(out[i]);
                have = 1;
            }
            for (uint32_t s = 0; s < S; s++) {
                const uint16_t v = (local != NULL && s == local_pos) ? local[i] : dec[s][i];
                acc = have ? acc + bf16_to_float(v) : bf16_to_float(v);
                have = 1;
            }
            out[i] = zo_round_bf16(acc);
        }
    }
    for (uint32_t s = 0; s < S; s++) free(dec[s]);
    free(dec);
    return st;
}

/* Exponent histogram of n BF16 values: hist[e] = how many have biased
 * exponent e (bits 7..14), for e = 0..255.  hist is overwritten. */
void zo_exponent_histogram(const uint16_t* x, uint64_t n, uint64_t hist[256])
{
    for (int e = 0; e < 256; e++) hist[e] = 0;
    for (uint64_t i = 0; i < n; i++) hist[(x[i] >> 7) & 0xFF]++;
}

/* A LUT measured from data, the alternative to the sigma rule that the page
 * sets aside for cost (ZipCCL 2.A: no online statistics pass) [R15]: the 7
 * exponents with the largest counts, in rank order (code 1 = most frequent),
 * ties to the smaller exponent; every exponent 0..255 is a candidate (a
 * data LUT may hold the zero/subnormal binade, unlike the sigma rule). */
int zo_lut_from_histogram(const uint64_t hist[256], uint8_t lut[7])
{
    if (hist == NULL || lut == NULL) return ZO_INVALID_ARG;
    int taken[256] = {0};
    for (int r = 0; r < 7; r++) {
        int best = -1;
        for (int e = 0; e < 256; e++) {
            if (taken[e]) continue;
            if (best < 0 || hist[e] > hist[best]) best = e;  /* strict: the smaller e wins ties */
        }
        taken[best] = 1;
        lut[r] = (uint8_t)best;
    }
    return ZO_OK;
}

// zccl_host.cu -- the C ABI of libzccl: argument validation, LUT derivation,
// workspace sizing and kernel launches.  Declarations and contracts are in
// include/zccl.h.
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.A (LUT
// from the layer's sigma instead of an online histogram) and 2.B-2.D (the
// operations this layer launches).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "zccl_common.cuh"
#include "zccl_internal.h"

using namespace zccl;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    std::once_flag once;
    int sms = 0;
    int compress_per_sm = 1;
    // the batched kernel's shared memory grows with the segment count: its
    // occupancy for 2^b segments, b = 0 .. log2(ZCCL_MAX_SEGMENTS)
    int compress_per_sm_batched[13] = {};
    int scan_per_sm = 1;
    int decompress_per_sm = 1;
    // the reduction's occupancy, [plain BF16 steps or not][S <= kSmallShards, any S <= ZCCL_MAX_SHARDS]
    int reduce_per_sm[2][2] = {{1, 1}, {1, 1}};
};
constexpr uint32_t kSmallShards = 32;
static_assert(ZCCL_MAX_SEGMENTS == 1u << 12, "one occupancy bucket per power of two up to the segment limit");
DeviceInfo g_dev[kMaxDevices];

// SM count and kernel occupancy of the current device, computed once.
const DeviceInfo* device_info()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&]() {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        d.sms = sms > 0 ? sms : 1;
        d.compress_per_sm = compress_ctas_per_sm(1);
        for (int b = 0; b < 13; ++b) d.compress_per_sm_batched[b] = compress_ctas_per_sm(1u << b);
        d.scan_per_sm = scan_ctas_per_sm();
        d.decompress_per_sm = decompress_ctas_per_sm();
        for (int plain = 0; plain < 2; ++plain) {
            d.reduce_per_sm[plain][0] = reduce_ctas_per_sm(kSmallShards, plain != 0);
            d.reduce_per_sm[plain][1] = reduce_ctas_per_sm(ZCCL_MAX_SHARDS, plain != 0);
        }
    });
    return &d;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

bool lut_ok(const zccl_lut_t* lut)
{
    if (lut == nullptr) return false;
    for (int i = 0; i < 7; ++i)
        for (int j = i + 1; j < 7; ++j)
            if (lut->exp[i] == lut->exp[j]) return false;
    return true;
}

uint64_t ranges_of(uint64_t units) { return (units + kRangeChunks - 1) / kRangeChunks; }

// Every workspace starts with the same prefix (kPrefixBytes): the control
// words, then the two parity sets of run flag words.  Each op leaves the
// scratch after it all zero, so a workspace can serve any op in any order.
static_assert(kFlagWords == kMaxGrid, "one flag word per CTA");

// Compression workspace: prefix | escape count per chunk | a 4096-byte
// escape staging slot per chunk.
struct CompressLayout {
    uint64_t counts, stage, total;
};
CompressLayout compress_layout(uint64_t units)
{
    CompressLayout l;
    l.counts = kPrefixBytes;
    l.stage = round_up(l.counts + 4 * units, 256);
    l.total = round_up(l.stage + (uint64_t)kChunk * units, 256);
    return l;
}

// Decompression workspace: prefix | one entry word per chunk.
struct DecompressLayout {
    uint64_t entry, total;
};
DecompressLayout decompress_layout(uint64_t units)
{
    DecompressLayout l;
    l.entry = kPrefixBytes;
    l.total = round_up(l.entry + 8 * units, 256);
    return l;
}

// Decompression / reduction workspace, per stream: look-back word per range |
// range base | chunk prefix within its range | quarter word per chunk.
struct ScanLayout {
    uint64_t lookback, bases, local, qinfo, total;
};
ScanLayout scan_layout(uint64_t units, uint64_t S)
{
    const uint64_t R = S * ranges_of(units);
    ScanLayout l;
    l.lookback = kPrefixBytes;
    l.bases = round_up(l.lookback + 8 * R, 16);
    l.local = round_up(l.bases + 8 * R, 16);
    l.qinfo = round_up(l.local + 4 * S * units, 16);
    l.total = round_up(l.qinfo + 8 * S * units, 256);
    return l;
}

uint64_t batched_max_units(uint64_t total_n, uint32_t n_segs) { return total_n / kChunk + n_segs; }

uint32_t grid_for(uint64_t units, int per_sm, int sms)
{
    const uint64_t cap = std::min<uint64_t>((uint64_t)per_sm * (uint64_t)sms, kMaxGrid);
    const uint64_t g = std::min<uint64_t>(units, cap);
    return (uint32_t)std::max<uint64_t>(g, 1);
}

// zccl_decompress and zccl_decompress_split: the frame (header + blocks) at
// `frame`, the zero-point array at `zp`, in_bytes = zp_offset + the bytes at zp.
zccl_status_t decompress_impl(const uint8_t* frame, const uint8_t* zp, uint64_t in_bytes, uint16_t* d_out,
                              uint64_t n, void* d_ws, uint64_t ws_bytes, uint32_t* d_status, cudaStream_t stream)
{
    if ((n > 0 && (d_out == nullptr || !aligned(d_out, 16))) || d_ws == nullptr || !aligned(d_ws, 16) ||
        !aligned(d_status, 4))
        return ZCCL_ERR_INVALID_ARG;
    const uint64_t units = units_of(n);
    const DecompressLayout l = decompress_layout(units);
    if (ws_bytes < l.total) return ZCCL_ERR_BUFFER_TOO_SMALL;
    const DeviceInfo* dev = device_info();
    if (dev == nullptr) return ZCCL_ERR_CUDA;

    DecompressArgs a{};
    a.in = frame;
    a.zp = zp;
    a.in_bytes = in_bytes;
    a.out = d_out;
    a.n = n;
    a.ctrl = reinterpret_cast<WsCtrl*>(d_ws);
    a.flags = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + kCtrlBytes);
    a.entry = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + l.entry);
    a.status = d_status;
    return launch_decompress(a, grid_for(units, dev->decompress_per_sm, dev->sms), stream) == cudaSuccess
               ? ZCCL_OK
               : ZCCL_ERR_CUDA;
}

}  // namespace

extern "C" {

zccl_status_t zccl_lut_from_sigma(double sigma, zccl_lut_t* lut)
{
    if (lut == nullptr || !(sigma > 0.0) || !std::isfinite(sigma)) return ZCCL_ERR_INVALID_ARG;
    // Gaussian mass of every normal binade E = 1..254, then the 7 largest.
    struct Cand {
        double mass;
        int e;
    };
    Cand c[254];
    const double inv = 1.0 / (sigma * std::sqrt(2.0));
    for (int e = 1; e <= 254; ++e) {
        const double a = std::ldexp(1.0, e - 127), b = std::ldexp(1.0, e - 126);
        // 2 (Phi(b/sigma) - Phi(a/sigma)) = erfc(a/(sigma sqrt 2)) - erfc(b/(sigma sqrt 2))
        c[e - 1] = Cand{std::erfc(a * inv) - std::erfc(b * inv), e};
    }
    std::partial_sort(c, c + 7, c + 254, [](const Cand& x, const Cand& y) {
        return x.mass != y.mass ? x.mass > y.mass : x.e < y.e;
    });
    for (int r = 0; r < 7; ++r) lut->exp[r] = (uint8_t)c[r].e;
    return ZCCL_OK;
}

uint64_t zccl_max_compressed_bytes(uint64_t n) { return stream_bytes_of(n, n); }

uint64_t zccl_zero_point_offset(uint64_t n) { return zp_offset_of(n); }

zccl_status_t zccl_workspace_bytes(int op, uint64_t n, uint32_t k, uint64_t* bytes)
{
    if (bytes == nullptr || n >= kMaxElems) return ZCCL_ERR_INVALID_ARG;
    switch (op) {
        case ZCCL_OP_COMPRESS: *bytes = compress_layout(units_of(n)).total; return ZCCL_OK;
        case ZCCL_OP_DECOMPRESS: *bytes = decompress_layout(units_of(n)).total; return ZCCL_OK;
        case ZCCL_OP_COMPRESS_BATCHED:
            if (k == 0 || k > ZCCL_MAX_SEGMENTS) return ZCCL_ERR_INVALID_ARG;
            *bytes = compress_layout(batched_max_units(n, k)).total;
            return ZCCL_OK;
        case ZCCL_OP_DECOMPRESS_REDUCE:
            if (k == 0 || k > ZCCL_MAX_SHARDS) return ZCCL_ERR_INVALID_ARG;
            *bytes = scan_layout(units_of(n), k).total;
            return ZCCL_OK;
        default: return ZCCL_ERR_INVALID_ARG;
    }
}

zccl_status_t zccl_workspace_init(void* d_ws, uint64_t ws_bytes, cudaStream_t stream)
{
    if (d_ws == nullptr || ws_bytes < kCtrlBytes) return ZCCL_ERR_INVALID_ARG;
    return cudaMemsetAsync(d_ws, 0, ws_bytes, stream) == cudaSuccess ? ZCCL_OK : ZCCL_ERR_CUDA;
}

zccl_status_t zccl_compress(const uint16_t* d_in, uint64_t n, const zccl_lut_t* lut, void* d_out,
                            uint64_t out_capacity, uint64_t* d_out_bytes, void* d_ws, uint64_t ws_bytes,
                            uint32_t* d_status, cudaStream_t stream)
{
    if (n >= kMaxElems || !lut_ok(lut) || d_out == nullptr || !aligned(d_out, 16) ||
        (n > 0 && (d_in == nullptr || !aligned(d_in, 16))) || d_out_bytes == nullptr ||
        !aligned(d_out_bytes, 8) || d_ws == nullptr || !aligned(d_ws, 16) || !aligned(d_status, 4))
        return ZCCL_ERR_INVALID_ARG;
    if (out_capacity < zccl_max_compressed_bytes(n)) return ZCCL_ERR_BUFFER_TOO_SMALL;
    const uint64_t units = units_of(n);
    const CompressLayout l = compress_layout(units);
    if (ws_bytes < l.total) return ZCCL_ERR_BUFFER_TOO_SMALL;
    const DeviceInfo* dev = device_info();
    if (dev == nullptr) return ZCCL_ERR_CUDA;

    CompressArgs a{};
    a.segs = nullptr;
    a.single = zccl_segment_t{d_in, n, d_out, out_capacity};
    a.n_segs = 1;
    a.max_units = (uint32_t)units;
    std::memcpy(a.lut, lut->exp, 7);
    a.out_bytes = d_out_bytes;
    a.ctrl = reinterpret_cast<WsCtrl*>(d_ws);
    a.flags = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + kCtrlBytes);
    a.counts = reinterpret_cast<uint32_t*>((uint8_t*)d_ws + l.counts);
    a.stage = (uint8_t*)d_ws + l.stage;
    a.status = d_status;
    return launch_compress(a, grid_for(units, dev->compress_per_sm, dev->sms), stream) == cudaSuccess
               ? ZCCL_OK
               : ZCCL_ERR_CUDA;
}

zccl_status_t zccl_compress_batched(const zccl_segment_t* d_segs, uint32_t n_segs, uint64_t total_n,
                                    const zccl_lut_t* lut, uint64_t* d_out_bytes, void* d_ws,
                                    uint64_t ws_bytes, uint32_t* d_status, cudaStream_t stream)
{
    if (n_segs == 0 || n_segs > ZCCL_MAX_SEGMENTS || total_n >= kMaxElems || !lut_ok(lut) ||
        d_segs == nullptr || !aligned(d_segs, 8) || d_out_bytes == nullptr || !aligned(d_out_bytes, 8) ||
        d_ws == nullptr || !aligned(d_ws, 16) || !aligned(d_status, 4))
        return ZCCL_ERR_INVALID_ARG;
    const uint64_t max_units = batched_max_units(total_n, n_segs);
    const CompressLayout l = compress_layout(max_units);
    if (ws_bytes < l.total) return ZCCL_ERR_BUFFER_TOO_SMALL;
    const DeviceInfo* dev = device_info();
    if (dev == nullptr) return ZCCL_ERR_CUDA;

    CompressArgs a{};
    a.segs = d_segs;
    a.n_segs = n_segs;
    a.max_units = (uint32_t)max_units;
    std::memcpy(a.lut, lut->exp, 7);
    a.out_bytes = d_out_bytes;
    a.ctrl = reinterpret_cast<WsCtrl*>(d_ws);
    a.flags = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + kCtrlBytes);
    a.counts = reinterpret_cast<uint32_t*>((uint8_t*)d_ws + l.counts);
    a.stage = (uint8_t*)d_ws + l.stage;
    a.status = d_status;
    // occupancy of the next power of two at or above n_segs: that needs at
    // least this call's shared memory, so the grid stays co-resident
    int b = 0;
    while ((1u << b) < n_segs) ++b;
    return launch_compress(a, grid_for(max_units, dev->compress_per_sm_batched[b], dev->sms), stream) == cudaSuccess
               ? ZCCL_OK
               : ZCCL_ERR_CUDA;
}

zccl_status_t zccl_decompress(const void* d_in, uint64_t in_bytes, uint16_t* d_out, uint64_t n, void* d_ws,
                              uint64_t ws_bytes, uint32_t* d_status, cudaStream_t stream)
{
    if (n >= kMaxElems || d_in == nullptr || !aligned(d_in, 16) || in_bytes < zp_offset_of(n))
        return ZCCL_ERR_INVALID_ARG;
    return decompress_impl(reinterpret_cast<const uint8_t*>(d_in),
                           reinterpret_cast<const uint8_t*>(d_in) + zp_offset_of(n), in_bytes, d_out, n, d_ws,
                           ws_bytes, d_status, stream);
}

zccl_status_t zccl_decompress_split(const void* d_frame, const void* d_tail, uint64_t tail_bytes, uint16_t* d_out,
                                    uint64_t n, void* d_ws, uint64_t ws_bytes, uint32_t* d_status,
                                    cudaStream_t stream)
{
    if (n >= kMaxElems || d_frame == nullptr || !aligned(d_frame, 16) || tail_bytes >= kMaxElems * 4 ||
        (tail_bytes > 0 && (d_tail == nullptr || !aligned(d_tail, 16))))
        return ZCCL_ERR_INVALID_ARG;
    return decompress_impl(reinterpret_cast<const uint8_t*>(d_frame), reinterpret_cast<const uint8_t*>(d_tail),
                           zp_offset_of(n) + tail_bytes, d_out, n, d_ws, ws_bytes, d_status, stream);
}

}  // extern "C"

namespace {

zccl_status_t reduce_impl(const void* const* d_streams, const uint64_t* d_in_bytes, uint32_t S,
                          const uint16_t* d_local, uint32_t local_pos, int accumulate, uint16_t* d_out, uint64_t n,
                          void* d_ws, uint64_t ws_bytes, uint32_t* d_status, cudaStream_t stream)
{
    if (S == 0 || S > ZCCL_MAX_SHARDS || n >= kMaxElems || d_streams == nullptr || !aligned(d_streams, 8) ||
        d_in_bytes == nullptr || !aligned(d_in_bytes, 8) || (n > 0 && (d_out == nullptr || !aligned(d_out, 16))) ||
        d_ws == nullptr || !aligned(d_ws, 16) || !aligned(d_status, 4) ||
        (d_local != nullptr && (local_pos >= S || !aligned(d_local, 16))))
        return ZCCL_ERR_INVALID_ARG;
    const uint64_t units = units_of(n);
    const ScanLayout l = scan_layout(units, S);
    if (ws_bytes < l.total) return ZCCL_ERR_BUFFER_TOO_SMALL;
    const DeviceInfo* dev = device_info();
    if (dev == nullptr) return ZCCL_ERR_CUDA;

    ScanArgs sc{};
    sc.streams = d_streams;
    sc.in_bytes_dev = d_in_bytes;
    sc.S = S;
    sc.skip = d_local != nullptr ? local_pos : S;
    sc.n = n;
    sc.ctrl = reinterpret_cast<WsCtrl*>(d_ws);
    sc.lookback = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + l.lookback);
    sc.bases = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + l.bases);
    sc.local = reinterpret_cast<uint32_t*>((uint8_t*)d_ws + l.local);
    sc.qinfo = reinterpret_cast<uint64_t*>((uint8_t*)d_ws + l.qinfo);
    sc.status = d_status;
    ReduceArgs a{};
    a.streams = d_streams;
    a.in_bytes = d_in_bytes;
    a.S = S;
    a.local = d_local;
    a.local_pos = d_local != nullptr ? local_pos : 0u;
    a.accumulate = accumulate ? 1u : 0u;
    a.out = d_out;
    a.n = n;
    a.ctrl = sc.ctrl;
    a.bases = sc.bases;
    a.lookback = sc.lookback;
    a.local_off = sc.local;
    a.qinfo = sc.qinfo;
    a.status = d_status;
    const int per_sm = dev->reduce_per_sm[(d_local != nullptr || accumulate) ? 1 : 0][S <= kSmallShards ? 0 : 1];
    return launch_reduce(sc, a, grid_for((uint64_t)S * ranges_of(units), dev->scan_per_sm, dev->sms),
                         grid_for(units, per_sm, dev->sms), stream) == cudaSuccess
               ? ZCCL_OK
               : ZCCL_ERR_CUDA;
}

}  // namespace

extern "C" {

zccl_status_t zccl_decompress_reduce(const void* const* d_streams, const uint64_t* d_in_bytes, uint32_t S,
                                     uint16_t* d_out, uint64_t n, void* d_ws, uint64_t ws_bytes,
                                     uint32_t* d_status, cudaStream_t stream)
{
    return reduce_impl(d_streams, d_in_bytes, S, nullptr, 0, 0, d_out, n, d_ws, ws_bytes, d_status, stream);
}

zccl_status_t zccl_decompress_reduce_local(const void* const* d_streams, const uint64_t* d_in_bytes, uint32_t S,
                                           const uint16_t* d_local, uint32_t local_pos, int accumulate,
                                           uint16_t* d_out, uint64_t n, void* d_ws, uint64_t ws_bytes,
                                           uint32_t* d_status, cudaStream_t stream)
{
    return reduce_impl(d_streams, d_in_bytes, S, d_local, local_pos, accumulate, d_out, n, d_ws, ws_bytes,
                       d_status, stream);
}

zccl_status_t zccl_exponent_histogram(const uint16_t* d_in, uint64_t n, uint64_t* d_hist, int accumulate,
                                      cudaStream_t stream)
{
    if (n >= kMaxElems || (n > 0 && (d_in == nullptr || !aligned(d_in, 16))) || d_hist == nullptr ||
        !aligned(d_hist, 8))
        return ZCCL_ERR_INVALID_ARG;
    const DeviceInfo* dev = device_info();
    if (dev == nullptr) return ZCCL_ERR_CUDA;
    return launch_histogram(d_in, n, d_hist, accumulate != 0, dev->sms, stream) == cudaSuccess ? ZCCL_OK
                                                                                           : ZCCL_ERR_CUDA;
}

zccl_status_t zccl_lut_from_histogram(const uint64_t* hist, zccl_lut_t* lut)
{
    if (hist == nullptr || lut == nullptr) return ZCCL_ERR_INVALID_ARG;
    bool used[256] = {};
    for (int r = 0; r < 7; ++r) {  // rank r: the largest count not yet taken, the smaller exponent on ties
        int pick = -1;
        for (int e = 0; e < 256; ++e)
            if (!used[e] && (pick < 0 || hist[e] > hist[pick])) pick = e;
        used[pick] = true;
        lut->exp[r] = (uint8_t)pick;
    }
    return ZCCL_OK;
}

zccl_status_t zccl_lut_from_data(const uint16_t* d_in, uint64_t n, uint64_t* d_hist, zccl_lut_t* lut,
                                 cudaStream_t stream)
{
    if (lut == nullptr) return ZCCL_ERR_INVALID_ARG;
    const zccl_status_t st = zccl_exponent_histogram(d_in, n, d_hist, 0, stream);
    if (st != ZCCL_OK) return st;
    uint64_t hist[256];
    if (cudaMemcpyAsync(hist, d_hist, sizeof(hist), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return ZCCL_ERR_CUDA;
    return zccl_lut_from_histogram(hist, lut);
}

zccl_status_t zccl_check_bounded_wait(uint32_t limit_us, uint32_t* d_status, cudaStream_t stream)
{
    if (d_status == nullptr || !aligned(d_status, 4) || limit_us == 0 || limit_us > 1000000)
        return ZCCL_ERR_INVALID_ARG;
    return launch_wait_check((uint64_t)limit_us * 1000, d_status, stream) == cudaSuccess ? ZCCL_OK : ZCCL_ERR_CUDA;
}

zccl_status_t zccl_check_bounded_poll(int kind, uint32_t limit_us, const void* d_word, uint32_t* d_status,
                                      cudaStream_t stream)
{
    if ((kind != ZCCL_POLL_COUNTER && kind != ZCCL_POLL_FLAG) || d_word == nullptr || !aligned(d_word, 8) ||
        d_status == nullptr || !aligned(d_status, 4) || limit_us == 0 || limit_us > 1000000)
        return ZCCL_ERR_INVALID_ARG;
    return launch_poll_check(kind, (uint64_t)limit_us * 1000, d_word, d_status, stream) == cudaSuccess
               ? ZCCL_OK
               : ZCCL_ERR_CUDA;
}

const char* zccl_status_string(zccl_status_t s)
{
    switch (s) {
        case ZCCL_OK: return "ok";
        case ZCCL_ERR_INVALID_ARG: return "invalid argument";
        case ZCCL_ERR_BUFFER_TOO_SMALL: return "buffer too small";
        case ZCCL_ERR_CORRUPT_STREAM: return "corrupt stream";
        case ZCCL_ERR_CUDA: return "CUDA runtime error";
        case ZCCL_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"

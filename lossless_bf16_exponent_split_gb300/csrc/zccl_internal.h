// zccl_internal.h -- launch interface between the C-ABI host layer and the
// kernels (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/zccl.h"

namespace zccl {

struct WsCtrl;

// Compression, one stream or a batch of segments (one cooperative kernel).
struct CompressArgs {
    const zccl_segment_t* segs;  // device descriptors (batched) or nullptr
    zccl_segment_t single;       // the one segment when segs == nullptr
    uint32_t n_segs;
    uint32_t max_units;          // chunks the workspace has room for
    uint8_t lut[8];
    uint64_t* out_bytes;         // device [n_segs]
    WsCtrl* ctrl;
    uint64_t* flags;             // [2][kFlagWords] run flag words, by call parity
    uint32_t* counts;            // [max_units] escapes per chunk
    uint8_t* stage;              // [max_units * 4096] escapes, chunk-local
    uint32_t* status;
};

// Escape-offset scan over S streams of n elements (decompress: S = 1).
struct ScanArgs {
    const void* const* streams;  // device [S], or nullptr with `single`
    const uint8_t* single;
    const uint64_t* in_bytes_dev;  // device [S], or nullptr with `in_bytes`
    uint64_t in_bytes;
    uint32_t S;
    uint32_t skip;               // a position holding plain BF16 (no stream), or S for none
    uint64_t n;
    WsCtrl* ctrl;
    uint64_t* lookback;          // [S][ranges per stream] look-back words (kLbState | value)
    uint64_t* bases;             // [S][ranges per stream] range offset in its stream
    uint32_t* local;             // [S][units] chunk offset within its range
    uint64_t* qinfo;             // [S][units] quarter word per chunk (quarter_before / quarter_end)
    uint32_t* status;
};

struct DecompressArgs {
    const uint8_t* in;           // header and chunk blocks (the frame)
    const uint8_t* zp;           // the zero-point array: in + zp_offset, or a separate tail buffer
    uint64_t in_bytes;           // zp_offset + the bytes available at zp
    uint16_t* out;
    uint64_t n;
    WsCtrl* ctrl;
    uint64_t* flags;             // [2][kFlagWords] run totals, by call parity
    uint64_t* entry;             // [units] flag | zero-point offset << 13 | escapes
    uint32_t* status;
};

struct ReduceArgs {
    const void* const* streams;  // device [S]
    const uint64_t* in_bytes;    // device [S]
    uint32_t S;
    const uint16_t* local;       // plain BF16 input at position local_pos, or nullptr
    uint32_t local_pos;
    uint32_t accumulate;         // nonzero: the fold starts from the values in out
    uint16_t* out;
    uint64_t n;
    WsCtrl* ctrl;
    uint64_t* bases;             // from the scan: [S][ranges per stream] (cleared by the last CTA)
    uint64_t* lookback;          // from the scan: [S][ranges per stream] (cleared by the last CTA)
    uint32_t* local_off;         // [S][units] chunk prefix within its range (cleared by the CTA that read it)
    uint64_t* qinfo;             // [S][units] quarter words (cleared by the CTA that read them)
    uint32_t* status;
};

// Launches `kernel` on `stream` so that it may start while the previous
// kernel on the stream finishes (programmatic dependent launch); the kernel
// itself waits (griddepcontrol.wait) before reading the previous kernel's
// results.
template <typename Args>
cudaError_t launch_dependent(void (*kernel)(Args), uint32_t grid, uint32_t threads, size_t smem,
                             cudaStream_t stream, const Args& a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Launches `kernel` cooperatively: all its CTAs are resident at once (the
// launch fails otherwise), so they may wait for one another at a grid
// barrier.
template <typename Args>
cudaError_t launch_cooperative(void (*kernel)(Args), uint32_t grid, uint32_t threads, size_t smem,
                               cudaStream_t stream, const Args& a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Largest grid the cooperative kernels use (sizes the per-CTA workspace arrays).
constexpr uint32_t kMaxGrid = 4096;

size_t compress_smem_bytes(uint32_t n_segs);
cudaError_t launch_compress(const CompressArgs& a, uint32_t grid, cudaStream_t stream);
int compress_ctas_per_sm(uint32_t n_segs);

cudaError_t launch_scan(const ScanArgs& a, uint32_t grid, cudaStream_t stream);
int scan_ctas_per_sm();
cudaError_t launch_decompress(const DecompressArgs& a, uint32_t grid, cudaStream_t stream);
int decompress_ctas_per_sm();

cudaError_t launch_reduce(const ScanArgs& s, const ReduceArgs& a, uint32_t grid_scan, uint32_t grid,
                          cudaStream_t stream);
int reduce_ctas_per_sm(uint32_t S, bool plain);

cudaError_t launch_histogram(const uint16_t* in, uint64_t n, uint64_t* hist, bool accumulate, int sms,
                             cudaStream_t stream);

cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* status, cudaStream_t stream);
cudaError_t launch_poll_check(int kind, uint64_t limit_ns, const void* word, uint32_t* status, cudaStream_t stream);

}  // namespace zccl

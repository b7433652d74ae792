// zccl_internal.h -- launch interface between the C-ABI host layer and the
// kernels (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/zccl.h"

namespace zccl {

struct WsCtrl;

struct CompressArgs {
    const zccl_segment_t* segs;  // device descriptors (batched) or nullptr
    zccl_segment_t single;       // the one segment when segs == nullptr
    uint32_t n_segs;
    uint32_t max_units;          // flag words available = chunk capacity
    uint8_t lut[8];
    uint64_t* out_bytes;         // device [n_segs]
    WsCtrl* ctrl;
    uint64_t* flags;
    uint64_t n_flag_words;
    uint32_t* status;
};

struct DecompressArgs {
    const uint8_t* in;
    uint64_t in_bytes;
    uint16_t* out;
    uint64_t n;
    WsCtrl* ctrl;
    uint64_t* flags;
    uint64_t n_flag_words;
    uint32_t* status;
};

struct ReduceArgs {
    const void* const* streams;  // device [S]
    const uint64_t* in_bytes;    // device [S]
    uint32_t S;
    uint16_t* out;
    uint64_t n;
    WsCtrl* ctrl;
    uint64_t* flags;             // [S][units]
    uint64_t n_flag_words;
    uint32_t* status;
};

size_t compress_smem_bytes(uint32_t n_segs);
cudaError_t launch_compress(const CompressArgs& a, uint32_t grid, cudaStream_t stream);
int compress_ctas_per_sm(uint32_t n_segs);

cudaError_t launch_decompress(const DecompressArgs& a, uint32_t grid, cudaStream_t stream);
int decompress_ctas_per_sm();

cudaError_t launch_reduce(const ReduceArgs& a, uint32_t grid, cudaStream_t stream);
int reduce_ctas_per_sm(uint32_t S);

}  // namespace zccl

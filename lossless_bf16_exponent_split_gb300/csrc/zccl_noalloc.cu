// zccl_noalloc.cu -- zccl_decompress_noalloc: decompression for callers that
// cannot allocate device memory.
//
// Some callers of a codec that sits inside a collective cannot call
// cudaMalloc: a communication library's progress thread or transport
// plugin, or a framework hook that must stay inside the framework's own
// memory pool, where an extra allocation can block on device-wide
// synchronisation, fail under a fixed memory budget, or fragment the pool
// mid-collective.  They still pass their own input and output buffers; this
// entry point supplies the workspace itself, from one static device array
// of kNoAllocScratchBytes compiled into the library.
//
// The array exists once per GPU that loads the library and lives until the
// process exits.  Its device address is looked up once per device (the
// first call made with that device current), so make that first call before
// any stream capture.  All calls share the array: calls whose execution
// overlaps on the GPU (e.g. on two streams) race and must not be issued.
#include <cstdint>
#include <mutex>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace {

constexpr uint64_t kNoAllocScratchBytes = 1ull << 20;  // 1 MiB; must match ZCCL_NOALLOC_SCRATCH_BYTES
static_assert(kNoAllocScratchBytes == ZCCL_NOALLOC_SCRATCH_BYTES, "header and library agree");

// The workspace of zccl_decompress_noalloc.  In host code this name is only
// a stand-in for the device array: its device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_address[kMaxDevices];  // per device; nullptr until a lookup succeeds

// Device address of the scratch array on the current device, or nullptr on
// failure.  Looked up with that device current; only a successful lookup is
// kept, so a failed one (say, a first call made during stream capture) is
// tried again by the next call.
void* scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_address[dev] = p;
    }
    return g_scratch_address[dev];
}

}  // namespace

extern "C" zccl_status_t zccl_decompress_noalloc(const void* d_in, uint64_t in_bytes, uint16_t* d_out, uint64_t n,
                                                 uint32_t* d_status, cudaStream_t stream)
{
    uint64_t need = 0;
    if (n > ZCCL_NOALLOC_MAX_ELEMS || zccl_workspace_bytes(ZCCL_OP_DECOMPRESS, n, 0, &need) != ZCCL_OK ||
        need > kNoAllocScratchBytes)
        return ZCCL_ERR_INVALID_ARG;  // beyond what the static scratch can hold
    // the argument checks of zccl_decompress, made here too so that a call it
    // would reject queues nothing at all
    if (d_in == nullptr || ((uintptr_t)d_in & 15) || (n > 0 && (d_out == nullptr || ((uintptr_t)d_out & 15))) ||
        ((uintptr_t)d_status & 3) || in_bytes < zccl_zero_point_offset(n))
        return ZCCL_ERR_INVALID_ARG;
    void* ws = scratch_on_current_device();
    if (ws == nullptr) return ZCCL_ERR_CUDA;
    // the part of the workspace the call uses must start at zero; a call that
    // stopped early (timeout) may have left it otherwise
    if (cudaMemsetAsync(ws, 0, need, stream) != cudaSuccess) return ZCCL_ERR_CUDA;
    return zccl_decompress(d_in, in_bytes, d_out, n, ws, kNoAllocScratchBytes, d_status, stream);
}

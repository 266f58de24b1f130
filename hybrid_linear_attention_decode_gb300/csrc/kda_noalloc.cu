// kda_noalloc.cu -- chunked prefill for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for the prefill workspace:
//   * a serving engine whose caching allocator already owns every free byte of the GPU, so an extra
//     cudaMalloc would fail or fragment the engine's pool, and which hands kernels only the tensors
//     it manages;
//   * plug-in or callback interfaces that pass input and output tensors but no allocator;
//   * processes that forbid device allocation after start-up (fixed memory budgets).
// For them, kda_prefill_chunked_noalloc runs the same kernels with a workspace taken from a fixed
// array compiled into this library.  The array lives in this file's device module: under CUDA's lazy
// module loading the driver allocates it on a device when the module first loads there, which is the first
// call's address lookup on that device.  That first call (one with nseq = 0 does only the set-up) belongs at
// start-up, before the caller reserves its memory and before any stream capture; the array is then held
// until the process exits.
#include <atomic>

#include <cuda_runtime.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

// The fixed scratch: one per device, shared by every call on that device.
static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device.  In host code the array's name is only a
// host-side stand-in, so the address is resolved once per device with cudaGetSymbolAddress while
// that device is current.  Returns nullptr on failure.
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_kda_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
    g_scratch_addr[dev].store(addr, std::memory_order_release);
    return addr;
}

}  // namespace

extern "C" KDA_API int kda_prefill_chunked_noalloc(
    const kda_pool *pool, const kda_params *prm, int32_t nseq, int64_t total_tokens, const int32_t *cu_seqlens,
    const int64_t *start_pos, const int32_t *src_slot, const int32_t *dst_slot, int32_t chunk, int64_t ckpt_interval,
    const int32_t *ckpt_offsets, const int32_t *ckpt_slots, const uint16_t *q, const uint16_t *k, const uint16_t *v,
    const uint16_t *a, const uint16_t *b, const uint16_t *z, uint16_t *y, int32_t *dev_status, kda_stream_t stream) {
    kda::clear_error();
    // The argument checks come first, so a bad call fails with its reason and touches no device.
    int rc = kda::check_prefill_args(pool, prm, nseq, total_tokens, cu_seqlens, start_pos, src_slot, dst_slot, chunk,
                                     ckpt_interval, ckpt_offsets, ckpt_slots, q, k, v, a, b, z, y, dev_status);
    if (rc != KDA_OK) return rc;
    // Problems whose workspace does not fit the fixed scratch are rejected before any device call.
    const size_t need = kda_prefill_workspace_bytes(pool, nseq, total_tokens, chunk);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES)
        return kda::fail(KDA_ERR_WORKSPACE, "prefill_noalloc: workspace larger than the static scratch");
    // Per-device set-up (the first call on a device): the scratch's device address, which loads this module
    // and with it the array, and the launchers' own one-time state (kernel attributes, the side stream and
    // events of segmented launches), so that no later call creates anything.
    void *scratch = scratch_on_current_device();
    if (!scratch) return kda::fail(KDA_ERR_CUDA, "prefill_noalloc: cudaGetSymbolAddress of the scratch failed");
    rc = kda::prefill_prepare();
    if (rc != KDA_OK || nseq == 0) return rc;
    // Every field of the workspace is written before it is read, so the contents left by an earlier
    // call need no clearing.
    return kda_prefill_chunked(pool, prm, nseq, total_tokens, cu_seqlens, start_pos, src_slot, dst_slot, chunk,
                               ckpt_interval, ckpt_offsets, ckpt_slots, q, k, v, a, b, z, y, scratch,
                               (size_t)KDA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}

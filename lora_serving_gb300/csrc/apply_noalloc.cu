// apply_noalloc.cu -- lora_apply without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call in: a serving
// engine that has already reserved nearly all free HBM for its KV-cache
// pool (so a cudaMalloc would fail), or a plug-in hosted by an engine that
// forbids allocations outside its own pool, or a latency-critical loop where
// cudaMalloc's implicit device synchronisation is not acceptable.  For them,
// lora_apply_noalloc keeps lora_apply's workspace (the intermediate v, fp32
// and as bf16 hi/lo planes) in a fixed scratch array compiled into this
// library, instead of a workspace the caller would have to allocate.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds LORA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the array's name as a device address (on the host
// it is only a stand-in), so the first call on each device looks the
// address up with cudaGetSymbolAddress, with that device current, and keeps
// it for the life of the process; a device reset (cudaDeviceReset, or a
// reset of the primary context) reloads the module and may move the array,
// after which the kept address is stale and this entry point must not be
// called again on that device.  Nothing in the array needs to start at zero: within one call, every
// element the expand reads has been written by that call's shrink.  All
// calls share the one array, so calls that may run at the same time on the
// GPU (on different streams, say) race on it.

#include <mutex>

#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_apply_scratch[LORA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_apply_scratch on the current device (looked up once).
lora_status_t scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_apply_scratch) != cudaSuccess || !p) return LORA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_apply_noalloc(lora_bf16_t* y, int ld_y, const lora_bf16_t* x, int ld_x, int h_in,
                                            const lora_proj_t* projs, int n_proj, int r_slot, int n_slots,
                                            const lora_meta_t* meta, uint32_t flags, int32_t* dev_status,
                                            lora_stream_t stream)
{
    if (!projs || !meta || n_proj <= 0 || n_proj > LORA_MAX_PROJ) return LORA_ERR_INVALID_ARG;
    // The counts lora_apply checks first, so a bad rank reports what
    // lora_apply would report rather than a scratch-size failure.
    if (meta->n_rows < 0 || n_slots <= 0 || r_slot <= 0) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    if (lora_apply_workspace_bytes(meta->n_rows, n_proj, r_slot) > LORA_NOALLOC_SCRATCH_BYTES)
        return LORA_ERR_WORKSPACE;   // batch too large for the built-in scratch
    void* scratch = nullptr;
    const lora_status_t st = scratch_address(&scratch);
    if (st != LORA_OK) return st;
    return lora_apply(y, ld_y, x, ld_x, h_in, projs, n_proj, r_slot, n_slots, meta, scratch,
                      LORA_NOALLOC_SCRATCH_BYTES, flags, dev_status, stream);
}

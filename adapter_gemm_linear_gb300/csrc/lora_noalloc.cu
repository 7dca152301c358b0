// lora_linear_forward_noalloc: the forward with its scratch memory taken from
// a fixed array that the library itself places in device memory, for callers
// that cannot allocate device memory (see include/lora.h).
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds LORA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the array's name as a device address (on the host the
// name denotes a host-side stand-in), so the real address is looked up with
// cudaGetSymbolAddress while that device is current, and that address is
// what the kernels receive.  The lookup is kept per device together with the
// CUDA context it was made in; after a device reset (a new primary context)
// the next call looks the address up again instead of using a stale one.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "lora.h"
#include "lora_internal.h"

namespace {

static __device__ __align__(256) unsigned char lora_noalloc_scratch[LORA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
uint64_t g_scratch_ctx[kMaxDevices] = {};  // context id of each lookup (0: unknown, look up again)

// Device address of this device's copy of the scratch array in the current
// context; the first call for a device (or context) does the lookup.
lora_status_t scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    const uint64_t ctx = lora::current_context_id();
    if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, lora_noalloc_scratch);
        if (e != cudaSuccess || !p) return LORA_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = lora::current_context_id();  // the lookup made the context current
    }
    *out = g_scratch_addr[dev];
    return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_linear_forward_noalloc(const lora_forward_args_t *args, void *stream) {
    if (!args) return LORA_ERR_INVALID_ARG;
    lora_forward_args_t a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    const size_t need = lora_forward_workspace_bytes(&a);
    if (need == 0) return lora_linear_forward(&a, stream);  // reports the invalid argument
    if (need > LORA_NOALLOC_SCRATCH_BYTES) return LORA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const lora_status_t s = scratch_for_current_device(&scratch);
    if (s != LORA_OK) return s;
    a.workspace = scratch;
    a.workspace_bytes = LORA_NOALLOC_SCRATCH_BYTES;
    return lora_linear_forward(&a, stream);
}

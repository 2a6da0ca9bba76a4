// Attention backward for callers that cannot allocate device memory.
//
// ulysses_attn_bwd needs a caller-provided workspace (an fp32 dQ accumulator and the
// per-row Delta). Some callers have no way to provide one: for example a plugin running
// inside a host framework whose device memory is owned entirely by that framework's pool,
// or a runtime whose memory plan is fixed at start-up and which may not call cudaMalloc
// afterwards. For them this file keeps the workspace in a file-scope device array of a
// fixed size, so that the call itself allocates nothing.
//
// The array is part of the library's device image: every GPU that loads the library holds
// its ULYSSES_BWD_NOALLOC_SCRATCH_BYTES until the process exits. In host code its name is
// only a host-side stand-in, so its device address is looked up once per device with
// cudaGetSymbolAddress and that address is what the kernels receive.
#include <mutex>

#include "common.cuh"
#include "ulysses_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[ULYSSES_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array; the first call on a device looks it up
// (with that device current) and caches it.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int ulysses_attn_bwd_noalloc(ulysses_shape_t shape, const ulysses_mask_t* mask, float softmax_scale,
                                        int io_layout, const void* q, const void* k, const void* v, const void* o,
                                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                        void* stream) {
    // a shape whose workspace does not fit the array is refused before anything else
    if (ulysses_attn_bwd_workspace_size(shape) > size_t(ULYSSES_BWD_NOALLOC_SCRATCH_BYTES))
        return ULYSSES_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (shape.B > 0 && shape.L > 0) {
        scratch = scratch_address();
        if (!scratch) return ULYSSES_ERR_CUDA;
    }
    // the regular entry point validates every other argument and launches the kernels
    return ulysses_attn_bwd(shape, mask, softmax_scale, io_layout, q, k, v, o, lse, dO, dq, dk, dv, scratch,
                            size_t(ULYSSES_BWD_NOALLOC_SCRATCH_BYTES), stream);
}

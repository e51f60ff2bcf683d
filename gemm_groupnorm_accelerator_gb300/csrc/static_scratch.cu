// An entry point for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocator) on the path that runs the
// operator: code running inside a host framework that owns every device allocation, a plugin whose
// host forbids allocation after initialisation, or a real-time loop where an allocation could
// block or fail. conv1d_norm_run_static_scratch() gives them the whole operator with no
// allocation at all: the scratch the kernels need (status word, packed weights, statistics) lives
// in one fixed-size array in device global memory that is part of this library's device image.
// Every GPU that loads the library holds this array until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "c1n_internal.h"

namespace {

// The shared scratch. Host code must not use this name as an address: on the host it is only a
// stand-in for the symbol. Its device address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_static_scratch[C1N_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" c1n_status conv1d_norm_run_static_scratch(c1n_desc* desc, const c1n_args* args, c1n_stream_t stream) {
    char msg[256];
    if (!desc || !args) {
        c1n::set_last_error("desc and args must be non-NULL");
        return C1N_ERR_INVALID_ARG;
    }
    if (args->workspace != nullptr) {
        c1n::set_last_error("args->workspace must be NULL: the fixed scratch is the workspace");
        return C1N_ERR_INVALID_ARG;
    }
    // Every descriptor packs its weights into the same array, so weights packed by an earlier call
    // may belong to another operator; the pack also resets the fused GroupNorm exchange words.
    // Every call therefore packs.
    if (args->flags & C1N_FLAG_WEIGHTS_PACKED) {
        c1n::set_last_error("C1N_FLAG_WEIGHTS_PACKED is not accepted here: the fixed scratch is shared by every "
                            "descriptor, so each call packs its own weights");
        return C1N_ERR_INVALID_ARG;
    }
    size_t need = 0;
    c1n_status st = conv1d_norm_workspace_size(desc, &need);
    if (st != C1N_OK) return st;
    if (need > (size_t)C1N_STATIC_SCRATCH_BYTES) {
        snprintf(msg, sizeof(msg), "this operator needs %zu bytes of scratch; the fixed scratch holds %u bytes",
                 need, (unsigned)C1N_STATIC_SCRATCH_BYTES);
        c1n::set_last_error(msg);
        return C1N_ERR_WORKSPACE;
    }
    void* ptr = nullptr;
    cudaError_t e = scratch_address(&ptr);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the fixed scratch failed: %s", cudaGetErrorString(e));
        c1n::set_last_error(msg);
        return C1N_ERR_CUDA;
    }
    // The status word must start at zero; everything else the kernels read is written first.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(ptr, 0, c1n::kWsStatusBytes, s);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "clearing the status word failed: %s", cudaGetErrorString(e));
        c1n::set_last_error(msg);
        return C1N_ERR_CUDA;
    }
    // Attach the array as the descriptor's workspace so conv1d_norm_check(desc, NULL, stream)
    // reads this call's status word.
    st = conv1d_norm_set_workspace(desc, ptr, (size_t)C1N_STATIC_SCRATCH_BYTES);
    if (st != C1N_OK) return st;
    c1n_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    return conv1d_norm_run_ex(desc, &a, stream);
}

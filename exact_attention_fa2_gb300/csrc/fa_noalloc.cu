// fa_noalloc.cu - fa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// fa_bwd needs a device workspace (D and the fp32 dQ accumulator) that the
// caller allocates.  Some callers cannot call cudaMalloc or any allocating
// routine at that point: code running inside a custom allocator's callbacks,
// runtimes that hand out only preallocated tensors and forbid allocation
// during a step, or plugins embedded in hosts that own all device memory.
// For them this entry point takes its workspace from a fixed array compiled
// into the library instead, so the call allocates nothing.

#include "fa_gb300.h"
#include "fa_launch.h"

#include <cstdio>
#include <mutex>

namespace {

// Built-in backward workspace.  Every GPU that loads the library holds these
// bytes until the process exits; all fa_bwd_noalloc calls on a device share
// them and they keep the last call's contents (fa_bwd rewrites D and zeroes
// the dQ accumulator on every call).
constexpr size_t kScratchBytes = (size_t)FA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the built-in scratch on the current device.  In host code
// `g_bwd_scratch` names a host-side stand-in, not device memory, so the
// address is looked up once per device with that device current.
int scratch_ptr(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fa::set_last_error(FA_ERR_CUDA, "fa_bwd_noalloc: cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return fa::set_last_error(FA_ERR_UNSUPPORTED, "fa_bwd_noalloc: device ordinal too large");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof(msg), "fa_bwd_noalloc: cudaGetSymbolAddress of the built-in scratch failed: %s",
                     cudaGetErrorString(e));
            return fa::set_last_error(FA_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_scratch_bytes(void) { return kScratchBytes; }

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int S, int d, int causal, float scale, int dtype, void* stream) {
    const size_t need = fa_bwd_workspace_size(B, H, S, d, dtype);
    if (need > kScratchBytes) {
        // fa_bwd's own argument checks come first: given no workspace they end
        // in FA_ERR_WORKSPACE, before any device call, when every other rule
        // holds; a call that breaks one of them gets that rule's code.
        const int rc = fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, nullptr, 0, B, H, S, d, causal, scale, dtype, stream);
        if (rc != FA_ERR_WORKSPACE) return rc;
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "fa_bwd_noalloc: this problem needs %zu bytes of workspace but the built-in scratch holds %zu; "
                 "call fa_bwd with a caller-allocated workspace instead", need, kScratchBytes);
        return fa::set_last_error(FA_ERR_WORKSPACE, msg);
    }
    void* ws = nullptr;
    if (need > 0) {
        int rc = scratch_ptr(&ws);
        if (rc != FA_OK) return rc;
    }
    // Same checks and kernels as fa_bwd, with the built-in array as workspace.
    return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, ws, need > 0 ? kScratchBytes : 0,
                  B, H, S, d, causal, scale, dtype, stream);
}

}  // extern "C"

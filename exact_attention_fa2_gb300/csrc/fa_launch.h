// fa_launch.h - host-side launch interface between the C ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <algorithm>
#include <atomic>

namespace fa {

enum { DT_BF16 = 0, DT_FP32 = 1 };

// Element strides of a [B, H, rows, d] view whose head dimension is
// contiguous (stride 1).
struct View {
    long long b, h, s;
    __host__ __device__ long long off(int bi, int hi, long long row) const { return bi * b + hi * h + row * s; }
};
inline View contiguous_view(int H, int rows, int d) {
    return View{(long long)H * rows * d, (long long)rows * d, (long long)d};
}

struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;             // contiguous [B, H, S] fp32
    int B, H, S, d;         // S = N_q, the number of query rows
    int causal;
    float scale;
    int dtype;
    cudaStream_t stream;
    unsigned int* status;   // device status word (timeouts, index checks)
    int Sk;                 // N_k, the number of key rows
    View vq, vk, vv, vo;    // strides of q, o ([B,H,S,d]) and k, v ([B,H,Sk,d])
};

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const void* dO;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    float* Dvec;            // [B*H*S] fp32, inside the workspace
    float* dQacc;           // [B*H*S*d] fp32, inside the workspace (null: deterministic backward)
    int B, H, S, d;         // S = N_q
    int causal;
    float scale;
    int dtype;
    cudaStream_t stream;
    unsigned int* status;
    int Sk;                 // N_k
    View vq, vk, vv, vo, vdo, vdq, vdk, vdv;   // q, o, dO, dq: [B,H,S,d]; k, v, dk, dv: [B,H,Sk,d]
};

// Raise `kern`'s dynamic shared-memory limit to `bytes`, once per device
// (the attribute persists in the context; setting it on every launch costs a
// driver call).  A cudaDeviceReset inside the process is not tracked: the
// next launch of the kernel then fails with a launch error.
template <auto KERN>
cudaError_t set_smem_limit(int bytes) {
    static std::atomic<unsigned long long> done{0};   // bit i: set on device i (< 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launch `kern` as a programmatic dependent of the previous kernel on the
// stream: its blocks may start while that kernel drains and must execute
// griddepcontrol.wait before reading anything the previous kernel writes (or
// writing anything it reads).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// fp32 (and generic) FMA-pipe kernels.
cudaError_t launch_fwd_simt(const FwdArgs& a);
cudaError_t launch_bwd_simt(const BwdArgs& a);

// Backward helpers: D = rowsum(O*dO) plus zeroing of dQacc; dQacc -> dq.
cudaError_t launch_bwd_preprocess(const BwdArgs& a);
cudaError_t launch_dq_convert(const BwdArgs& a);
// dK = dV = 0 on key rows [row0, Sk): keys no query attends (no query rows
// at all, or causal keys past the last query tile).
cudaError_t launch_zero_rows(const BwdArgs& a, int row0);

// Record `msg` as the calling thread's last error (read by fa_get_last_error)
// and return `code`.
int set_last_error(int code, const char* msg);

// bf16 tensor-core (tcgen05) kernels.
cudaError_t launch_fwd_tc(const FwdArgs& a);
// Partial forward over keys [key_begin, key_end) (key_begin a multiple of
// 128): normalised fp32 O into o32, L into a.lse (-inf where no key).
cudaError_t launch_fwd_tc_partial(const FwdArgs& a, int key_begin, int key_end, float* o32);
cudaError_t launch_fwd_simt_partial(const FwdArgs& a, int key_begin, int key_end, float* o32);
// Merge of two partial results over disjoint key sets.
struct MergeArgs {
    const float* o_a;
    const float* lse_a;
    const float* o_b;
    const float* lse_b;
    void* o;
    float* lse;
    long long rows;
    int d;
    int dtype;
    cudaStream_t stream;
};
cudaError_t launch_merge(const MergeArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a);

// Deterministic backward: dK/dV without dQ, then a query-tile-outer dQ pass
// that writes dq directly (no dQacc, no atomics).
cudaError_t launch_bwd_tc_dkdv(const BwdArgs& a);
cudaError_t launch_bwd_dq_tc(const BwdArgs& a);
cudaError_t launch_bwd_dq_simt(const BwdArgs& a);

}  // namespace fa

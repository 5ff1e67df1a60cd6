// fa_api.cu - the C ABI (include/fa_gb300.h): argument checks, workspace
// layout, kernel selection and error reporting.  No device memory is
// allocated here; the only device state is one status word per device that
// kernels set when a bounded wait runs out or an index check fails.

#include "fa_gb300.h"
#include "fa_common.cuh"
#include "fa_launch.h"
#include "sm103_ptx.cuh"

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

namespace {

__device__ unsigned int g_status_word;

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};

// Device address of this device's status word (looked up once per device).
int status_ptr(unsigned int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_status_ptr[dev];
    return FA_OK;
}

bool supported_d(int d) {
    return d == 16 || d == 32 || d == 64 || d == 80 || d == 96 || d == 128;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks shared by forward and backward.  Returns FA_OK, an error code, or 1
// for a valid empty problem (nothing to launch).
int check_sizes(int B, int H, int S, int d, float scale, int dtype) {
    if (B < 0 || H < 0 || S < 0)
        return fail(FA_ERR_INVALID_ARG, "negative size: B=%d H=%d S=%d", B, H, S);
    if (dtype != FA_BF16 && dtype != FA_FP32)
        return fail(FA_ERR_UNSUPPORTED, "dtype %d is not FA_BF16 or FA_FP32", dtype);
    if (!supported_d(d))
        return fail(FA_ERR_UNSUPPORTED, "head dim %d not in {16,32,64,80,96,128}", d);
    if (!std::isfinite(scale))
        return fail(FA_ERR_INVALID_ARG, "scale is not finite");
    const long long n = (long long)B * H * S * d;
    if (n >= (1LL << 31))
        return fail(FA_ERR_UNSUPPORTED, "B*H*S*d = %lld elements exceeds 2^31-1", n);
    if ((long long)B * H > 65535LL)
        return fail(FA_ERR_UNSUPPORTED, "B*H = %lld exceeds 65535", (long long)B * H);
    if ((long long)B * H * S == 0) return 1;
    return FA_OK;
}

int check_ptr(const void* p, const char* name) {
    if (!p) return fail(FA_ERR_INVALID_ARG, "%s is null", name);
    if (!aligned16(p)) return fail(FA_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    return FA_OK;
}

// The view of a [B, H, rows, d] array from a host array of element strides
// {batch, head, row} (NULL: contiguous).  A stride whose dimension has more
// than one index must be positive and a multiple of 16 bytes.
int get_view(const long long* st, int B, int H, int rows, int d, int dtype, const char* name, fa::View* out) {
    if (!st) {
        *out = fa::contiguous_view(H, rows, d);
        return FA_OK;
    }
    const long long elt = dtype == FA_BF16 ? 2 : 4;
    const int ext[3] = {B, H, rows};
    static const char* dims[3] = {"batch", "head", "row"};
    for (int i = 0; i < 3; ++i) {
        if (ext[i] <= 1) continue;
        if (st[i] <= 0)
            return fail(FA_ERR_INVALID_ARG, "%s %s stride %lld is not positive", name, dims[i], st[i]);
        if ((st[i] * elt) % 16 != 0 || st[i] * elt >= (1LL << 40))
            return fail(FA_ERR_MISALIGNED, "%s %s stride %lld elements is not a multiple of 16 bytes (or too large)",
                        name, dims[i], st[i]);
    }
    *out = fa::View{st[0], st[1], st[2]};
    return FA_OK;
}

// Sizes of a call with N_q = Sq query rows and N_k = Sk key rows.  Returns
// FA_OK, an error code, or 1 when there is nothing to compute.
int check_sizes_qk(int B, int H, int Sq, int Sk, int d, float scale, int dtype) {
    int rq = check_sizes(B, H, Sq, d, scale, dtype);
    if (rq < 0) return rq;
    int rk = check_sizes(B, H, Sk, d, scale, dtype);
    if (rk < 0) return rk;
    if ((long long)B * H == 0 || Sq == 0) return 1;
    if (Sk == 0) return fail(FA_ERR_INVALID_ARG, "no key rows (Sk = 0) for %d query rows", Sq);
    return FA_OK;
}

// ---- optional kernel timing (fa_profile_enable / fa_profile_read)
enum { PROF_FWD = 0, PROF_PRE = 1, PROF_BWD = 2, PROF_CONV = 3, PROF_DQ = 4, PROF_KINDS = 5 };
struct ProfRec { cudaEvent_t a, b; int kind; };
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_ev_pool;

cudaEvent_t prof_event() {
    if (!g_ev_pool.empty()) {
        cudaEvent_t e = g_ev_pool.back();
        g_ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Runs `launch` on `stream`, bracketed by timing events when profiling is on.
template <typename F>
cudaError_t timed(int kind, cudaStream_t stream, F&& launch) {
    cudaEvent_t a = nullptr, b = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        if (g_prof_on) { a = prof_event(); b = prof_event(); }
    }
    if (a && b) cudaEventRecord(a, stream);
    cudaError_t e = launch();
    if (a && b) {
        cudaEventRecord(b, stream);
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_prof_pending.push_back({a, b, kind});
    }
    return e;
}

// One non-blocking helper stream per (device, caller stream), created on first
// use by fa_fwd_bwd_host and kept for the life of the process.
std::mutex g_side_mu;
std::map<std::pair<int, void*>, cudaStream_t> g_side;

int side_stream(void* user, cudaStream_t* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_side_mu);
    auto it = g_side.find({dev, user});
    if (it == g_side.end()) {
        cudaStream_t st = nullptr;
        e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
        it = g_side.emplace(std::make_pair(dev, user), st).first;
    }
    *out = it->second;
    return FA_OK;
}

// Device layout of fa_fwd_bwd_host's buffer: q, k, v, dO, o, dq, dk, dv, lse,
// then the backward workspace, each starting on a 256-byte boundary.
struct HostStepLayout {
    size_t arr, lse, ws, total;
};
HostStepLayout host_step_layout(int B, int H, int S, int d, int dtype) {
    const size_t rows = (size_t)B * H * S;
    const size_t elt = dtype == FA_BF16 ? 2 : 4;
    HostStepLayout L;
    L.arr = align_up(rows * d * elt, 256);
    L.lse = align_up(rows * sizeof(float), 256);
    L.ws = fa_bwd_workspace_size(B, H, S, d, dtype);
    L.total = 8 * L.arr + L.lse + L.ws;
    return L;
}

}  // namespace

int fa::set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

extern "C" {

int fa_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = on != 0;
    return FA_OK;
}

int fa_profile_read(double* ms, int* launches) {
    if (!ms || !launches) return fail(FA_ERR_INVALID_ARG, "null output array");
    std::vector<ProfRec> recs;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        recs.swap(g_prof_pending);
    }
    int rc = FA_OK;
    for (const ProfRec& r : recs) {
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.a, r.b);
        if (e != cudaSuccess) { rc = cuda_fail(e, "profile event"); continue; }
        ms[r.kind] += t;
        launches[r.kind] += 1;
    }
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (const ProfRec& r : recs) { g_ev_pool.push_back(r.a); g_ev_pool.push_back(r.b); }
    return rc;
}


int fa_version(void) { return 100; }

const char* fa_get_last_error(void) { return g_err; }

}  // extern "C"

namespace {

int fwd_common(const void* q, const long long* sq, const void* k, const long long* sk, const void* v,
               const long long* sv, void* o, const long long* so, float* lse, int B, int H, int Sq, int Sk, int d,
               int causal, float scale, int dtype, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes_qk(B, H, Sq, Sk, d, scale, dtype);
    if (rc == 1) return FA_OK;
    if (rc) return rc;
    if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
        (rc = check_ptr(o, "o")) || (rc = check_ptr(lse, "lse")))
        return rc;
    fa::FwdArgs a{q, k, v, o, lse, B, H, Sq, d, causal ? 1 : 0, scale, dtype,
                  static_cast<cudaStream_t>(stream), nullptr};
    a.Sk = Sk;
    if ((rc = get_view(sq, B, H, Sq, d, dtype, "q", &a.vq)) || (rc = get_view(sk, B, H, Sk, d, dtype, "k", &a.vk)) ||
        (rc = get_view(sv, B, H, Sk, d, dtype, "v", &a.vv)) || (rc = get_view(so, B, H, Sq, d, dtype, "o", &a.vo)))
        return rc;
    if ((rc = status_ptr(&a.status))) return rc;
    cudaError_t e = timed(PROF_FWD, a.stream, [&] {
        return dtype == FA_BF16 ? fa::launch_fwd_tc(a) : fa::launch_fwd_simt(a);
    });
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int S, int d, int causal, float scale, int dtype, void* stream) {
    return fwd_common(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, B, H, S, S, d, causal, scale, dtype,
                      stream);
}

int fa_fwd_strided(const void* q, const long long* q_strides, const void* k, const long long* k_strides,
                   const void* v, const long long* v_strides, void* o, const long long* o_strides, float* lse,
                   int B, int H, int Sq, int Sk, int d, int causal, float scale, int dtype, void* stream) {
    return fwd_common(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, B, H, Sq, Sk, d, causal, scale,
                      dtype, stream);
}

int fa_fwd_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                   int B, int H, int S, int d, int key_begin, int key_end, int causal, float scale, int dtype,
                   void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(B, H, S, d, scale, dtype);
    if (rc == 1) return FA_OK;
    if (rc) return rc;
    if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
        (rc = check_ptr(o_part, "o_part")) || (rc = check_ptr(lse_part, "lse_part")))
        return rc;
    if (key_begin < 0 || key_end > S || key_begin >= key_end)
        return fail(FA_ERR_INVALID_ARG, "key window [%d, %d) is empty or outside [0, %d)", key_begin, key_end, S);
    if (key_begin % 128 != 0)
        return fail(FA_ERR_UNSUPPORTED, "key_begin %d is not a multiple of 128", key_begin);
    fa::FwdArgs a{q, k, v, nullptr, lse_part, B, H, S, d, causal ? 1 : 0, scale, dtype,
                  static_cast<cudaStream_t>(stream), nullptr};
    a.Sk = S;
    a.vq = a.vk = a.vv = a.vo = fa::contiguous_view(H, S, d);
    if ((rc = status_ptr(&a.status))) return rc;
    cudaError_t e = timed(PROF_FWD, a.stream, [&] {
        return dtype == FA_BF16 ? fa::launch_fwd_tc_partial(a, key_begin, key_end, o_part)
                                : fa::launch_fwd_simt_partial(a, key_begin, key_end, o_part);
    });
    if (e != cudaSuccess) return cuda_fail(e, "partial forward launch");
    return FA_OK;
}

int fa_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b, void* o, float* lse,
             int B, int H, int S, int d, int dtype, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(B, H, S, d, 1.f, dtype);
    if (rc == 1) return FA_OK;
    if (rc) return rc;
    if ((rc = check_ptr(o_a, "o_a")) || (rc = check_ptr(lse_a, "lse_a")) || (rc = check_ptr(o_b, "o_b")) ||
        (rc = check_ptr(lse_b, "lse_b")) || (rc = check_ptr(o, "o")) || (rc = check_ptr(lse, "lse")))
        return rc;
    fa::MergeArgs a{o_a, lse_a, o_b, lse_b, o, lse, (long long)B * H * S, d, dtype, static_cast<cudaStream_t>(stream)};
    cudaError_t e = fa::launch_merge(a);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return FA_OK;
}

size_t fa_bwd_workspace_size(int B, int H, int S, int d, int dtype) {
    if (B <= 0 || H <= 0 || S <= 0 || !supported_d(d) || (dtype != FA_BF16 && dtype != FA_FP32))
        return 0;
    const size_t rows = (size_t)B * H * S;
    return align_up(rows * sizeof(float), 256) + rows * (size_t)d * sizeof(float);
}

}  // extern "C"

namespace {

// Every backward entry point: the same checks, D preprocess and dK/dV loop;
// dQ either by atomics into dQacc plus a convert, or (det) by its own
// query-tile-outer pass.
int bwd_common(const void* q, const long long* sq, const void* k, const long long* sk, const void* v,
               const long long* sv, const void* o, const long long* so, const void* dO, const long long* sdo,
               const float* lse, void* dq, const long long* sdq, void* dk, const long long* sdk, void* dv,
               const long long* sdv, void* workspace, size_t workspace_bytes, int B, int H, int Sq, int Sk, int d,
               int causal, float scale, int dtype, void* stream, bool det) {
    g_err[0] = 0;
    int rc = check_sizes_qk(B, H, Sq, Sk, d, scale, dtype);
    const bool keys_only = rc == 1 && (long long)B * H > 0 && Sk > 0;   // no queries: dK = dV = 0
    if (rc == 1 && !keys_only) return FA_OK;
    if (rc < 0) return rc;
    if ((rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv"))) return rc;
    fa::BwdArgs a{q, k, v, o, dO, lse, dq, dk, dv, nullptr, nullptr, B, H, Sq, d, causal ? 1 : 0, scale,
                  dtype, static_cast<cudaStream_t>(stream), nullptr};
    a.Sk = Sk;
    if ((rc = get_view(sdk, B, H, Sk, d, dtype, "dk", &a.vdk)) || (rc = get_view(sdv, B, H, Sk, d, dtype, "dv", &a.vdv)))
        return rc;
    if (keys_only) {
        cudaError_t e = fa::launch_zero_rows(a, 0);
        if (e != cudaSuccess) return cuda_fail(e, "zero dk/dv launch");
        return FA_OK;
    }
    if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
        (rc = check_ptr(o, "o")) || (rc = check_ptr(dO, "dO")) || (rc = check_ptr(lse, "lse")) ||
        (rc = check_ptr(dq, "dq")))
        return rc;
    if ((rc = get_view(sq, B, H, Sq, d, dtype, "q", &a.vq)) || (rc = get_view(sk, B, H, Sk, d, dtype, "k", &a.vk)) ||
        (rc = get_view(sv, B, H, Sk, d, dtype, "v", &a.vv)) || (rc = get_view(so, B, H, Sq, d, dtype, "o", &a.vo)) ||
        (rc = get_view(sdo, B, H, Sq, d, dtype, "dO", &a.vdo)) || (rc = get_view(sdq, B, H, Sq, d, dtype, "dq", &a.vdq)))
        return rc;
    const size_t rows = (size_t)B * H * Sq;
    const size_t need = det ? rows * sizeof(float) : fa_bwd_workspace_size(B, H, Sq, d, dtype);
    if (!workspace || workspace_bytes < need)
        return fail(FA_ERR_WORKSPACE, "workspace %p of %zu bytes, need %zu", workspace, workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(FA_ERR_MISALIGNED, "workspace is not 256-byte aligned");
    a.Dvec = static_cast<float*>(workspace);
    a.dQacc = det ? nullptr
                  : reinterpret_cast<float*>(static_cast<char*>(workspace) + align_up(rows * sizeof(float), 256));
    if ((rc = status_ptr(&a.status))) return rc;
    cudaError_t e = timed(PROF_PRE, a.stream, [&] { return fa::launch_bwd_preprocess(a); });
    if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
    e = timed(PROF_BWD, a.stream, [&] {
        if (dtype != FA_BF16) return fa::launch_bwd_simt(a);
        return det ? fa::launch_bwd_tc_dkdv(a) : fa::launch_bwd_tc(a);
    });
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    if (causal && dtype == FA_BF16) {
        // The tensor-core kernel covers the key tiles some query reaches under
        // the causal mask; the key rows of the tiles past the last query tile
        // get zero gradients here.
        e = fa::launch_zero_rows(a, ((Sq + 127) / 128) * 128);
        if (e != cudaSuccess) return cuda_fail(e, "zero dk/dv launch");
    }
    if (det) {
        e = timed(PROF_DQ, a.stream, [&] {
            return dtype == FA_BF16 ? fa::launch_bwd_dq_tc(a) : fa::launch_bwd_dq_simt(a);
        });
        if (e != cudaSuccess) return cuda_fail(e, "dq pass launch");
    } else {
        e = timed(PROF_CONV, a.stream, [&] { return fa::launch_dq_convert(a); });
        if (e != cudaSuccess) return cuda_fail(e, "dq convert launch");
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv,
           void* workspace, size_t workspace_bytes,
           int B, int H, int S, int d, int causal, float scale, int dtype, void* stream) {
    return bwd_common(q, nullptr, k, nullptr, v, nullptr, o, nullptr, dO, nullptr, lse, dq, nullptr, dk, nullptr, dv,
                      nullptr, workspace, workspace_bytes, B, H, S, S, d, causal, scale, dtype, stream, false);
}

int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes,
                         int B, int H, int S, int d, int causal, float scale, int dtype, void* stream) {
    return bwd_common(q, nullptr, k, nullptr, v, nullptr, o, nullptr, dO, nullptr, lse, dq, nullptr, dk, nullptr, dv,
                      nullptr, workspace, workspace_bytes, B, H, S, S, d, causal, scale, dtype, stream, true);
}

int fa_bwd_strided(const void* q, const long long* q_strides, const void* k, const long long* k_strides,
                   const void* v, const long long* v_strides, const void* o, const long long* o_strides,
                   const void* dO, const long long* do_strides, const float* lse,
                   void* dq, const long long* dq_strides, void* dk, const long long* dk_strides,
                   void* dv, const long long* dv_strides, void* workspace, size_t workspace_bytes,
                   int B, int H, int Sq, int Sk, int d, int causal, float scale, int dtype, int deterministic,
                   void* stream) {
    return bwd_common(q, q_strides, k, k_strides, v, v_strides, o, o_strides, dO, do_strides, lse, dq, dq_strides,
                      dk, dk_strides, dv, dv_strides, workspace, workspace_bytes, B, H, Sq, Sk, d, causal, scale,
                      dtype, stream, deterministic != 0);
}

size_t fa_fwd_bwd_host_buffer_size(int B, int H, int S, int d, int dtype) {
    if (B <= 0 || H <= 0 || S <= 0 || !supported_d(d) || (dtype != FA_BF16 && dtype != FA_FP32))
        return 0;
    return host_step_layout(B, H, S, d, dtype).total;
}

int fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO,
                    void* o, float* lse, void* dq, void* dk, void* dv,
                    void* dev_buf, size_t dev_buf_bytes,
                    int B, int H, int S, int d, int causal, float scale, int dtype, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(B, H, S, d, scale, dtype);
    if (rc == 1) return FA_OK;
    if (rc) return rc;
    const void* in[4] = {q, k, v, dO};
    void* out[5] = {o, lse, dq, dk, dv};
    const char* in_name[4] = {"q", "k", "v", "dO"};
    const char* out_name[5] = {"o", "lse", "dq", "dk", "dv"};
    for (int i = 0; i < 4; ++i)
        if (!in[i]) return fail(FA_ERR_INVALID_ARG, "%s is null", in_name[i]);
    for (int i = 0; i < 5; ++i)
        if (!out[i]) return fail(FA_ERR_INVALID_ARG, "%s is null", out_name[i]);
    const HostStepLayout L = host_step_layout(B, H, S, d, dtype);
    if (!dev_buf || dev_buf_bytes < L.total)
        return fail(FA_ERR_WORKSPACE, "device buffer %p of %zu bytes, need %zu", dev_buf, dev_buf_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(dev_buf) & 255u)
        return fail(FA_ERR_MISALIGNED, "device buffer is not 256-byte aligned");
    const size_t rows = (size_t)B * H * S;
    const size_t bytes = rows * d * (dtype == FA_BF16 ? 2 : 4);
    char* base = static_cast<char*>(dev_buf);
    void* dev[8];
    for (int i = 0; i < 8; ++i) dev[i] = base + i * L.arr;          // q, k, v, dO, o, dq, dk, dv
    float* lse_d = reinterpret_cast<float*>(base + 8 * L.arr);
    void* ws = base + 8 * L.arr + L.lse;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t side = nullptr;
    if ((rc = side_stream(stream, &side))) return rc;
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};             // call start, dO copied, o/lse copied
    for (int i = 0; i < 3; ++i) {
        cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return cuda_fail(e, "cudaEventCreateWithFlags");
        }
    }
    cudaEvent_t ev_fwd = nullptr;
    cudaError_t e = cudaEventCreateWithFlags(&ev_fwd, cudaEventDisableTiming);
    auto done = [&](int r) {
        for (int i = 0; i < 3; ++i) cudaEventDestroy(ev[i]);   // released once they have completed
        if (ev_fwd) cudaEventDestroy(ev_fwd);
        return r;
    };
    if (e != cudaSuccess) return done(cuda_fail(e, "cudaEventCreateWithFlags"));
    // Inputs: q, k, v on the caller's stream; dO on the helper stream, after
    // the caller's earlier work on the buffer.
    e = cudaEventRecord(ev[0], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev[0], 0);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaMemcpyAsync(dev[i], in[i], bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dev[3], dO, bytes, cudaMemcpyHostToDevice, side);
    if (e == cudaSuccess) e = cudaEventRecord(ev[1], side);
    if (e != cudaSuccess) return done(cuda_fail(e, "host-to-device copies"));
    if ((rc = fa_fwd(dev[0], dev[1], dev[2], dev[4], lse_d, B, H, S, d, causal, scale, dtype, stream))) return done(rc);
    // O and L go back on the helper stream while the backward runs.
    e = cudaEventRecord(ev_fwd, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev_fwd, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o, dev[4], bytes, cudaMemcpyDeviceToHost, side);
    if (e == cudaSuccess) e = cudaMemcpyAsync(lse, lse_d, rows * sizeof(float), cudaMemcpyDeviceToHost, side);
    if (e == cudaSuccess) e = cudaEventRecord(ev[2], side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[1], 0);
    if (e != cudaSuccess) return done(cuda_fail(e, "forward output copies"));
    if ((rc = fa_bwd(dev[0], dev[1], dev[2], dev[4], dev[3], lse_d, dev[5], dev[6], dev[7], ws, L.ws,
                     B, H, S, d, causal, scale, dtype, stream)))
        return done(rc);
    void* host_out[3] = {dq, dk, dv};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
        e = cudaMemcpyAsync(host_out[i], dev[5 + i], bytes, cudaMemcpyDeviceToHost, st);
    // The call is complete on the caller's stream once the helper's copies are.
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[2], 0);
    if (e != cudaSuccess) return done(cuda_fail(e, "gradient copies"));
    return done(FA_OK);
}

}  // extern "C"

namespace {

// One thread waits, through the bounded wait every kernel uses, for an
// mbarrier phase that nothing completes; it gives up after limit_ns, sets
// the status word and returns.
__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        fa::sm103::mbar_init(fa::sm103::smem_u32(&bar), 1);
        abort_flag = 0;
        fa::sm103::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) fa::sm103::mbar_wait(fa::sm103::smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

}  // namespace

extern "C" {

int fa_selftest_bounded_wait(unsigned long long limit_ns, void* stream) {
    g_err[0] = 0;
    if (limit_ns == 0 || limit_ns > 10000000000ull)
        return fail(FA_ERR_INVALID_ARG, "limit %llu ns is outside (0, 10 s]", limit_ns);
    unsigned int* status = nullptr;
    int rc = status_ptr(&status);
    if (rc) return rc;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return FA_OK;
}

int fa_check_status(void* stream) {
    g_err[0] = 0;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (word == 0) return FA_OK;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    if (word & FA_DEV_STATUS_TIMEOUT)
        return fail(FA_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (status 0x%x)", word);
    return fail(FA_ERR_DEVICE_BOUNDS, "a kernel caught an out-of-range index (status 0x%x)", word);
}

}  // extern "C"

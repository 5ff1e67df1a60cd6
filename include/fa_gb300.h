/*
 * fa_gb300.h - C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The library computes exact scaled-dot-product attention
 *     O = softmax(Q K^T * scale) V,   L_i = log sum_j exp((Q K^T * scale)_ij)
 * in the FlashAttention-2 manner (tiled over keys with an online softmax; the
 * S x S score matrix is never written to memory), and its recompute backward
 * (dQ, dK, dV from Q, K, V, O, dO and L, using D = rowsum(O * dO)).
 *
 * Sources for the operations:
 *   - "Stanford CS336 Assignment 2 (Systems)" handout, section 4
 *     "FlashAttention-2": Eq. 4-6 (forward), Eq. 12 (logsumexp L), Eq. 13-19
 *     (backward with recomputation and D), Algorithm 1 (tiled forward),
 *     Algorithm 2 (tiled backward), problem flash_forward (c) (causal mask).
 *   - "CS336 Assignment 2: Systems" blog, FlashAttention-2 section: the
 *     autograd contract forward(Q, K, V, is_causal) -> O saving L, and
 *     backward(dO) -> dQ, dK, dV.
 *   - "Phase T14: fused Flash-Attention kernel - design document" (xtrain):
 *     launch entry points over a C FFI and an fp32 logsumexp.
 *
 * Conventions shared by every entry point
 *   Layout   q, k, v, o, dO, dq, dk, dv are contiguous [B, H, S, d] arrays of
 *            the element type `dtype` (row-major, d fastest).  lse is a
 *            contiguous [B, H, S] fp32 array holding the natural-log L.
 *            Queries and keys share the length S, except in fa_fwd_strided /
 *            fa_bwd_strided, which take N_q query rows and N_k key rows and
 *            strided views (see there).
 *   Causal   causal != 0 keeps key j for query i only when j <= i
 *            (top-left aligned, square).
 *   Pointers every array argument is a DEVICE pointer of the current CUDA
 *            device, 16-byte aligned.  `stream` is a cudaStream_t passed as
 *            void* (NULL = the legacy default stream).  All work is enqueued
 *            asynchronously on that stream; nothing is synchronised.
 *   Ownership the caller allocates and owns every buffer it passes,
 *            including the backward workspace; no call allocates device
 *            memory.  The library's own device state is static and comes
 *            with the module when it loads on a device: one status word
 *            (bounded-wait timeouts, caught indices) and the built-in
 *            workspace of fa_bwd_noalloc (FA_NOALLOC_SCRATCH_BYTES).  Host
 *            side it caches kernel attributes and those two arrays' device
 *            addresses per device, so no cudaDeviceReset may come between
 *            two calls of this library in one process.
 *   Sizes    B, H, S >= 0 (a zero size is a valid empty problem and returns
 *            FA_OK without launching); d in {16, 32, 64, 80, 96, 128};
 *            B*H <= 65535 and B*H*S*d < 2^31 elements per array.  Any S >= 1 is accepted
 *            (a ragged last tile is masked).
 *   Errors   every call returns FA_OK (0) or a negative fa_status code and
 *            never aborts or traps; fa_get_last_error() describes the last
 *            failure of the calling thread.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_BF16 = 0,   /* bfloat16 storage, fp32 accumulation, tcgen05 tensor cores */
    FA_FP32 = 1    /* fp32 storage and arithmetic on the FMA pipes (tight checks) */
} fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,     /* null pointer, negative size, non-finite scale */
    FA_ERR_UNSUPPORTED = -2,     /* head dim or dtype outside the supported set, or too large */
    FA_ERR_MISALIGNED = -3,      /* an array pointer is not 16-byte aligned */
    FA_ERR_WORKSPACE = -4,       /* workspace null or smaller than fa_bwd_workspace_size() */
    FA_ERR_CUDA = -5,            /* a CUDA runtime/driver call or a launch failed */
    FA_ERR_DEVICE_TIMEOUT = -6,  /* a kernel gave up a bounded wait (reported by fa_check_status) */
    FA_ERR_DEVICE_BOUNDS = -7    /* a kernel caught an out-of-range index (reported by fa_check_status) */
} fa_status;

/*
 * Forward pass: handout Eq. 4-6 and Eq. 12, computed as in Algorithm 1.
 *   q, k, v  [B,H,S,d] dtype, read only.
 *   o        [B,H,S,d] dtype, fully overwritten with softmax(QK^T*scale)V,
 *            rounded to nearest even from the fp32 accumulator.
 *   lse      [B,H,S] fp32, fully overwritten with L (natural log).
 *   scale    the score scale (1/sqrt(d) in the handout); any finite value.
 * bf16 rounds the unnormalised probabilities to bf16 before the PV product
 * (handout, flash_forward (b): cast P to V's dtype); fp32 keeps them fp32.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int S, int d, int causal, float scale, int dtype, void* stream);

/*
 * Forward pass on general shapes (handout Algorithm 1 as stated: Q in
 * R^{N_q x d}, K, V in R^{N_k x d}), with strided operands.
 *   q, o       [B, H, Sq, d] views; k, v [B, H, Sk, d] views.  Each view is
 *              given by a HOST array of three element strides {batch, head,
 *              row}; the head dimension is contiguous (stride 1).  NULL
 *              means contiguous.  A stride whose dimension has more than one
 *              index must be positive and a multiple of 16 bytes (8 bf16 or 4
 *              fp32 elements); FA_ERR_MISALIGNED otherwise.  o must not
 *              overlap itself or the inputs.
 *   lse        contiguous [B, H, Sq] fp32.
 *   Sq, Sk     N_q >= 0 and N_k >= 1 (N_k = 0 with N_q > 0 is
 *              FA_ERR_INVALID_ARG: the softmax over no key is undefined).
 *   causal     keeps key j for query i when j <= i (indices from 0 in both,
 *              top-left aligned): with Sk > Sq the last keys are never seen,
 *              with Sq > Sk the last queries see every key.
 * Everything else as fa_fwd; fa_fwd(...) equals fa_fwd_strided with NULL
 * strides and Sq = Sk = S.
 */
int fa_fwd_strided(const void* q, const long long* q_strides, const void* k, const long long* k_strides,
                   const void* v, const long long* v_strides, void* o, const long long* o_strides, float* lse,
                   int B, int H, int Sq, int Sk, int d, int causal, float scale, int dtype, void* stream);

/*
 * Split-KV building block ("[Attention] FlashAttention/Ring-Attention/...统一
 * 原理": attention over a subset of the keys, merged exactly afterwards).
 *
 * fa_fwd_partial: every query attends only to keys [key_begin, key_end)
 * (causal: also key <= query, in whole-sequence positions).
 *   q, k, v      [B,H,S,d] dtype, the whole sequence, read only.
 *   o_part       [B,H,S,d] fp32, overwritten with the output normalised over
 *                the window's keys (0 for a query with no admissible key).
 *   lse_part     [B,H,S] fp32, overwritten with the natural-log logsumexp of
 *                the window's scores (-inf for a query with no admissible key).
 *   key_begin    a multiple of 128; 0 <= key_begin < key_end <= S.
 * Same conventions as fa_fwd otherwise (bf16 on the tensor cores, P rounded to
 * bf16 before its product; fp32 on the FMA pipes).
 *
 * fa_merge: combine two partial results over disjoint key sets of the same
 * queries: L = log(e^lse_a + e^lse_b), o = e^(lse_a - L) o_a + e^(lse_b - L) o_b.
 *   o_a, o_b     [B,H,S,d] fp32 (fa_fwd_partial outputs, or merges of them).
 *   lse_a, lse_b [B,H,S] fp32.
 *   o            [B,H,S,d] dtype (bf16 rounded to nearest even, or fp32).
 *   lse          [B,H,S] fp32.
 * o may alias o_a (or o_b) when dtype is FA_FP32, so merges can chain; lse
 * must not alias lse_a or lse_b.  Merging the partials of key windows that
 * tile [0, S) gives fa_fwd's result up to rounding.
 */
int fa_fwd_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                   int B, int H, int S, int d, int key_begin, int key_end, int causal, float scale, int dtype,
                   void* stream);
int fa_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b, void* o, float* lse,
             int B, int H, int S, int d, int dtype, void* stream);

/*
 * Bytes of device workspace fa_bwd needs.  The workspace holds, in order,
 *   D      [B,H,S] fp32   D_i = rowsum(O * dO)_i (handout, "backward pass with
 *                         recomputation"; Algorithm 2, before its loops), written by fa_bwd;
 *   (zero padding to a 256-byte boundary)
 *   dQacc  [B,H,S,d] fp32 the dQ accumulator that the key-tile-outer kernel adds
 *                         into with fp32 atomic adds (bf16: TMA bulk reduce-adds
 *                         of whole staged tiles), zeroed by fa_bwd itself.
 * Returns 0 for invalid or empty sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int S, int d, int dtype);

/*
 * Backward pass: handout Eq. 13-19 with Algorithm 2's key-tile-outer loop for
 * dK and dV; dQ is reduced across key tiles with fp32 atomics into dQacc and
 * converted to dtype at the end (its last bits may differ from run to run).
 *   q, k, v, o, dO  [B,H,S,d] dtype, read only; o must be the fa_fwd output.
 *   lse             [B,H,S] fp32 from fa_fwd, read only.
 *   dq, dk, dv      [B,H,S,d] dtype, fully overwritten.
 *   workspace       device buffer of >= fa_bwd_workspace_size() bytes, 256-byte
 *                   aligned; contents on entry are ignored, D is left in it.
 * Same B, H, S, d, causal, scale and dtype as the forward call.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv,
           void* workspace, size_t workspace_bytes,
           int B, int H, int S, int d, int causal, float scale, int dtype, void* stream);

/*
 * Deterministic backward: the same results as fa_bwd up to rounding, and
 * bitwise identical from run to run.  Algorithm 2 of the handout as it is
 * written: the key-tile-outer loop computes dK and dV only, and a separate
 * query-tile-outer loop recomputes P, dP and dS to sum each dQ row in one
 * fixed order (Eq. 18), with no atomics and no dQ accumulator.  It does more
 * arithmetic than fa_bwd (S and dP are formed twice per tile pair).
 *   Arguments as fa_bwd; dk and dv are bitwise equal to fa_bwd's.
 *   workspace  device buffer of >= B*H*S*4 bytes (fa_bwd_workspace_size() is
 *              always enough), 256-byte aligned; D is left at its start.
 */
int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes,
                         int B, int H, int S, int d, int causal, float scale, int dtype, void* stream);

/*
 * Backward pass on general shapes and strided operands; the counterpart of
 * fa_fwd_strided (same view, size and causal conventions).
 *   q, o, dO, dq   [B, H, Sq, d] views; k, v, dk, dv [B, H, Sk, d] views, each
 *                  with its own host stride array (NULL: contiguous).
 *   lse            contiguous [B, H, Sq] fp32 from the forward.
 *   workspace      >= fa_bwd_workspace_size(B, H, Sq, d, dtype) bytes
 *                  (B*H*Sq*4 with deterministic != 0), 256-byte aligned.
 *   deterministic  0: dQ by fp32 atomics as fa_bwd; otherwise dQ by its own
 *                  pass as fa_bwd_deterministic.
 * With Sq = 0 and Sk > 0 only dk and dv are written (zeros).  Keys that no
 * query attends under the causal mask get dk = dv = 0.
 */
int fa_bwd_strided(const void* q, const long long* q_strides, const void* k, const long long* k_strides,
                   const void* v, const long long* v_strides, const void* o, const long long* o_strides,
                   const void* dO, const long long* do_strides, const float* lse,
                   void* dq, const long long* dq_strides, void* dk, const long long* dk_strides,
                   void* dv, const long long* dv_strides, void* workspace, size_t workspace_bytes,
                   int B, int H, int Sq, int Sk, int d, int causal, float scale, int dtype, int deterministic,
                   void* stream);

/*
 * Backward pass for callers that cannot allocate device memory.
 * The pages describe no counterpart of this entry point; it exists for users
 * of this library that cannot call cudaMalloc (or any allocating routine,
 * PyTorch's caching allocator included) when they run the backward: code
 * inside an allocator's own callbacks, runtimes that forbid allocation during
 * a step, or plugins whose host owns all device memory.
 *
 * Same arguments and results as fa_bwd, minus the workspace: the workspace is
 * a fixed array of FA_NOALLOC_SCRATCH_BYTES bytes compiled into the library
 * (every GPU that loads the library holds it until the process exits).  The
 * call allocates nothing.
 *   - Problems whose fa_bwd_workspace_size() exceeds FA_NOALLOC_SCRATCH_BYTES
 *     are rejected with FA_ERR_WORKSPACE and a message naming both sizes.
 *     fa_bwd's argument checks run first, so a call that also breaks one of
 *     them (a null or misaligned pointer, a size out of range) gets that
 *     rule's code instead.
 *   - The array's device address is cached per device after the first call:
 *     no cudaDeviceReset may come between calls (the cached address would
 *     then name memory of a context that no longer exists).
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents (D stays readable there; the dQ accumulator is zeroed by every
 *     call).  Calls whose work overlaps on the GPU (different streams, or
 *     host threads, without ordering between them) race on it and give wrong
 *     results: order them on one stream.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int S, int d, int causal, float scale, int dtype, void* stream);

/* Size in bytes of the built-in scratch used by fa_bwd_noalloc. */
size_t fa_bwd_noalloc_scratch_bytes(void);

/*
 * One training step of attention on HOST buffers: copy q, k, v, dO to the
 * device, run fa_fwd and fa_bwd there, copy o, lse, dq, dk, dv back.  The
 * pages describe no counterpart; it is the end-to-end path for callers whose
 * tensors live in host memory (and the one the benchmark's end-to-end figure
 * goes through).
 *   q, k, v, dO         HOST [B,H,S,d] dtype, read only.
 *   o, dq, dk, dv       HOST [B,H,S,d] dtype, lse HOST [B,H,S] fp32, overwritten.
 *                       Pinned (page-locked) host memory makes every copy
 *                       asynchronous; pageable memory works but the copies
 *                       then synchronise with the host.
 *   dev_buf             DEVICE buffer of >= fa_fwd_bwd_host_buffer_size()
 *                       bytes, 256-byte aligned, owned by the caller; it holds
 *                       device copies of all nine arrays and the backward
 *                       workspace (q, k, v, dO, o, dq, dk, dv, lse, workspace,
 *                       each on a 256-byte boundary).
 * All work is ordered on `stream`: the call returns after enqueueing, and the
 * outputs are valid once `stream` has reached the point of the call.  o and
 * lse are copied back on a helper stream (one per caller stream, created on
 * first use) while the backward runs, and dO is copied in on it while the
 * forward runs; the call's work on `stream` waits for both.  Consecutive
 * calls on different streams with different dev_buf overlap their copies and
 * kernels.  Same size, dtype and error conventions as fa_fwd / fa_bwd;
 * FA_ERR_WORKSPACE when dev_buf is null or too small.
 */
size_t fa_fwd_bwd_host_buffer_size(int B, int H, int S, int d, int dtype);
int fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO,
                    void* o, float* lse, void* dq, void* dk, void* dv,
                    void* dev_buf, size_t dev_buf_bytes,
                    int B, int H, int S, int d, int causal, float scale, int dtype, void* stream);

/* Message for the calling thread's last non-zero return ("" if none). */
const char* fa_get_last_error(void);

/*
 * Synchronise `stream` and read, then clear, the current device's status word
 * that kernels set when a bounded wait runs out or an index check fails.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_BOUNDS or FA_ERR_CUDA.
 */
int fa_check_status(void* stream);

/*
 * Self-test of device-side failure detection.  Every wait inside the
 * library's kernels is bounded: after its limit (2 s) the kernel sets the
 * device status word, the CTA's other roles give up too, and the kernel
 * returns, leaving the CUDA context usable; fa_check_status then reports
 * FA_ERR_DEVICE_TIMEOUT.  This call enqueues one tiny kernel on `stream` whose
 * single wait can never complete (a barrier phase nothing arrives at) and
 * gives up after limit_ns nanoseconds (0 < limit_ns <= 10 s), exercising that
 * path.  Returns FA_OK once enqueued; FA_ERR_INVALID_ARG for a bad limit.
 */
int fa_selftest_bounded_wait(unsigned long long limit_ns, void* stream);

/* Library version as 10000*major + 100*minor + patch. */
int fa_version(void);

/*
 * Kernel timing for benchmarks (not needed to compute attention).  While
 * enabled, every fa_fwd / fa_bwd / fa_bwd_deterministic call records a pair of CUDA events on its
 * stream directly around each of its kernels.  fa_profile_read waits for the
 * recorded events, adds their elapsed times since the previous read into
 * ms[5] and the number of timed launches into launches[5], indexed by
 *   0 = forward kernel, 1 = backward preprocess (D, dQacc zeroing),
 *   2 = backward main kernel, 3 = dQ conversion, 4 = deterministic dQ pass,
 * and forgets them.  Both return FA_OK or FA_ERR_CUDA / FA_ERR_INVALID_ARG.
 * Events come from a host-side pool; no device memory is allocated.
 */
int fa_profile_enable(int on);
int fa_profile_read(double* ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

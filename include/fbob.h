/*
 * fbob.h - C ABI of the GB300 FlashBoB library (libfbob.so).
 *
 * FlashBoB ("FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
 * Attention", Abstract) computes the exact backward-over-backward (BoB) of
 * softmax attention without writing any N x N tensor to device memory.  This
 * library exposes that computation and the two calls it builds on:
 *
 *   fbob_forward   O = softmax(c Q K^T) V and the row log-sum-exp LSE
 *                  (the FlashAttention forward the abstract builds on)
 *   fbob_backward  dQ, dK, dV of <dO, O>          (the first backward)
 *   fbob_bob       the gradient of L = <gQ,dQ> + <gK,dK> + <gV,dV> with
 *                  respect to Q, K, V and dO       (the BoB, Abstract)
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Layout: every [B,H,N,d] tensor is dense and row-major (d fastest), of
 *    the call's dtype; LSE and the row scalars are fp32 [B,H,N].  Device
 *    pointers must be 16-byte aligned.  Outputs must not alias inputs.
 *  - Masking: with causal != 0 key j is visible to query i iff j <= i
 *    (square, top-left aligned).  The scale c is passed in shape->scale
 *    (1/sqrt(d) is the usual choice) and is a constant, not differentiated.
 *  - Derivative convention: O and LSE are the forward's outputs for the same
 *    Q, K, V (not independent inputs); BoB is the total derivative.
 *  - Ownership: the caller owns every buffer, including the workspace `ws`
 *    of at least fbob_workspace_size() bytes.  The library allocates and
 *    frees nothing.
 *  - Asynchrony: every call only enqueues work on `stream` (a cudaStream_t,
 *    or NULL for the legacy default stream) and returns.  The return value
 *    reports errors detected on the host (bad arguments, launch failures).
 *    Device-side failures (a bounded wait that ran out) are recorded in the
 *    workspace's status word and read back with fbob_status().
 *  - Threading: calls are re-entrant as long as concurrent calls use distinct
 *    workspaces.  The process-wide settings (fbob_force_path,
 *    fbob_set_profile_events) are not synchronised.
 *  - Supported shapes: N >= 1, B*H <= 65535.  fp32: 1 <= d <= 128, computed
 *    on CUDA cores.  bf16: 1 <= d <= 128; d = 64 and d = 128 run the
 *    tensor-core (tcgen05) kernels, other d run on CUDA cores.
 */
#ifndef FBOB_H_
#define FBOB_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FBOB_BF16 = 0, FBOB_FP32 = 1 } fbob_dtype_t;

typedef enum {
  FBOB_OK = 0,
  FBOB_ERR_INVALID_ARG = 1, /* null pointer, misalignment, bad size/flag    */
  FBOB_ERR_UNSUPPORTED = 2, /* shape or dtype outside the supported set     */
  FBOB_ERR_WORKSPACE = 3,   /* ws_bytes smaller than fbob_workspace_size()  */
  FBOB_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed         */
  FBOB_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out           */
} fbob_status_t;

typedef enum {
  FBOB_OP_FORWARD = 0,
  FBOB_OP_BACKWARD = 1,
  FBOB_OP_BOB = 2
} fbob_op_t;

/* Kernel family that serves a call (see fbob_path). */
typedef enum { FBOB_PATH_SIMT = 0, FBOB_PATH_TCGEN05 = 1 } fbob_path_t;

/* Problem description.  B batches x H heads of length-N sequences with head
 * dimension d; dtype is an fbob_dtype_t; causal is 0 or 1; scale is the
 * factor c in S = c Q K^T. */
typedef struct {
  int B, H, N, d;
  int dtype;
  int causal;
  float scale;
} fbob_shape_t;

/* Bytes of workspace that `op` needs for `shape` (0 if the shape is invalid).
 * The workspace holds a status word, the fp32 row scalars and, on the
 * tensor-core path, an fp32 [B,H,N,d] accumulator for dQ / gradQ. */
size_t fbob_workspace_size(int op, const fbob_shape_t* shape);

/* Forward: O = softmax(c Q K^T) V and LSE_i = log sum_j exp(c Q_i.K_j).
 *   q, k, v : [B,H,N,d] inputs            o : [B,H,N,d] output
 *   lse     : [B,H,N] fp32 output (natural log, scaled scores)
 * FlashAttention forward, cited as the base of FlashBoB (Abstract). */
int fbob_forward(const fbob_shape_t* shape, const void* q, const void* k,
                 const void* v, void* o, float* lse, void* ws,
                 size_t ws_bytes, void* stream);

/* First backward of attention for upstream gradient dO:
 *   D = rowsum(dO * O), dS = P * (dO V^T - D),
 *   dQ = c dS K,  dK = c dS^T Q,  dV = P^T dO.
 *   q, k, v, o, dO : [B,H,N,d] inputs; lse : [B,H,N] fp32 from fbob_forward
 *   dq, dk, dv     : [B,H,N,d] outputs
 * The "first backward pass" of the FlashBoB abstract. */
int fbob_backward(const fbob_shape_t* shape, const void* q, const void* k,
                  const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, void* ws,
                  size_t ws_bytes, void* stream);

/* Backward-over-backward: given cotangents gQ, gK, gV on the first
 * backward's outputs dQ, dK, dV, returns the gradient of
 *   L = <gQ,dQ> + <gK,dK> + <gV,dV>
 * with respect to Q, K, V and dO (gradq, gradk, gradv, graddo).
 *   q, k, v, o, dO, gq, gk, gv : [B,H,N,d] inputs
 *   lse                        : [B,H,N] fp32 from fbob_forward
 *   gradq, gradk, gradv, graddo: [B,H,N,d] outputs (fully overwritten)
 * Any of gq, gk, gv may be NULL: that cotangent is zero (a loss that reads
 * only some of dQ, dK, dV).  The kernels then skip its loads and the MMAs
 * it feeds.  With all three NULL, L = 0 and the four outputs are zeroed.
 * Exact BoB, "FlashBoB: I/O-Efficient Exact Backward-over-Backward for
 * Softmax Attention", Abstract: two row-wise scalars per query (r and sigma,
 * reduced in a row-stationary pass) determine every output through affine
 * maps, which a second, key-stationary pass applies.  No N x N tensor is
 * written. */
int fbob_bob(const fbob_shape_t* shape, const void* q, const void* k,
             const void* v, const void* o, const float* lse, const void* dO,
             const void* gq, const void* gk, const void* gv, void* gradq,
             void* gradk, void* gradv, void* graddo, void* ws,
             size_t ws_bytes, void* stream);

/* Size of the fixed device scratch array behind fbob_bob_noalloc: 32 MiB. */
#define FBOB_NOALLOC_SCRATCH_BYTES (32u << 20)

/* fbob_bob for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this call.  It exists for callers that are
 * handed only their input and output buffers: plugin or custom-operator
 * hosts that give a kernel no allocator and no workspace, and code that must
 * not call cudaMalloc / cudaFree, which can stall the whole device or fail
 * when a caching allocator already holds the free memory.  Arguments and
 * results are those of fbob_bob without `ws` / `ws_bytes`; this call itself
 * allocates nothing.
 *
 * Scratch comes from one array of FBOB_NOALLOC_SCRATCH_BYTES in the
 * library's device memory, which every GPU that loads the library keeps
 * reserved until the process exits.  The first call on a device (with that
 * device current) looks up the array's device address; make that first call
 * before any stream capture.  Problems whose fbob_workspace_size(
 * FBOB_OP_BOB, shape) exceeds FBOB_NOALLOC_SCRATCH_BYTES are rejected with
 * FBOB_ERR_WORKSPACE (the tensor-core path needs about B*H*N*(d+3)*4 bytes,
 * i.e. at most about 125,000 rows B*H*N at d = 64 or 63,000 at d = 128; the
 * CUDA-core path needs about B*H*N*12 bytes).  All calls share the one
 * array, so calls that can overlap on the GPU (different streams, or host
 * threads) race on it: serialise them.  Each call clears what must start at
 * zero, so contents left by an earlier call do not affect the result.  The
 * status word that device-side bounded waits write lives in that array:
 * read it with fbob_noalloc_status(), not fbob_status().  The array's
 * address is kept for the life of the process, so calls after a device
 * reset (cudaDeviceReset) are not supported. */
int fbob_bob_noalloc(const fbob_shape_t* shape, const void* q, const void* k,
                     const void* v, const void* o, const float* lse,
                     const void* dO, const void* gq, const void* gk,
                     const void* gv, void* gradq, void* gradk, void* gradv,
                     void* graddo, void* stream);

/* Status of the last fbob_bob_noalloc call on the current device: synchronises
 * `stream` (the stream that call used), then returns the first device-side
 * error it recorded in the scratch array's status word (FBOB_OK if none), or
 * FBOB_ERR_CUDA if the stream reports an error or the array cannot be reached.
 * Like fbob_bob_noalloc, it has no counterpart in the paper. */
int fbob_noalloc_status(void* stream);

/* Synchronises `stream`, then returns the first error recorded in the
 * workspace's status word by the last call that used `ws` (FBOB_OK if none),
 * or FBOB_ERR_CUDA if the stream itself reports an error. */
int fbob_status(const void* ws, void* stream);

/* Static description of a status code. */
const char* fbob_strerror(int code);

/* Kernel family (fbob_path_t) that serves `op` for `shape`, or -1 if the
 * shape is not supported. */
int fbob_path(int op, const fbob_shape_t* shape);

/* Process-wide override of the kernel family: -1 = automatic (default),
 * FBOB_PATH_SIMT = always CUDA cores.  Forcing FBOB_PATH_TCGEN05 on a shape
 * it cannot serve makes calls return FBOB_ERR_UNSUPPORTED.  Returns the
 * previous setting.  Intended for tests and benchmarks. */
int fbob_force_path(int path);

/* Benchmark hook.  With count >= 1, later fbob_bob / fbob_backward /
 * fbob_forward calls record events[0] before their first kernel and
 * events[m] after their m-th kernel (m < count), on the call's stream.
 * `events` are cudaEvent_t created by the caller; pass count = 0 to turn
 * the hook off.  Returns FBOB_OK or FBOB_ERR_INVALID_ARG. */
int fbob_set_profile_events(void* const* events, int count);

/* Process-wide limit, in nanoseconds, of one device-side bounded wait in the
 * tensor-core kernels (default 2 s, far above any legitimate wait).  A wait
 * that runs out records FBOB_ERR_TIMEOUT in the call's status word; every
 * role of that thread block then stops early, waits (with a fixed 100 ms
 * limit of its own) for the copies and MMAs it has in flight, and exits, and
 * the call's outputs are undefined.  The limit is checked each time the
 * waiting thread wakes, at least every 10 us.  ns = 0 restores the default;
 * 1 <= ns <= 6e10 sets it.
 * Applies to calls enqueued afterwards.  Returns the previous limit, or -1
 * (nothing changed) for a value out of range.  Not synchronised. */
long long fbob_set_wait_limit(long long ns);

/* Number of kernels the last enqueued call launched (for launch counting). */
int fbob_last_launch_count(void);

/* Failure-detection self-test: launches one block that waits, with the same
 * bounded wait the tensor-core kernels use, on a barrier that nothing ever
 * completes, giving up after `limit_us` microseconds (1..10^6) and recording
 * FBOB_ERR_TIMEOUT in the status word of `ws` (>= 256 bytes).  The GPU is
 * never hung.  Read the result with fbob_status(). */
int fbob_selftest_wait_timeout(void* ws, size_t ws_bytes, int limit_us,
                               void* stream);

/* Library ABI version (major*100 + minor). */
int fbob_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FBOB_H_ */

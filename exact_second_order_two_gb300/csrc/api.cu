// Host entry points of libfbob.so (the C ABI declared in include/fbob.h):
// argument validation, workspace carving, kernel-family dispatch.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "fbob.h"
#include "internal.h"

namespace fbob {
namespace {

int g_force_path = -1;
// 2 s: far above any legitimate wait inside a kernel (microseconds), far
// below anything that would look like a hang.
constexpr long long kDefaultWaitLimitNs = 2000000000ll;
long long g_wait_limit_ns = kDefaultWaitLimitNs;
cudaEvent_t g_events[16];
int g_event_count = 0;
int g_last_launches = 0;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int check_shape(const fbob_shape_t* s, Problem* out) {
  if (!s) return FBOB_ERR_INVALID_ARG;
  if (s->B < 1 || s->H < 1 || s->N < 1 || s->d < 1) return FBOB_ERR_INVALID_ARG;
  if (s->causal != 0 && s->causal != 1) return FBOB_ERR_INVALID_ARG;
  if (s->dtype != FBOB_BF16 && s->dtype != FBOB_FP32) return FBOB_ERR_UNSUPPORTED;
  if (s->d > 128) return FBOB_ERR_UNSUPPORTED;
  if ((long long)s->B * s->H > 65535) return FBOB_ERR_UNSUPPORTED;
  if (!(s->scale == s->scale) || s->scale == 0.f) return FBOB_ERR_INVALID_ARG;
  const long long elems = (long long)s->B * s->H * s->N * (long long)s->d;
  if (elems > (1ll << 40)) return FBOB_ERR_UNSUPPORTED;
  Problem p;
  p.B = s->B; p.H = s->H; p.N = s->N; p.d = s->d;
  p.bf16 = s->dtype == FBOB_BF16;
  p.causal = s->causal;
  p.scale = s->scale;
  *out = p;
  return FBOB_OK;
}

// Kernel family for a validated problem.
int choose_path(int op, const Problem& p) {
  // the tensor-core family serves bf16 at d = 64 and 128 (all three ops);
  // everything else runs on CUDA cores
  const bool tc = tc_supported(p);
  if (g_force_path == FBOB_PATH_SIMT) return FBOB_PATH_SIMT;
  if (g_force_path == FBOB_PATH_TCGEN05) return tc ? FBOB_PATH_TCGEN05 : -1;
  return tc ? FBOB_PATH_TCGEN05 : FBOB_PATH_SIMT;
}

// Workspace layout: [status 256 B][r][sigma][D][acc], each region aligned.
size_t carve(int op, const Problem& p, int path, char* base, Workspace* ws) {
  size_t off = kAlign;  // status word region
  const size_t vec = align_up(p.rows() * sizeof(float));
  const size_t mat = align_up(p.elems() * sizeof(float));
  if (ws) ws->status = reinterpret_cast<int*>(base);
  if (op == FBOB_OP_BOB) {
    if (ws) {
      ws->r = reinterpret_cast<float*>(base + off);
      ws->sigma = reinterpret_cast<float*>(base + off + vec);
      ws->D = reinterpret_cast<float*>(base + off + 2 * vec);
    }
    off += 3 * vec;
  } else if (op == FBOB_OP_BACKWARD) {
    if (ws) ws->D = reinterpret_cast<float*>(base + off);
    off += vec;
  }
  if (path == FBOB_PATH_TCGEN05 && (op == FBOB_OP_BOB || op == FBOB_OP_BACKWARD)) {
    if (ws) ws->acc = reinterpret_cast<float*>(base + off);
    off += mat;
  }
  if (ws) ws->bytes = off;
  return off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int to_status(cudaError_t e) { return e == cudaSuccess ? FBOB_OK : FBOB_ERR_CUDA; }

// Common prologue: validate, pick the path, carve the workspace, reset the
// status word.
int prologue(int op, const fbob_shape_t* shape, void* ws_ptr, size_t ws_bytes,
             cudaStream_t stream, Problem* p, int* path, Workspace* ws) {
  int st = check_shape(shape, p);
  if (st != FBOB_OK) return st;
  *path = choose_path(op, *p);
  if (*path < 0) return FBOB_ERR_UNSUPPORTED;
  if (!ws_ptr || !aligned16(ws_ptr)) return FBOB_ERR_INVALID_ARG;
  const size_t need = carve(op, *p, *path, static_cast<char*>(ws_ptr), ws);
  if (ws_bytes < need) return FBOB_ERR_WORKSPACE;
  if (cudaMemsetAsync(ws->status, 0, sizeof(int), stream) != cudaSuccess)
    return FBOB_ERR_CUDA;
  return FBOB_OK;
}

bool ptrs_ok(std::initializer_list<const void*> ps) {
  for (const void* q : ps)
    if (!q || !aligned16(q)) return false;
  return true;
}

bool opt_ptrs_ok(std::initializer_list<const void*> ps) {
  for (const void* q : ps)
    if (q && !aligned16(q)) return false;
  return true;
}

}  // namespace

unsigned long long wait_limit_ns() { return (unsigned long long)g_wait_limit_ns; }

void LaunchLog::mark() {
  ++launches;
  if (launches < g_event_count) cudaEventRecord(g_events[launches], stream);
}

}  // namespace fbob

using namespace fbob;

extern "C" {

int fbob_version(void) { return 100; }

const char* fbob_strerror(int code) {
  switch (code) {
    case FBOB_OK: return "ok";
    case FBOB_ERR_INVALID_ARG: return "invalid argument";
    case FBOB_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case FBOB_ERR_WORKSPACE: return "workspace too small";
    case FBOB_ERR_CUDA: return "CUDA error";
    case FBOB_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

size_t fbob_workspace_size(int op, const fbob_shape_t* shape) {
  Problem p;
  if (op < FBOB_OP_FORWARD || op > FBOB_OP_BOB) return 0;
  if (check_shape(shape, &p) != FBOB_OK) return 0;
  const int path = choose_path(op, p);
  if (path < 0) return 0;
  return carve(op, p, path, nullptr, nullptr);
}

int fbob_path(int op, const fbob_shape_t* shape) {
  Problem p;
  if (op < FBOB_OP_FORWARD || op > FBOB_OP_BOB) return -1;
  if (check_shape(shape, &p) != FBOB_OK) return -1;
  return choose_path(op, p);
}

int fbob_force_path(int path) {
  const int old = g_force_path;
  if (path == -1 || path == FBOB_PATH_SIMT || path == FBOB_PATH_TCGEN05) g_force_path = path;
  return old;
}

int fbob_set_profile_events(void* const* events, int count) {
  if (count < 0 || count > 16 || (count > 0 && !events)) return FBOB_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) g_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_event_count = count;
  return FBOB_OK;
}

int fbob_last_launch_count(void) { return g_last_launches; }

long long fbob_set_wait_limit(long long ns) {
  const long long old = g_wait_limit_ns;
  if (ns == 0) g_wait_limit_ns = kDefaultWaitLimitNs;
  else if (ns > 0 && ns <= 60000000000ll) g_wait_limit_ns = ns;
  else return -1;
  return old;
}

int fbob_forward(const fbob_shape_t* shape, const void* q, const void* k,
                 const void* v, void* o, float* lse, void* ws_ptr,
                 size_t ws_bytes, void* stream) {
  Problem p;
  int path;
  Workspace ws;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!ptrs_ok({q, k, v, o, lse})) return FBOB_ERR_INVALID_ARG;
  int st = prologue(FBOB_OP_FORWARD, shape, ws_ptr, ws_bytes, s, &p, &path, &ws);
  if (st != FBOB_OK) return st;
  LaunchLog log{s};
  if (g_event_count > 0) cudaEventRecord(g_events[0], s);
  cudaError_t e = path == FBOB_PATH_TCGEN05 ? tc_forward(p, q, k, v, o, lse, ws, log)
                                            : simt_forward(p, q, k, v, o, lse, log);
  g_last_launches = log.launches;
  return to_status(e);
}

int fbob_backward(const fbob_shape_t* shape, const void* q, const void* k,
                  const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, void* ws_ptr,
                  size_t ws_bytes, void* stream) {
  Problem p;
  int path;
  Workspace ws;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!ptrs_ok({q, k, v, o, lse, dO, dq, dk, dv})) return FBOB_ERR_INVALID_ARG;
  int st = prologue(FBOB_OP_BACKWARD, shape, ws_ptr, ws_bytes, s, &p, &path, &ws);
  if (st != FBOB_OK) return st;
  LaunchLog log{s};
  if (g_event_count > 0) cudaEventRecord(g_events[0], s);
  cudaError_t e =
      path == FBOB_PATH_TCGEN05
          ? tc_backward(p, q, k, v, o, lse, dO, dq, dk, dv, ws, log)
          : simt_backward(p, q, k, v, o, lse, dO, dq, dk, dv, ws, log);
  g_last_launches = log.launches;
  return to_status(e);
}

int fbob_bob(const fbob_shape_t* shape, const void* q, const void* k,
             const void* v, const void* o, const float* lse, const void* dO,
             const void* gq, const void* gk, const void* gv, void* gradq,
             void* gradk, void* gradv, void* graddo, void* ws_ptr,
             size_t ws_bytes, void* stream) {
  Problem p;
  int path;
  Workspace ws;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // gq, gk, gv may be null (a zero cotangent); present ones must be aligned
  if (!ptrs_ok({q, k, v, o, lse, dO, gradq, gradk, gradv, graddo}) || !opt_ptrs_ok({gq, gk, gv}))
    return FBOB_ERR_INVALID_ARG;
  int st = prologue(FBOB_OP_BOB, shape, ws_ptr, ws_bytes, s, &p, &path, &ws);
  if (st != FBOB_OK) return st;
  LaunchLog log{s};
  if (g_event_count > 0) cudaEventRecord(g_events[0], s);
  if (!gq && !gk && !gv) {  // L = 0: every output is zero
    const size_t bytes = p.elems() * (p.bf16 ? 2 : 4);
    cudaError_t e = cudaSuccess;
    for (void* out : {gradq, gradk, gradv, graddo})
      if (e == cudaSuccess) e = cudaMemsetAsync(out, 0, bytes, s);
    g_last_launches = 0;
    return to_status(e);
  }
  cudaError_t e =
      path == FBOB_PATH_TCGEN05
          ? tc_bob(p, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk, gradv, graddo, ws, log)
          : simt_bob(p, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk, gradv, graddo, ws, log);
  g_last_launches = log.launches;
  return to_status(e);
}

int fbob_status(const void* ws_ptr, void* stream) {
  if (!ws_ptr) return FBOB_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FBOB_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return FBOB_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ws_ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FBOB_ERR_CUDA;
  return word;
}

int fbob_selftest_wait_timeout(void* ws_ptr, size_t ws_bytes, int limit_us,
                               void* stream) {
  if (!ws_ptr || !aligned16(ws_ptr) || ws_bytes < 256) return FBOB_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return FBOB_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(ws_ptr);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return FBOB_ERR_CUDA;
  g_last_launches = 1;
  return to_status(launch_wait_timeout_selftest(status, 1000ll * limit_us, s));
}

}  // extern "C"

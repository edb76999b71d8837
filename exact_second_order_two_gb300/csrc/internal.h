// Internal declarations shared by the host entry points (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fbob {

// Problem description after validation (see fbob_shape_t).
struct Problem {
  int B, H, N, d;
  int bf16;    // 1 = bf16 tensors, 0 = fp32 tensors
  int causal;  // 0 / 1
  float scale;
  int BH() const { return B * H; }
  size_t rows() const { return (size_t)B * H * N; }
  size_t elems() const { return rows() * (size_t)d; }
};

// Workspace carving.  The first 256 bytes hold the status word (int32 at
// offset 0); every other region is 256-byte aligned.
struct Workspace {
  int* status = nullptr;
  float* r = nullptr;      // [B,H,N] row scalar r_i   (BoB)
  float* sigma = nullptr;  // [B,H,N] row scalar sigma_i (BoB)
  float* D = nullptr;      // [B,H,N] D_i = dO_i . O_i (backward, BoB)
  float* acc = nullptr;    // [B,H,N,d] fp32 dQ / gradQ accumulator (tcgen05)
  size_t bytes = 0;
};

// Kernel launch bookkeeping: optional profiling events and a launch count.
struct LaunchLog {
  cudaStream_t stream;
  int launches = 0;
  void mark();  // records the next profiling event if the hook is set
};

// ---- CUDA-core (SIMT) kernels, any d <= 128, fp32 or bf16 ---------------
cudaError_t simt_forward(const Problem& p, const void* q, const void* k,
                         const void* v, void* o, float* lse, LaunchLog& log);
cudaError_t simt_backward(const Problem& p, const void* q, const void* k,
                          const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv,
                          const Workspace& ws, LaunchLog& log);
cudaError_t simt_bob(const Problem& p, const void* q, const void* k,
                     const void* v, const void* o, const float* lse,
                     const void* dO, const void* gq, const void* gk,
                     const void* gv, void* gradq, void* gradk, void* gradv,
                     void* graddo, const Workspace& ws, LaunchLog& log);

// ---- tensor-core (tcgen05 / TMEM / TMA) kernels, bf16, d in {64, 128} ----
bool tc_supported(const Problem& p);
cudaError_t tc_forward(const Problem& p, const void* q, const void* k,
                       const void* v, void* o, float* lse, const Workspace& ws,
                       LaunchLog& log);
cudaError_t tc_backward(const Problem& p, const void* q, const void* k,
                        const void* v, const void* o, const float* lse,
                        const void* dO, void* dq, void* dk, void* dv,
                        const Workspace& ws, LaunchLog& log);
// scale * fp32 accumulator [elems] -> bf16 output (elems a multiple of 8).
cudaError_t launch_acc_to_bf16(const float* acc, void* out, size_t elems, float scale,
                               LaunchLog& log);
cudaError_t tc_bob(const Problem& p, const void* q, const void* k,
                   const void* v, const void* o, const float* lse,
                   const void* dO, const void* gq, const void* gk,
                   const void* gv, void* gradq, void* gradk, void* gradv,
                   void* graddo, const Workspace& ws, LaunchLog& log);

// Limit of one device-side bounded wait, in nanoseconds (process-wide;
// fbob_set_wait_limit).  Every tensor-core kernel receives it as an argument.
unsigned long long wait_limit_ns();

// Failure-detection self-test kernel (bounded wait that must run out).
cudaError_t launch_wait_timeout_selftest(int* status, long long limit_ns,
                                         cudaStream_t stream);

}  // namespace fbob

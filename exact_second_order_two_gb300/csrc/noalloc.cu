// fbob_bob_noalloc: the BoB call for callers that cannot allocate device
// memory.
//
// Some callers get only their input and output buffers and have no way to
// obtain device memory: plugin and custom-operator hosts that pass a kernel
// its tensors but no allocator or workspace, and code that must not call
// cudaMalloc / cudaFree because those calls can stall the whole device or
// fail when a caching allocator already holds the free memory.  For them this
// entry point takes its scratch (status word, row scalars r / sigma / D and,
// on the tensor-core path, the fp32 gradQ accumulator) from a fixed array in
// the library's own device memory instead of from a caller workspace.
//
// The array is a file-scope __device__ variable, so each GPU that loads this
// library keeps FBOB_NOALLOC_SCRATCH_BYTES of its memory reserved until the
// process exits.  In host code the variable's name is only a host-side
// stand-in: its device address is fetched once per device with
// cudaGetSymbolAddress, on the first call made while that device is current,
// and kept for the life of the process (a device reset, which can move the
// array, is not supported).
#include <cuda_runtime.h>
#include <mutex>

#include "fbob.h"

namespace {

static __device__ __align__(256) unsigned char g_bob_scratch[FBOB_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on
// failure).  The first call per device does the lookup.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bob_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int fbob_bob_noalloc(const fbob_shape_t* shape, const void* q, const void* k,
                                const void* v, const void* o, const float* lse, const void* dO,
                                const void* gq, const void* gk, const void* gv, void* gradq,
                                void* gradk, void* gradv, void* graddo, void* stream) {
  const size_t need = fbob_workspace_size(FBOB_OP_BOB, shape);
  if (need == 0) {
    // invalid or unsupported shape: the regular entry point reports which
    return fbob_bob(shape, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk, gradv, graddo,
                    nullptr, 0, stream);
  }
  if (need > (size_t)FBOB_NOALLOC_SCRATCH_BYTES) return FBOB_ERR_WORKSPACE;
  void* scratch = scratch_for_current_device();
  if (!scratch) return FBOB_ERR_CUDA;
  // fbob_bob clears the status word and the gradQ accumulator itself and
  // fully overwrites the row scalars, so stale contents of the shared array
  // from an earlier call do not leak into this one.
  return fbob_bob(shape, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk, gradv, graddo, scratch,
                  (size_t)FBOB_NOALLOC_SCRATCH_BYTES, stream);
}

// The status word that device-side bounded waits write sits at the start of
// the scratch array, where the caller cannot read it: this returns it.
extern "C" int fbob_noalloc_status(void* stream) {
  void* scratch = scratch_for_current_device();
  if (!scratch) return FBOB_ERR_CUDA;
  return fbob_status(scratch, stream);
}

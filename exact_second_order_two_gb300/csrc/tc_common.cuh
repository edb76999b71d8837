// Shared pieces of the tensor-core kernels (BoB passes, forward, first
// backward): bounded waits, tile visiting order, TMA tile loads, descriptor
// offset arithmetic, and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm103.cuh"

namespace fbob {
namespace tc {

using namespace sm103;

constexpr float kLog2e = 1.4426950408889634f;

// MN-major operand descriptor convention: LBO = stride between 64-element
// groups along M/N, SBO = stride between 8-row groups along K.

// Per-CTA abort state in shared memory: the flag that tells every role of
// the CTA to stop, and the time limit of one bounded wait (a kernel argument,
// written once before the CTA's first barrier).
struct Abort {
  volatile int flag;
  int pad;
  uint64_t limit_ns;
};

// Bounded wait that also gives up as soon as another role has aborted.  A
// failed poll sleeps until the phase completes or 10 us pass (less for a
// shorter limit); the abort flag and the time limit are checked after each.
constexpr uint32_t kPollSleepNs = 10000;
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Abort* ab, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  const uint64_t limit = ab->limit_ns;
  const uint32_t sleep = limit < kPollSleepNs ? (uint32_t)limit : kPollSleepNs;
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, sleep)) return true;
    if (ab->flag) return false;
    if (global_ns() - t0 > limit) {
      report_status(status, FBOB_ERR_TIMEOUT);
      ab->flag = 1;
      return false;
    }
  }
}

// Warp-uniform bounded wait: tcgen05.ld is .sync.aligned, so every lane of
// a warp must take the same branch after a wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Abort* ab, int* status) {
  const bool ok = wait_bar(bar, parity, ab, status);
  return __all_sync(0xffffffffu, ok);
}

// Named barrier over the first THREADS threads of the CTA (id != 0).
template <int THREADS>
__device__ __forceinline__ void named_sync(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(THREADS) : "memory");
}

// One-dimensional grid of nblk * BH CTAs.  Heads are taken in groups of G;
// within a group the block index varies slowest, so block 0 of every head
// of the group starts before block 1 of any.  With the heaviest block of a
// head numbered 0, the long CTAs start first and short ones fill the tail,
// while the CTAs that run at the same time belong to a few heads only, whose
// streamed tiles stay in L2.  G is chosen on the host (cta_group_heads).
struct CtaCoord {
  int bh, blk;
};
__device__ __forceinline__ CtaCoord cta_coord(int BH, int G, int nblk) {
  const int i = (int)blockIdx.x;
  const int per_group = G * nblk;
  const int g = i / per_group;
  const int j = i - g * per_group;
  const int gs = min(G, BH - g * G);  // heads in this (possibly last) group
  return {g * G + j % gs, j / gs};
}

// Number of SMs of the current device (looked up once per process).
inline int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
  });
  return n;
}

// Heads per group: enough that a group holds at least two waves of CTAs.
inline int cta_group_heads(int BH, int nblk, int sms) {
  int G = 1;
  while (G < BH && (long long)G * nblk < 2ll * sms) G *= 2;
  return G < BH ? G : BH;
}

// Adds this thread's NC fp32 partials (consecutive columns, STRIDE elements
// apart in the accumulator) with one global reduction each; only the first
// `valid` are inside the sequence.  The scale factor of dQ / gradQ is applied
// once, when the accumulator is converted to bf16.
template <int STRIDE, int NC>
__device__ __forceinline__ void red_columns(float* base, const uint32_t (&v)[NC], int valid) {
  if (valid >= NC) {
#pragma unroll
    for (int c = 0; c < NC; ++c) atomicAdd(base + (size_t)c * STRIDE, __uint_as_float(v[c]));
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (c < valid) atomicAdd(base + (size_t)c * STRIDE, __uint_as_float(v[c]));
  }
}

// Tile visited at step t when a CTA starts its loop at tile `rot` and wraps:
// CTAs of one head sweep the shared operand tiles out of phase, so the L2
// serves a tile to a few SMs at a time instead of to all of them at once.
// Every sum over tiles is order-independent.
__device__ __forceinline__ int rotated(int t, int rot, int T) {
  const int u = t + rot;
  return u >= T ? u - T : u;
}

// One TMA box per [rows][D] tile: the 4-D tensor view (64 features, rows,
// D/64 feature halves, heads) lands it as D/64 consecutive [rows][64] blocks.
__device__ __forceinline__ void load_tile(void* dst, const CUtensorMap* map, uint64_t* bar, int row,
                                          int bh) {
  tma_load_4d(dst, map, bar, 0, row, 0, bh);
}

// K-major tile [rows][D] stored as D/64 boxes of [rows][64] (128 B rows,
// 128-byte swizzle): offset of the k-th 16-element slice along D, in
// descriptor units (16 bytes), to add to the tile's descriptor low word.
__host__ __device__ constexpr uint32_t kslice_off(int rows, int k) {
  return (uint32_t)(((k >> 2) * rows * 128 + (k & 3) * 32) >> 4);
}
// MN-major operand: the k-th 16-row step along K (16 rows x 128 B).
__host__ __device__ constexpr uint32_t kstep_off(int k) { return (uint32_t)(k * 2048 >> 4); }
// A value the compiler must treat as new on every evaluation: keeps
// `base + constant` descriptor words inside the tile loop (one add each)
// instead of hoisting every unrolled offset into its own register.
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
  asm volatile("" : "+r"(x));
  return x;
}
// Descriptor low words (see sdesc_lo).
__device__ __forceinline__ uint32_t lo_kmajor(uint32_t saddr) { return sdesc_lo(saddr, 16); }
__device__ __forceinline__ uint32_t lo_mnmajor(uint32_t saddr, uint32_t mn_group_stride) {
  return sdesc_lo(saddr, mn_group_stride);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B*H, N, D] bf16 tensor viewed 4-D as (64 features, N rows, D/64 halves,
// B*H heads); one box = box_rows rows x all D features, landing in shared
// memory as D/64 consecutive [box_rows][64] blocks with 128-byte swizzle.
// Rows past N read as zero.
// With one_half the box spans a single 64-feature half (for interleaved pairs).
inline bool make_map(CUtensorMap* m, const void* ptr, const Problem& p, int box_rows,
                     bool one_half = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)p.N, (cuuint64_t)(p.d / 64), (cuuint64_t)p.BH()};
  cuuint64_t strides[3] = {(cuuint64_t)p.d * 2, 128, (cuuint64_t)p.N * p.d * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, one_half ? 1u : (cuuint32_t)(p.d / 64), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B*H, N, D] fp32 accumulator viewed 3-D as (D features, N rows, B*H
// heads); one box = box_rows rows x the first box_cols features,
// [box_rows][box_cols] fp32 rows in shared memory without swizzle.  A
// reduce-add skips rows past N.
inline bool make_acc_map(CUtensorMap* m, float* ptr, const Problem& p, int box_cols,
                         int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.N, (cuuint64_t)p.BH()};
  cuuint64_t strides[2] = {(cuuint64_t)p.d * 4, (cuuint64_t)p.N * p.d * 4};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace fbob

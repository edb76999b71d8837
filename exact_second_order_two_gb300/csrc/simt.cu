// CUDA-core kernels for attention forward, first backward and BoB.
//
// These serve fp32 tensors (where bf16 tensor-core products would miss an
// fp32 accuracy budget) and any head dimension d <= 128.  Arithmetic is fp32
// throughout.  Design: one warp owns one query row (row kernels) or one key
// row (column kernels); the other operand streams through shared memory in
// tiles of 32 rows, one row per lane for the score dot products, and the
// per-lane scores are then broadcast with shuffles to accumulate d-wide
// outputs with lane = column.
//
// BoB here uses three passes (FlashBoB, Abstract: "two row-wise scalars
// determine all outputs through affine transformations"):
//   row pass 1  r_i = sum_j P_ij G_ij, graddO_i = P gV + (P*G) V - r_i O_i,
//               sigma_i = dO_i . graddO_i, D_i = dO_i . O_i
//   column pass gradK_j, gradV_j from the now-known row scalars
//   row pass 2  gradQ_i (rows cannot be accumulated from the column pass
//               without atomics, which CUDA-core throughput cannot afford)
// with G = c (Q gK^T + gQ K^T) and H = dO gV^T never stored.

#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace fbob {
namespace {

constexpr int kWarps = 8;   // rows per block
constexpr int kTile = 32;   // streamed rows per shared-memory tile
constexpr int kMaxD = 128;
constexpr int kSlots = kMaxD / 32;

enum RowMode { kRowForward = 0, kRowBwdDq = 1, kRowBob1 = 2, kRowBobGradq = 3 };
enum ColMode { kColBwdDkdv = 0, kColBob2 = 1 };

struct RowArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const void* gq;
  const void* gk;
  const void* gv;
  const float* lse;  // read (all modes but forward)
  const float* D;    // read (bwd-dq, bob-gradq)
  const float* r;    // read (bob-gradq)
  const float* sigma;
  void* out;         // O, dQ, graddO or gradQ
  float* lse_out;    // forward
  float* r_out;      // bob1
  float* sigma_out;  // bob1
  float* D_out;      // bob1
  int N, d, causal;
  float scale;
};

struct ColArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dO;
  const void* gq;
  const void* gk;
  const void* gv;
  const float* lse;
  const float* D;
  const float* r;
  const float* sigma;
  void* out_k;  // dK or gradK
  void* out_v;  // dV or gradV
  int N, d, causal;
  float scale;
};

template <typename T>
__device__ __forceinline__ float ldx(const void* p, size_t i) {
  return to_f32<T>(static_cast<const T*>(p)[i]);
}

template <typename T>
__device__ __forceinline__ void stx(void* p, size_t i, float x) {
  static_cast<T*>(p)[i] = from_f32<T>(x);
}

// ----------------------------------------------------------------------------
// Row-stationary kernel: warp w owns query row i = blockIdx.x*kWarps + w.
// ----------------------------------------------------------------------------
template <typename T, int MODE>
__global__ void __launch_bounds__(kWarps * 32)
    row_kernel(RowArgs a) {
  constexpr bool kNeedGq = (MODE == kRowBob1 || MODE == kRowBobGradq);
  constexpr bool kNeedDo = (MODE == kRowBwdDq || MODE == kRowBobGradq);
  constexpr bool kNeedGkv = (MODE == kRowBob1 || MODE == kRowBobGradq);
  extern __shared__ float sm[];
  const int d = a.d, ldk = d + 1, N = a.N;
  float* qs = sm;                      // [kWarps][d]
  float* gqs = qs + kWarps * d;        // [kWarps][d]
  float* dos = gqs + kWarps * d;       // [kWarps][d]
  float* ks = dos + kWarps * d;        // [kTile][d+1]
  float* vs = ks + kTile * ldk;
  float* gks = vs + kTile * ldk;
  float* gvs = gks + kTile * ldk;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t bh = blockIdx.y;
  const size_t base = bh * (size_t)N * d;
  const int row0 = blockIdx.x * kWarps;
  const int i = row0 + warp;
  const bool row_ok = i < N;
  const size_t srow = bh * (size_t)N + (row_ok ? i : 0);

  for (int e = threadIdx.x; e < kWarps * d; e += blockDim.x) {
    const int ii = row0 + e / d, c = e % d;
    const bool ok = ii < N;
    const size_t off = base + (size_t)(ok ? ii : 0) * d + c;
    qs[e] = ok ? ldx<T>(a.q, off) : 0.f;
    if (kNeedGq) gqs[e] = ok && a.gq ? ldx<T>(a.gq, off) : 0.f;  // null: zero cotangent
    if (kNeedDo) dos[e] = ok ? ldx<T>(a.dO, off) : 0.f;
  }
  float lse_i = 0.f, D_i = 0.f, r_i = 0.f, sig_i = 0.f;
  if (MODE != kRowForward && row_ok) lse_i = a.lse[srow];
  if ((MODE == kRowBwdDq || MODE == kRowBobGradq) && row_ok) D_i = a.D[srow];
  if (MODE == kRowBobGradq && row_ok) {
    r_i = a.r[srow];
    sig_i = a.sigma[srow];
  }

  float acc[kSlots];
#pragma unroll
  for (int t = 0; t < kSlots; ++t) acc[t] = 0.f;
  float m_run = -INFINITY, l_run = 0.f, r_part = 0.f;

  const int kend = a.causal ? min(N, row0 + kWarps) : N;
  for (int j0 = 0; j0 < kend; j0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int jj = e / d, c = e % d, j = j0 + jj;
      const bool ok = j < N;
      const size_t off = base + (size_t)(ok ? j : 0) * d + c;
      ks[jj * ldk + c] = ok ? ldx<T>(a.k, off) : 0.f;
      vs[jj * ldk + c] = ok ? ldx<T>(a.v, off) : 0.f;
      if (kNeedGkv) {
        gks[jj * ldk + c] = ok && a.gk ? ldx<T>(a.gk, off) : 0.f;
        gvs[jj * ldk + c] = ok && a.gv ? ldx<T>(a.gv, off) : 0.f;
      }
    }
    __syncthreads();

    const int j = j0 + lane;
    const bool valid = row_ok && j < N && (!a.causal || j <= i);
    const float* qrow = qs + warp * d;
    const float* krow = ks + lane * ldk;
    float s = 0.f, g1 = 0.f, g2 = 0.f, dp = 0.f, h = 0.f;
    for (int c = 0; c < d; ++c) {
      const float kc = krow[c];
      s = fmaf(qrow[c], kc, s);
      if (kNeedGq) {
        g1 = fmaf(qrow[c], gks[lane * ldk + c], g1);
        g2 = fmaf(gqs[warp * d + c], kc, g2);
      }
      if (kNeedDo) dp = fmaf(dos[warp * d + c], vs[lane * ldk + c], dp);
      if (MODE == kRowBobGradq) h = fmaf(dos[warp * d + c], gvs[lane * ldk + c], h);
    }
    s *= a.scale;

    if (MODE == kRowForward) {
      const float sm_ = valid ? s : -INFINITY;
      const float m_new = fmaxf(m_run, warp_max(sm_));
      const float p = valid ? expf(s - m_new) : 0.f;
      const float alpha = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
      l_run = l_run * alpha + warp_sum(p);
      m_run = m_new;
#pragma unroll
      for (int t = 0; t < kSlots; ++t) acc[t] *= alpha;
      for (int jj = 0; jj < kTile; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const int c = lane + 32 * t;
          if (c < d) acc[t] = fmaf(pj, vs[jj * ldk + c], acc[t]);
        }
      }
    } else if (MODE == kRowBwdDq) {
      const float p = valid ? expf(s - lse_i) : 0.f;
      const float ds = p * (dp - D_i);
      for (int jj = 0; jj < kTile; ++jj) {
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const int c = lane + 32 * t;
          if (c < d) acc[t] = fmaf(dsj, ks[jj * ldk + c], acc[t]);
        }
      }
    } else if (MODE == kRowBob1) {
      const float p = valid ? expf(s - lse_i) : 0.f;
      const float g = a.scale * (g1 + g2);
      const float pg = p * g;
      r_part += pg;
      for (int jj = 0; jj < kTile; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const float pgj = __shfl_sync(0xffffffffu, pg, jj);
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const int c = lane + 32 * t;
          if (c < d)
            acc[t] = fmaf(pj, gvs[jj * ldk + c], fmaf(pgj, vs[jj * ldk + c], acc[t]));
        }
      }
    } else {  // kRowBobGradq
      const float p = valid ? expf(s - lse_i) : 0.f;
      const float g = a.scale * (g1 + g2);
      const float ds = p * (dp - D_i);
      const float gs = p * (h + (g - r_i) * (dp - D_i) - sig_i);
      for (int jj = 0; jj < kTile; ++jj) {
        const float gsj = __shfl_sync(0xffffffffu, gs, jj);
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const int c = lane + 32 * t;
          if (c < d)
            acc[t] = fmaf(gsj, ks[jj * ldk + c], fmaf(dsj, gks[jj * ldk + c], acc[t]));
        }
      }
    }
  }

  if (!row_ok) return;  // no block-wide barrier follows
  const size_t obase = base + (size_t)i * d;
  if (MODE == kRowForward) {
    const float inv = 1.f / l_run;
#pragma unroll
    for (int t = 0; t < kSlots; ++t) {
      const int c = lane + 32 * t;
      if (c < d) stx<T>(a.out, obase + c, acc[t] * inv);
    }
    if (lane == 0) a.lse_out[srow] = m_run + logf(l_run);
  } else if (MODE == kRowBwdDq || MODE == kRowBobGradq) {
#pragma unroll
    for (int t = 0; t < kSlots; ++t) {
      const int c = lane + 32 * t;
      if (c < d) stx<T>(a.out, obase + c, a.scale * acc[t]);
    }
  } else {  // kRowBob1 epilogue: graddO = W - r O, sigma = dO . graddO
    const float r = warp_sum(r_part);
    float dd = 0.f, sg = 0.f;
    float gdo[kSlots];
#pragma unroll
    for (int t = 0; t < kSlots; ++t) {
      const int c = lane + 32 * t;
      gdo[t] = 0.f;
      if (c < d) {
        const float ov = ldx<T>(a.o, obase + c);
        const float dov = ldx<T>(a.dO, obase + c);
        gdo[t] = acc[t] - r * ov;
        dd = fmaf(dov, ov, dd);
        sg = fmaf(dov, gdo[t], sg);
        stx<T>(a.out, obase + c, gdo[t]);
      }
    }
    dd = warp_sum(dd);
    sg = warp_sum(sg);
    if (lane == 0) {
      a.r_out[srow] = r;
      a.sigma_out[srow] = sg;
      a.D_out[srow] = dd;
    }
  }
}

// ----------------------------------------------------------------------------
// Column-stationary kernel: warp w owns key row j = blockIdx.x*kWarps + w.
// ----------------------------------------------------------------------------
template <typename T, int MODE>
__global__ void __launch_bounds__(kWarps * 32)
    col_kernel(ColArgs a) {
  constexpr bool kBob = (MODE == kColBob2);
  extern __shared__ float sm[];
  const int d = a.d, ldk = d + 1, N = a.N;
  float* ks = sm;                     // [kWarps][d]
  float* vs = ks + kWarps * d;
  float* gks = vs + kWarps * d;
  float* gvs = gks + kWarps * d;
  float* qs = gvs + kWarps * d;       // [kTile][d+1]
  float* dos = qs + kTile * ldk;
  float* gqs = dos + kTile * ldk;
  float* sc = gqs + kTile * ldk;      // [4][kTile]: lse, D, r, sigma

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t bh = blockIdx.y;
  const size_t base = bh * (size_t)N * d;
  const size_t sbase = bh * (size_t)N;
  const int col0 = blockIdx.x * kWarps;
  const int j = col0 + warp;
  const bool col_ok = j < N;

  for (int e = threadIdx.x; e < kWarps * d; e += blockDim.x) {
    const int jj = col0 + e / d, c = e % d;
    const bool ok = jj < N;
    const size_t off = base + (size_t)(ok ? jj : 0) * d + c;
    ks[e] = ok ? ldx<T>(a.k, off) : 0.f;
    vs[e] = ok ? ldx<T>(a.v, off) : 0.f;
    if (kBob) {
      gks[e] = ok && a.gk ? ldx<T>(a.gk, off) : 0.f;
      gvs[e] = ok && a.gv ? ldx<T>(a.gv, off) : 0.f;
    }
  }

  float acc_k[kSlots], acc_v[kSlots];
#pragma unroll
  for (int t = 0; t < kSlots; ++t) acc_k[t] = acc_v[t] = 0.f;

  const int istart = a.causal ? (col0 / kTile) * kTile : 0;
  for (int i0 = istart; i0 < N; i0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int ii = e / d, c = e % d, i = i0 + ii;
      const bool ok = i < N;
      const size_t off = base + (size_t)(ok ? i : 0) * d + c;
      qs[ii * ldk + c] = ok ? ldx<T>(a.q, off) : 0.f;
      dos[ii * ldk + c] = ok ? ldx<T>(a.dO, off) : 0.f;
      if (kBob) gqs[ii * ldk + c] = ok && a.gq ? ldx<T>(a.gq, off) : 0.f;
    }
    if (threadIdx.x < kTile) {
      const int i = i0 + threadIdx.x;
      const bool ok = i < N;
      sc[threadIdx.x] = ok ? a.lse[sbase + i] : 0.f;
      sc[kTile + threadIdx.x] = ok ? a.D[sbase + i] : 0.f;
      if (kBob) {
        sc[2 * kTile + threadIdx.x] = ok ? a.r[sbase + i] : 0.f;
        sc[3 * kTile + threadIdx.x] = ok ? a.sigma[sbase + i] : 0.f;
      }
    }
    __syncthreads();

    const int i = i0 + lane;
    const bool valid = col_ok && i < N && (!a.causal || i >= j);
    const float* krow = ks + warp * d;
    const float* qrow = qs + lane * ldk;
    const float* dorow = dos + lane * ldk;
    float s = 0.f, dp = 0.f, g1 = 0.f, g2 = 0.f, h = 0.f;
    for (int c = 0; c < d; ++c) {
      const float qc = qrow[c], doc = dorow[c];
      s = fmaf(krow[c], qc, s);
      dp = fmaf(vs[warp * d + c], doc, dp);
      if (kBob) {
        g1 = fmaf(gks[warp * d + c], qc, g1);
        g2 = fmaf(krow[c], gqs[lane * ldk + c], g2);
        h = fmaf(gvs[warp * d + c], doc, h);
      }
    }
    s *= a.scale;
    const float lse_i = sc[lane], D_i = sc[kTile + lane];
    const float p = valid ? expf(s - lse_i) : 0.f;
    const float ds = p * (dp - D_i);
    if (!kBob) {
      for (int ii = 0; ii < kTile; ++ii) {
        const float pi = __shfl_sync(0xffffffffu, p, ii);
        const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const int c = lane + 32 * t;
          if (c < d) {
            acc_v[t] = fmaf(pi, dos[ii * ldk + c], acc_v[t]);
            acc_k[t] = fmaf(dsi, qs[ii * ldk + c], acc_k[t]);
          }
        }
      }
    } else {
      const float r_i = sc[2 * kTile + lane], sig_i = sc[3 * kTile + lane];
      const float g = a.scale * (g1 + g2);
      const float gdp = p * (g - r_i);
      const float gs = p * (h + (g - r_i) * (dp - D_i) - sig_i);
      for (int ii = 0; ii < kTile; ++ii) {
        const float gdpi = __shfl_sync(0xffffffffu, gdp, ii);
        const float gsi = __shfl_sync(0xffffffffu, gs, ii);
        const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const int c = lane + 32 * t;
          if (c < d) {
            acc_v[t] = fmaf(gdpi, dos[ii * ldk + c], acc_v[t]);
            acc_k[t] = fmaf(gsi, qs[ii * ldk + c], fmaf(dsi, gqs[ii * ldk + c], acc_k[t]));
          }
        }
      }
    }
  }

  if (!col_ok) return;
  const size_t obase = base + (size_t)j * d;
#pragma unroll
  for (int t = 0; t < kSlots; ++t) {
    const int c = lane + 32 * t;
    if (c < d) {
      stx<T>(a.out_k, obase + c, a.scale * acc_k[t]);
      stx<T>(a.out_v, obase + c, acc_v[t]);
    }
  }
}

// D_i = dO_i . O_i, one warp per row.
template <typename T>
__global__ void __launch_bounds__(256)
    row_dot_kernel(const void* o, const void* dO, float* D, size_t rows, int d) {
  const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32)
    acc = fmaf(ldx<T>(o, row * d + c), ldx<T>(dO, row * d + c), acc);
  acc = warp_sum(acc);
  if (lane == 0) D[row] = acc;
}

size_t row_smem(int d) {
  return sizeof(float) * (3 * kWarps * d + 4 * kTile * (d + 1));
}
size_t col_smem(int d) {
  return sizeof(float) * (4 * kWarps * d + 3 * kTile * (d + 1) + 4 * kTile);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

template <typename T, int MODE>
cudaError_t launch_row(const Problem& p, const RowArgs& a, LaunchLog& log) {
  const size_t smem = row_smem(p.d);
  cudaError_t e = set_smem(row_kernel<T, MODE>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.N + kWarps - 1) / kWarps, p.BH());
  row_kernel<T, MODE><<<grid, kWarps * 32, smem, log.stream>>>(a);
  e = cudaGetLastError();
  log.mark();
  return e;
}

template <typename T, int MODE>
cudaError_t launch_col(const Problem& p, const ColArgs& a, LaunchLog& log) {
  const size_t smem = col_smem(p.d);
  cudaError_t e = set_smem(col_kernel<T, MODE>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.N + kWarps - 1) / kWarps, p.BH());
  col_kernel<T, MODE><<<grid, kWarps * 32, smem, log.stream>>>(a);
  e = cudaGetLastError();
  log.mark();
  return e;
}

template <typename T>
cudaError_t forward_t(const Problem& p, const void* q, const void* k,
                      const void* v, void* o, float* lse, LaunchLog& log) {
  RowArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = o; a.lse_out = lse;
  a.N = p.N; a.d = p.d; a.causal = p.causal; a.scale = p.scale;
  return launch_row<T, kRowForward>(p, a, log);
}

template <typename T>
cudaError_t backward_t(const Problem& p, const void* q, const void* k,
                       const void* v, const void* o, const float* lse,
                       const void* dO, void* dq, void* dk, void* dv,
                       const Workspace& ws, LaunchLog& log) {
  const size_t rows = p.rows();
  row_dot_kernel<T><<<(unsigned)((rows + 7) / 8), 256, 0, log.stream>>>(o, dO, ws.D, rows, p.d);
  cudaError_t e = cudaGetLastError();
  log.mark();
  if (e != cudaSuccess) return e;
  RowArgs a{};
  a.q = q; a.k = k; a.v = v; a.dO = dO; a.lse = lse; a.D = ws.D; a.out = dq;
  a.N = p.N; a.d = p.d; a.causal = p.causal; a.scale = p.scale;
  e = launch_row<T, kRowBwdDq>(p, a, log);
  if (e != cudaSuccess) return e;
  ColArgs c{};
  c.q = q; c.k = k; c.v = v; c.dO = dO; c.lse = lse; c.D = ws.D;
  c.out_k = dk; c.out_v = dv;
  c.N = p.N; c.d = p.d; c.causal = p.causal; c.scale = p.scale;
  return launch_col<T, kColBwdDkdv>(p, c, log);
}

template <typename T>
cudaError_t bob_t(const Problem& p, const void* q, const void* k, const void* v,
                  const void* o, const float* lse, const void* dO,
                  const void* gq, const void* gk, const void* gv, void* gradq,
                  void* gradk, void* gradv, void* graddo, const Workspace& ws,
                  LaunchLog& log) {
  RowArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.dO = dO; a.gq = gq; a.gk = gk; a.gv = gv;
  a.lse = lse; a.out = graddo; a.r_out = ws.r; a.sigma_out = ws.sigma; a.D_out = ws.D;
  a.N = p.N; a.d = p.d; a.causal = p.causal; a.scale = p.scale;
  cudaError_t e = launch_row<T, kRowBob1>(p, a, log);
  if (e != cudaSuccess) return e;
  ColArgs c{};
  c.q = q; c.k = k; c.v = v; c.dO = dO; c.gq = gq; c.gk = gk; c.gv = gv;
  c.lse = lse; c.D = ws.D; c.r = ws.r; c.sigma = ws.sigma;
  c.out_k = gradk; c.out_v = gradv;
  c.N = p.N; c.d = p.d; c.causal = p.causal; c.scale = p.scale;
  e = launch_col<T, kColBob2>(p, c, log);
  if (e != cudaSuccess) return e;
  RowArgs b = a;
  b.o = nullptr; b.D = ws.D; b.r = ws.r; b.sigma = ws.sigma; b.out = gradq;
  b.r_out = b.sigma_out = b.D_out = nullptr;
  return launch_row<T, kRowBobGradq>(p, b, log);
}

}  // namespace

cudaError_t simt_forward(const Problem& p, const void* q, const void* k,
                         const void* v, void* o, float* lse, LaunchLog& log) {
  return p.bf16 ? forward_t<__nv_bfloat16>(p, q, k, v, o, lse, log)
                : forward_t<float>(p, q, k, v, o, lse, log);
}

cudaError_t simt_backward(const Problem& p, const void* q, const void* k,
                          const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv,
                          const Workspace& ws, LaunchLog& log) {
  return p.bf16 ? backward_t<__nv_bfloat16>(p, q, k, v, o, lse, dO, dq, dk, dv, ws, log)
                : backward_t<float>(p, q, k, v, o, lse, dO, dq, dk, dv, ws, log);
}

cudaError_t simt_bob(const Problem& p, const void* q, const void* k,
                     const void* v, const void* o, const float* lse,
                     const void* dO, const void* gq, const void* gk,
                     const void* gv, void* gradq, void* gradk, void* gradv,
                     void* graddo, const Workspace& ws, LaunchLog& log) {
  return p.bf16 ? bob_t<__nv_bfloat16>(p, q, k, v, o, lse, dO, gq, gk, gv, gradq,
                                       gradk, gradv, graddo, ws, log)
                : bob_t<float>(p, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk,
                               gradv, graddo, ws, log);
}

}  // namespace fbob

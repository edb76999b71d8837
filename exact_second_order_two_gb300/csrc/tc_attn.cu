// Tensor-core (tcgen05 / TMEM / TMA) kernels for sm_103a: the attention
// forward and first backward whose outputs the backward-over-backward of
// FlashBoB ("FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention", Abstract) consumes.  With c the scale:
//   S = c Q K^T,  LSE_i = log sum_j exp(S_ij),  P = exp(S - LSE),  O = P V;
//   dP = dO V^T,  D_i = dO_i . O_i,  dS = P*(dP - D),
//   dQ = c dS K,  dK = c dS^T Q,  dV = P^T dO.
//
// forward (row-stationary, 128 query rows per CTA, 128-key tiles): one sweep
//   over the key tiles with an online softmax.  S goes into TMEM; bf16
//   P = 2^(S c log2 e - m) is written over it and O += P V accumulates in
//   TMEM.  The reference maximum m moves only when a tile's maximum exceeds
//   it by more than 8 (log2 units), and O is then rescaled in TMEM; the
//   epilogue divides by the row sum and writes LSE.  At d = 128 the four
//   column slices of a row share m (agreed per tile through shared memory);
//   at d = 64 each slice has its own m and its own O, combined in the
//   epilogue.
// first backward (key-stationary, 128 key rows per CTA, 64-query tiles):
//   S^T and dP^T into TMEM; bf16 P^T and dS^T written back into the S^T
//   columns as the A operands of dV += P^T dO and dK += dS^T Q; the next
//   tile's scores are issued before this tile's dQ^T = K^T dS^T, which the
//   elementwise warps read out one tile late and stage in shared memory; a
//   TMA reduce-add carries it into an fp32 accumulator (at d = 128 half of
//   the features, the other half by red.global), then converted.
//
// Warp roles as in the BoB kernels: elementwise warps own TMEM lanes, one TMA
// producer warp, one MMA warp (TMEM allocator; elect.sync picks the issuing
// lane), and in the first backward a warp issuing the reduce-adds.  Every
// mbarrier wait is bounded, and every warp-collective operation sits in
// warp-uniform control flow.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "sm103.cuh"
#include "tc_common.cuh"

namespace fbob {

using namespace sm103;
using namespace tc;

namespace {

// Forward warp roles: warps 0-15 elementwise (warp w: TMEM lane quadrant
// w % 4, 32-key slice w / 4 of the 128-key tile), warp 16 TMA producer,
// warp 17 TMEM allocator and MMA issuer.
constexpr int kFwdConsumerWarps = 16;
constexpr int kFwdConsumers = kFwdConsumerWarps * 32;
constexpr int kFwdProducerWarp = kFwdConsumerWarps;
constexpr int kFwdMmaWarp = kFwdConsumerWarps + 1;
constexpr int kFwdThreads = (kFwdConsumerWarps + 2) * 32;
constexpr int kFwdSlices = kFwdConsumerWarps / 4;  // column slices per row
constexpr int kFwdCols = 128 / kFwdSlices;          // key columns per thread
constexpr float kLn2 = 0.6931471805599453f;

// ===========================================================================
// Forward: row-stationary, one sweep over the key tiles with an online
// softmax.
// ===========================================================================
template <int D>
struct Fwd {
  static constexpr int BM = 128, BN = 128;
  static constexpr int KSTAGES = D == 128 ? 3 : 4, VSTAGES = D == 128 ? 2 : 3;
  static constexpr uint32_t QB = BM * D * 2;   // stationary Q tile
  static constexpr uint32_t KB = BN * D * 2;   // one streamed K or V tile
  static constexpr uint32_t OFF_Q = 0, OFF_K = QB, OFF_V = OFF_K + KSTAGES * KB;
  // [2][slices][128] per-tile row maxima, then [slices][128] row sums
  static constexpr uint32_t OFF_RED = OFF_V + VSTAGES * KB;
  static constexpr uint32_t OFF_MISC = OFF_RED + 3 * kFwdSlices * 128 * 4;
  static constexpr uint32_t MISC = 512;
  static constexpr uint32_t SMEM = OFF_MISC + MISC;
  static_assert(SMEM <= 232448, "forward shared memory budget");
  // TMEM columns: S (two buffers of 128), O, bf16 Q as the A operand of
  // S = Q K^T (at d = 64: four O's, one per slice, and Q stays in shared
  // memory).  Each elementwise thread writes bf16 P over the first 16 of
  // the 32 S columns it read: keys 32s + 2c, + 1 of slice s in column
  // 32s + c, so 16-key step k of P V sits at p_col(k).
  static constexpr uint32_t T_O = 256, TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t T_S(int b) { return 128u * b; }
  __host__ __device__ static constexpr uint32_t p_col(int k) { return 32u * (k >> 1) + 8u * (k & 1); }
  static constexpr uint32_t T_QA = 256 + D;
  static_assert(T_QA + D / 2 <= TMEM_COLS, "forward TMEM budget");
  // The running row maximum m (log2 domain) only moves when a tile's maximum
  // exceeds it by more than kRescale: P = 2^(S c log2 e - m) then stays
  // below 2^kRescale, and O is rescaled in TMEM only on those rare moves.
  static constexpr float kRescale = 8.f;
  // d = 64: one O accumulator per column slice (columns 256 + 64 s), each
  // with its own reference maximum, combined in the epilogue.  At d = 64 the
  // tile's MMAs (about 640 cycles) do not hide a per-tile exchange of the
  // row maximum between the slices; without it the forward at 4 x 262144
  // went from 45.3 to 42.8 ms.  S = Q K^T then takes Q from shared memory:
  // the TMEM columns of its copy hold the fourth O, and an N=128 MMA costs
  // the same with both operands in shared memory.
  static constexpr bool PSO = D == 64;
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int* status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int N, causal;
  int BH, G;  // batch * heads, heads per CTA group (cta_coord)
  float scale;
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_row_pass(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                 const __grid_constant__ CUtensorMap mV, FwdParams prm) {
  using C = Fwd<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report_status(prm.status, FBOB_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;                   // [KSTAGES]
  uint64_t* k_empty = k_full + C::KSTAGES;       // [KSTAGES]
  uint64_t* v_full = k_empty + C::KSTAGES;       // [VSTAGES]
  uint64_t* v_empty = v_full + C::VSTAGES;       // [VSTAGES]
  uint64_t* s_full = v_empty + C::VSTAGES;       // [2]
  uint64_t* s_empty = s_full + 2;                // [2]: S read out of TMEM
  uint64_t* p_full = s_empty + 2;                // [2]: bf16 P written over S, O rescaled
  uint64_t* o_ready = p_full + 2;                // one phase per tile: P V MMAs done
  uint64_t* red_full = o_ready + 1;              // [2]: the slices' tile maxima written
  uint64_t* q_tmem = red_full + 2;
  uint64_t* drain = q_tmem + 1;
  static_assert((12 + 2 * C::KSTAGES + 2 * C::VSTAGES) * 8 <= 256,
                "barriers end below the TMEM slot");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 256);
  Abort* abort_st = reinterpret_cast<Abort*>(smem + C::OFF_MISC + 264);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = prm.N;
  const int nblk = (prm.N + C::BM - 1) / C::BM;
  const CtaCoord cc = cta_coord(prm.BH, prm.G, nblk);
  const int bh = cc.bh;
  // heavy (late) row blocks first under a causal mask
  const int blk = prm.causal ? (nblk - 1 - cc.blk) : cc.blk;
  const int i0 = blk * C::BM;
  const int kend = prm.causal ? min(N, i0 + C::BM) : N;
  const int T = (kend + C::BN - 1) / C::BN;
  // every CTA walks the key tiles from the first, so the CTAs of one head
  // share them in L2 (as in BoB pass 1)
  const int rot = 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::KSTAGES; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(s_empty + b, kFwdConsumers);
      mbar_init(p_full + b, kFwdConsumers);
    }
    mbar_init(o_ready, 1);
    mbar_init(red_full + 0, kFwdConsumers);
    mbar_init(red_full + 1, kFwdConsumers);
    mbar_init(q_tmem, kFwdConsumers);
    mbar_init(drain, 1);
    abort_st->flag = 0;
    abort_st->limit_ns = prm.wait_ns;
    fence_mbar_init();
  }
  if (warp == kFwdMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kFwdProducerWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, C::QB);
      load_tile(smem + C::OFF_Q, &mQ, q_full, i0, bh);
      int k_issued = 0, v_issued = 0;
      // K runs ahead of V: S(t) needs K(t) one tile before P V(t) needs V(t)
      auto load_k = [&](int t) -> bool {
        const int s = t % C::KSTAGES;
        if (t >= C::KSTAGES &&
            !wait_bar(k_empty + s, ((t / C::KSTAGES) - 1) & 1, abort_st, prm.status))
          return false;
        mbar_arrive_expect_tx(k_full + s, C::KB);
        load_tile(smem + C::OFF_K + s * C::KB, &mK, k_full + s, rotated(t, rot, T) * C::BN, bh);
        ++k_issued;
        return true;
      };
      auto load_v = [&](int t) -> bool {
        const int s = t % C::VSTAGES;
        if (t >= C::VSTAGES &&
            !wait_bar(v_empty + s, ((t / C::VSTAGES) - 1) & 1, abort_st, prm.status))
          return false;
        mbar_arrive_expect_tx(v_full + s, C::KB);
        load_tile(smem + C::OFF_V + s * C::KB, &mV, v_full + s, rotated(t, rot, T) * C::BN, bh);
        ++v_issued;
        return true;
      };
      bool pok = load_k(0);
      for (int t = 0; pok && t < T; ++t) {
        if (t + 1 < T && !load_k(t + 1)) break;
        if (!load_v(t)) break;
      }
      // every load this thread issued has landed before the CTA exits (after
      // an abort some were never awaited); each phase waited for is the last
      // of its barrier, so on the normal path these return at once
      mbar_wait_bounded(q_full, 0, prm.status, 100000000ull);
      for (int t = max(0, k_issued - C::KSTAGES); t < k_issued; ++t)
        mbar_wait_bounded(k_full + (t % C::KSTAGES), (t / C::KSTAGES) & 1, prm.status,
                          100000000ull);
      for (int t = max(0, v_issued - C::VSTAGES); t < v_issued; ++t)
        mbar_wait_bounded(v_full + (t % C::VSTAGES), (t / C::VSTAGES) & 1, prm.status,
                          100000000ull);
    }
  } else if (warp == kFwdMmaWarp) {
    {  // the whole warp: warp-uniform waits, elect.sync issues each MMA
      constexpr uint32_t id_s = idesc_bf16(128, C::BN, false, false);  // S = Q K^T: N = BN
      constexpr uint32_t id_o = idesc_bf16(128, D, false, true);       // O += P V: N = D, B MN
      const uint32_t t_o = tmem + C::T_O, t_q = tmem + C::T_QA;
      bool ok = warp_wait(q_tmem, 0, abort_st, prm.status);
      // O += P(t) V(t), A = bf16 P from TMEM (in S buffer t & 1), contraction
      // over the tile's keys; o_ready completes once per tile
      auto issue_pv = [&](int t) -> bool {
        const int pb = t & 1, vs = t % C::VSTAGES;
        if (!warp_wait(p_full + pb, (t >> 1) & 1, abort_st, prm.status)) return false;
        if (!warp_wait(v_full + vs, (t / C::VSTAGES) & 1, abort_st, prm.status)) return false;
        tc_fence_after();
        const uint32_t v_mn = opaque(lo_mnmajor(sb + C::OFF_V + vs * C::KB, C::BN * 128));
        const uint32_t t_p = tmem + C::T_S(pb);
#pragma unroll
        for (int k = 0; k < C::BN / 16; ++k) {
          // PSO: key steps 2s, 2s + 1 are slice s's, into its own O
          const uint32_t to = C::PSO ? t_o + 64u * (uint32_t)(k >> 1) : t_o;
          const bool chained = C::PSO ? (k & 1) != 0 : k > 0;
          mma_ts_w(to, t_p + C::p_col(k), v_mn + kstep_off(k), id_o, (t > 0 || chained) ? 1u : 0u);
        }
        mma_commit_w(v_empty + vs);
        mma_commit_w(o_ready);
        return true;
      };
      // S(t) reuses the buffer of tile t - 2: read out (s_empty) and its P
      // consumed by the P V MMAs of tile t - 2, issued before S(t)
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % C::KSTAGES, b = t & 1;
        if (!warp_wait(k_full + s, (t / C::KSTAGES) & 1, abort_st, prm.status)) { ok = false; break; }
        if (t >= 2 && !warp_wait(s_empty + b, ((t >> 1) - 1) & 1, abort_st, prm.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_lo = opaque(lo_kmajor(sb + C::OFF_K + s * C::KB));
        const uint32_t q_lo = opaque(lo_kmajor(sb + C::OFF_Q));
        const uint32_t t_s = tmem + C::T_S(b);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          if (C::PSO)
            mma_ss_w(t_s, q_lo + kslice_off(C::BM, k), k_lo + kslice_off(C::BN, k), id_s,
                     k > 0 ? 1u : 0u);
          else
            mma_ts_w(t_s, t_q + 8 * k, k_lo + kslice_off(C::BN, k), id_s, k > 0 ? 1u : 0u);
        }
        mma_commit_w(s_full + b);
        mma_commit_w(k_empty + s);
        if (t >= 1 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(T - 1);
      // every MMA this thread issued has completed before TMEM is released
      mma_commit_w(drain);
      mbar_wait_bounded(drain, 0, prm.status, 100000000ull);
    }
  } else {
    // ---------------- elementwise warps: thread = query row --------------
    constexpr int NC = kFwdCols, NS = kFwdSlices;
    const int row = 32 * (warp & 3) + lane;
    const int slice = warp >> 2;  // key columns [NC*slice, NC*slice + NC) of a tile
    const int i = i0 + row;
    const bool row_ok = i < N;
    const size_t srow = (size_t)bh * N + (row_ok ? i : 0);
    const float sc2 = prm.scale * kLog2e;
    const f2 sc2_2 = {sc2, sc2};
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    bool ok = warp_wait(q_full, 0, abort_st, prm.status);
    if (ok) {
      // stationary Q row -> TMEM (bf16 pairs, lower half = even feature): one
      // 64-feature half-row per thread of slices 0 .. D/64 - 1
      if (!C::PSO && slice < D / 64) {
        const uint32_t src = C::OFF_Q + slice * C::BM * 128 + row * 128;
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(smem + src + ((c ^ (row & 7)) << 4));
          uint32_t* dst = c < 4 ? lo + 4 * c : hi + 4 * (c - 4);
          dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
        }
        const uint32_t dst = tmem + lane_off + C::T_QA + 32 * slice;
        tmem_st16(dst, lo);
        tmem_st16(dst + 16, hi);
      }
      tc_fence_before();
      mbar_arrive(q_tmem);
    }
    // m: the row's reference maximum (log2 domain), the same in all slices;
    // l: this slice's sum of 2^(S c log2 e - m)
    float m = -INFINITY, l = 0.f;
    for (int t = 0; ok && t < T; ++t) {
      const int b = t & 1;
      if (!warp_wait(s_full + b, (t >> 1) & 1, abort_st, prm.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[NC];
      tmem_ld32(tmem + lane_off + C::T_S(b) + NC * slice, sr);
      tc_fence_before();
      mbar_arrive(s_empty + b);
      const int j0 = rotated(t, rot, T) * C::BN + NC * slice;
      const bool need_mask = !row_ok || (j0 + NC > N) || (prm.causal && j0 + NC - 1 > i);
      // this slice's raw maximum (c log2 e > 0 keeps the order); masked
      // entries become -inf, so they give 2^-inf = 0 below
      float mx = -INFINITY;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int j = j0 + c;
          const bool in = row_ok && j < N && (!prm.causal || j <= i);
          const float v = in ? __uint_as_float(sr[c]) : -INFINITY;
          sr[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      } else {
#pragma unroll
        for (int c = 0; c < NC; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      }
      // the row's maximum over the tile, through shared memory and a bounded
      // wait on an mbarrier (one buffer per tile parity: a buffer is
      // rewritten only after every thread has arrived for the next tile,
      // hence after it read this one)
      float mt = mx * sc2;  // PSO: this slice's own maximum is its reference
      if (!C::PSO) {
        float* rt = red + b * NS * 128;
        rt[slice * 128 + row] = mt;
        mbar_arrive(red_full + b);
        if (!warp_wait(red_full + b, (t >> 1) & 1, abort_st, prm.status)) { ok = false; break; }
        mt = -INFINITY;
#pragma unroll
        for (int u = 0; u < NS; ++u) mt = fmaxf(mt, rt[u * 128 + row]);
      }
      // the reference maximum moves (the same decision in every slice of a
      // row; rows, i.e. lanes, decide independently)
      const bool move = mt > m + C::kRescale;
      const float alpha = move ? ex2_approx(m - mt) : 1.f;  // 0 while m is still -inf
      l *= alpha;
      // O (this slice's D/NS columns of the row) holds the P V sums of the
      // earlier tiles: rescale it once their MMAs are done.  The wait and the
      // TMEM accesses are warp-collective, so the whole warp takes this
      // branch when any lane needs it; the other lanes scale by 1.
      const bool scale_o = move && t >= 1 && m > -INFINITY;
      if (__any_sync(0xffffffffu, scale_o)) {
        if (!warp_wait(o_ready, (t - 1) & 1, abort_st, prm.status)) { ok = false; break; }
        tc_fence_after();
        const float f = scale_o ? alpha : 1.f;
        constexpr int PART = C::PSO ? D : D / NS;  // PSO: the slice's whole O
#pragma unroll
        for (int cc = 0; cc < PART; cc += 16) {
          uint32_t v[16];
          const uint32_t ta = tmem + lane_off + C::T_O + PART * slice + cc;
          tmem_ld16(ta, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
          tmem_st16(ta, v);
        }
      }
      if (move) m = mt;
      uint32_t pw[NC / 2];
      if (m > -INFINITY) {
        const f2 nm = {-m, -m};
        f2 acc = {0.f, 0.f};
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
          const f2 x = fma2({__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, sc2_2, nm);
          const f2 p = {ex2_approx(x.x), ex2_approx(x.y)};
          acc = add2(acc, p);
          pw[c >> 1] = pack_bf16(p.x, p.y);
        }
        l += acc.x + acc.y;
      } else {
#pragma unroll
        for (int c = 0; c < NC / 2; ++c) pw[c] = 0u;
      }
      // bf16 P over the first 16 of the 32 S columns this thread read: keys
      // NC*slice + 2c, + 1 in column NC*slice + c (two 16-key MMA steps)
      tmem_st16(tmem + lane_off + C::T_S(b) + NC * slice, pw);
      tc_fence_before();
      mbar_arrive(p_full + b);
    }
    // ---- epilogue: O / l (bf16) and LSE (natural log) ----
    // the slices' sums share the reference maximum m; every consumer thread
    // gets to this barrier, also after a failed wait
    float* part = red + 2 * NS * 128;
    part[slice * 128 + row] = l;
    if (C::PSO) red[slice * 128 + row] = m;
    named_sync<kFwdConsumers>(1);
    float L = 0.f;
    float fs[NS];  // PSO: weight of slice u's O and sum against the row maximum
    if (C::PSO) {
      float M = -INFINITY;
#pragma unroll
      for (int u = 0; u < NS; ++u) M = fmaxf(M, red[u * 128 + row]);
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        const float mu = red[u * 128 + row];
        fs[u] = mu > -INFINITY ? ex2_approx(mu - M) : 0.f;
        L += part[u * 128 + row] * fs[u];
      }
      m = M;
    } else {
#pragma unroll
      for (int u = 0; u < NS; ++u) L += part[u * 128 + row];
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = warp_wait(o_ready, (T - 1) & 1, abort_st, prm.status);
    tc_fence_after();
    if (ok) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      constexpr int PART = D / NS;  // output features per thread
      uint4* op = reinterpret_cast<uint4*>(prm.o + srow * D + PART * slice);
#pragma unroll
      for (int cc = 0; cc < PART; cc += 16) {
        uint32_t v[16];
        if (C::PSO) {
          float a[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) a[e] = 0.f;
#pragma unroll
          for (int u = 0; u < NS; ++u) {
            tmem_ld16(tmem + lane_off + C::T_O + 64u * u + PART * slice + cc, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) a[e] = fmaf(fs[u], __uint_as_float(v[e]), a[e]);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(a[e]);
        } else {
          tmem_ld16(tmem + lane_off + C::T_O + PART * slice + cc, v);
        }
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 2; ++q)
            op[cc / 8 + q] = make_uint4(
                pack_bf16(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv),
                pack_bf16(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv),
                pack_bf16(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv),
                pack_bf16(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv));
        }
      }
      if (slice == 0 && row_ok) prm.lse[srow] = (m > -INFINITY && L > 0.f) ? (m + log2f(L)) * kLn2 : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ===========================================================================
// First backward: key-stationary.
// ===========================================================================
template <int D>
struct Bwd {
  static constexpr int BM = 128, BN = 64;
  // Q (+ row scalars) ring and dO ring: three stages each, because the next
  // tile's S^T and dP^T are issued while this tile's elementwise phase runs,
  // before this tile's dK / dV MMAs have released its Q and dO
  static constexpr int STAGES = 3, DSTAGES = 3;
  static constexpr uint32_t KB = BM * D * 2;     // stationary K, V tile
  static constexpr uint32_t QB = BN * D * 2;     // streamed Q, dO tile
  static constexpr uint32_t XB = BM * BN * 2;    // dS^T tile (dQ^T B operand)
  static constexpr uint32_t OFF_K = 0, OFF_V = KB, OFF_Q = 2 * KB;
  static constexpr uint32_t OFF_DO = OFF_Q + STAGES * QB;
  static constexpr uint32_t OFF_DS = OFF_DO + DSTAGES * QB;
  static constexpr uint32_t OFF_SC = OFF_DS + XB;            // [STAGES][2][BN] fp32
  // dQ^T partials go from TMEM to global memory through shared memory: the
  // elementwise warps write a tile's partial as [BN][SF] fp32 rows into one
  // of two staging buffers and a TMA reduce-add carries it into the
  // accumulator.  At d = 128 the staging carries features 0-63 only; the
  // threads holding features 64-127 add theirs with red.global.  Shared
  // memory is this kernel's limit (MMA operand reads, the dS^T stores and
  // the staging round trip), and halving the staged bytes took the
  // benchmark workload's first backward from 4.70 to 4.51 ms.
  static constexpr int SF = D == 128 ? 64 : D;  // features staged per row
  static constexpr uint32_t STGB = BN * SF * 4;
  static constexpr int SBUF = 2;
  static constexpr uint32_t OFF_STG = (OFF_SC + STAGES * 2 * BN * 4 + 1023) / 1024 * 1024;
  static constexpr uint32_t OFF_MISC = OFF_STG + SBUF * STGB;
  static constexpr uint32_t MISC = 512;
  static constexpr uint32_t SMEM = OFF_MISC + MISC;
  static_assert(SMEM <= 232448, "backward shared memory budget");
  // TMEM columns.  S^T has two buffers, so the next tile's S^T (and dP^T,
  // once its predecessor has been read out) is computed while the
  // elementwise warps work on this tile: they start the next tile as soon
  // as they are done with this one, and the dK / dV / dQ^T MMAs of a tile
  // run during the next tile's elementwise phase.  After reading a tile's
  // scores the elementwise warps write, inside the 16 S^T columns each of
  // them read, bf16 P^T (first 8) and dS^T (last 8): the A operands of the
  // dV / dK MMAs.
  __host__ __device__ static constexpr uint32_t T_S(int b) { return 64u * b; }
  static constexpr uint32_t T_DP = 128, T_DK = 192, T_DV = 192 + D, T_DQ = 192 + 2 * D;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(T_DQ + 64 <= TMEM_COLS, "backward TMEM budget");
};

struct BwdParams {
  const float* lse;
  const float* Dv;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int N, causal;
  int BH, G;  // batch * heads, heads per CTA group (cta_coord)
  float scale;
  float* acc;  // fp32 dQ accumulator, for the features the staging does not carry
};

// Warps 0-15 elementwise, 16 TMA producer, 17 MMA issuer, 18 issues the TMA
// reduce-add of each staged dQ^T partial (per-thread atomics for the whole
// partial kept the elementwise warps issuing for over a thousand cycles per
// tile; at d = 128 they carry half of it, which relieves shared memory).
constexpr int kBwdConsumerWarps = 16;
constexpr int kBwdConsumers = kBwdConsumerWarps * 32;
constexpr int kBwdProducerWarp = kBwdConsumerWarps;
constexpr int kBwdMmaWarp = kBwdConsumerWarps + 1;
constexpr int kBwdReduceWarp = kBwdConsumerWarps + 2;
constexpr int kBwdThreads = (kBwdConsumerWarps + 3) * 32;
constexpr int kBwdCols = 16;  // query columns per elementwise thread

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_col_pass(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                 const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mDO,
                 const __grid_constant__ CUtensorMap mACC, BwdParams prm) {
  using C = Bwd<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {
    if (threadIdx.x == 0) report_status(prm.status, FBOB_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;                  // [STAGES]: Q landed, scalars written
  uint64_t* q_empty = q_full + C::STAGES;       // [STAGES]: dK MMAs done with Q
  uint64_t* do_full = q_empty + C::STAGES;      // [DSTAGES]
  uint64_t* do_empty = do_full + C::DSTAGES;    // [DSTAGES]: dV MMAs done with dO
  uint64_t* s_full = do_empty + C::DSTAGES;     // [2]: S^T of a buffer in TMEM
  uint64_t* dp_full = s_full + 2;               // dP^T in TMEM
  uint64_t* dp_read = dp_full + 1;              // elementwise warps hold S^T and dP^T
  uint64_t* ds_full = dp_read + 1;
  uint64_t* dq_full = ds_full + 1;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* acc_done = dq_empty + 1;
  uint64_t* drain = acc_done + 1;
  uint64_t* stg_full = drain + 1;               // [SBUF]: a dQ^T partial staged
  uint64_t* stg_free = stg_full + 2;            // [SBUF]: its reduce-add has read it
  static_assert((15 + 2 * C::STAGES + 2 * C::DSTAGES) * 8 <= 256,
                "barriers end below the TMEM slot");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 256);
  Abort* abort_st = reinterpret_cast<Abort*>(smem + C::OFF_MISC + 264);
  float* scal = reinterpret_cast<float*>(smem + C::OFF_SC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = prm.N;
  const CtaCoord cc = cta_coord(prm.BH, prm.G, (prm.N + C::BM - 1) / C::BM);
  const int bh = cc.bh;
  const int j0 = cc.blk * C::BM;
  const int qstart = prm.causal ? (j0 / C::BN) * C::BN : 0;
  const int T = (N - qstart + C::BN - 1) / C::BN;
  // every CTA walks the query tiles from its first (unlike BoB pass 2,
  // where rotated start tiles measured faster at long N)
  const int rot = 0;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    for (int s = 0; s < C::DSTAGES; ++s) {
      mbar_init(do_full + s, 1);
      mbar_init(do_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_full + 1, 1);
    mbar_init(dp_full, 1);
    mbar_init(dp_read, kBwdConsumers);
    mbar_init(ds_full, kBwdConsumers);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, kBwdConsumers);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    for (int b = 0; b < C::SBUF; ++b) {
      mbar_init(stg_full + b, kBwdConsumers);
      mbar_init(stg_free + b, 1);
    }
    abort_st->flag = 0;
    abort_st->limit_ns = prm.wait_ns;
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdProducerWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::KB);
      load_tile(smem + C::OFF_K, &mK, kv_full, j0, bh);
      load_tile(smem + C::OFF_V, &mV, kv_full, j0, bh);
    }
    // row scalars (LSE pre-scaled by log2 e, D) of the next query tile are
    // fetched into registers one tile ahead
    constexpr int PER = C::BN / 32;
    float pre[2][PER];
    auto fetch = [&](int q0) {
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int q = q0 + lane + 32 * u;
        const bool in = q < N;
        const size_t idx = (size_t)bh * N + (in ? q : 0);
        pre[0][u] = in ? prm.lse[idx] * kLog2e : 0.f;
        pre[1][u] = in ? prm.Dv[idx] : 0.f;
      }
    };
    fetch(qstart + rotated(0, rot, T) * C::BN);
    int q_issued = 0, do_issued = 0;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::STAGES, ds = t % C::DSTAGES;
      const int q0 = qstart + rotated(t, rot, T) * C::BN;
      bool w = true;
      if (lane == 0) {
        if (t >= C::DSTAGES)
          w = wait_bar(do_empty + ds, ((t / C::DSTAGES) - 1) & 1, abort_st, prm.status);
        if (w) {
          mbar_arrive_expect_tx(do_full + ds, C::QB);
          load_tile(smem + C::OFF_DO + ds * C::QB, &mDO, do_full + ds, q0, bh);
          ++do_issued;
        }
        if (w && t >= C::STAGES)
          w = wait_bar(q_empty + s, ((t / C::STAGES) - 1) & 1, abort_st, prm.status);
      }
      if (__shfl_sync(0xffffffffu, w ? 1 : 0, 0) == 0) break;
      // the stage's scalars were last read by the elementwise warps of tile
      // t - STAGES, which finished before the dK MMAs that freed the stage;
      // stored negated, since both are subtracted
      float* sc = scal + s * 2 * C::BN;
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int u = 0; u < PER; ++u) sc[a * C::BN + lane + 32 * u] = -pre[a][u];
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full + s, C::QB);
        load_tile(smem + C::OFF_Q + s * C::QB, &mQ, q_full + s, q0, bh);
        ++q_issued;
      }
      if (t + 1 < T) fetch(qstart + rotated(t + 1, rot, T) * C::BN);
    }
    // every load this warp issued has landed before the CTA exits (after an
    // abort some were never awaited); each phase waited for is the last of
    // its barrier, so on the normal path these return at once
    if (lane == 0) {
      mbar_wait_bounded(kv_full, 0, prm.status, 100000000ull);
      for (int t = max(0, q_issued - C::STAGES); t < q_issued; ++t)
        mbar_wait_bounded(q_full + (t % C::STAGES), (t / C::STAGES) & 1, prm.status,
                          100000000ull);
      for (int t = max(0, do_issued - C::DSTAGES); t < do_issued; ++t)
        mbar_wait_bounded(do_full + (t % C::DSTAGES), (t / C::DSTAGES) & 1, prm.status,
                          100000000ull);
    }
  } else if (warp == kBwdReduceWarp) {
    if (lane == 0) {
      // one reduce-add per tile, in tile order: the partial of tile u sits
      // in staging buffer u % SBUF
      for (int u = 0; u < T; ++u) {
        const int b = u % C::SBUF;
        if (!wait_bar(stg_full + b, (u / C::SBUF) & 1, abort_st, prm.status)) break;
        tma_reduce_add_3d(&mACC, smem + C::OFF_STG + b * C::STGB, 0,
                          qstart + rotated(u, rot, T) * C::BN, bh);
        bulk_commit_group();
        bulk_wait_read_all();  // the buffer may be refilled
        mbar_arrive(stg_free + b);
      }
      bulk_wait_all();  // every reduce-add has landed before the CTA exits
    }
  } else if (warp == kBwdMmaWarp) {
    {  // the whole warp: warp-uniform waits, elect.sync issues each MMA
      constexpr uint32_t id_sc = idesc_bf16(128, 64, false, false);  // scores: M=128 N=64
      constexpr uint32_t id_out = idesc_bf16(128, D, false, true);   // dK/dV: N=D, B MN
      constexpr uint32_t id_dq = idesc_bf16(D, 64, true, true);      // dQ^T: M=D, A,B MN
      const uint32_t k_lo = lo_kmajor(sb + C::OFF_K), v_lo = lo_kmajor(sb + C::OFF_V);
      const uint32_t k_mn = lo_mnmajor(sb + C::OFF_K, C::BM * 128);
      const uint32_t ds_mn = lo_mnmajor(sb + C::OFF_DS, 1024);
      const uint32_t t_dp = tmem + C::T_DP, t_dk = tmem + C::T_DK, t_dv = tmem + C::T_DV,
                     t_dq = tmem + C::T_DQ;
      // dP^T of tile t (needs dO(t) and the previous tile's dP^T read out),
      // then its commit
      auto issue_dp = [&](int t) -> bool {
        const int ds = t % C::DSTAGES;
        const uint32_t do_lo = opaque(lo_kmajor(sb + C::OFF_DO + ds * C::QB));
        const uint32_t v_l = opaque(v_lo);
        if (!warp_wait(do_full + ds, (t / C::DSTAGES) & 1, abort_st, prm.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_w(t_dp, v_l + kslice_off(C::BM, k), do_lo + kslice_off(C::BN, k), id_sc,
                 k > 0 ? 1u : 0u);
        mma_commit_w(dp_full);
        return true;
      };
      // S^T of tile t into buffer t & 1 (needs Q(t); overwrites the A
      // operands of tile t - 2, whose dK / dV MMAs were issued before), then
      // its commit
      auto issue_s = [&](int t) -> bool {
        const int s = t % C::STAGES;
        const uint32_t q_lo = opaque(lo_kmajor(sb + C::OFF_Q + s * C::QB));
        const uint32_t k_l = opaque(k_lo);
        if (!warp_wait(q_full + s, (t / C::STAGES) & 1, abort_st, prm.status)) return false;
        tc_fence_after();
        const uint32_t t_s = tmem + C::T_S(t & 1);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_w(t_s, k_l + kslice_off(C::BM, k), q_lo + kslice_off(C::BN, k), id_sc,
                 k > 0 ? 1u : 0u);
        mma_commit_w(s_full + (t & 1));
        return true;
      };
      bool ok = warp_wait(kv_full, 0, abort_st, prm.status) && issue_dp(0) && issue_s(0);
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % C::STAGES, ds = t % C::DSTAGES;
        // ---- next tile's dP^T and S^T while the elementwise warps work ----
        if (t + 1 < T) {
          if (!warp_wait(dp_read, t & 1, abort_st, prm.status)) { ok = false; break; }
          tc_fence_after();
          if (!issue_dp(t + 1) || !issue_s(t + 1)) { ok = false; break; }
        }
        if (!warp_wait(ds_full, t & 1, abort_st, prm.status)) { ok = false; break; }
        tc_fence_after();
        // dQ^T of tile t first, once the previous one has been read out of
        // TMEM: the next tile's elementwise phase drains it, and issued
        // before dK / dV it is ready sooner (dK / dV only free ring stages
        // and this tile's S^T buffer, which are not needed yet)
        if (t >= 1) {
          if (!warp_wait(dq_empty, (t - 1) & 1, abort_st, prm.status)) { ok = false; break; }
          tc_fence_after();
        }
        {
          const uint32_t k_m = opaque(k_mn), ds_m = opaque(ds_mn);
#pragma unroll
          for (int k = 0; k < C::BM / 16; ++k)  // contraction over the 128 keys
            mma_ss_w(t_dq, k_m + kstep_off(k), ds_m + kstep_off(k), id_dq, k > 0 ? 1u : 0u);
          mma_commit_w(dq_full);
        }
        {
          const uint32_t q_mn = opaque(lo_mnmajor(sb + C::OFF_Q + s * C::QB, C::BN * 128));
          const uint32_t do_mn = opaque(lo_mnmajor(sb + C::OFF_DO + ds * C::QB, C::BN * 128));
          const uint32_t t_s = tmem + C::T_S(t & 1);
          const uint32_t first = t > 0 ? 1u : 0u;
          // dK += dS^T Q first: it releases the Q stage
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k)
            mma_ts_w(t_dk, t_s + 16 * k + 8, q_mn + kstep_off(k), id_out, k > 0 ? 1u : first);
          mma_commit_w(q_empty + s);
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k)
            mma_ts_w(t_dv, t_s + 16 * k, do_mn + kstep_off(k), id_out, k > 0 ? 1u : first);
          mma_commit_w(do_empty + ds);
        }
      }
      if (ok) mma_commit_w(acc_done);
      mma_commit_w(drain);
      mbar_wait_bounded(drain, 0, prm.status, 100000000ull);
    }
  } else {
    // ---------------- elementwise warps: thread = key row -----------------
    constexpr int NC = kBwdCols;
    const int row = 32 * (warp & 3) + lane;
    const int slice = warp >> 2;  // query columns [NC*slice, NC*slice + NC)
    const int j = j0 + row;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sc2 = prm.scale * kLog2e;
    const f2 sc2_2 = {sc2, sc2};
    // dQ^T partial of a finished tile (TMEM lane = feature index, column =
    // query) into the fp32 accumulator
    auto drain_dq = [&](int t, uint32_t (&dq)[NC]) -> bool {
      if (!warp_wait(dq_full, t & 1, abort_st, prm.status)) return false;
      tc_fence_after();
      tmem_ld16(tmem + lane_off + C::T_DQ + NC * slice, dq);
      tc_fence_before();
      mbar_arrive(dq_empty);
      return true;
    };
    // dQ^T partial of tile u into staging buffer u % SBUF as [BN][SF] fp32
    // rows (query column c, feature f at c * SF + f; a warp's lanes write
    // consecutive words) once the reduce-add that last used the buffer has
    // read it, then the arrival that hands it to the reduce warp.  Features
    // from SF on (d = 128) go to the accumulator directly.
    auto stage_dq = [&](int u, const uint32_t (&dq)[NC]) -> bool {
      const int b = u % C::SBUF;
      if (u >= C::SBUF &&
          !warp_wait(stg_free + b, ((u / C::SBUF) - 1) & 1, abort_st, prm.status))
        return false;
      // M = 64 accumulator at d = 64: rows 16w' + x (w' = warp & 3, x < 16)
      // live in lanes 32w' + x; the upper 16 lanes of each warp hold nothing
      const int f = D == 128 ? row : 16 * (warp & 3) + lane;
      if (D == 128 && f >= C::SF) {
        const int qa = qstart + rotated(u, rot, T) * C::BN + NC * slice;
        red_columns<D, NC>(prm.acc + ((size_t)bh * N + qa) * D + f, dq, N - qa);
      } else if (D == 128 || lane < 16) {
        const uint32_t base = sb + C::OFF_STG + b * C::STGB + (uint32_t)(NC * slice * C::SF + f) * 4u;
#pragma unroll
        for (int i = 0; i < NC; ++i) st_shared_u32(base + (uint32_t)(i * C::SF * 4), dq[i]);
      }
      fence_async_smem();
      mbar_arrive(stg_full + b);
      return true;
    };
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::STAGES;
      const int q0 = qstart + rotated(t, rot, T) * C::BN;
      if (!warp_wait(s_full + (t & 1), (t >> 1) & 1, abort_st, prm.status) ||
          !warp_wait(dp_full, t & 1, abort_st, prm.status)) {
        ok = false;
        break;
      }
      if (!warp_wait(q_full + s, (t / C::STAGES) & 1, abort_st, prm.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[NC], dpr[NC];
      const uint32_t tl = tmem + lane_off + NC * slice;
      const uint32_t ts = tl + C::T_S(t & 1);
      tmem_ld16x2(ts, tl + C::T_DP, sr, dpr);
      // the loads above have completed: the dP^T columns are free
      tc_fence_before();
      mbar_arrive(dp_read);
      const float4* sc4 = reinterpret_cast<const float4*>(scal + s * 2 * C::BN + NC * slice);
      const int qa = q0 + NC * slice;
      const bool need_mask = (qa + NC > N) || (j0 + C::BM > N) || (prm.causal && qa < j0 + C::BM);
      uint32_t pw[NC / 2], dsw[NC / 2];
      auto body = [&](auto masked) {
#pragma unroll
        for (int c4 = 0; c4 < NC / 4; ++c4) {  // 4 query columns per step
          // negated row scalars of the 4 queries: -LSE log2 e, -D
          const float4 L = sc4[c4], Dd = sc4[C::BN / 4 + c4];
          const f2 nl[2] = {{L.x, L.y}, {L.z, L.w}}, nd[2] = {{Dd.x, Dd.y}, {Dd.z, Dd.w}};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // query columns cc, cc + 1: one packed pair
            const int cc = 4 * c4 + 2 * hh;
            const f2 x = fma2({__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])}, sc2_2, nl[hh]);
            f2 p = {ex2_approx(x.x), ex2_approx(x.y)};
            if (decltype(masked)::value) {
              const int q = qa + cc;
              p.x = (q < N && j < N && (!prm.causal || q >= j)) ? p.x : 0.f;
              p.y = (q + 1 < N && j < N && (!prm.causal || q + 1 >= j)) ? p.y : 0.f;
            }
            const f2 ds = mul2(p, add2({__uint_as_float(dpr[cc]), __uint_as_float(dpr[cc + 1])}, nd[hh]));
            pw[cc >> 1] = pack_bf16(p.x, p.y);
            dsw[cc >> 1] = pack_bf16(ds.x, ds.y);
          }
        }
      };
      if (need_mask)
        body(std::true_type{});
      else
        body(std::false_type{});
      // A operands of the dV / dK MMAs: bf16 pairs (low half = even query),
      // P^T in the first 8 and dS^T in the last 8 of the 16 S^T columns this
      // thread read
      tmem_st8x2(ts, pw, ts + 8, dsw);
      // the previous tile's dQ^T MMAs read the dS^T tile below: drain their
      // result first
      uint32_t dq[NC];
      if (t >= 1 && !drain_dq(t - 1, dq)) { ok = false; break; }
      // dS^T also goes to shared memory as the dQ^T B operand.  This
      // thread's columns are 16-byte chunks [NC*slice/8, +NC/8) of its row.
#pragma unroll
      for (int q = 0; q < NC / 8; ++q) {
        const uint32_t chunk = (NC / 8) * slice + q;
        st_shared_v4(sb + C::OFF_DS + sw128_offset(row, chunk), dsw[4 * q], dsw[4 * q + 1],
                     dsw[4 * q + 2], dsw[4 * q + 3]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(ds_full);
      if (t >= 1 && !stage_dq(t - 1, dq)) { ok = false; break; }
    }
    if (ok && T >= 1) {
      uint32_t dq[NC];
      ok = drain_dq(T - 1, dq) && stage_dq(T - 1, dq);
    }
    // ---- epilogue: dK (scaled), dV; each thread D/4 features ----
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = warp_wait(acc_done, 0, abort_st, prm.status);
    tc_fence_after();
    if (ok) {
      constexpr int PART = D / 4;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = which == 0 ? prm.dk : prm.dv;
        const float mul = which == 0 ? prm.scale : 1.f;
        const uint32_t tcol = (which == 0 ? C::T_DK : C::T_DV) + PART * slice;
        uint4* op = reinterpret_cast<uint4*>(out + ((size_t)bh * N + j) * D + PART * slice);
#pragma unroll
        for (int cc = 0; cc < PART; cc += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_off + tcol + cc, v);
          if (j < N) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16(__uint_as_float(v[8 * q + 2 * e]) * mul,
                                  __uint_as_float(v[8 * q + 2 * e + 1]) * mul);
              op[cc / 8 + q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// D_i = dO_i . O_i (fp32) for every row, and the row's fp32 dQ accumulator
// cleared: D/8 threads per row, 8 bf16 elements each.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_prep(const uint4* __restrict__ o, const uint4* __restrict__ dO, float* __restrict__ Dout,
             float4* __restrict__ acc, size_t rows) {
  constexpr int G = D / 8;  // threads per row (a power of two dividing 32)
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t r = t / G;
  const int c = (int)(t % G);
  float s = 0.f;
  if (r < rows) {
    const uint4 ov = o[r * G + c], dv = dO[r * G + c];
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 of = __bfloat1622float2(o2[e]);
      const float2 df = __bfloat1622float2(d2[e]);
      s = fmaf(of.x, df.x, fmaf(of.y, df.y, s));
    }
    acc[(r * G + c) * 2] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[(r * G + c) * 2 + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (r < rows && c == 0) Dout[r] = s;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int D>
cudaError_t forward_d(const Problem& p, const void* q, const void* k, const void* v, void* o,
                      float* lse, const Workspace& ws, LaunchLog& log) {
  using C = Fwd<D>;
  CUtensorMap mQ, mK, mV;
  if (!make_map(&mQ, q, p, C::BM) || !make_map(&mK, k, p, C::BN) || !make_map(&mV, v, p, C::BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_row_pass<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::SMEM);
  if (e != cudaSuccess) return e;
  FwdParams fp;
  fp.o = static_cast<__nv_bfloat16*>(o);
  fp.lse = lse;
  fp.status = ws.status;
  fp.wait_ns = wait_limit_ns();
  fp.N = p.N;
  fp.BH = p.BH();
  fp.G = cta_group_heads(p.BH(), (p.N + C::BM - 1) / C::BM, sm_count());
  fp.causal = p.causal;
  fp.scale = p.scale;
  dim3 grid((unsigned)(((p.N + C::BM - 1) / C::BM) * p.BH()));
  fwd_row_pass<D><<<grid, kFwdThreads, C::SMEM, log.stream>>>(mQ, mK, mV, fp);
  e = cudaGetLastError();
  log.mark();
  return e;
}

template <int D>
cudaError_t backward_d(const Problem& p, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* dO, void* dq, void* dk,
                       void* dv, const Workspace& ws, LaunchLog& log) {
  using C = Bwd<D>;
  const size_t rows = p.rows();
  const size_t threads = rows * (D / 8);
  bwd_prep<D><<<(unsigned)((threads + 255) / 256), 256, 0, log.stream>>>(
      static_cast<const uint4*>(o), static_cast<const uint4*>(dO), ws.D,
      reinterpret_cast<float4*>(ws.acc), rows);
  cudaError_t e = cudaGetLastError();
  log.mark();
  if (e != cudaSuccess) return e;

  CUtensorMap mK, mV, mQ, mDO;
  if (!make_map(&mK, k, p, C::BM) || !make_map(&mV, v, p, C::BM) ||
      !make_map(&mQ, q, p, C::BN) || !make_map(&mDO, dO, p, C::BN))
    return cudaErrorInvalidValue;
  CUtensorMap mAcc;
  if (!make_acc_map(&mAcc, ws.acc, p, C::SF, C::BN)) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(bwd_col_pass<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::SMEM);
  if (e != cudaSuccess) return e;
  BwdParams bp;
  bp.acc = ws.acc;
  bp.lse = lse;
  bp.Dv = ws.D;
  bp.dk = static_cast<__nv_bfloat16*>(dk);
  bp.dv = static_cast<__nv_bfloat16*>(dv);
  bp.status = ws.status;
  bp.wait_ns = wait_limit_ns();
  bp.N = p.N;
  bp.BH = p.BH();
  bp.G = cta_group_heads(p.BH(), (p.N + C::BM - 1) / C::BM, sm_count());
  bp.causal = p.causal;
  bp.scale = p.scale;
  dim3 grid((unsigned)(((p.N + C::BM - 1) / C::BM) * p.BH()));
  bwd_col_pass<D><<<grid, kBwdThreads, C::SMEM, log.stream>>>(mK, mV, mQ, mDO, mAcc, bp);
  e = cudaGetLastError();
  log.mark();
  if (e != cudaSuccess) return e;
  return launch_acc_to_bf16(ws.acc, dq, p.elems(), p.scale, log);
}

}  // namespace

cudaError_t tc_forward(const Problem& p, const void* q, const void* k, const void* v, void* o,
                       float* lse, const Workspace& ws, LaunchLog& log) {
  if (p.d == 128) return forward_d<128>(p, q, k, v, o, lse, ws, log);
  return forward_d<64>(p, q, k, v, o, lse, ws, log);
}

cudaError_t tc_backward(const Problem& p, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dO, void* dq, void* dk,
                        void* dv, const Workspace& ws, LaunchLog& log) {
  if (p.d == 128) return backward_d<128>(p, q, k, v, o, lse, dO, dq, dk, dv, ws, log);
  return backward_d<64>(p, q, k, v, o, lse, dO, dq, dk, dv, ws, log);
}

}  // namespace fbob

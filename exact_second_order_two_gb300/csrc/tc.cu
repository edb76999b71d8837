// Tensor-core (tcgen05 / TMEM / TMA) kernels for sm_103a: the two-pass
// exact backward-over-backward of softmax attention.
//
// FlashBoB ("FlashBoB: I/O-Efficient Exact Backward-over-Backward for
// Softmax Attention", Abstract) observes that two row-wise scalars determine
// every BoB output through affine maps.  With c the scale,
//   S = c Q K^T, P = exp(S - LSE), dP = dO V^T, D_i = dO_i . O_i,
//   G = c (Q gK^T + gQ K^T)   (cotangent of dS),   H = dO gV^T,
//   r_i = sum_j P_ij G_ij,
//   graddO = P gV + (P*G) V - r O,      sigma_i = dO_i . graddO_i,
//   dS  = P*(dP - D),  gdP = P*(G - r),  gS = P*(H + (G - r)*(dP - D) - sigma),
//   gradQ = c (gS K + dS gK),  gradK = c (gS^T Q + dS^T gQ),  gradV = gdP^T dO.
// (Derived for this library; the pages print no equations.)  The schedule:
//
//   pass 1 (row-stationary, 128 query rows per CTA, 64-key tiles streamed):
//     S and G on the tensor cores into one of two TMEM buffers; P and P*G in
//     registers, written back as bf16 into the S / G columns just read;
//     W += P gV + (P*G) V into TMEM with those as A operands (at d = 64 two
//     MMA warps take alternate tiles, each into its own W); epilogue r, D,
//     sigma, graddO = W - r O.
//   pass 2 (key-stationary, 128 key rows per CTA, 64-query tiles streamed):
//     S^T, dP^T, G^T, H^T into TMEM; dS^T, gdP^T, gS^T in registers, written
//     back as bf16 into TMEM (A operands of gradV += gdP^T dO and gradK +=
//     gS^T Q + dS^T gQ) and dS^T, gS^T also into shared memory (B operands
//     of the gradQ^T partial K^T gS^T + gK^T dS^T, reduced into an fp32
//     accumulator with red.global.add).  At d = 64 TMEM holds two S^T / G^T
//     buffers, so the next tile's scores run during this tile's
//     elementwise phase.
//   convert: fp32 gradQ accumulator -> bf16.
//
// No N x N tensor ever leaves TMEM / shared memory / registers.  Warp roles
// per CTA: elementwise warps (thread = TMEM lane), TMA producer warps (one
// issuing thread each), a warp that allocates TMEM and issues tcgen05.mma
// with all its lanes (elect.sync picks the issuing lane), and in pass 1 a
// helper warp that folds the MMA warp's waits.  In pass 2 the control warps
// form one warpgroup (with an idle fourth warp) that hands registers to the
// elementwise warpgroups (setmaxnreg).  Every wait is bounded (see
// common.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "sm103.cuh"
#include "tc_common.cuh"

namespace fbob {

using namespace sm103;
using namespace tc;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Waits for a tile's operands (P from the elementwise warps, V and the K two
// tiles ahead from TMA) and signals them to the MMA warp as one barrier: an
// mbarrier test by the MMA warp costs hundreds of cycles while the tensor
// pipe streams its operands, and the pipe holds only a few MMAs of work to
// cover it, so one wait per tile leaves it idle far less than three.
constexpr int kHelperWarp = 10;
// At d = 64 a second MMA warp takes the odd tiles (Row::TWO_MMA).
constexpr int kMmaWarp2 = 11;
constexpr int kConsumers = kConsumerWarps * 32;
__device__ __forceinline__ void consumer_sync() { named_sync<kConsumers>(1); }

// Two [rows][D] tiles A and B interleaved per 64-feature half (A_h, B_h,
// A_h+1, ...): each half holds 2*rows rows, so one N = 2*rows MMA sees A and B
// stacked; maps with one feature half per box.  B ([K|gK] or [Q|gQ] with gK /
// gQ as B) is skipped when its cotangent is absent: the MMAs then read only
// the first `rows` rows of each half.
template <int D>
__device__ __forceinline__ void load_pair_opt(uint8_t* dst, const CUtensorMap* mapA,
                                              const CUtensorMap* mapB, bool with_b, uint64_t* bar,
                                              int rows, int row, int bh) {
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    tma_load_4d(dst + h * 2 * rows * 128, mapA, bar, 0, row, h, bh);
    if (with_b) tma_load_4d(dst + h * 2 * rows * 128 + rows * 128, mapB, bar, 0, row, h, bh);
  }
}

// ===========================================================================
// Pass 1: row-stationary.
// ===========================================================================
template <int D>
struct Row {
  static constexpr int BM = 128, BN = 64;
  // Two decoupled rings: [K|gK] (read by the S/G MMAs, freed early) and
  // [V|gV] (read by the W MMAs of the same tile, freed one tile later).
  static constexpr int STAGES = D == 128 ? 3 : 4;    // [K|gK] ring
  static constexpr int VSTAGES = D == 128 ? 2 : 3;   // [V|gV] ring
  static constexpr uint32_t QB = BM * D * 2;        // Q or gQ tile
  static constexpr uint32_t KB = BN * D * 2;        // one streamed key-side tile
  // [K|gK] stage: interleaved per 64-feature half (one N=128 MMA sees K and
  // gK stacked); [V|gV] stage: V then gV, one box each
  static constexpr uint32_t SB = 2 * KB;
  static constexpr uint32_t OFF_Q = 0, OFF_GQ = QB, OFF_KG = 2 * QB;
  static constexpr uint32_t OFF_V = OFF_KG + STAGES * SB;
  static constexpr uint32_t OFF_PART = OFF_V + VSTAGES * SB;  // epilogue sums [4][128]
  static constexpr uint32_t OFF_MISC = OFF_PART + 4 * 128 * 4;  // barriers, slot, flag
  static constexpr uint32_t MISC = 512;
  static constexpr uint32_t SMEM = OFF_MISC + MISC;
  static_assert(SMEM <= 232448, "pass 1 shared memory budget");
  // TMEM columns: two [S | G] buffers (64 + 64 columns), W, and the
  // stationary bf16 Q and gQ as MMA A operands (D/2 columns each).  The
  // elementwise warps write bf16 P and P*G back into the first 16 of the 32 S
  // and G columns each of them read: the A operands of the W MMAs.  While
  // they work on one buffer, the S/G MMAs of the next tile fill the other.
  static constexpr uint32_t T_W = 256, TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t T_S(int b) { return 128u * b; }
  __host__ __device__ static constexpr uint32_t T_G(int b) { return 128u * b + 64u; }
  // bf16 P (or P*G) of keys [16k, 16k + 16): column offset in the S (G) block
  __host__ __device__ static constexpr uint32_t p_col(int k) { return 32u * (k >> 1) + 8u * (k & 1); }
  static constexpr uint32_t T_QA = 256 + D, T_GQA = 256 + D + D / 2;
  // d = 64: two MMA warps, one per tile parity, each with its own W
  // accumulator (summed in the epilogue).  Every MMA warp stalls for a few
  // hundred cycles after each tile's burst of MMAs; with two, one warp's
  // stall is covered by the other's burst.  Buffer t % 2 and ready[t % 2]
  // already belong to one parity, so the warps share nothing else that
  // needs ordering.  At d = 128 TMEM has no room for a second W.
  static constexpr bool TWO_MMA = D == 64;
  static constexpr uint32_t T_W2 = T_GQA + D / 2;
  static_assert(T_GQA + D / 2 + (TWO_MMA ? D : 0) <= TMEM_COLS, "pass 1 TMEM budget");
  static constexpr int THREADS = (TWO_MMA ? 12 : 11) * 32;
};

struct RowParams {
  const float* lse;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  __nv_bfloat16* graddo;
  float* r_out;
  float* sigma_out;
  float* D_out;
  float* acc_zero;  // fp32 gradQ accumulator rows to clear (may be null)
  int* status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int N, causal;
  int BH, G;  // batch * heads, heads per CTA group (cta_coord)
  float scale;
  // which cotangents are present (an absent one is zero: its loads and MMAs
  // are skipped); at least one is
  int has_gq, has_gk, has_gv;
};

template <int D, bool ALL>
__global__ void __launch_bounds__(Row<D>::THREADS, 1)
    bob_row_pass(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mGQ,
                 const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mGK,
                 const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mGV,
                 RowParams prm) {
  using C = Row<D>;
  // cotangents present: ALL (every one) is the compiled fast path; otherwise
  // the flags decide at run time
  const bool has_gq = ALL || prm.has_gq != 0, has_gk = ALL || prm.has_gk != 0,
             has_gv = ALL || prm.has_gv != 0;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report_status(prm.status, FBOB_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  uint64_t* q_full = bars + 0;
  uint64_t* kg_full = bars + 1;                  // [STAGES]
  uint64_t* kg_empty = kg_full + C::STAGES;      // [STAGES]
  uint64_t* v_full = kg_empty + C::STAGES;       // [VSTAGES]
  uint64_t* v_empty = v_full + C::VSTAGES;       // [VSTAGES]
  uint64_t* sg_full = v_empty + C::VSTAGES;      // [2]: S, G of a buffer in TMEM
  uint64_t* p_full = sg_full + 2;                // [2]: bf16 P, P*G of a buffer in TMEM
  uint64_t* w_done = p_full + 2;
  uint64_t* q_tmem = w_done + 2;                  // Q, gQ copied into TMEM
  uint64_t* drain = w_done + 1;
  uint64_t* ready = q_tmem + 1;                   // [2]: P(t), V(t), K(t+2) all in place
  uint64_t* drain2 = ready + 2;                   // TWO_MMA: the second MMA warp's drain
  static_assert((1 + 2 * C::STAGES + 2 * C::VSTAGES + 10) * 8 <= 256,
                "barriers end below the TMEM slot");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 256);
  Abort* abort_st = reinterpret_cast<Abort*>(smem + C::OFF_MISC + 264);
  float* part = reinterpret_cast<float*>(smem + C::OFF_PART);

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
  // Every CTA walks the key tiles from the first: the CTAs of one head then
  // read the same K / V tiles at about the same time and share them in L2.
  // (Pass 2 starts each CTA at a different query tile instead; there that
  // measured faster at long N, here slower.)
  const int rot = 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kg_full + s, 1);
      mbar_init(kg_empty + s, 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sg_full + b, 1);
      mbar_init(p_full + b, kConsumers);
    }
    mbar_init(w_done, C::TWO_MMA ? 2 : 1);
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    mbar_init(q_tmem, kConsumers);
    mbar_init(ready, 1);
    mbar_init(ready + 1, 1);
    abort_st->flag = 0;
    abort_st->limit_ns = prm.wait_ns;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      mbar_arrive_expect_tx(q_full, (has_gq ? 2 : 1) * C::QB);
      load_tile(smem + C::OFF_Q, &mQ, q_full, i0, bh);
      if (has_gq) load_tile(smem + C::OFF_GQ, &mGQ, q_full, i0, bh);
      // [K|gK] runs one tile ahead of [V|gV]: the S/G MMAs of tile t+1 need
      // only K/gK, which are released as soon as the S/G MMAs of tile t-1 end
      int kg_issued = 0, v_issued = 0;
      auto load_kg = [&](int t) -> bool {
        const int s = t % C::STAGES;
        if (t >= C::STAGES &&
            !wait_bar(kg_empty + s, ((t / C::STAGES) - 1) & 1, abort_st, prm.status))
          return false;
        uint8_t* st = smem + C::OFF_KG + s * C::SB;
        mbar_arrive_expect_tx(kg_full + s, has_gk ? C::SB : C::SB / 2);
        const int kt = rotated(t, rot, T) * C::BN;
        load_pair_opt<D>(st, &mK, &mGK, has_gk, kg_full + s, C::BN, kt, bh);
        ++kg_issued;
        return true;
      };
      auto load_v = [&](int t) -> bool {
        const int s = t % C::VSTAGES;
        if (t >= C::VSTAGES &&
            !wait_bar(v_empty + s, ((t / C::VSTAGES) - 1) & 1, abort_st, prm.status))
          return false;
        uint8_t* st = smem + C::OFF_V + s * C::SB;
        mbar_arrive_expect_tx(v_full + s, has_gv ? C::SB : C::KB);
        const int kt = rotated(t, rot, T) * C::BN;
        load_tile(st, &mV, v_full + s, kt, bh);
        if (has_gv) load_tile(st + C::KB, &mGV, v_full + s, kt, bh);
        ++v_issued;
        return true;
      };
      bool pok = load_kg(0);
      for (int t = 0; pok && t < T; ++t) {
        if (t + 1 < T && !load_kg(t + 1)) break;
        if (!load_v(t)) break;
      }
      // every load this thread issued has landed before the CTA exits (after
      // an abort some were never awaited); each phase waited for is the last
      // of its barrier, so on the normal path these return at once
      mbar_wait_bounded(q_full, 0, prm.status, 100000000ull);
      for (int t = max(0, kg_issued - C::STAGES); t < kg_issued; ++t)
        mbar_wait_bounded(kg_full + (t % C::STAGES), (t / C::STAGES) & 1, prm.status,
                          100000000ull);
      for (int t = max(0, v_issued - C::VSTAGES); t < v_issued; ++t)
        mbar_wait_bounded(v_full + (t % C::VSTAGES), (t / C::VSTAGES) & 1, prm.status,
                          100000000ull);
    }
  } else if (warp == kMmaWarp || (C::TWO_MMA && warp == kMmaWarp2)) {
    {  // the whole warp: warp-uniform waits, elect.sync issues each MMA
      // tiles par, par + step, ...: all of them, or (TWO_MMA) one parity
      const int par = warp == kMmaWarp ? 0 : 1, step = C::TWO_MMA ? 2 : 1;
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);    // gQ K^T: M=128 N=64
      constexpr uint32_t id_sg = idesc_bf16(128, 128, false, false);  // Q [K;gK]^T: N=128
      constexpr uint32_t id_w = idesc_bf16(128, D, false, true);    // W: N=D, B MN-major
      bool ok = warp_wait(q_tmem, 0, abort_st, prm.status);
      const uint32_t tw = tmem + (par == 0 ? C::T_W : C::T_W2), tq = tmem + C::T_QA,
                     tgq = tmem + C::T_GQA;
      // S and G of tile t into buffer t & 1
      auto wait_sg = [&](int t) -> bool {
        return warp_wait(kg_full + t % C::STAGES, (t / C::STAGES) & 1, abort_st, prm.status);
      };
      auto issue_sg = [&](int t) {
        const int s = t % C::STAGES, b = t & 1;
        // [K;gK] per half, 2*BN rows
        const uint32_t kgk_lo = opaque(lo_kmajor(sb + C::OFF_KG + s * C::SB));
        const uint32_t ts = tmem + C::T_S(b), tg = tmem + C::T_G(b);
        // [S | Q gK^T] = Q [K; gK]^T in one N=128 MMA chain (T_G = T_S + 64),
        // A = Q from TMEM; S = Q K^T alone (N=64) without gK
        const uint32_t id_first = has_gk ? id_sg : id_s;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ts_w(ts, tq + 8 * k, kgk_lo + kslice_off(2 * C::BN, k), id_first, k > 0 ? 1u : 0u);
        // G += gQ K^T (the first BN rows of each [K;gK] half are K), A = gQ from TMEM
        if (has_gq) {
          const uint32_t g0 = has_gk ? 1u : 0u;  // without gK this starts G
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ts_w(tg, tgq + 8 * k, kgk_lo + kslice_off(2 * C::BN, k), id_s, k > 0 ? 1u : g0);
        }
        mma_commit_w(sg_full + b);
        mma_commit_w(kg_empty + s);
      };
      // W += P gV + (P*G) V for tile t: A operands (bf16 P, P*G) from TMEM
      auto issue_w = [&](int t) {
        const int s = t % C::VSTAGES, b = t & 1;
        const uint32_t st = sb + C::OFF_V + s * C::SB;
        const uint32_t v_lo = opaque(lo_mnmajor(st, C::BN * 128)),
                       gv_lo = opaque(lo_mnmajor(st + C::KB, C::BN * 128));
        const uint32_t tp = tmem + C::T_S(b), tpg = tmem + C::T_G(b);
        const uint32_t first = t >= step ? 1u : 0u;  // this warp's first tile starts its W
        // without gV only (P*G) V; without gQ and gK, G = 0 and only P gV
        const bool use_gv = has_gv, use_g = has_gq || has_gk;
#pragma unroll
        for (int k = 0; k < C::BN / 16; ++k) {  // contraction over the 64 keys
          const uint32_t acc = k > 0 ? 1u : first;
          if (use_gv) mma_ts_w(tw, tp + C::p_col(k), gv_lo + kstep_off(k), id_w, acc);
          if (use_g) mma_ts_w(tw, tpg + C::p_col(k), v_lo + kstep_off(k), id_w, use_gv ? 1u : acc);
        }
        mma_commit_w(v_empty + s);
      };
      // Buffer b holds tile t until the W MMAs of t have read its P: the S/G
      // MMAs of tile t + 2 are issued after them, and MMAs from one thread
      // run in issue order.
      for (int t = par; ok && t < 2 && t < T; t += step) {
        ok = wait_sg(t);
        if (ok) {
          tc_fence_after();
          issue_sg(t);
        }
      }
      // One wait per tile, on the helper warp's combined barrier.  Tile t's
      // phase of ready[t & 1] cannot be signalled before the MMA warp has
      // passed its wait for tile t - 2: the helper first needs P(t), which
      // needs S(t), issued only after that wait.
      for (int t = par; ok && t < T; t += step) {
        if (!warp_wait(ready + (t & 1), (t >> 1) & 1, abort_st, prm.status)) { ok = false; break; }
        tc_fence_after();
        issue_w(t);
        if (t + 2 < T) issue_sg(t + 2);
      }
      if (ok) mma_commit_w(w_done);
      // every MMA this thread issued has completed before TMEM is released
      uint64_t* dr = par == 0 ? drain : drain2;
      mma_commit_w(dr);
      mbar_wait_bounded(dr, 0, prm.status, 100000000ull);
    }
  } else if (warp == kHelperWarp) {
    if (lane == 0) {
      for (int t = 0; t < T; ++t) {
        if (!wait_bar(p_full + (t & 1), (t >> 1) & 1, abort_st, prm.status) ||
            !wait_bar(v_full + t % C::VSTAGES, (t / C::VSTAGES) & 1, abort_st, prm.status) ||
            (t + 2 < T && !wait_bar(kg_full + (t + 2) % C::STAGES, ((t + 2) / C::STAGES) & 1,
                                    abort_st, prm.status)))
          break;
        mbar_arrive(ready + (t & 1));
      }
    }
  } else {
    // ---------------- elementwise warps: thread = query row --------------
    const int row = 32 * (warp & 3) + lane;
    const int half = warp >> 2;  // columns [32*half, 32*half + 32) of a tile
    const int i = i0 + row;
    const bool row_ok = i < N;
    const size_t srow = (size_t)bh * N + (row_ok ? i : 0);
    const float lse2 = row_ok ? prm.lse[srow] * kLog2e : 0.f;
    const float sc2 = prm.scale * kLog2e;
    const f2 sc2_2 = {sc2, sc2}, nlse2 = {-lse2, -lse2}, scale_2 = {prm.scale, prm.scale};
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const bool has_g = has_gq || has_gk;
    f2 r_acc = {0.f, 0.f};  // even and odd keys summed apart
    bool ok = warp_wait(q_full, 0, abort_st, prm.status);
    if (ok) {
      // stationary Q and gQ rows -> TMEM (bf16 pairs, lower half = even
      // feature): one 64-feature half-row per thread and tensor
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const int h = D == 128 ? half : 0;          // feature half copied
        if (D == 64 && which != half) continue;     // d = 64: half 0 -> Q, half 1 -> gQ
        if (which == 1 && !has_gq) continue;    // no gQ: its TMEM copy is never read
        const uint32_t src = sb + (which == 0 ? C::OFF_Q : C::OFF_GQ) + h * C::BM * 128 + row * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(
              smem + (src - sb) + ((c ^ (row & 7)) << 4));
          w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
        const uint32_t dst = tmem + lane_off + (which == 0 ? C::T_QA : C::T_GQA) + 32 * h;
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) { lo[c] = w[c]; hi[c] = w[16 + c]; }
        tmem_st16(dst, lo);
        tmem_st16(dst + 16, hi);
      }
      tc_fence_before();
      mbar_arrive(q_tmem);
    }
    for (int t = 0; ok && t < T; ++t) {
      const int b = t & 1;
      // buffer b last held tile t - 2, whose W MMAs completed before the S/G
      // MMAs of tile t (issued after them) signalled sg_full
      if (!warp_wait(sg_full + b, (t >> 1) & 1, abort_st, prm.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[32], gr[32];
      const uint32_t ts = tmem + lane_off + C::T_S(b) + 32 * half,
                     tg = tmem + lane_off + C::T_G(b) + 32 * half;
      tmem_ld32x2(ts, tg, sr, gr);
      const int j0 = rotated(t, rot, T) * C::BN + 32 * half;
      const bool need_mask = !row_ok || (j0 + 32 > N) || (prm.causal && j0 + 31 > i0);
      uint32_t pw[16], pgw[16];
      auto body = [&](auto masked) {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {  // keys c, c + 1: one packed pair
          const f2 x = fma2({__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, sc2_2, nlse2);
          f2 p = {ex2_approx(x.x), ex2_approx(x.y)};
          if (decltype(masked)::value) {
            const int jj = j0 + c;
            p.x = (row_ok && jj < N && (!prm.causal || jj <= i)) ? p.x : 0.f;
            p.y = (row_ok && jj + 1 < N && (!prm.causal || jj + 1 <= i)) ? p.y : 0.f;
          }
          // G is zero (and its TMEM columns unwritten) without gQ and gK
          const f2 pg = has_g ? mul2(p, mul2({__uint_as_float(gr[c]), __uint_as_float(gr[c + 1])},
                                             scale_2))
                              : f2{0.f, 0.f};
          r_acc = add2(r_acc, pg);
          pw[c >> 1] = pack_bf16(p.x, p.y);
          pgw[c >> 1] = pack_bf16(pg.x, pg.y);
        }
      };
      if (need_mask)
        body(std::true_type{});
      else
        body(std::false_type{});
      // bf16 P and P*G of this thread's 32 keys into the first 16 of the S and
      // G columns it just read (keys 32*half + 2c, + 1 in column c)
      tmem_st16(ts, pw);
      tmem_st16(tg, pgw);
      tc_fence_before();
      mbar_arrive(p_full + b);
    }
    // ---- epilogue: r, D, sigma, graddO = W - r O ----
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = warp_wait(w_done, 0, abort_st, prm.status);
    tc_fence_after();
    part[half * 128 + row] = r_acc.x + r_acc.y;
    consumer_sync();
    const float r = part[row] + part[128 + row];
    float dd = 0.f, sg = 0.f;
    if (ok) {
      constexpr int HALF = D / 2;
      const size_t obase = srow * D + HALF * half;
#pragma unroll
      for (int cc = 0; cc < HALF; cc += 32) {
        uint32_t wr[32];
        tmem_ld32(tmem + lane_off + C::T_W + HALF * half + cc, wr);
        if (C::TWO_MMA && T >= 2) {  // the odd tiles' share, from the second MMA warp
          uint32_t w2[32];
          tmem_ld32(tmem + lane_off + C::T_W2 + HALF * half + cc, w2);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            wr[e] = __float_as_uint(__uint_as_float(wr[e]) + __uint_as_float(w2[e]));
        }
        if (row_ok) {
          const uint4* op = reinterpret_cast<const uint4*>(prm.o + obase + cc);
          const uint4* dp = reinterpret_cast<const uint4*>(prm.dO + obase + cc);
          uint4* gp = reinterpret_cast<uint4*>(prm.graddo + obase + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 ov = op[v], dv = dp[v];
            const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
            const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
            uint32_t outw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 of = __bfloat1622float2(o2[e]);
              const float2 df = __bfloat1622float2(d2[e]);
              const float w0 = __uint_as_float(wr[8 * v + 2 * e]) - r * of.x;
              const float w1 = __uint_as_float(wr[8 * v + 2 * e + 1]) - r * of.y;
              dd = fmaf(df.x, of.x, fmaf(df.y, of.y, dd));
              sg = fmaf(df.x, w0, fmaf(df.y, w1, sg));
              outw[e] = pack_bf16(w0, w1);
            }
            gp[v] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
          }
        }
      }
    }
    tc_fence_before();
    consumer_sync();  // everyone has read `part` for r
    part[half * 128 + row] = dd;
    part[256 + half * 128 + row] = sg;
    consumer_sync();
    if (ok && half == 0 && row_ok) {
      prm.r_out[srow] = r;
      prm.D_out[srow] = part[row] + part[128 + row];
      prm.sigma_out[srow] = part[256 + row] + part[384 + row];
    }
    // clear this row's fp32 gradQ accumulator for the key-stationary pass
    if (prm.acc_zero && row_ok) {
      float4* a = reinterpret_cast<float4*>(prm.acc_zero + srow * D + (D / 2) * half);
#pragma unroll
      for (int v = 0; v < D / 8; ++v) a[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ===========================================================================
// Pass 2: key-stationary.
// ===========================================================================
template <int D>
struct Col {
  static constexpr int BM = 128, BN = 64;
  // At d = 64 two score buffers (SG2 below) put the next tile's S^T / G^T
  // ahead of this tile's gradK / gradV, so both rings hold three tiles.
  static constexpr int STAGES = D == 128 ? 1 : 3;    // [Q|gQ] (+ row scalars) ring
  static constexpr int DSTAGES = D == 128 ? 2 : 3;   // dO ring
  static constexpr uint32_t KB = BM * D * 2;     // stationary K, gK, V, gV tile
  static constexpr uint32_t QB = BN * D * 2;     // streamed Q, gQ, dO tile
  static constexpr uint32_t XB = BM * BN * 2;    // dS^T / gS^T tile (gradQ^T B operands)
  static constexpr uint32_t OFF_K = 0, OFF_GK = KB, OFF_V = 2 * KB, OFF_GV = 3 * KB;
  static constexpr uint32_t OFF_QG = 4 * KB;                     // [STAGES][2 * QB]
  static constexpr uint32_t OFF_DO = OFF_QG + STAGES * 2 * QB;   // [DSTAGES][QB]
  static constexpr uint32_t OFF_DS = OFF_DO + DSTAGES * QB, OFF_GS = OFF_DS + XB;
  // row scalars: one buffer more than [Q|gQ] stages, so the producer can
  // write a tile's scalars before its stage is free
  static constexpr int SCSTAGES = STAGES + 1;
  static constexpr uint32_t OFF_SC = OFF_GS + XB;          // [SCSTAGES][4][BN] fp32
  static constexpr uint32_t OFF_MISC = OFF_SC + SCSTAGES * 4 * BN * 4;
  static constexpr uint32_t MISC = 512;
  static constexpr uint32_t SMEM = OFF_MISC + MISC;
  static_assert(SMEM <= 232448, "pass 2 shared memory budget");
  // TMEM columns
  // S^T and G^T adjacent: one N=128 MMA chain writes [S^T | K gQ^T].  Once
  // the elementwise warps have read a tile's four score blocks, the next
  // tile's dP^T and H^T are computed into their columns while the
  // elementwise phase runs.  The bf16 A operands of the gradK / gradV MMAs go
  // inside the 16 columns each thread read: gS^T into the first 8 and dS^T
  // into the last 8 of S^T, gdP^T into the first 8 of G^T.  The gradQ^T
  // partial of a tile (64 columns) goes into its S^T columns once the gradK
  // MMAs have read them.
  // d = 128: one S^T / G^T buffer.  The MMA order per tile is gradK, gradQ^T,
  // gradV, then the next tile's S^T / G^T, which wait for the elementwise
  // warps to drain the partial at the end of their tile.
  // d = 64 (SG2): TMEM also holds a second S^T / G^T buffer (tile t in
  // buffer t % 2).  The next tile's S^T / G^T go first, into the other
  // buffer, as soon as the elementwise warps have drained the partial of
  // the tile before (which they do as they hand over this tile's A
  // operands), so they run while those warps reduce that partial; then
  // gradK, gradV and gradQ^T of this tile, during the next tile's
  // elementwise phase.
  static constexpr bool SG2 = (D == 64);
  __host__ __device__ static constexpr uint32_t T_S(int b) { return SG2 ? 128u * b : 0u; }
  __host__ __device__ static constexpr uint32_t T_G(int b) { return T_S(b) + 64u; }
  static constexpr uint32_t T_DP = SG2 ? 256 : 128, T_H = T_DP + 64, T_GK = T_H + 64,
                            T_GV = T_GK + D;
  static_assert(T_GV + D == 512, "pass 2 TMEM layout fills 512 columns");
  static constexpr uint32_t TMEM_COLS = 512;
  // Registers per thread after the split: 640 threads launch with 96 each
  // (five warps share each SM sub-partition's 64 KB register file), and the
  // control warpgroup gives the elementwise warps its surplus.  More would
  // overdraw the launch's registers, and a claim that cannot be met waits
  // forever, so the host checks the kernel's register count first.  The
  // elementwise phase at 96 spills and is latency-bound: 104 removes the
  // d = 128 spills (pass 2 9.36 -> 8.93 ms at the benchmark workload).  The
  // control split differs per d only because ptxas spills less that way.
  static constexpr int REGS_ELEMENTWISE = 104, REGS_CONTROL = D == 128 ? 56 : 64;
  static constexpr int REGS_NEEDED = 16 * 32 * REGS_ELEMENTWISE + 4 * 32 * REGS_CONTROL;
};

struct ColParams {
  const float* lse;
  const float* Dv;
  const float* r;
  const float* sigma;
  __nv_bfloat16* gradk;
  __nv_bfloat16* gradv;
  float* acc;  // fp32 [B,H,N,D] gradQ accumulator
  int* status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int N, causal;
  int BH, G;  // batch * heads, heads per CTA group (cta_coord)
  float scale;
  int has_gq, has_gk, has_gv;  // as in RowParams
};

// Pass 2 warp roles: warps 0-15 elementwise (warp w: TMEM lane quadrant w%4,
// 16-column slice w/4 of the 64-query tile, which is also the 16-query
// contraction step w/4 of the gradK / gradV MMAs), warp 16 TMA producer of
// the stationary tiles, the [Q|gQ] stages and the row scalars, warp 17 TMEM
// allocator and MMA issuer, warp 18 TMA producer of the dO ring.  dO has a
// warp of its own so that its loads run as far ahead as its ring allows:
// the next tile's dP^T / H^T MMAs wait for it while the elementwise phase
// runs, and the [Q|gQ] producer spends most of each tile waiting for the
// gradK MMAs to free its stage.  The MMA warp waits for the elementwise
// warps itself: these waits gate the next MMAs directly, and folding them
// through a helper warp (as in pass 1) added a hand-off to every tile.
// Warp 19 has no role: it completes warps 16-19 to a warpgroup, the unit in
// which setmaxnreg moves registers (see Col::REGS_*).
constexpr int kColConsumerWarps = 16;
constexpr int kColConsumers = kColConsumerWarps * 32;
constexpr int kColProducerWarp = kColConsumerWarps;
constexpr int kColMmaWarp = kColConsumerWarps + 1;
constexpr int kColDoWarp = kColConsumerWarps + 2;
constexpr int kColThreads = (kColConsumerWarps + 4) * 32;
constexpr int kColCols = 64 / (kColConsumerWarps / 4);  // columns per elementwise thread
static_assert(kColCols == 16, "one 16-query MMA step per column slice");

template <int D, bool ALL>
__global__ void __launch_bounds__(kColThreads, 1)
    bob_col_pass(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mGK,
                 const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mGV,
                 const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mGQ,
                 const __grid_constant__ CUtensorMap mDO, ColParams prm) {
  using C = Col<D>;
  // cotangents present: ALL (every one) is the compiled fast path; otherwise
  // the flags decide at run time
  const bool has_gq = ALL || prm.has_gq != 0, has_gk = ALL || prm.has_gk != 0,
             has_gv = ALL || prm.has_gv != 0;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report_status(prm.status, FBOB_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  uint64_t* kv_full = bars + 0;
  uint64_t* qg_full = bars + 1;                 // [STAGES]: [Q|gQ] landed, scalars written
  uint64_t* qg_empty = qg_full + C::STAGES;     // [STAGES]: gradK MMAs done with [Q|gQ]
  uint64_t* do_full = qg_empty + C::STAGES;     // [DSTAGES]
  uint64_t* do_empty = do_full + C::DSTAGES;    // [DSTAGES]: gradV MMAs done with dO
  uint64_t* sc_full = do_empty + C::DSTAGES;    // scores in TMEM
  uint64_t* sc_read = sc_full + 1;              // elementwise warps hold the scores
  uint64_t* ds_full = sc_read + 1;              // A operands in TMEM, dS^T / gS^T in smem
  uint64_t* gq_full = ds_full + 1;
  uint64_t* gq_empty = gq_full + 1;
  uint64_t* acc_done = gq_empty + 1;
  uint64_t* drain = acc_done + 1;
  static_assert((8 + 2 * C::STAGES + 2 * C::DSTAGES) * 8 <= 256,
                "barriers end below the TMEM slot");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 256);
  Abort* abort_st = reinterpret_cast<Abort*>(smem + C::OFF_MISC + 264);
  float* scal = reinterpret_cast<float*>(smem + C::OFF_SC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = prm.N;
  const CtaCoord cc = cta_coord(prm.BH, prm.G, (prm.N + C::BM - 1) / C::BM);
  const int bh = cc.bh;
  const int j0 = cc.blk * C::BM;  // low key blocks (most query tiles) first
  const int qstart = prm.causal ? (j0 / C::BN) * C::BN : 0;
  const int T = (N - qstart + C::BN - 1) / C::BN;
  const int rot = cc.blk % T;  // start tile of this CTA's query loop

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(qg_full + s, 1);
      mbar_init(qg_empty + s, 1);
    }
    for (int s = 0; s < C::DSTAGES; ++s) {
      mbar_init(do_full + s, 1);
      mbar_init(do_empty + s, 1);
    }
    mbar_init(sc_full, 1);
    mbar_init(sc_read, kColConsumers);
    mbar_init(ds_full, kColConsumers);
    mbar_init(gq_full, 1);
    mbar_init(gq_empty, kColConsumers);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    abort_st->flag = 0;
    abort_st->limit_ns = prm.wait_ns;
    fence_mbar_init();
  }
  if (warp == kColMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kColConsumerWarps) {
    // control warpgroup (warps 16-19): it hands registers to the
    // elementwise warpgroups as one, then splits into its roles; warp 19
    // only completes the warpgroup
    regs_release<C::REGS_CONTROL>();
    if (warp == kColProducerWarp) {
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, (2 + (has_gk ? 1 : 0) + (has_gv ? 1 : 0)) * C::KB);
        load_tile(smem + C::OFF_K, &mK, kv_full, j0, bh);
        if (has_gk) load_tile(smem + C::OFF_GK, &mGK, kv_full, j0, bh);
        load_tile(smem + C::OFF_V, &mV, kv_full, j0, bh);
        if (has_gv) load_tile(smem + C::OFF_GV, &mGV, kv_full, j0, bh);
      }
      bool ok = true;
      // row scalars (lse pre-scaled by log2 e, D, r, sigma) of the next query
      // tile are fetched into registers one tile ahead, off the critical path
      constexpr int PER = C::BN / 32;
      float pre[4][PER];
      auto fetch = [&](int q0) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int q = q0 + lane + 32 * u;
          const bool in = q < N;
          const size_t idx = (size_t)bh * N + (in ? q : 0);
          pre[0][u] = in ? prm.lse[idx] * kLog2e : 0.f;
          pre[1][u] = in ? prm.Dv[idx] : 0.f;
          pre[2][u] = in ? prm.r[idx] : 0.f;
          pre[3][u] = in ? prm.sigma[idx] : 0.f;
        }
      };
      fetch(qstart + rotated(0, rot, T) * C::BN);
      int qg_issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % C::STAGES;
        const int q0 = qstart + rotated(t, rot, T) * C::BN;
        const int q_next = qstart + rotated(t + 1 < T ? t + 1 : 0, rot, T) * C::BN;
        // Row scalars of tile t, stored negated (every one of them is
        // subtracted).  Their buffer was last read by the elementwise warps of
        // tile t - SCSTAGES, which finished before that tile's gradK MMAs
        // released its [Q|gQ] stage, awaited in the previous iteration.
        float* sc = scal + (t % C::SCSTAGES) * 4 * C::BN;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int u = 0; u < PER; ++u) sc[a * C::BN + lane + 32 * u] = -pre[a][u];
        __syncwarp();
        // the next tile's scalars are in flight while this warp waits below
        if (t + 1 < T) fetch(q_next);
        bool w = true;
        if (lane == 0 && t >= C::STAGES)
          w = wait_bar(qg_empty + s, ((t / C::STAGES) - 1) & 1, abort_st, prm.status);
        ok = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (lane == 0) {
          // this arrival publishes the scalars written above with the stage
          mbar_arrive_expect_tx(qg_full + s, (has_gq ? 2 : 1) * C::QB);
          load_pair_opt<D>(smem + C::OFF_QG + s * 2 * C::QB, &mQ, &mGQ, has_gq, qg_full + s,
                           C::BN, q0, bh);
          ++qg_issued;
          if (t + 1 < T) {  // warm L2 with the next query tile
            tma_prefetch_l2_4d(&mQ, 0, q_next, 0, bh);
            if (has_gq) tma_prefetch_l2_4d(&mGQ, 0, q_next, 0, bh);
          }
        }
      }
      // every load this warp issued has landed before the CTA exits (after an
      // abort some were never awaited); each phase waited for is the last of
      // its barrier, so on the normal path these return at once
      if (lane == 0) {
        mbar_wait_bounded(kv_full, 0, prm.status, 100000000ull);
        for (int t = max(0, qg_issued - C::STAGES); t < qg_issued; ++t)
          mbar_wait_bounded(qg_full + (t % C::STAGES), (t / C::STAGES) & 1, prm.status,
                            100000000ull);
      }
    } else if (warp == kColDoWarp) {
      if (lane == 0) {
        int do_issued = 0;
        for (int t = 0; t < T; ++t) {
          const int ds = t % C::DSTAGES;
          if (t >= C::DSTAGES &&
              !wait_bar(do_empty + ds, ((t / C::DSTAGES) - 1) & 1, abort_st, prm.status))
            break;
          mbar_arrive_expect_tx(do_full + ds, C::QB);
          load_tile(smem + C::OFF_DO + ds * C::QB, &mDO, do_full + ds,
                    qstart + rotated(t, rot, T) * C::BN, bh);
          ++do_issued;
          if (t + 1 < T)  // warm L2 with the next dO tile
            tma_prefetch_l2_4d(&mDO, 0, qstart + rotated(t + 1, rot, T) * C::BN, 0, bh);
        }
        // every load this thread issued has landed before the CTA exits
        for (int t = max(0, do_issued - C::DSTAGES); t < do_issued; ++t)
          mbar_wait_bounded(do_full + (t % C::DSTAGES), (t / C::DSTAGES) & 1, prm.status,
                            100000000ull);
      }
    } else if (warp == kColMmaWarp) {
      {  // the whole warp: warp-uniform waits, elect.sync issues each MMA
        constexpr uint32_t id_sc = idesc_bf16(128, 64, false, false);  // scores: M=128 N=64
        constexpr uint32_t id_sg = idesc_bf16(128, 128, false, false);  // K [Q;gQ]^T: N=128
        constexpr uint32_t id_out = idesc_bf16(128, D, false, true);   // gradK/V: N=D, B MN
        constexpr uint32_t id_gq = idesc_bf16(D, 64, true, true);      // gradQ^T: M=D, A,B MN
        // descriptor low words of the stationary tiles: K-major for the score
        // MMAs, MN-major (64-feature groups BM*128 bytes apart) for gradQ^T
        const uint32_t k_lo = lo_kmajor(sb + C::OFF_K), gk_lo = lo_kmajor(sb + C::OFF_GK),
                       v_lo = lo_kmajor(sb + C::OFF_V), gv_lo = lo_kmajor(sb + C::OFF_GV);
        const uint32_t k_mn = lo_mnmajor(sb + C::OFF_K, C::BM * 128),
                       gk_mn = lo_mnmajor(sb + C::OFF_GK, C::BM * 128);
        const uint32_t ds_mn = lo_mnmajor(sb + C::OFF_DS, 1024), gs_mn = lo_mnmajor(sb + C::OFF_GS, 1024);
        const uint32_t t_dp = tmem + C::T_DP, t_h = tmem + C::T_H, t_gk = tmem + C::T_GK,
                       t_gv = tmem + C::T_GV;
        // dP^T and H^T of tile t (need dO(t) and the previous tile's scores
        // read out of TMEM)
        auto issue_dh = [&](int t) -> bool {
          const int ds = t % C::DSTAGES;
          const uint32_t do_lo = opaque(lo_kmajor(sb + C::OFF_DO + ds * C::QB));
          const uint32_t v_l = opaque(v_lo), gv_l = opaque(gv_lo);
          if (!warp_wait(do_full + ds, (t / C::DSTAGES) & 1, abort_st, prm.status)) return false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss_w(t_dp, v_l + kslice_off(C::BM, k), do_lo + kslice_off(C::BN, k), id_sc, k > 0 ? 1u : 0u);
          if (has_gv) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss_w(t_h, gv_l + kslice_off(C::BM, k), do_lo + kslice_off(C::BN, k), id_sc,
                     k > 0 ? 1u : 0u);
          }
          return true;
        };
        // S^T and G^T of tile t into buffer t % 2 (need Q, gQ; overwrite the
        // A operands and the gradQ^T partial of the tile that last used the
        // buffer: t - 1 at d = 128, t - 2 with SG2), then the commit that
        // covers all four score blocks
        auto issue_sg = [&](int t) -> bool {
          const int s = t % C::STAGES;
          const uint32_t qgq_lo = opaque(lo_kmajor(sb + C::OFF_QG + s * 2 * C::QB));  // [Q;gQ] per half
          const uint32_t k_l = opaque(k_lo), gk_l = opaque(gk_lo);
          const uint32_t t_s = tmem + C::T_S(t & 1), t_g = tmem + C::T_G(t & 1);
          const int prev = C::SG2 ? t - 2 : t - 1;  // the buffer's previous tile
          if (!warp_wait(qg_full + s, (t / C::STAGES) & 1, abort_st, prm.status)) return false;
          if (prev >= 0 && !warp_wait(gq_empty, prev & 1, abort_st, prm.status)) return false;
          tc_fence_after();
          // [S^T | K gQ^T] = K [Q; gQ]^T (S^T = K Q^T alone without gQ), then
          // G^T += gK Q^T (the first BN rows of each [Q;gQ] half are Q)
          const uint32_t id_first = has_gq ? id_sg : id_sc;
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss_w(t_s, k_l + kslice_off(C::BM, k), qgq_lo + kslice_off(2 * C::BN, k), id_first,
                   k > 0 ? 1u : 0u);
          if (has_gk) {
            const uint32_t g0 = has_gq ? 1u : 0u;  // without gQ this starts G^T
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss_w(t_g, gk_l + kslice_off(C::BM, k), qgq_lo + kslice_off(2 * C::BN, k), id_sc,
                     k > 0 ? 1u : g0);
          }
          mma_commit_w(sc_full);
          return true;
        };
        bool ok = warp_wait(kv_full, 0, abort_st, prm.status) && issue_dh(0) && issue_sg(0);
        for (int t = 0; ok && t < T; ++t) {
          const int s = t % C::STAGES, ds = t % C::DSTAGES;
          // ---- next tile's dP^T, H^T while the elementwise warps work ----
          if (t + 1 < T) {
            if (!warp_wait(sc_read, t & 1, abort_st, prm.status)) { ok = false; break; }
            tc_fence_after();
            if (!issue_dh(t + 1)) { ok = false; break; }
          }
          // ---- SG2: next tile's S^T, G^T into the other buffer ----
          if (C::SG2 && t + 1 < T && !issue_sg(t + 1)) { ok = false; break; }
          // ---- outputs: A operands (bf16 gS^T, dS^T, gdP^T) from TMEM ----
          if (!warp_wait(ds_full, t & 1, abort_st, prm.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t t_s = tmem + C::T_S(t & 1), t_g = tmem + C::T_G(t & 1);
          const uint32_t qgq_s = sb + C::OFF_QG + s * 2 * C::QB;
          // B operands MN-major: 64-feature groups 2*BN*128 bytes apart in the
          // interleaved [Q;gQ] stage, BN*128 apart in the dO tile
          const uint32_t q_mn = opaque(lo_mnmajor(qgq_s, 2 * C::BN * 128)),
                         gq_mn = opaque(lo_mnmajor(qgq_s + C::BN * 128, 2 * C::BN * 128));
          const uint32_t do_mn = opaque(lo_mnmajor(sb + C::OFF_DO + ds * C::QB, C::BN * 128));
          const uint32_t first = t > 0 ? 1u : 0u;
          // gradK first: it releases the [Q|gQ] stage that the next tile waits for
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k) {  // contraction over the 64 queries
            mma_ts_w(t_gk, t_s + 16 * k, q_mn + kstep_off(k), id_out, k > 0 ? 1u : first);
            if (has_gq) mma_ts_w(t_gk, t_s + 16 * k + 8, gq_mn + kstep_off(k), id_out, 1u);
          }
          mma_commit_w(qg_empty + s);
          // gradQ^T of tile t into its S^T columns, whose A operands the gradK
          // MMAs above read first (MMAs from one thread run in issue order).
          // The partial that used them before was drained before this tile's
          // S^T / G^T were issued.
          auto issue_gq = [&]() {
            const uint32_t k_m = opaque(k_mn), gk_m = opaque(gk_mn), ds_m = opaque(ds_mn),
                           gs_m = opaque(gs_mn);
#pragma unroll
            for (int k = 0; k < C::BM / 16; ++k) {  // contraction over the 128 keys
              mma_ss_w(t_s, k_m + kstep_off(k), gs_m + kstep_off(k), id_gq, k > 0 ? 1u : 0u);
              if (has_gk) mma_ss_w(t_s, gk_m + kstep_off(k), ds_m + kstep_off(k), id_gq, 1u);
            }
            mma_commit_w(gq_full);
          };
          // at d = 128 gradQ^T goes before gradV: its partial is drained sooner,
          // and the next tile's scores wait for that drain
          if (!C::SG2) issue_gq();
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k)
            mma_ts_w(t_gv, t_g + 16 * k, do_mn + kstep_off(k), id_out, k > 0 ? 1u : first);
          mma_commit_w(do_empty + ds);
          if (C::SG2) {
            issue_gq();
          } else if (t + 1 < T && !issue_sg(t + 1)) {
            ok = false;
            break;
          }
        }
        if (ok) mma_commit_w(acc_done);
        mma_commit_w(drain);
        mbar_wait_bounded(drain, 0, prm.status, 100000000ull);
      }
    }
  } else {
    regs_claim<C::REGS_ELEMENTWISE>();
    // ---------------- elementwise warps: thread = key row -----------------
    constexpr int NC = kColCols;           // query columns per thread
    const int row = 32 * (warp & 3) + lane;
    const int slice = warp >> 2;           // columns [NC*slice, NC*slice + NC)
    const int j = j0 + row;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sc2 = prm.scale * kLog2e;
    const f2 sc2_2 = {sc2, sc2}, scale_2 = {prm.scale, prm.scale};
    const bool has_g = has_gq || has_gk, has_h = has_gv;
    // gradQ^T partial of tile t (TMEM lane = feature index, column = query),
    // in the S^T columns of its buffer, once gq_full(t) has been awaited
    auto load_gq = [&](int t, uint32_t (&gq)[NC]) {
      tc_fence_after();
      tmem_ld16(tmem + lane_off + C::T_S(t & 1) + NC * slice, gq);
      tc_fence_before();
      mbar_arrive(gq_empty);  // TMEM region free; the reductions follow
    };
    auto reduce_gq = [&](int t, const uint32_t (&gq)[NC]) {
      const int qa = qstart + rotated(t, rot, T) * C::BN + NC * slice;
      if (D == 128) {
        red_columns<D, NC>(prm.acc + ((size_t)bh * N + qa) * D + row, gq, N - qa);
      } else {
        // M = 64 accumulator: rows 16w' + x (w' = warp & 3, x < 16) live in
        // lanes 32w' + x; the upper 16 lanes of each warp hold nothing.
        if (lane < 16) {
          red_columns<D, NC>(prm.acc + ((size_t)bh * N + qa) * D + 16 * (warp & 3) + lane, gq, N - qa);
        }
      }
    };
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::STAGES;
      const int q0 = qstart + rotated(t, rot, T) * C::BN;
      if (!warp_wait(sc_full, t & 1, abort_st, prm.status)) { ok = false; break; }
      // the stage's row scalars were published with qg_full (already complete)
      if (!warp_wait(qg_full + s, (t / C::STAGES) & 1, abort_st, prm.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[NC], dpr[NC], gr[NC], hr[NC];
      const uint32_t tl = tmem + lane_off + NC * slice;
      const uint32_t ts = tl + C::T_S(t & 1), tg = tl + C::T_G(t & 1);
      tmem_ld16x4(ts, tl + C::T_DP, tg, tl + C::T_H, sr, dpr, gr, hr);
      // the loads above have completed: dP^T, H^T are free
      tc_fence_before();
      mbar_arrive(sc_read);
      const float4* sc4 =
          reinterpret_cast<const float4*>(scal + (t % C::SCSTAGES) * 4 * C::BN + NC * slice);
      const int qa = q0 + NC * slice;
      const bool need_mask = (qa + NC > N) || (j0 + C::BM > N) || (prm.causal && qa < j0 + C::BM);
      uint32_t dsw[NC / 2], gdw[NC / 2], gsw[NC / 2];
      // one body per mask case, so the unmasked bulk carries no per-element
      // branches
      auto body = [&](auto masked) {
#pragma unroll
        for (int c4 = 0; c4 < NC / 4; ++c4) {  // 4 query columns per step
          // negated row scalars of the 4 queries: -LSE log2 e, -D, -r, -sigma
          const float4 L = sc4[c4], Dd = sc4[C::BN / 4 + c4], R = sc4[C::BN / 2 + c4],
                       Sg = sc4[3 * C::BN / 4 + c4];
          const f2 nl[2] = {{L.x, L.y}, {L.z, L.w}}, nd[2] = {{Dd.x, Dd.y}, {Dd.z, Dd.w}},
                   nr[2] = {{R.x, R.y}, {R.z, R.w}}, ns[2] = {{Sg.x, Sg.y}, {Sg.z, Sg.w}};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // query columns cc, cc + 1: one packed pair
            const int cc = 4 * c4 + 2 * hh;
            const f2 sv2 = {__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])};
            const f2 x = fma2(sv2, sc2_2, nl[hh]);
            f2 p = {ex2_approx(x.x), ex2_approx(x.y)};
            if (decltype(masked)::value) {
              const int q = qa + cc;
              p.x = (q < N && j < N && (!prm.causal || q >= j)) ? p.x : 0.f;
              p.y = (q + 1 < N && j < N && (!prm.causal || q + 1 >= j)) ? p.y : 0.f;
            }
            const f2 dpm = add2({__uint_as_float(dpr[cc]), __uint_as_float(dpr[cc + 1])}, nd[hh]);
            // G^T (H^T) is zero, its TMEM columns unwritten, without gQ and gK (gV)
            const f2 gm = has_g ? fma2({__uint_as_float(gr[cc]), __uint_as_float(gr[cc + 1])},
                                       scale_2, nr[hh])
                                : nr[hh];
            const f2 hv = has_h ? f2{__uint_as_float(hr[cc]), __uint_as_float(hr[cc + 1])}
                                : f2{0.f, 0.f};
            const f2 ds = mul2(p, dpm), gd = mul2(p, gm);
            const f2 gs = mul2(p, add2(fma2(gm, dpm, hv), ns[hh]));
            dsw[cc >> 1] = pack_bf16(ds.x, ds.y);
            gdw[cc >> 1] = pack_bf16(gd.x, gd.y);
            gsw[cc >> 1] = pack_bf16(gs.x, gs.y);
          }
        }
      };
      if (need_mask)
        body(std::true_type{});
      else
        body(std::false_type{});
      // A operands of the gradK / gradV MMAs: bf16 pairs (low half = even
      // query), gS^T and dS^T in the 16 columns this thread read from S^T,
      // gdP^T in the first 8 it read from G^T; one 16-query contraction step
      // per slice
      tmem_st8x3(ts, gsw, ts + 8, dsw, tg, gdw);
      // With SG2 the previous tile's gradQ^T MMAs read the dS^T / gS^T tiles
      // below: wait for them first.  At d = 128 that wait ended the previous
      // iteration.
      if (C::SG2 && t >= 1 && !warp_wait(gq_full, (t - 1) & 1, abort_st, prm.status)) {
        ok = false;
        break;
      }
      // dS^T and gS^T also go to shared memory as the gradQ^T B operands.
      // This thread's columns are 16-byte chunks [NC*slice/8, +NC/8) of its row.
#pragma unroll
      for (int q = 0; q < NC / 8; ++q) {
        const uint32_t chunk = (NC / 8) * slice + q;
        st_shared_v4(sb + C::OFF_DS + sw128_offset(row, chunk), dsw[4 * q], dsw[4 * q + 1],
                     dsw[4 * q + 2], dsw[4 * q + 3]);
        st_shared_v4(sb + C::OFF_GS + sw128_offset(row, chunk), gsw[4 * q], gsw[4 * q + 1],
                     gsw[4 * q + 2], gsw[4 * q + 3]);
      }
      if (C::SG2 && t >= 1) {
        // drain the previous tile's partial now, which frees the other
        // buffer for the next tile's scores
        uint32_t gq[NC];
        load_gq(t - 1, gq);
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(ds_full);
        reduce_gq(t - 1, gq);
      } else {
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(ds_full);
        if (!C::SG2) {
          if (!warp_wait(gq_full, t & 1, abort_st, prm.status)) { ok = false; break; }
          uint32_t gq[NC];
          load_gq(t, gq);
          reduce_gq(t, gq);
        }
      }
    }
    if (C::SG2 && ok && T >= 1) {
      ok = warp_wait(gq_full, (T - 1) & 1, abort_st, prm.status);
      if (ok) {
        uint32_t gq[NC];
        load_gq(T - 1, gq);
        reduce_gq(T - 1, gq);
      }
    }
    // ---- epilogue: gradK (scaled), gradV; each thread D/4 features ----
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = warp_wait(acc_done, 0, abort_st, prm.status);
    tc_fence_after();
    if (ok) {  // warp-uniform: every lane loads TMEM, rows past N do not store
      constexpr int PART = D / 4;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = which == 0 ? prm.gradk : prm.gradv;
        const float mul = which == 0 ? prm.scale : 1.f;
        const uint32_t tcol = (which == 0 ? C::T_GK : C::T_GV) + PART * slice;
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
  if (warp == kColMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// scale * fp32 accumulator -> bf16, 8 elements per thread.
__global__ void __launch_bounds__(256) gradq_convert(const float4* __restrict__ acc,
                                                     uint4* __restrict__ out, size_t n8,
                                                     float scale) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    out[i] = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                        pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Whether the pass-2 kernel's launch registers (per thread, as compiled)
// cover the warpgroup split it performs; looked up once per instantiation.
template <int D>
bool col_regs_cover_split(bool all) {
  auto covers = [](const void* fn) {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, fn) == cudaSuccess &&
           (long long)fa.numRegs * kColThreads >= Col<D>::REGS_NEEDED;
  };
  static const bool ok_all = covers(reinterpret_cast<const void*>(bob_col_pass<D, true>));
  static const bool ok_some = covers(reinterpret_cast<const void*>(bob_col_pass<D, false>));
  return all ? ok_all : ok_some;
}

template <int D>
cudaError_t bob_d(const Problem& p, const void* q, const void* k, const void* v, const void* o,
                  const float* lse, const void* dO, const void* gq, const void* gk,
                  const void* gv, void* gradq, void* gradk, void* gradv, void* graddo,
                  const Workspace& ws, LaunchLog& log) {
  using R = Row<D>;
  using Cc = Col<D>;
  // an absent cotangent (null pointer) is zero: its map is a placeholder the
  // kernels never load through
  const int has_gq = gq != nullptr, has_gk = gk != nullptr, has_gv = gv != nullptr;
  CUtensorMap mQr, mGQr, mKr, mGKr, mVr, mGVr;
  if (!make_map(&mQr, q, p, R::BM) || !make_map(&mGQr, has_gq ? gq : q, p, R::BM) ||
      !make_map(&mKr, k, p, R::BN, true) || !make_map(&mGKr, has_gk ? gk : k, p, R::BN, true) ||
      !make_map(&mVr, v, p, R::BN) || !make_map(&mGVr, has_gv ? gv : v, p, R::BN))
    return cudaErrorInvalidValue;
  CUtensorMap mKc, mGKc, mVc, mGVc, mQc, mGQc, mDOc;
  if (!make_map(&mKc, k, p, Cc::BM) || !make_map(&mGKc, has_gk ? gk : k, p, Cc::BM) ||
      !make_map(&mVc, v, p, Cc::BM) || !make_map(&mGVc, has_gv ? gv : v, p, Cc::BM) ||
      !make_map(&mQc, q, p, Cc::BN, true) || !make_map(&mGQc, has_gq ? gq : q, p, Cc::BN, true) ||
      !make_map(&mDOc, dO, p, Cc::BN))
    return cudaErrorInvalidValue;

  const bool all = has_gq && has_gk && has_gv;
  auto row_kernel = all ? bob_row_pass<D, true> : bob_row_pass<D, false>;
  auto col_kernel = all ? bob_col_pass<D, true> : bob_col_pass<D, false>;
  // pass 2 moves registers between its warpgroups; refuse to launch a build
  // whose register count cannot cover that split (the claim would not end)
  if (!col_regs_cover_split<D>(all)) return cudaErrorLaunchOutOfResources;
  cudaError_t e = cudaFuncSetAttribute(row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)R::SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(col_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)Cc::SMEM);
  if (e != cudaSuccess) return e;

  RowParams rp;
  rp.lse = lse;
  rp.o = static_cast<const __nv_bfloat16*>(o);
  rp.dO = static_cast<const __nv_bfloat16*>(dO);
  rp.graddo = static_cast<__nv_bfloat16*>(graddo);
  rp.r_out = ws.r;
  rp.sigma_out = ws.sigma;
  rp.D_out = ws.D;
  rp.acc_zero = ws.acc;
  rp.status = ws.status;
  rp.wait_ns = wait_limit_ns();
  rp.N = p.N;
  rp.BH = p.BH();
  rp.G = cta_group_heads(p.BH(), (p.N + R::BM - 1) / R::BM, sm_count());
  rp.causal = p.causal;
  rp.scale = p.scale;
  rp.has_gq = has_gq;
  rp.has_gk = has_gk;
  rp.has_gv = has_gv;
  dim3 g1((unsigned)(((p.N + R::BM - 1) / R::BM) * p.BH()));
  row_kernel<<<g1, R::THREADS, R::SMEM, log.stream>>>(mQr, mGQr, mKr, mGKr, mVr, mGVr, rp);
  e = cudaGetLastError();
  log.mark();
  if (e != cudaSuccess) return e;

  ColParams cp;
  cp.lse = lse;
  cp.Dv = ws.D;
  cp.r = ws.r;
  cp.sigma = ws.sigma;
  cp.gradk = static_cast<__nv_bfloat16*>(gradk);
  cp.gradv = static_cast<__nv_bfloat16*>(gradv);
  cp.acc = ws.acc;
  cp.status = ws.status;
  cp.wait_ns = wait_limit_ns();
  cp.N = p.N;
  cp.BH = p.BH();
  cp.G = cta_group_heads(p.BH(), (p.N + Cc::BM - 1) / Cc::BM, sm_count());
  cp.causal = p.causal;
  cp.scale = p.scale;
  cp.has_gq = has_gq;
  cp.has_gk = has_gk;
  cp.has_gv = has_gv;
  dim3 g2((unsigned)(((p.N + Cc::BM - 1) / Cc::BM) * p.BH()));
  col_kernel<<<g2, kColThreads, Cc::SMEM, log.stream>>>(mKc, mGKc, mVc, mGVc, mQc, mGQc, mDOc, cp);
  e = cudaGetLastError();
  log.mark();
  if (e != cudaSuccess) return e;

  return launch_acc_to_bf16(ws.acc, gradq, p.elems(), p.scale, log);
}

// One thread waits on an mbarrier whose phase nothing completes; the bounded
// wait gives up after limit_ns and records FBOB_ERR_TIMEOUT.
__global__ void wait_timeout_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* status, long long limit_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

bool tc_supported(const Problem& p) { return p.bf16 && (p.d == 64 || p.d == 128); }

cudaError_t launch_acc_to_bf16(const float* acc, void* out, size_t elems, float scale,
                               LaunchLog& log) {
  const size_t n8 = elems / 8;
  const unsigned blocks = (unsigned)std::min<size_t>((n8 + 255) / 256, 152 * 16);
  gradq_convert<<<blocks, 256, 0, log.stream>>>(reinterpret_cast<const float4*>(acc),
                                                static_cast<uint4*>(out), n8, scale);
  const cudaError_t e = cudaGetLastError();
  log.mark();
  return e;
}

cudaError_t tc_bob(const Problem& p, const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dO, const void* gq, const void* gk,
                   const void* gv, void* gradq, void* gradk, void* gradv, void* graddo,
                   const Workspace& ws, LaunchLog& log) {
  if (p.d == 128)
    return bob_d<128>(p, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk, gradv, graddo, ws, log);
  return bob_d<64>(p, q, k, v, o, lse, dO, gq, gk, gv, gradq, gradk, gradv, graddo, ws, log);
}

}  // namespace fbob

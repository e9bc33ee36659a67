// Fused backward at d = 128 for moderate key lengths (gist.science technical
// summary, "Metodologia" section 2, kernel fusion paragraph: one kernel visits
// every (query tile, key tile) pair once and accumulates dQ across key tiles
// with atomics). Probabilities are regenerated tile by tile from Q, K and the
// saved LSEs, P_t = exp(S_t - LSE_t).
//
// CTA = one (batch-head, 128-key tile); it sweeps 64-row query steps (causal:
// from the diagonal down):
//   T_t     = K_t Q_t^T       (M = 128 keys, N = 64 queries, K = d)
//   dS_t    from T_t          (softmax warps; bf16 to shared memory, row = key)
//   dK_t   += dS_t Q_t        (M = 128 keys, N = d, K = 64 queries; TMEM)
//   dQ_t^T  = K_t^T dS_t      (M = d, N = 64 queries, K = 128 keys; TMEM)
// Against the separate dK and dQ kernels this regenerates S1, S2 and forms dS
// once per pair (8d FLOPs per pair and set instead of 12d). Each step's dQ
// goes from TMEM (lane = d column) through a shared-memory staging tile
// (row = query, 128-byte swizzle: a warp's stores are one contiguous 128-byte
// row piece) and TMA bulk reductions (add) into the fp32 accumulator
// [BH][N_Q][d] (zeroed by the caller): 4 d bytes per pair and set, so the
// kernel pays off only while the keys are few enough that those reductions
// stay below the work saved. dK leaves once at the end through the staging
// tile and TMA stores.
//
// The kernel is bound by its step's dependency chain, not by one unit: a
// tcgen05.mma of M = 128 costs ~45 cycles whatever N <= 64 (timed alone), so
// the N = 64 GEMMs run at two thirds of the tensor rate at best. With one
// gradient set the T GEMMs take K from TMEM (copied there once per CTA by the
// softmax warps) and the freed K tile becomes a second dQ staging tile.
//
// Gradients of L = sum_i g_i KL_i, with s = scale * q.k (g and scale folded
// into dS):
//   configuration 1 (teacher P1 fixed):  dS2 = g * (P2 - P1)
//   configuration 2 (student P2 fixed):  dS1 = g * P1 * (log(P1/P2) - KL)
// with log(P1/P2) - KL = scale (s1 - s2) - (LSE1 - LSE2 + KL) from logits and
// the saved LSEs (section 3, numerical stability).
//
// Warps: 0 = TMA producer (lane 0) and the per-query constant table of each Q
// stage (all lanes); 1 = TMEM owner + MMA issuer; 2..17 = softmax and
// read-outs: warp w reads TMEM lanes [32 (w%4), +32) and serves column group
// g = (w-2)/4 (T: thread = key row, query columns [16g, 16g+16); dQ^T
// read-out: thread = d column, queries [16g, 16g+16); dK read-out: thread =
// key row, d columns [32g, 32g+32)); 18 = TMA reductions and stores (lane 0).
// TMEM: T1 [0,64) T2 [64,128) | dK per set (128 columns) | dQ^T per set (64)
// | one set: K1, K2 as packed bf16 pairs (64 columns each).
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

// the bulk copy groups of this thread, but the most recent one, have finished
// reading shared memory
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

constexpr int kF2Threads = 608;  // 19 warps
constexpr int kF2SoftmaxWarps = 16;
constexpr int kF2StoreWarp = 18;
constexpr int kF2D = 128;
constexpr int kF2Step = 64;       // query rows per step
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSet2 = 1, kSet1 = 2;

template <int SETS>
struct Fused128Layout {
  static constexpr int NSETS = SETS == (kSet1 | kSet2) ? 2 : 1;
  static constexpr int KT = kBlockN * kF2D * 2;        // one K tile: 2 boxes of 128 rows x 128 B
  static constexpr int QT = kF2Step * kF2D * 2;        // one Q tile: 2 boxes of 64 rows x 128 B
  static constexpr int STAGES = NSETS == 2 ? 2 : 3;    // Q1, Q2 stages
  static constexpr int DST = kBlockN * kF2Step * 2;    // one dS tile: 128 key rows x 128 B
  static constexpr int STG = kF2Step * kF2D * 4;       // one set's fp32 dQ rows: 4 boxes of 8 KB
  static_assert(STG >= kBlockN * kF2D * 2, "the staging tile also holds one set's bf16 dK");
  static constexpr int TAB = 4 * kF2Step * 4;          // per stage: 4 x 64 floats
  // one gradient set: K1, K2 also in TMEM (64 packed columns each), the A
  // operand of the T GEMMs, which then read only Q from shared memory. The K
  // tile that the dQ GEMMs do not read (K1 for configuration 1, K2 for
  // configuration 2) is free after that copy and becomes a second staging
  // tile, so that a step's dQ read-out does not wait for the previous step's
  // reductions to leave shared memory.
  static constexpr bool KTM = NSETS == 1;
  static constexpr int NSTG = KTM ? 2 : 1;             // staging tiles
  static constexpr int OFF_K = 0;                      // K1, K2
  static constexpr int OFF_STG1 = OFF_K + (SETS == kSet2 ? 0 : KT);  // second staging tile
  static constexpr int OFF_Q = 2 * KT;                 // stage s: Q1 at +2s QT, Q2 at +(2s+1) QT
  static constexpr int OFF_DS = OFF_Q + STAGES * 2 * QT;  // slot t: the t-th computed set
  static constexpr int OFF_STG = OFF_DS + NSETS * DST;
  static constexpr int OFF_TAB = OFF_STG + STG;
  static constexpr int OFF_BAR = OFF_TAB + STAGES * TAB;
  // k_full, q_full[S], q_empty[S], t_full, t_free, ds_full, dq_full, dq_free,
  // dk_full, stg_full, stg_empty, drain, kt_full, then stg_full and stg_empty
  // of staging tile 1
  static constexpr int NBAR = 1 + 2 * STAGES + 12;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr uint32_t COL_T = 0, COL_DK = 2 * kF2Step, COL_DQ = COL_DK + NSETS * kF2D;
  static constexpr uint32_t COL_K = COL_DQ + NSETS * kF2Step;
  static_assert(COL_K + (KTM ? kF2D : 0) <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(OFF_Q % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_STG % 1024 == 0 && OFF_STG1 % 1024 == 0,
                "swizzled tiles on 1024-byte boundaries");
};

template <int SETS>
__global__ void __launch_bounds__(kF2Threads, 1)
    streamkl_bwd_fused128_kernel(const __grid_constant__ CUtensorMap tm_q1,
                                 const __grid_constant__ CUtensorMap tm_k1,
                                 const __grid_constant__ CUtensorMap tm_q2,
                                 const __grid_constant__ CUtensorMap tm_k2,
                                 const __grid_constant__ CUtensorMap tm_dq2,
                                 const __grid_constant__ CUtensorMap tm_dq1,
                                 const __grid_constant__ CUtensorMap tm_dk2,
                                 const __grid_constant__ CUtensorMap tm_dk1, int NQ, int NK,
                                 int causal, float scale, int BH, const float* __restrict__ kl_in,
                                 const float* __restrict__ lse1_in,
                                 const float* __restrict__ lse2_in, const float* __restrict__ g_in,
                                 int* dev_status, uint64_t timeout_ns) {
  using L = Fused128Layout<SETS>;
  constexpr bool HAS2 = SETS & kSet2, HAS1 = SETS & kSet1;
  constexpr int D = kF2D, STEP = kF2Step;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kt = static_cast<int>(blockIdx.x);  // key tile (causal: key tile 0 is the heaviest)
  const int bh = static_cast<int>(blockIdx.y);
  const int off = NK - NQ;                      // causal: key j visible to query i iff j <= i + off
  const int k0 = kt * kBlockN;
  const int nqs = (NQ + STEP - 1) / STEP;
  // query steps with a row that sees some key of this tile
  const int qs0 = causal ? max(0, k0 - off) / STEP : 0;
  int n = (k0 < NK && !(causal && NQ > NK)) ? max(0, nqs - qs0) : 0;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t k_full = bar0;
  auto q_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto q_empty = [&](int s) { return bar0 + 8u * (1 + L::STAGES + s); };
  const uint32_t t_full = bar0 + 8u * (1 + 2 * L::STAGES);
  const uint32_t t_free = t_full + 8, ds_full = t_full + 16;
  // dq_full: the step's dQ^T GEMMs, the last readers of its dS tiles, are
  // done (one commit serves both: a commit costs the tensor pipe about as
  // much as an MMA)
  const uint32_t dq_full = t_full + 24, dq_free = t_full + 32, dk_full = t_full + 40;
  const uint32_t stg_full = t_full + 48, stg_empty = t_full + 56, drain = t_full + 64;
  const uint32_t kt_full = t_full + 72;  // K rows copied into TMEM
  static_assert(1 + 2 * L::STAGES + 12 == L::NBAR, "barrier region holds every barrier");
  // staging use u (one per set and step, then one per set for dK) goes
  // through tile u % NSTG
  constexpr int NSTG = L::NSTG;
  auto stg_full_b = [&](int u) { return u % NSTG ? t_full + 80 : stg_full; };
  auto stg_empty_b = [&](int u) { return u % NSTG ? t_full + 88 : stg_empty; };
  auto stg_tile = [&](int u) { return sb + (u % NSTG ? L::OFF_STG1 : L::OFF_STG); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);
  // per stage and query column: -LSE1 log2e, -LSE2 log2e, g scale, -(LSE1 - LSE2 + KL)
  float* tab = reinterpret_cast<float*>(gb + L::OFF_TAB);

  CheckCtx ck{sb, sb + L::OFF_BAR, sb + L::OFF_BAR, sb + L::OFF_BAR + L::NBAR * 8, 0, 0,
              abort_flag, dev_status};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    bool lay_ok = true;
    if (kDeviceChecks) {  // every barrier address inside the barrier region
      lay_ok = check_bar(ck, k_full, __LINE__) && check_bar(ck, t_full, __LINE__) &&
               check_bar(ck, drain, __LINE__) && check_bar(ck, stg_empty_b(1), __LINE__);
      for (int s = 0; s < L::STAGES; ++s)
        lay_ok = lay_ok && check_bar(ck, q_full(s), __LINE__) && check_bar(ck, q_empty(s), __LINE__);
    }
    if (lay_ok) {
      mbar_init(k_full, 1);
      for (int s = 0; s < L::STAGES; ++s) {
        mbar_init(q_full(s), 1);
        mbar_init(q_empty(s), 1);
      }
      mbar_init(t_full, 1);
      mbar_init(t_free, kF2SoftmaxWarps);
      mbar_init(ds_full, kF2SoftmaxWarps);
      mbar_init(dq_full, 1);
      mbar_init(dq_free, kF2SoftmaxWarps);
      mbar_init(dk_full, 1);
      mbar_init(stg_full, kF2SoftmaxWarps);
      mbar_init(stg_empty, 1);
      mbar_init(drain, 1);
      mbar_init(kt_full, kF2SoftmaxWarps);
      mbar_init(stg_full_b(1), kF2SoftmaxWarps);
      mbar_init(stg_empty_b(1), 1);
    }
    // a failure recorded earlier (this launch or a previous one), or a
    // failed layout check, skips the work
    *skip_flag = !lay_ok || *reinterpret_cast<volatile int*>(dev_status) != 0;
    if (causal && NQ > NK) atomicCAS(dev_status, 0, kStatusInvalidArg);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q1);
    tma_prefetch_desc(&tm_k1);
    tma_prefetch_desc(&tm_q2);
    tma_prefetch_desc(&tm_k2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (*skip_flag) n = 0;
  const WaitCtx wc{abort_flag, dev_status, timeout_ns};
  ck.tmem = tmem;
  ck.tmem_cols = 512;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int j = 0;
    if (n > 0) {
      if (lane == 0) {
        if (kDeviceChecks)
          for (int t = 0; t < 2; ++t)
            for (int b = 0; b < 2; ++b)
              ok = ok && check_tma(ck, sb + L::OFF_K + t * L::KT + b * 16384, 16384, k_full, b * 64, D,
                                   k0, NK, kBlockN, bh, BH, __LINE__);
        if (ok) {
          mbar_arrive_expect_tx(k_full, 2 * L::KT);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_load_3d(sb + L::OFF_K + t * L::KT + b * 16384, t == 0 ? &tm_k1 : &tm_k2, k_full,
                          b * 64, k0, bh);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (; ok && j < n; ++j) {
        const int s = j % L::STAGES;
        const int q0 = (qs0 + j) * STEP;
        // this lane's table entries (query rows q0 + lane + 32 e), loaded before the wait
        float4 ce[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = q0 + lane + 32 * e;
          ce[e] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (q < NQ) {
            const size_t o = static_cast<size_t>(bh) * NQ + q;
            const float l1 = lse1_in[o], l2 = lse2_in[o];
            ce[e] = make_float4(-l1 * kLog2e, -l2 * kLog2e, g_in[o] * scale, -(l1 - l2 + kl_in[o]));
          }
        }
        bool good = true;
        if (lane == 0) good = wait_bounded(q_empty(s), ((j / L::STAGES) & 1) ^ 1, wc);
        if (!(ok = __shfl_sync(0xffffffffu, good, 0))) break;
        float* ts = tab + s * 4 * STEP;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = lane + 32 * e;
          ts[q] = ce[e].x;
          ts[STEP + q] = ce[e].y;
          ts[2 * STEP + q] = ce[e].z;
          ts[3 * STEP + q] = ce[e].w;
        }
        __syncwarp();  // the arrive below publishes the whole warp's entries
        if (lane == 0) {
          const uint32_t dst = sb + L::OFF_Q + s * 2 * L::QT;
          if (kDeviceChecks)
            for (int t = 0; t < 2; ++t)
              for (int b = 0; b < 2; ++b)
                good = good && check_tma(ck, dst + t * L::QT + b * 8192, 8192, q_full(s), b * 64, D, q0,
                                         NQ, STEP, bh, BH, __LINE__);
          if (good) {
            mbar_arrive_expect_tx(q_full(s), 2 * L::QT);
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
              for (int b = 0; b < 2; ++b)
                tma_load_3d(dst + t * L::QT + b * 8192, t == 0 ? &tm_q1 : &tm_q2, q_full(s), b * 64,
                            q0, bh);
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, good, 0))) break;
      }
      // let every copy this thread issued land before the CTA can exit
      if (lane == 0) {
        wait_drain(k_full, 0, timeout_ns);
        for (int i = max(0, j - L::STAGES); i < j; ++i)
          wait_drain(q_full(i % L::STAGES), (i / L::STAGES) & 1, timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      // the whole of TMEM is this CTA's, so its base address is 0; a
      // compile-time base keeps the MMA operand addresses constants (checked
      // in every build: a nonzero base stops the CTA with a device-check
      // status instead of issuing MMAs to the wrong columns)
      constexpr uint32_t tmem = 0;
      const bool base_zero = *tmem_slot == 0u;
      if (!base_zero) {
        *abort_flag = 1;
        atomicCAS(dev_status, 0, kStatusDeviceCheck);
      }
      constexpr uint32_t id_t = idesc_bf16(kBlockN, STEP, 0, 0);  // T = K Q^T
      constexpr uint32_t id_dk = idesc_bf16(kBlockN, D, 0, 1);    // dK = dS Q
      constexpr uint32_t id_dq = idesc_bf16(D, STEP, 1, 1);       // dQ^T = K^T dS
      bool ok = check_tmem(ck, tmem + L::COL_T, 128, 2 * STEP, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DK, 128, L::NSETS * D, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DQ, 128, L::NSETS * STEP, __LINE__) &&
                (!L::KTM || check_tmem(ck, tmem + L::COL_K, 128, D, __LINE__)) &&
                base_zero && wait_bounded(k_full, 0, wc) && (!L::KTM || wait_bounded(kt_full, 0, wc));
      const uint32_t k1s = sb + L::OFF_K, k2s = k1s + L::KT;
      // T of step j: two K-major GEMMs (A = K tile, B = Q tile), k-steps interleaved
      auto issue_t = [&](int j) {
        const uint32_t qs = sb + L::OFF_Q + (j % L::STAGES) * 2 * L::QT;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32, qo = (k >> 2) * 8192 + (k & 3) * 32;
          if constexpr (L::KTM) {
            mma_bf16_ts(tmem + L::COL_T, tmem + L::COL_K + 8 * k, smem_desc_sw128(qs + qo, 16, 1024), id_t,
                        k > 0);
            mma_bf16_ts(tmem + L::COL_T + STEP, tmem + L::COL_K + D / 2 + 8 * k,
                        smem_desc_sw128(qs + L::QT + qo, 16, 1024), id_t, k > 0);
          } else {
            mma_bf16(tmem + L::COL_T, smem_desc_sw128(k1s + ko, 16, 1024),
                     smem_desc_sw128(qs + qo, 16, 1024), id_t, k > 0);
            mma_bf16(tmem + L::COL_T + STEP, smem_desc_sw128(k2s + ko, 16, 1024),
                     smem_desc_sw128(qs + L::QT + qo, 16, 1024), id_t, k > 0);
          }
        }
        mma_commit(t_full);
      };
      bool t_issued = false;  // T of step j already issued
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % L::STAGES;
        if (!t_issued) {
          if (!(ok = wait_bounded(q_full(s), (j / L::STAGES) & 1, wc))) break;
          if (j > 0 && !(ok = wait_bounded(t_free, (j - 1) & 1, wc))) break;
          tc_fence_after();
          issue_t(j);
        }
        // the gradient GEMMs of step j once its dS is in shared memory; T of
        // step j+1 goes in whenever its Q tile has landed and T of step j has
        // been loaded (the softmax warps need it before they need this dQ)
        t_issued = false;
        const int sn = (j + 1) % L::STAGES;
        const uint32_t phn = ((j + 1) / L::STAGES) & 1;
        auto try_next = [&]() {
          if (j + 1 < n && !t_issued && mbar_test_wait(q_full(sn), phn) && mbar_test_wait(t_free, j & 1)) {
            tc_fence_after();
            issue_t(j + 1);
            t_issued = true;
          }
        };
        if (!(ok = wait_bounded_idle(ds_full, j & 1, wc, try_next))) break;
        tc_fence_after();
        const uint32_t qs = sb + L::OFF_Q + s * 2 * L::QT;
        // dK_t += dS_t Q_t: A = dS (K-major, one 64-query box), B = Q_t
        // (MN-major: the two 64-column boxes of d are 8 KB apart)
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          const bool set2 = HAS2 && t == 0;
          const uint32_t ds = sb + L::OFF_DS + t * L::DST;
          const uint32_t qt = qs + (set2 ? L::QT : 0);
#pragma unroll
          for (int kk = 0; kk < STEP / 16; ++kk)
            mma_bf16(tmem + L::COL_DK + t * D, smem_desc_sw128(ds + kk * 32, 16, 1024),
                     smem_desc_sw128(qt + kk * 2048, 8192, 1024), id_dk, (j > 0 || kk > 0));
        }
        mma_commit(q_empty(s));
        try_next();
        // dQ_t^T = K_t^T dS_t: A = K^T (MN-major: the two 64-column boxes of
        // d are 16 KB apart), B = dS (MN-major); the previous step's dQ^T has
        // been read out of TMEM
        if (j > 0 && !(ok = wait_bounded_idle(dq_free, (j - 1) & 1, wc, try_next))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          const bool set2 = HAS2 && t == 0;
          const uint32_t ds = sb + L::OFF_DS + t * L::DST;
          const uint32_t kts = set2 ? k2s : k1s;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_bf16(tmem + L::COL_DQ + t * STEP, smem_desc_sw128(kts + kk * 2048, 16384, 1024),
                     smem_desc_sw128(ds + kk * 2048, 8192, 1024), id_dq, kk > 0);
        }
        mma_commit(dq_full);
      }
      mma_commit(dk_full);  // after every MMA of this CTA (dK complete)
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    }
  } else if (warp == kF2StoreWarp) {
    // ------------------------------------------------------------ TMA reductions / stores
    if (lane == 0 && n > 0) {
      bool ok = true;
      int u = 0;  // staging uses so far
      // after issuing the copies of use u: the tile of use u - (NSTG - 1) has
      // been read (at most NSTG - 1 copy groups still reading) and may be
      // written again
      auto release_stage = [&](int uu) {
        bulk_commit_group();
        if constexpr (NSTG == 2) {
          bulk_wait_read_le1();
          if (uu >= 1) mbar_arrive(stg_empty_b(uu - 1));
        } else {
          bulk_wait_read_all();
          mbar_arrive(stg_empty_b(uu));
        }
      };
      for (int j = 0; ok && j < n; ++j) {
        const int q0 = (qs0 + j) * STEP;
        for (int t = 0; t < L::NSETS; ++t, ++u) {
          if (!(ok = wait_bounded(stg_full_b(u), (u / NSTG) & 1, wc))) break;
          if (!(ok = dcheck(ck, q0 < NQ && bh < BH, __LINE__))) break;
          const CUtensorMap* m = (HAS2 && t == 0) ? &tm_dq2 : &tm_dq1;
          // rows past N_Q (the last step's tail) are not reduced into
#pragma unroll
          for (int b = 0; b < D / 32; ++b) tma_reduce_add_3d(m, stg_tile(u) + b * 8192, b * 32, q0, bh);
          release_stage(u);
        }
      }
      // dK rows of each set, through the same staging tile
      for (int t = 0; ok && t < L::NSETS; ++t, ++u) {
        if (!(ok = wait_bounded(stg_full_b(u), (u / NSTG) & 1, wc))) break;
        if (!(ok = dcheck(ck, k0 < NK && bh < BH, __LINE__))) break;
        const CUtensorMap* m = (HAS2 && t == 0) ? &tm_dk2 : &tm_dk1;
        tma_store_3d(m, stg_tile(u), 0, k0, bh);
        tma_store_3d(m, stg_tile(u) + 16384, 64, k0, bh);
        release_stage(u);
      }
      bulk_wait_all();  // every reduction and store is in global memory before the CTA exits
    }
  } else {
    // ------------------------------------------------------------ softmax / read-outs
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row of T and dK (TMEM lane); d column of dQ^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const int key = k0 + r;
    const int qlo = causal ? key - off : 0;  // queries >= qlo see this key (all, when non-causal)
    bool ok = true;
    int u = 0;  // staging uses so far
    // staging tile u % NSTG is free again (the store warp has read use u - NSTG)
    auto stage_free = [&]() {
      return u < NSTG || __all_sync(0xffffffffu, wait_bounded(stg_empty_b(u), (u / NSTG - 1) & 1, wc));
    };
    // dQ^T of step j (thread = d column r, queries [16 grp, 16 grp + 16)) ->
    // staging rows q, fp32 (box r/32 of 32 columns x 64 rows, 4-byte slot r%32
    // of the row, 16-byte chunks swizzled by the row) -> TMA reduction
    auto read_dq = [&](int j) {
      if (!__all_sync(0xffffffffu, wait_bounded(dq_full, j & 1, wc))) return false;
      tc_fence_after();
      const int cb = (r & 31) * 4;  // byte of this column within a 128-byte row
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t, ++u) {
        float v[16];
        if (!check_tmem(ck, tmem + lane_off + L::COL_DQ + t * STEP + grp * 16, 32, 16, __LINE__))
          return false;
        tmem_ld16(tmem + lane_off + L::COL_DQ + t * STEP + grp * 16, v);
        tmem_wait_ld();
        if (t + 1 == L::NSETS) {  // the next step's dQ^T GEMMs may overwrite this dQ^T
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dq_free);
        }
        if (!stage_free()) return false;
        const uint32_t col = stg_tile(u) + static_cast<uint32_t>((r >> 5) * 8192);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int q = grp * 16 + k;
          st_shared_b32(col + q * 128 + ((((cb >> 4) ^ (q & 7))) << 4) + (cb & 15), __float_as_uint(v[k]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full_b(u));
      }
      return true;
    };
    if constexpr (L::KTM) {
      // K1, K2 row r into TMEM lane r: this thread's 32 d values of each (the
      // 64-column box grp/2, 16-byte chunks 4 (grp%2) .. +4 of the swizzled
      // row) -> packed columns [16 grp, +16)
      if (n > 0 && (ok = __all_sync(0xffffffffu, wait_bounded(k_full, 0, wc)) &&
                         check_tmem(ck, tmem + lane_off + L::COL_K + 16 * grp, 32, D / 2 + 16, __LINE__))) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t rowk = sb + L::OFF_K + t * L::KT + static_cast<uint32_t>((grp >> 1) * 16384 + r * 128);
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ld_shared_v4(rowk + (((4 * (grp & 1) + q) ^ (r & 7)) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                         w[4 * q + 3]);
          tmem_st_cols<16>(tmem + lane_off + L::COL_K + t * (D / 2) + 16 * grp, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(kt_full);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      const int s = j % L::STAGES;
      const int q0 = (qs0 + j) * STEP + grp * 16;  // this thread's first query column
      // the stage's Q barrier also publishes its constant table; its phase
      // completed before these T GEMMs were issued
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(q_full(s), (j / L::STAGES) & 1, wc) &&
                                             wait_bounded(t_full, j & 1, wc))))
        break;
      if (!(ok = check_tmem(ck, tmem + lane_off + L::COL_T + grp * 16, 32, 16, __LINE__) &&
                 check_tmem(ck, tmem + lane_off + L::COL_T + STEP + grp * 16, 32, 16, __LINE__)))
        break;
      tc_fence_after();
      float a[16], b[16];
      tmem_ld16(tmem + lane_off + L::COL_T + grp * 16, a);
      tmem_ld16(tmem + lane_off + L::COL_T + STEP + grp * 16, b);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(t_free);
      // visible (key, query) pairs of this thread's 16 columns
      const bool full = key < NK && q0 >= qlo && q0 + 16 <= NQ;
      const float* tq = tab + s * 4 * STEP + grp * 16;
      uint32_t d2p[8], d1p[8];
      const float2 c2 = make_float2(c, c), sc2 = make_float2(scale, scale);
      const float2 m1 = make_float2(-1.f, -1.f);
      float4 q1c, q2c, qgc, qec;  // 4 columns of each constant, one 16-byte load each
#pragma unroll
      for (int k = 0; k < 16; k += 2) {
        const bool lo = (k & 3) == 0;
        if (lo) {
          q1c = *reinterpret_cast<const float4*>(tq + k);
          q2c = *reinterpret_cast<const float4*>(tq + STEP + k);
          qgc = *reinterpret_cast<const float4*>(tq + 2 * STEP + k);
          if (HAS1) qec = *reinterpret_cast<const float4*>(tq + 3 * STEP + k);
        }
        const float2 nb1 = lo ? make_float2(q1c.x, q1c.y) : make_float2(q1c.z, q1c.w);
        const float2 nb2 = lo ? make_float2(q2c.x, q2c.y) : make_float2(q2c.z, q2c.w);
        const float2 gs = lo ? make_float2(qgc.x, qgc.y) : make_float2(qgc.z, qgc.w);
        const float2 s1 = make_float2(a[k], a[k + 1]), s2 = make_float2(b[k], b[k + 1]);
        const float2 x1 = __ffma2_rn(s1, c2, nb1);
        float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
        float2 p2 = p1;
        if constexpr (HAS2) {
          const float2 x2 = __ffma2_rn(s2, c2, nb2);
          p2 = make_float2(ex2(x2.x), ex2(x2.y));
        }
        if (!full) {
          const bool v0 = key < NK && q0 + k < NQ && q0 + k >= qlo;
          const bool v1 = key < NK && q0 + k + 1 < NQ && q0 + k + 1 >= qlo;
          if (!v0) p1.x = p2.x = 0.f;
          if (!v1) p1.y = p2.y = 0.f;
        }
        if constexpr (HAS2) {
          const float2 d2 = __fmul2_rn(__ffma2_rn(p1, m1, p2), gs);  // g (P2 - P1)
          d2p[k >> 1] = pack_bf16x2(d2.x, d2.y);
        }
        if constexpr (HAS1) {
          const float2 ne = lo ? make_float2(qec.x, qec.y) : make_float2(qec.z, qec.w);
          // g P1 (log(P1/P2) - KL), log(P1/P2) - KL = scale (s1 - s2) - e
          const float2 lr = __ffma2_rn(__ffma2_rn(s2, m1, s1), sc2, ne);
          const float2 d1 = __fmul2_rn(__fmul2_rn(p1, gs), lr);
          d1p[k >> 1] = pack_bf16x2(d1.x, d1.y);
        }
      }
      // the previous step's gradient GEMMs have read the dS tiles
      if (j > 0 && !(ok = __all_sync(0xffffffffu, wait_bounded(dq_full, (j - 1) & 1, wc)))) break;
      // row r of each dS tile: 128 bytes = 64 queries; this thread's 32 bytes
      // are 16-byte chunks 2 grp and 2 grp + 1, swizzled by the row
      const uint32_t row = sb + L::OFF_DS + static_cast<uint32_t>(r * 128);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        const uint32_t* v = (HAS2 && t == 0) ? d2p : d1p;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          st_shared_v4(row + t * L::DST + (((2 * grp + h) ^ (r & 7)) << 4), v[4 * h], v[4 * h + 1],
                       v[4 * h + 2], v[4 * h + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      // the previous step's dQ out, while this step's gradient GEMMs run
      if (j > 0 && !(ok = read_dq(j - 1))) break;
    }
    if (ok && n > 0) ok = read_dq(n - 1);
    // dK rows (thread = key row r, d columns [32 grp, 32 grp + 32)) -> the
    // staging tile as bf16 (box grp/2 of 64 columns x 128 rows, 16-byte
    // chunks 4 (grp%2) .. +4 of the row) -> the store warp's TMA stores
    if (ok && n > 0 && __all_sync(0xffffffffu, wait_bounded(dk_full, 0, wc))) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t, ++u) {
        const uint32_t row = stg_tile(u) + static_cast<uint32_t>((grp >> 1) * 16384 + r * 128);
        float v[32];
        if (!check_tmem(ck, tmem + lane_off + L::COL_DK + t * D + grp * 32, 32, 32, __LINE__)) break;
        tmem_ld32(tmem + lane_off + L::COL_DK + t * D + grp * 32, v);
        tmem_wait_ld();
        if (!stage_free()) break;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(row + (((4 * (grp & 1) + q) ^ (r & 7)) << 4), pack_bf16x2(v[8 * q], v[8 * q + 1]),
                       pack_bf16x2(v[8 * q + 2], v[8 * q + 3]), pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                       pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full_b(u));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int SETS>
cudaError_t launch_fused128_t(const BwdArgs& a, cudaStream_t stream) {
  using L = Fused128Layout<SETS>;
  auto kern = streamkl_bwd_fused128_kernel<SETS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  if (!a.tm_dq2 || !a.tm_dq1 || !a.tm_dk2 || !a.tm_dk1) return cudaErrorInvalidValue;
  dim3 grid((a.NK + kBlockN - 1) / kBlockN, a.BH, 1);
  kern<<<grid, kF2Threads, L::ALLOC, stream>>>(*a.tm_q1, *a.tm_k1, *a.tm_q2, *a.tm_k2, *a.tm_dq2,
                                               *a.tm_dq1, *a.tm_dk2, *a.tm_dk1, a.NQ, a.NK, a.causal,
                                               a.scale, a.BH, a.kl, a.lse1, a.lse2, a.g, a.dev_status,
                                               a.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused128(const BwdArgs& a, cudaStream_t stream) {
  if (a.d != kF2D) return cudaErrorInvalidValue;
  return a.grad1 ? launch_fused128_t<kSet1 | kSet2>(a, stream) : launch_fused128_t<kSet2>(a, stream);
}

}  // namespace skl

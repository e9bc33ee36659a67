// Fused backward at d = 64 (gist.science technical summary, "Metodologia"
// section 2, kernel fusion paragraph: one kernel visits every (query tile, key
// tile) pair once and accumulates dQ across key tiles with atomics).
// Probabilities are regenerated tile by tile from Q, K and the saved LSEs,
// P_t = exp(S_t - LSE_t).
//
// At d = 64 a (query, key) pair costs half the tensor work of d = 128 for the
// same two exponentials, so the separate dK and dQ kernels, which each
// regenerate P1, P2 and dS, are bound by that softmax work. Here it is done
// once per pair. CTA = one (batch-head, 128-key tile); it sweeps the 128-row
// query blocks that see its keys (causal: from the diagonal down):
//   T_t   = K_t Q_t^T         (M = 128 keys, N = 128 queries, K = d)
//   dS_t  from T_t            (softmax warps; bf16 to shared memory, row = key)
//   dK_t += dS_t Q_t          (M = 128 keys, N = d, K = 128 queries; TMEM)
//   dQ_t  = dS_t^T K_t        (M = 128 queries, N = d, K = 128 keys; TMEM)
// Each query block's dQ_t goes from TMEM through a shared-memory staging tile
// (128-byte swizzle) and a TMA bulk reduction (add) into the fp32 accumulator
// [BH][N_Q][d] (zeroed by the caller), one 128-byte line per row piece; dK
// leaves once at the end through the same staging and TMA stores.
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
// g = (w-2)/4 (T: thread = key row, query columns [32g, 32g+32); dQ read-out:
// thread = query row, d columns [16g, 16g+16); dK read-out: thread = key row,
// d columns [16g, 16g+16)); 18 = TMA reductions and stores (lane 0).
// TMEM: T1 [0,128) T2 [128,256) | dK per set (64 columns) | dQ per set.
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kFuThreads = 608;  // 19 warps
constexpr int kFuSoftmaxWarps = 16;
constexpr int kFuStoreWarp = 18;
constexpr int kFuD = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSet2 = 1, kSet1 = 2;

template <int SETS>
struct FusedLayout {
  static constexpr int NSETS = SETS == (kSet1 | kSet2) ? 2 : 1;
  static constexpr int TILE = kBlockM * kFuD * 2;      // 128 rows x 128 B (one box)
  static constexpr int STAGES = NSETS == 2 ? 2 : 3;    // Q1, Q2 stages
  static constexpr int DST = kBlockN * kBlockM * 2;    // one dS tile: 128 key rows x 256 B
  static constexpr int STG = kBlockM * kFuD * 4;       // one set's fp32 dQ rows: 2 boxes of 16 KB
  static constexpr int TAB = 4 * kBlockM * 4;          // per stage: 4 x 128 floats
  static constexpr int OFF_K = 0;                      // K1, K2
  static constexpr int OFF_Q = 2 * TILE;               // stage s: Q1 at +2s TILE, Q2 at +(2s+1) TILE
  static constexpr int OFF_DS = OFF_Q + STAGES * 2 * TILE;  // slot t: the t-th computed set
  static constexpr int OFF_STG = OFF_DS + NSETS * DST;
  static constexpr int OFF_TAB = OFF_STG + STG;
  static constexpr int OFF_BAR = OFF_TAB + STAGES * TAB;
  // k_full, q_full[S], q_empty[S], t_full, t_free, ds_full, dq_full, dq_free,
  // dk_full, stg_full, stg_empty, dke_full, drain, kt_full
  static constexpr int NBAR = 1 + 2 * STAGES + 11;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr uint32_t COL_T = 0, COL_DK = 256, COL_DQ = 256 + NSETS * kFuD;
  // one gradient set: K1, K2 also in TMEM (32 packed columns each), the A
  // operand of the T GEMMs, which then read only Q from shared memory
  static constexpr bool KTM = NSETS == 1;
  static constexpr uint32_t COL_K = COL_DQ + NSETS * kFuD;
  static_assert(COL_K + (KTM ? kFuD : 0) <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(OFF_Q % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_STG % 1024 == 0,
                "swizzled tiles on 1024-byte boundaries");
};

template <int SETS>
__global__ void __launch_bounds__(kFuThreads, 1)
    streamkl_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q1,
                              const __grid_constant__ CUtensorMap tm_k1,
                              const __grid_constant__ CUtensorMap tm_q2,
                              const __grid_constant__ CUtensorMap tm_k2,
                              const __grid_constant__ CUtensorMap tm_dq2,
                              const __grid_constant__ CUtensorMap tm_dq1,
                              const __grid_constant__ CUtensorMap tm_dk2,
                              const __grid_constant__ CUtensorMap tm_dk1, int NQ, int NK,
                              int causal, float scale, int BH, const float* __restrict__ kl_in,
                              const float* __restrict__ lse1_in, const float* __restrict__ lse2_in,
                              const float* __restrict__ g_in, int* dev_status, uint64_t timeout_ns) {
  using L = FusedLayout<SETS>;
  constexpr bool HAS2 = SETS & kSet2, HAS1 = SETS & kSet1;
  constexpr int D = kFuD;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kt = static_cast<int>(blockIdx.x);  // key tile (causal: key tile 0 is the heaviest)
  const int bh = static_cast<int>(blockIdx.y);
  const int off = NK - NQ;                      // causal: key j visible to query i iff j <= i + off
  const int k0 = kt * kBlockN;
  const int nqb = (NQ + kBlockM - 1) / kBlockM;
  // query blocks with a row that sees some key of this tile
  const int qb0 = causal ? max(0, k0 - off) / kBlockM : 0;
  int n = (k0 < NK && !(causal && NQ > NK)) ? max(0, nqb - qb0) : 0;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t k_full = bar0;
  auto q_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto q_empty = [&](int s) { return bar0 + 8u * (1 + L::STAGES + s); };
  const uint32_t t_full = bar0 + 8u * (1 + 2 * L::STAGES);
  const uint32_t t_free = t_full + 8, ds_full = t_full + 16;
  // dq_full: the step's dQ GEMMs, the last readers of its dS tiles, are done
  // (one commit serves both: a commit costs the tensor pipe about as much as
  // an MMA)
  const uint32_t dq_full = t_full + 24, dq_free = t_full + 32, dk_full = t_full + 40;
  const uint32_t stg_full = t_full + 48, stg_empty = t_full + 56, dke_full = t_full + 64;
  const uint32_t drain = t_full + 72, kt_full = t_full + 80;
  static_assert(1 + 2 * L::STAGES + 11 == L::NBAR, "barrier region holds every barrier");
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
               check_bar(ck, drain, __LINE__);
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
      mbar_init(t_free, kFuSoftmaxWarps);
      mbar_init(ds_full, kFuSoftmaxWarps);
      mbar_init(dq_full, 1);
      mbar_init(dq_free, kFuSoftmaxWarps);
      mbar_init(dk_full, 1);
      mbar_init(stg_full, kFuSoftmaxWarps);
      mbar_init(stg_empty, 1);
      mbar_init(dke_full, kFuSoftmaxWarps);
      mbar_init(drain, 1);
      mbar_init(kt_full, kFuSoftmaxWarps);
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
          ok = check_tma(ck, sb + L::OFF_K, L::TILE, k_full, 0, D, k0, NK, kBlockN, bh, BH, __LINE__) &&
               check_tma(ck, sb + L::OFF_K + L::TILE, L::TILE, k_full, 0, D, k0, NK, kBlockN, bh, BH,
                         __LINE__);
        if (ok) {
          mbar_arrive_expect_tx(k_full, 2 * L::TILE);
          tma_load_3d(sb + L::OFF_K, &tm_k1, k_full, 0, k0, bh);
          tma_load_3d(sb + L::OFF_K + L::TILE, &tm_k2, k_full, 0, k0, bh);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (; ok && j < n; ++j) {
        const int s = j % L::STAGES;
        const int q0 = (qb0 + j) * kBlockM;
        // this lane's table entries (query rows q0 + lane + 32 e), loaded before the wait
        float4 ce[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
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
        float* ts = tab + s * 4 * kBlockM;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = lane + 32 * e;
          ts[q] = ce[e].x;
          ts[kBlockM + q] = ce[e].y;
          ts[2 * kBlockM + q] = ce[e].z;
          ts[3 * kBlockM + q] = ce[e].w;
        }
        __syncwarp();  // the arrive below publishes the whole warp's entries
        if (lane == 0) {
          const uint32_t dst = sb + L::OFF_Q + s * 2 * L::TILE;
          if (kDeviceChecks)
            good = check_tma(ck, dst, L::TILE, q_full(s), 0, D, q0, NQ, kBlockM, bh, BH, __LINE__) &&
                   check_tma(ck, dst + L::TILE, L::TILE, q_full(s), 0, D, q0, NQ, kBlockM, bh, BH,
                             __LINE__);
          if (good) {
            mbar_arrive_expect_tx(q_full(s), 2 * L::TILE);
            tma_load_3d(dst, &tm_q1, q_full(s), 0, q0, bh);
            tma_load_3d(dst + L::TILE, &tm_q2, q_full(s), 0, q0, bh);
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
      constexpr uint32_t id_t = idesc_bf16(kBlockN, kBlockM, 0, 0);  // T = K Q^T
      constexpr uint32_t id_dk = idesc_bf16(kBlockN, D, 0, 1);       // dK = dS Q
      constexpr uint32_t id_dq = idesc_bf16(kBlockM, D, 1, 1);       // dQ = dS^T K
      bool ok = check_tmem(ck, tmem + L::COL_T, 128, 256, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DK, 128, L::NSETS * D, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DQ, 128, L::NSETS * D, __LINE__) &&
                (!L::KTM || check_tmem(ck, tmem + L::COL_K, 128, D, __LINE__)) &&
                wait_bounded(k_full, 0, wc) && (!L::KTM || wait_bounded(kt_full, 0, wc));
      const uint32_t k1s = sb + L::OFF_K, k2s = k1s + L::TILE;
      // T of step j: two K-major GEMMs (A = K tile, B = Q tile), k-steps interleaved
      auto issue_t = [&](int j) {
        const uint32_t qs = sb + L::OFF_Q + (j % L::STAGES) * 2 * L::TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          if constexpr (L::KTM) {
            mma_bf16_ts(tmem + L::COL_T, tmem + L::COL_K + 8 * k, smem_desc_sw128(qs + k * 32, 16, 1024),
                        id_t, k > 0);
            mma_bf16_ts(tmem + L::COL_T + 128, tmem + L::COL_K + D / 2 + 8 * k,
                        smem_desc_sw128(qs + L::TILE + k * 32, 16, 1024), id_t, k > 0);
          } else {
            mma_bf16(tmem + L::COL_T, smem_desc_sw128(k1s + k * 32, 16, 1024),
                     smem_desc_sw128(qs + k * 32, 16, 1024), id_t, k > 0);
            mma_bf16(tmem + L::COL_T + 128, smem_desc_sw128(k2s + k * 32, 16, 1024),
                     smem_desc_sw128(qs + L::TILE + k * 32, 16, 1024), id_t, k > 0);
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
        // the gradient GEMMs of step j once its dS is in shared memory; while
        // the softmax warps still compute it, T of step j+1 goes in if its Q
        // tile has landed and T of step j has been loaded
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
        const uint32_t qs = sb + L::OFF_Q + s * 2 * L::TILE;
        // dK_t += dS_t Q_t: A = dS (K-major, two 64-query boxes), B = Q_t (MN-major)
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          const bool set2 = HAS2 && t == 0;
          const uint32_t ds = sb + L::OFF_DS + t * L::DST;
          const uint32_t qt = qs + (set2 ? L::TILE : 0);
#pragma unroll
          for (int kk = 0; kk < kBlockM / 16; ++kk)
            mma_bf16(tmem + L::COL_DK + t * D,
                     smem_desc_sw128(ds + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                     smem_desc_sw128(qt + kk * 2048, 8192, 1024), id_dk, (j > 0 || kk > 0));
        }
        mma_commit(q_empty(s));
        // dQ_t = dS_t^T K_t: A = dS^T (MN-major), B = K_t (MN-major); the
        // previous step's dQ has been read out of TMEM (T of step j+1 still
        // goes in first if it can: the softmax warps need it sooner)
        try_next();
        if (j > 0 && !(ok = wait_bounded_idle(dq_free, (j - 1) & 1, wc, try_next))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          const bool set2 = HAS2 && t == 0;
          const uint32_t ds = sb + L::OFF_DS + t * L::DST;
          const uint32_t kts = set2 ? k2s : k1s;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_bf16(tmem + L::COL_DQ + t * D, smem_desc_sw128(ds + kk * 2048, 16384, 1024),
                     smem_desc_sw128(kts + kk * 2048, 8192, 1024), id_dq, kk > 0);
        }
        mma_commit(dq_full);
      }
      mma_commit(dk_full);  // after every MMA of this CTA (dK complete, dS no longer read)
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    }
  } else if (warp == kFuStoreWarp) {
    // ------------------------------------------------------------ TMA reductions / stores
    if (lane == 0 && n > 0) {
      bool ok = true;
      int u = 0;  // staging uses so far
      for (int j = 0; ok && j < n; ++j) {
        const int q0 = (qb0 + j) * kBlockM;
        for (int t = 0; t < L::NSETS; ++t, ++u) {
          if (!(ok = wait_bounded(stg_full, u & 1, wc))) break;
          if (!(ok = dcheck(ck, q0 < NQ && bh < BH, __LINE__))) break;
          const CUtensorMap* m = (HAS2 && t == 0) ? &tm_dq2 : &tm_dq1;
          // rows past N_Q (the last block's tail) are not reduced into
          tma_reduce_add_3d(m, sb + L::OFF_STG, 0, q0, bh);
          tma_reduce_add_3d(m, sb + L::OFF_STG + 16384, 32, q0, bh);
          bulk_commit_group();
          bulk_wait_read_all();  // the staging tile may be written again
          mbar_arrive(stg_empty);
        }
      }
      // dK rows, staged in the dS tiles once every MMA has run
      if (ok && (ok = wait_bounded(dke_full, 0, wc)) && dcheck(ck, k0 < NK && bh < BH, __LINE__)) {
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t)
          tma_store_3d((HAS2 && t == 0) ? &tm_dk2 : &tm_dk1, sb + L::OFF_DS + t * L::DST, 0, k0, bh);
        bulk_commit_group();
      }
      bulk_wait_all();  // every reduction and store is in global memory before the CTA exits
    }
  } else {
    // ------------------------------------------------------------ softmax / read-outs
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row of T and dK (TMEM lane); query row of dQ
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const int key = k0 + r;
    const int qlo = causal ? key - off : 0;  // queries >= qlo see this key (all, when non-causal)
    bool ok = true;
    int u = 0;  // staging uses so far
    // dQ of step j (thread = query row r, d columns [16 grp, 16 grp + 16)) ->
    // staging tile (box grp/2, 16-byte chunks 4 (grp%2) .. +4 of the row) ->
    // the store warp's TMA reduction
    auto read_dq = [&](int j) {
      if (!__all_sync(0xffffffffu, wait_bounded(dq_full, j & 1, wc))) return false;
      tc_fence_after();
      const uint32_t srow = sb + L::OFF_STG + static_cast<uint32_t>((grp >> 1) * 16384 + r * 128);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t, ++u) {
        float v[16];
        if (!check_tmem(ck, tmem + lane_off + L::COL_DQ + t * D + grp * 16, 32, 16, __LINE__))
          return false;
        tmem_ld16(tmem + lane_off + L::COL_DQ + t * D + grp * 16, v);
        tmem_wait_ld();
        if (t + 1 == L::NSETS) {  // the next step's dQ GEMMs may overwrite this dQ
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dq_free);
        }
        if (u > 0 && !__all_sync(0xffffffffu, wait_bounded(stg_empty, (u - 1) & 1, wc))) return false;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(srow + (((4 * (grp & 1) + q) ^ (r & 7)) << 4), __float_as_uint(v[4 * q]),
                       __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                       __float_as_uint(v[4 * q + 3]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full);
      }
      return true;
    };
    if constexpr (L::KTM) {
      // K1, K2 row r into TMEM lane r: this thread's 16 d values of each (16-byte
      // chunks 2 grp, 2 grp + 1 of the swizzled row) -> packed columns [8 grp, +8)
      if (n > 0 && (ok = __all_sync(0xffffffffu, wait_bounded(k_full, 0, wc)) &&
                         check_tmem(ck, tmem + lane_off + L::COL_K + 8 * grp, 32, D / 2 + 8, __LINE__))) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t rowk = sb + L::OFF_K + t * L::TILE + static_cast<uint32_t>(r * 128);
          uint32_t w[8];
          ld_shared_v4(rowk + (((2 * grp) ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
          ld_shared_v4(rowk + (((2 * grp + 1) ^ (r & 7)) << 4), w[4], w[5], w[6], w[7]);
          tmem_st_cols<8>(tmem + lane_off + L::COL_K + t * (D / 2) + 8 * grp, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(kt_full);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      const int s = j % L::STAGES;
      const int q0 = (qb0 + j) * kBlockM + grp * 32;  // this thread's first query column
      // the stage's Q barrier also publishes its constant table; its phase
      // completed before these T GEMMs were issued
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(q_full(s), (j / L::STAGES) & 1, wc) &&
                                             wait_bounded(t_full, j & 1, wc))))
        break;
      if (!(ok = check_tmem(ck, tmem + lane_off + L::COL_T + grp * 32, 32, 32, __LINE__) &&
                 check_tmem(ck, tmem + lane_off + L::COL_T + 128 + grp * 32, 32, 32, __LINE__)))
        break;
      tc_fence_after();
      float a[32], b[32];
      tmem_ld32(tmem + lane_off + L::COL_T + grp * 32, a);
      tmem_ld32(tmem + lane_off + L::COL_T + 128 + grp * 32, b);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(t_free);
      // visible (key, query) pairs of this thread's 32 columns
      const bool full = key < NK && q0 >= qlo && q0 + 32 <= NQ;
      const float* tq = tab + s * 4 * kBlockM + grp * 32;
      uint32_t d2p[16], d1p[16];
      const float2 c2 = make_float2(c, c), sc2 = make_float2(scale, scale);
      const float2 m1 = make_float2(-1.f, -1.f);
      float4 q1c, q2c, qgc, qec;  // 4 columns of each constant, one 16-byte load each
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const bool lo = (k & 3) == 0;
        if (lo) {
          q1c = *reinterpret_cast<const float4*>(tq + k);
          q2c = *reinterpret_cast<const float4*>(tq + kBlockM + k);
          qgc = *reinterpret_cast<const float4*>(tq + 2 * kBlockM + k);
          if (HAS1) qec = *reinterpret_cast<const float4*>(tq + 3 * kBlockM + k);
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
      // row r of each dS tile: 256 bytes = 128 queries in two 64-query boxes;
      // this thread's 64 bytes are 16-byte chunks 4 (grp%2) .. +4 of box grp/2
      const uint32_t row = sb + L::OFF_DS + static_cast<uint32_t>((grp >> 1) * 16384 + r * 128);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        const uint32_t* v = (HAS2 && t == 0) ? d2p : d1p;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(row + t * L::DST + (((4 * (grp & 1) + q) ^ (r & 7)) << 4), v[4 * q], v[4 * q + 1],
                       v[4 * q + 2], v[4 * q + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      // the previous step's dQ out, while this step's gradient GEMMs run
      if (j > 0 && !(ok = read_dq(j - 1))) break;
    }
    if (ok && n > 0) ok = read_dq(n - 1);
    // dK rows (thread = key row r, d columns [16 grp, 16 grp + 16)) -> the dS
    // tiles, free once every MMA has run -> the store warp's TMA stores
    if (ok && n > 0 && __all_sync(0xffffffffu, wait_bounded(dk_full, 0, wc))) {
      tc_fence_after();
      const uint32_t row = sb + L::OFF_DS + static_cast<uint32_t>(r * 128);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        float v[16];
        if (!check_tmem(ck, tmem + lane_off + L::COL_DK + t * D + grp * 16, 32, 16, __LINE__)) break;
        tmem_ld16(tmem + lane_off + L::COL_DK + t * D + grp * 16, v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 2; ++q)
          st_shared_v4(row + t * L::DST + (((2 * grp + q) ^ (r & 7)) << 4), pack_bf16x2(v[8 * q], v[8 * q + 1]),
                       pack_bf16x2(v[8 * q + 2], v[8 * q + 3]), pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                       pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(dke_full);
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
cudaError_t launch_fused_t(const BwdArgs& a, cudaStream_t stream) {
  using L = FusedLayout<SETS>;
  auto kern = streamkl_bwd_fused_kernel<SETS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  if (!a.tm_dq2 || !a.tm_dq1 || !a.tm_dk2 || !a.tm_dk1) return cudaErrorInvalidValue;
  dim3 grid((a.NK + kBlockN - 1) / kBlockN, a.BH, 1);
  kern<<<grid, kFuThreads, L::ALLOC, stream>>>(*a.tm_q1, *a.tm_k1, *a.tm_q2, *a.tm_k2, *a.tm_dq2,
                                               *a.tm_dq1, *a.tm_dk2, *a.tm_dk1, a.NQ, a.NK, a.causal,
                                               a.scale, a.BH, a.kl, a.lse1, a.lse2, a.g, a.dev_status,
                                               a.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused64(const BwdArgs& a, cudaStream_t stream) {
  if (a.d != kFuD) return cudaErrorInvalidValue;
  return a.grad1 ? launch_fused_t<kSet1 | kSet2>(a, stream) : launch_fused_t<kSet2>(a, stream);
}

}  // namespace skl

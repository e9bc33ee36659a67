// Backward pass of the attention-KL primitive (gist.science technical summary,
// "Metodologia" section 2): probabilities are regenerated tile by tile from Q,
// K and the saved LSEs, P_t = exp(S_t - LSE_t); the kernel visits each
// (query tile, key tile) pair once, keeps dK for its key tile in TMEM and
// accumulates dQ in an fp32 buffer with global reductions (the pages' "atomics
// for dQ" choice; the buffer is one head's [N_Q, d] fp32 slice at a time).
//
// Gradients of L = sum_i g_i KL_i, with s = scale * q.k:
//   configuration 1 (teacher P1 fixed):  dS2 = g * (P2 - P1)
//   configuration 2 (student P2 fixed):  dS1 = g * P1 * (log(P1/P2) - KL)
// where log(P1/P2) = (s1 - LSE1) - (s2 - LSE2) is formed from logits and the
// saved LSEs (section 3, numerical stability), never from logs of
// probabilities. dQ_t = scale * dS_t K_t, dK_t = scale * dS_t^T Q_t.
//
// CTA = one (batch*head, 128-key tile); it loops over the 128-row query tiles
// that can see its keys (causal: from the diagonal down).
//   warp 0       TMA: K1/K2 once, Q1/Q2 per query tile through a ring
//   warp 1       TMEM owner + MMA issuer:
//                  S1 = Q1 K1^T, S2 = Q2 K2^T               (M=128 rows, N=128 keys)
//                  dK_t += dS_t^T Q_t   (A, B MN-major)     (M=128 keys, N=d)
//                  dQ_t  = dS_t K_t     (A K-major, B MN)   (M=128 rows, N=d)
//   warps 4..11  thread = query row; warpgroup w owns key columns [64w, 64w+64)
//                of S and dS, and d columns [w d/2, (w+1) d/2) of dQ/dK
//                readouts.
// dS (scale and g folded in) is rounded to bf16 and written to shared memory in
// the 128-byte-swizzled layout that both gradient MMAs read.
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kBwdThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool GRAD1>
struct BwdLayout {
  static constexpr int KB = D / 64;
  static constexpr int TILE = kBlockM * D * 2;
  static constexpr int QSTAGES = (D == 128 && GRAD1) ? 1 : 2;
  static constexpr int DS_TILE = kBlockM * kBlockN * 2;  // 32 KB bf16
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = TILE;
  static constexpr int OFF_Q = 2 * TILE;  // stage s: Q1 at +2s*TILE, Q2 at +(2s+1)*TILE
  static constexpr int OFF_DS2 = OFF_Q + QSTAGES * 2 * TILE;
  static constexpr int OFF_DS1 = OFF_DS2 + DS_TILE;
  static constexpr int OFF_BAR = OFF_DS2 + (GRAD1 ? 2 : 1) * DS_TILE;
  // k_full, q_full[QS], q_empty[QS], s_full, s_free, ds_full, ds_free,
  // dq_full, dq_free, dk_full, drain
  static constexpr int NBAR = 1 + 2 * QSTAGES + 8;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  // TMEM columns
  static constexpr bool ALIAS = (D == 128 && GRAD1);  // dQ reuses S columns
  static constexpr bool DQT = (D == 128);  // dQ held transposed (lanes = d)
  static constexpr uint32_t COL_S1 = 0, COL_S2 = 128;
  static constexpr uint32_t COL_DK2 = 256;
  static constexpr uint32_t COL_DK1 = 256 + D;
  static constexpr uint32_t COL_DQ2 = ALIAS ? COL_S2 : (GRAD1 ? 256 + 2 * D + D : 256 + D);
  static constexpr uint32_t COL_DQ1 = ALIAS ? COL_S1 : 256 + 2 * D;
  static_assert(ALIAS || COL_DQ2 + D <= 512, "TMEM budget");
  static_assert(BYTES + 1024 <= 232448, "shared memory budget");
};

template <int D, bool GRAD1>
__global__ void __launch_bounds__(kBwdThreads, 1)
    streamkl_bwd_kernel(const __grid_constant__ CUtensorMap tm_q1,
                        const __grid_constant__ CUtensorMap tm_k1,
                        const __grid_constant__ CUtensorMap tm_q2,
                        const __grid_constant__ CUtensorMap tm_k2, int NQ, int NK, int causal,
                        float scale, const float* __restrict__ kl_in,
                        const float* __restrict__ lse1_in, const float* __restrict__ lse2_in,
                        const float* __restrict__ g_in, float* __restrict__ dq2acc,
                        float* __restrict__ dq1acc, __nv_bfloat16* __restrict__ dk2,
                        __nv_bfloat16* __restrict__ dk1, int* dev_status, uint64_t timeout_ns) {
  using L = BwdLayout<D, GRAD1>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kb = static_cast<int>(blockIdx.x);
  const int bh = static_cast<int>(blockIdx.y);
  const int nqb = (NQ + kBlockM - 1) / kBlockM;
  const int off = NK - NQ;
  // first query tile with a row that may see key kb*128: row i sees keys <= i + off
  const int qb0 = causal ? max(0, kb * kBlockN - off) / kBlockM : 0;
  int n_iter = nqb - qb0;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t k_full = bar0;
  auto q_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto q_empty = [&](int s) { return bar0 + 8u * (1 + L::QSTAGES + s); };
  const uint32_t s_full = bar0 + 8u * (1 + 2 * L::QSTAGES);
  const uint32_t s_free = s_full + 8;
  const uint32_t ds_full = s_full + 16;
  const uint32_t ds_free = s_full + 24;
  const uint32_t dq_full = s_full + 32;
  const uint32_t dq_free = s_full + 40;
  const uint32_t dk_full = s_full + 48;
  const uint32_t drain = s_full + 56;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);

  // debug build: the layout's regions (TMEM fields are set once allocated)
  CheckCtx ck{sb, sb + L::OFF_DS2, sb + L::OFF_BAR, sb + L::OFF_BAR + L::NBAR * 8, 0, 0,
              abort_flag, dev_status};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    bool lay_ok = true;
    if (kDeviceChecks) {  // every barrier address inside the barrier region
      lay_ok = check_bar(ck, k_full, __LINE__) && check_bar(ck, s_full, __LINE__) &&
               check_bar(ck, s_free, __LINE__) && check_bar(ck, ds_full, __LINE__) &&
               check_bar(ck, ds_free, __LINE__) && check_bar(ck, dq_full, __LINE__) &&
               check_bar(ck, dq_free, __LINE__) && check_bar(ck, dk_full, __LINE__) &&
               check_bar(ck, drain, __LINE__);
      for (int s = 0; s < L::QSTAGES; ++s)
        lay_ok = lay_ok && check_bar(ck, q_full(s), __LINE__) && check_bar(ck, q_empty(s), __LINE__);
    }
    if (lay_ok) {
      mbar_init(k_full, 1);
      for (int s = 0; s < L::QSTAGES; ++s) {
        mbar_init(q_full(s), 1);
        mbar_init(q_empty(s), 1);
      }
      mbar_init(s_full, 1);
      mbar_init(s_free, 8);
      mbar_init(ds_full, 8);
      mbar_init(ds_free, 1);
      mbar_init(dq_full, 1);
      mbar_init(dq_free, 8);
      mbar_init(dk_full, 1);
      mbar_init(drain, 1);
    }
    // a failure recorded earlier (this launch or a previous one), or a
    // failed layout check, skips the work
    *skip_flag = !lay_ok || *reinterpret_cast<volatile int*>(dev_status) != 0;
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
  if (*skip_flag) n_iter = 0;
  const WaitCtx wc{abort_flag, dev_status, timeout_ns};
  ck.tmem = tmem;
  ck.tmem_cols = 512;
  const int z_hi = static_cast<int>(gridDim.y);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool k_ok = true;
    if (kDeviceChecks && lane == 0 && n_iter > 0)
      for (int b = 0; b < L::KB; ++b)
        k_ok = k_ok &&
               check_tma(ck, sb + L::OFF_K1 + b * 16384, 16384, k_full, b * 64, D, kb * kBlockN,
                         NK, kBlockN, bh, z_hi, __LINE__) &&
               check_tma(ck, sb + L::OFF_K2 + b * 16384, 16384, k_full, b * 64, D, kb * kBlockN,
                         NK, kBlockN, bh, z_hi, __LINE__);
    if (lane == 0 && n_iter > 0 && k_ok) {
      mbar_arrive_expect_tx(k_full, 2 * L::TILE);
#pragma unroll
      for (int b = 0; b < L::KB; ++b) {
        tma_load_3d(sb + L::OFF_K1 + b * 16384, &tm_k1, k_full, b * 64, kb * kBlockN, bh);
        tma_load_3d(sb + L::OFF_K2 + b * 16384, &tm_k2, k_full, b * 64, kb * kBlockN, bh);
      }
      int it = 0;
      for (; it < n_iter; ++it) {
        const int s = it % L::QSTAGES;
        const uint32_t ph = (it / L::QSTAGES) & 1;
        if (!wait_bounded(q_empty(s), ph ^ 1, wc)) break;
        const int qrow = (qb0 + it) * kBlockM;
        const uint32_t dst = sb + L::OFF_Q + s * 2 * L::TILE;
        bool q_ok = true;
        if (kDeviceChecks)
          for (int b = 0; b < L::KB; ++b)
            q_ok = q_ok &&
                   check_tma(ck, dst + b * 16384, 16384, q_full(s), b * 64, D, qrow, NQ, kBlockM,
                             bh, z_hi, __LINE__) &&
                   check_tma(ck, dst + L::TILE + b * 16384, 16384, q_full(s), b * 64, D, qrow, NQ,
                             kBlockM, bh, z_hi, __LINE__);
        if (!q_ok) break;
        mbar_arrive_expect_tx(q_full(s), 2 * L::TILE);
#pragma unroll
        for (int b = 0; b < L::KB; ++b) {
          tma_load_3d(dst + b * 16384, &tm_q1, q_full(s), b * 64, qrow, bh);
          tma_load_3d(dst + L::TILE + b * 16384, &tm_q2, q_full(s), b * 64, qrow, bh);
        }
      }
      wait_drain(k_full, 0, timeout_ns);
      for (int j = max(0, it - L::QSTAGES); j < it; ++j)
        wait_drain(q_full(j % L::QSTAGES), (j / L::QSTAGES) & 1, timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t id_s = idesc_bf16(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t id_dk = idesc_bf16(kBlockN, D, 1, 1);
      constexpr uint32_t id_dq = idesc_bf16(kBlockM, D, 0, 1);
      constexpr uint32_t id_dqt = idesc_bf16(D, kBlockM, 1, 0);
      // S, dK and dQ accumulators inside the allocation (dQ^T: lanes = d)
      bool ok = check_tmem(ck, tmem + L::COL_S1, 128, 128, __LINE__) &&
                check_tmem(ck, tmem + L::COL_S2, 128, 128, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DK2, 128, D, __LINE__) &&
                (!GRAD1 || check_tmem(ck, tmem + L::COL_DK1, 128, D, __LINE__)) &&
                check_tmem(ck, tmem + L::COL_DQ2, L::DQT ? D : 128, L::DQT ? kBlockM : D, __LINE__) &&
                (!GRAD1 || check_tmem(ck, tmem + L::COL_DQ1, L::DQT ? D : 128,
                                      L::DQT ? kBlockM : D, __LINE__));
      ok = ok && wait_bounded(k_full, 0, wc);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % L::QSTAGES;
        const uint32_t ph = (it / L::QSTAGES) & 1;
        const uint32_t par = it & 1;
        if (!wait_bounded(q_full(s), ph, wc)) break;
        if (!wait_bounded(s_free, par ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t q1s = sb + L::OFF_Q + s * 2 * L::TILE;
        const uint32_t q2s = q1s + L::TILE;
        // S_t = Q_t K_t^T, both operands K-major (d contiguous); the two GEMMs'
        // k-steps interleaved so that independent accumulators overlap
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
          mma_bf16(tmem + L::COL_S1, smem_desc_sw128(q1s + koff, 16, 1024),
                   smem_desc_sw128(sb + L::OFF_K1 + koff, 16, 1024), id_s, k > 0);
          mma_bf16(tmem + L::COL_S2, smem_desc_sw128(q2s + koff, 16, 1024),
                   smem_desc_sw128(sb + L::OFF_K2 + koff, 16, 1024), id_s, k > 0);
        }
        mma_commit(s_full);
        if (!wait_bounded(ds_full, par, wc)) break;
        tc_fence_after();
        // dK_t += dS_t^T Q_t, 8 k-steps over the tile's 128 query rows:
        // A = dS_t viewed MN-major (keys contiguous), B = Q_t MN-major (d contiguous).
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mma_bf16(tmem + L::COL_DK2, smem_desc_sw128(sb + L::OFF_DS2 + k * 2048, 16384, 1024),
                   smem_desc_sw128(q2s + k * 2048, 16384, 1024), id_dk, (it > 0 || k > 0));
          if (GRAD1)
            mma_bf16(tmem + L::COL_DK1, smem_desc_sw128(sb + L::OFF_DS1 + k * 2048, 16384, 1024),
                     smem_desc_sw128(q1s + k * 2048, 16384, 1024), id_dk, (it > 0 || k > 0));
        }
        mma_commit(q_empty(s));  // the Q tile is no longer read: start the next load
        if (!L::ALIAS && !wait_bounded(dq_free, par ^ 1, wc)) break;
        tc_fence_after();
        // dQ, 8 k-steps over the tile's 128 keys.
        //  d == 128: dQ_t^T = K_t^T dS_t^T (M = d, N = query rows; A = K_t MN-major,
        //            B = dS_t K-major): a TMEM lane then holds one d column, so
        //            the readout reduces whole 128-byte row segments at once.
        //  d == 64:  dQ_t = dS_t K_t (M = query rows, N = d; A = dS_t K-major,
        //            B = K_t MN-major).
        auto mma_dq = [&](uint32_t col, uint32_t ds, uint32_t ks, int k) {
          const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
          if (L::DQT)
            mma_bf16(tmem + col, smem_desc_sw128(ks + k * 2048, 16384, 1024),
                     smem_desc_sw128(ds + koff, 16, 1024), id_dqt, k > 0);
          else
            mma_bf16(tmem + col, smem_desc_sw128(ds + koff, 16, 1024),
                     smem_desc_sw128(ks + k * 2048, 16384, 1024), id_dq, k > 0);
        };
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mma_dq(L::COL_DQ2, sb + L::OFF_DS2, sb + L::OFF_K2, k);
          if (GRAD1) mma_dq(L::COL_DQ1, sb + L::OFF_DS1, sb + L::OFF_K1, k);
        }
        mma_commit(dq_full);
        mma_commit(ds_free);
      }
      mma_commit(dk_full);
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dS / epilogues
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const int key0 = kb * kBlockN + wg * 64;  // first key of this thread's S columns
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const uint32_t par = it & 1;
      const int qrow = (qb0 + it) * kBlockM + r;
      float b1 = 0.f, b2 = 0.f, gs = 0.f, e = 0.f;
      if (qrow < NQ) {
        const size_t o = static_cast<size_t>(bh) * NQ + qrow;
        const float l1 = lse1_in[o], l2 = lse2_in[o];
        b1 = l1 * kLog2e;
        b2 = l2 * kLog2e;
        gs = g_in[o] * scale;
        e = l1 - l2 + kl_in[o];
      }
      const int lim = causal ? min(NK, qrow + 1 + off) : NK;
      if (!(ok = wait_bounded(s_full, par, wc))) break;
      if (!(ok = check_tmem(ck, tmem + lane_off + L::COL_S1 + wg * 64, 32, 64, __LINE__) &&
                 check_tmem(ck, tmem + lane_off + L::COL_S2 + wg * 64, 32, 64, __LINE__)))
        break;
      tc_fence_after();
      float a[64], b[64];
      tmem_ld32(tmem + lane_off + L::COL_S1 + wg * 64, *reinterpret_cast<float(*)[32]>(&a[0]));
      tmem_ld32(tmem + lane_off + L::COL_S1 + wg * 64 + 32, *reinterpret_cast<float(*)[32]>(&a[32]));
      tmem_ld32(tmem + lane_off + L::COL_S2 + wg * 64, *reinterpret_cast<float(*)[32]>(&b[0]));
      tmem_ld32(tmem + lane_off + L::COL_S2 + wg * 64 + 32, *reinterpret_cast<float(*)[32]>(&b[32]));
      tmem_wait_ld();
      if (!L::ALIAS) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
      }
      if (!(ok = wait_bounded(ds_free, par ^ 1, wc))) break;
      const bool full = key0 + 64 <= lim;
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        float p1 = ex2(fmaf(a[k], c, -b1));
        float p2 = ex2(fmaf(b[k], c, -b2));
        if (!full && key0 + k >= lim) {
          p1 = 0.f;
          p2 = 0.f;
        }
        const float d2 = gs * (p2 - p1);
        if (GRAD1) {
          const float lr = fmaf(scale, a[k] - b[k], -e);  // log(P1/P2) - KL
          a[k] = gs * p1 * lr;
        }
        b[k] = d2;
      }
      // bf16 dS rows into the swizzled tiles: row r, 16-byte chunk j of half wg
      const uint32_t row_base = static_cast<uint32_t>(wg * 16384 + r * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t o = row_base + static_cast<uint32_t>(((j ^ (r & 7)) << 4));
        st_shared_v4(sb + L::OFF_DS2 + o, pack_bf16x2(b[8 * j], b[8 * j + 1]),
                     pack_bf16x2(b[8 * j + 2], b[8 * j + 3]), pack_bf16x2(b[8 * j + 4], b[8 * j + 5]),
                     pack_bf16x2(b[8 * j + 6], b[8 * j + 7]));
        if (GRAD1)
          st_shared_v4(sb + L::OFF_DS1 + o, pack_bf16x2(a[8 * j], a[8 * j + 1]),
                       pack_bf16x2(a[8 * j + 2], a[8 * j + 3]),
                       pack_bf16x2(a[8 * j + 4], a[8 * j + 5]),
                       pack_bf16x2(a[8 * j + 6], a[8 * j + 7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      // dQ readout and reduction into the fp32 accumulator
      if (!(ok = wait_bounded(dq_full, par, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int set = 0; set < (GRAD1 ? 2 : 1); ++set) {
        float* acc = (set == 0 ? dq2acc : dq1acc);
        if (L::DQT) {
          // lane = d column (32*quarter + lane); warpgroup w takes query rows
          // [64w, 64w+64) of the tile; one red per row covers 128 contiguous bytes
          const uint32_t col = (set == 0 ? L::COL_DQ2 : L::COL_DQ1) + wg * 64;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[32];
            if (!check_tmem(ck, tmem + lane_off + col + h * 32, 32, 32, __LINE__)) continue;
            tmem_ld32(tmem + lane_off + col + h * 32, v);
            tmem_wait_ld();
            const int row0 = (qb0 + it) * kBlockM + wg * 64 + h * 32;
            float* dst = acc + (static_cast<size_t>(bh) * NQ + row0) * D + quarter * 32 + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (row0 + j < NQ) red_add_f32(dst + static_cast<size_t>(j) * D, v[j]);
          }
        } else {
          // lane = query row; this thread's d columns [wg*D/2, (wg+1)*D/2)
          const uint32_t col = (set == 0 ? L::COL_DQ2 : L::COL_DQ1) + wg * (D / 2);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            float v[32];
            if (!check_tmem(ck, tmem + lane_off + col + h * 32, 32, 32, __LINE__)) continue;
            tmem_ld32(tmem + lane_off + col + h * 32, v);
            tmem_wait_ld();
            if (qrow < NQ) {
              float* dst = acc + (static_cast<size_t>(bh) * NQ + qrow) * D + wg * (D / 2) + h * 32;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                red_add_v4(dst + 4 * j, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(L::ALIAS ? s_free : dq_free);
    }
    // dK readout: this thread's key row, d columns [wg*D/2, (wg+1)*D/2)
    if (ok && n_iter > 0 && wait_bounded(dk_full, 0, wc)) {
      tc_fence_after();
      const int key = kb * kBlockN + r;
#pragma unroll
      for (int set = 0; set < (GRAD1 ? 2 : 1); ++set) {
        const uint32_t col = (set == 0 ? L::COL_DK2 : L::COL_DK1) + wg * (D / 2);
        __nv_bfloat16* out = (set == 0 ? dk2 : dk1);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          float v[32];
          if (!check_tmem(ck, tmem + lane_off + col + h * 32, 32, 32, __LINE__)) continue;
          tmem_ld32(tmem + lane_off + col + h * 32, v);
          tmem_wait_ld();
          if (key < NK) {
            uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * NK + key) * D +
                                                  wg * (D / 2) + h * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                  pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                  pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                  pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
          }
        }
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

// fp32 dQ accumulator -> bf16, 8 elements per thread (n is a multiple of 8).
__global__ void streamkl_dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ out,
                                           long long n8) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    out[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                        pack_bf16x2(b.z, b.w));
  }
}

// Waits on an mbarrier that nothing ever arrives on; exercises the bounded
// wait's timeout path (status word set, kernel returns).
__global__ void streamkl_wait_selftest_kernel(int* dev_status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, dev_status, timeout_ns};
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0, wc);
  __syncthreads();
}

// Runs one range check that must fail: a TMEM range past the 512 columns of
// a (never made) allocation. Only the debug build records anything.
__global__ void streamkl_check_selftest_kernel(int* dev_status) {
  __shared__ int abort_flag;
  abort_flag = 0;
  const CheckCtx ck{0, 0, 0, 0, 0, 512, &abort_flag, dev_status};
  check_tmem(ck, 500, 32, 32, __LINE__);
}

template <int D, bool GRAD1>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayout<D, GRAD1>;
  auto kern = streamkl_bwd_kernel<D, GRAD1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const int nkb = (a.NK + kBlockN - 1) / kBlockN;
  dim3 grid(nkb, a.BH, 1);
  kern<<<grid, kBwdThreads, L::ALLOC, stream>>>(
      *a.tm_q1, *a.tm_k1, *a.tm_q2, *a.tm_k2, a.NQ, a.NK, a.causal, a.scale, a.kl, a.lse1, a.lse2,
      a.g, a.dq2acc, a.dq1acc, static_cast<__nv_bfloat16*>(a.dk2),
      static_cast<__nv_bfloat16*>(a.dk1), a.dev_status, a.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_smem_bytes(int d, int grad1) {
  if (d == 128) return grad1 ? BwdLayout<128, true>::ALLOC : BwdLayout<128, false>::ALLOC;
  return grad1 ? BwdLayout<64, true>::ALLOC : BwdLayout<64, false>::ALLOC;
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 128) return a.grad1 ? launch_bwd_t<128, true>(a, stream) : launch_bwd_t<128, false>(a, stream);
  return a.grad1 ? launch_bwd_t<64, true>(a, stream) : launch_bwd_t<64, false>(a, stream);
}

cudaError_t launch_dq_convert(const float* acc, void* out_bf16, long long n, cudaStream_t stream) {
  const long long n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (n8 + threads - 1) / threads;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  streamkl_dq_convert_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      reinterpret_cast<const float4*>(acc), static_cast<uint4*>(out_bf16), n8);
  return cudaGetLastError();
}

cudaError_t launch_check_selftest(int* dev_status, cudaStream_t stream) {
  streamkl_check_selftest_kernel<<<1, 1, 0, stream>>>(dev_status);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* dev_status, uint64_t timeout_ns, cudaStream_t stream) {
  streamkl_wait_selftest_kernel<<<1, 32, 0, stream>>>(dev_status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace skl

// Fused backward for short query sweeps (gist.science technical summary,
// "Metodologia" section 2, kernel fusion paragraph: one kernel visits every
// (query tile, key tile) pair once; dQ is accumulated across key tiles; the
// pages measure the fused kernel fastest when N_Q is small, "Resultados
// Experimentales", ablation). Probabilities are regenerated tile by tile from
// Q, K and the saved LSEs, P_t = exp(S_t - LSE_t).
//
// With at most 64 query rows (decode-like shapes) against long keys the
// backward is bound by reading K1, K2 and writing dK, which the separate dK and
// dQ kernels each pay for. Here a persistent grid (one CTA per SM) takes a
// contiguous range of (batch-head, 128-key tile) items. Per item:
//   T_t   = K_t Q_t^T                 (M = 128 keys, N = 64 queries, K = d)
//   dS_t  from T_t (softmax warps; bf16, into shared memory, row = key)
//   dK_t  = dS_t Q_t                  (M = 128 keys, N = d, K = 64)  -> bf16 out
//   dQ_t^T += K_t^T dS_t              (M = d, N = 64 queries, K = 128 keys)
// dQ^T stays in TMEM across all items of one batch-head that the CTA takes and
// is added to an fp32 accumulator (global reductions, zeroed by the caller)
// only when the batch-head changes, so its reductions are a few per CTA
// instead of one per key tile. Q1, Q2 of the current batch-head stay in
// shared memory; K tiles stream through a two-stage ring.
//
// Gradients of L = sum_i g_i KL_i, with s = scale * q.k (g and scale folded
// into dS):
//   configuration 1 (teacher P1 fixed):  dS2 = g * (P2 - P1)
//   configuration 2 (student P2 fixed):  dS1 = g * P1 * (log(P1/P2) - KL)
// with log(P1/P2) - KL = scale (s1 - s2) - (LSE1 - LSE2 + KL) from logits and
// the saved LSEs (section 3, numerical stability).
//
// Warps: 0 = TMA producer (lane 0) and, at each batch-head change, the per-query
// constant table (all lanes); 1 = TMEM owner + MMA issuer; 2..17 = softmax and
// epilogues: warp w reads TMEM lanes [32 (w%4), +32) and serves column group
// g = (w-2)/4; thread = key row (TMEM lane) of T, owning query columns
// [16g, 16g+16), and d columns [32g, 32g+32) of its dK row; for the dQ^T
// read-out, thread = one d column (lane), queries [16g, 16g+16); 18 = dK
// stores (lane 0). dK leaves through a 32 KB staging tile in shared memory
// (128-byte swizzle, the softmax warps write their rows' pieces) and two TMA
// stores per tile, so the writes are whole lines instead of one 16-byte piece
// of a different row per thread.
// TMEM: T1 [0,64) T2 [64,128) | dK set 2 [128,256) set 1 [256,384) |
// dQ^T set 2 [384,448) set 1 [448,512).
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kShThreads = 608;  // 19 warps
constexpr int kShSoftmaxWarps = 16;
constexpr int kShStoreWarp = 18;
constexpr int kShQ = 64;          // query rows per item (padded with zero rows)
constexpr int kShD = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSet2 = 1, kSet1 = 2;

template <int SETS>
struct ShortLayout {
  static constexpr int NSETS = SETS == (kSet1 | kSet2) ? 2 : 1;
  static constexpr int QT = kShQ * kShD * 2;       // one Q tensor: 2 boxes of 64 rows x 128 B
  static constexpr int KT = kBlockN * kShD * 2;    // one K tile: 2 boxes of 128 rows x 128 B
  static constexpr int STAGES = 2;
  static constexpr int DST = kBlockN * kShQ * 2;   // one dS tile: 128 key rows x 128 B
  static constexpr int OFF_Q = 0;                  // Q1, Q2
  static constexpr int OFF_K = 2 * QT;             // stage s: K1 at +2s KT, K2 at +(2s+1) KT
  static constexpr int OFF_DS = OFF_K + STAGES * 2 * KT;  // slot t: the t-th computed set
  static constexpr int STG = kBlockN * kShD * 2;          // dK staging: 2 boxes of 128 rows x 128 B
  static constexpr int OFF_STG = OFF_DS + NSETS * DST;
  static constexpr int OFF_TAB = OFF_STG + STG;           // [4][64] float
  static constexpr int OFF_BAR = OFF_TAB + 4 * kShQ * 4;
  // q_full, q_empty, tab_free, k_full[2], k_empty[2], t_full, t_free, ds_full,
  // ds_free, dk_full, dk_free, dq_full, dq_free, drain, st_full, st_empty
  static constexpr int NBAR = 3 + 2 * STAGES + 11;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr uint32_t COL_T = 0, COL_DK = 128, COL_DQ = 384;
  static_assert(COL_DQ + NSETS * kShQ <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(OFF_DS % 1024 == 0 && OFF_K % 1024 == 0 && OFF_STG % 1024 == 0,
                "swizzled tiles on 1024-byte boundaries");
};

template <int SETS>
__global__ void __launch_bounds__(kShThreads, 1)
    streamkl_bwd_short_kernel(const __grid_constant__ CUtensorMap tm_q1,
                              const __grid_constant__ CUtensorMap tm_k1,
                              const __grid_constant__ CUtensorMap tm_q2,
                              const __grid_constant__ CUtensorMap tm_k2, int NQ, int NK,
                              int causal, float scale, int BH, int items_per_cta,
                              const float* __restrict__ kl_in, const float* __restrict__ lse1_in,
                              const float* __restrict__ lse2_in, const float* __restrict__ g_in,
                              const __grid_constant__ CUtensorMap tm_dk2,
                              const __grid_constant__ CUtensorMap tm_dk1,
                              float* __restrict__ dq2acc, float* __restrict__ dq1acc,
                              int* dev_status, uint64_t timeout_ns) {
  using L = ShortLayout<SETS>;
  constexpr bool HAS2 = SETS & kSet2, HAS1 = SETS & kSet1;
  constexpr int D = kShD;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_kt = (NK + kBlockN - 1) / kBlockN;  // key tiles per batch-head
  const long long n_items = static_cast<long long>(BH) * n_kt;
  const long long i0 = static_cast<long long>(blockIdx.x) * items_per_cta;
  const long long i1 = min(n_items, i0 + items_per_cta);
  int n = static_cast<int>(max(0LL, i1 - i0));
  const int off = NK - NQ;  // causal: key j visible to query i iff j <= i + off
  // item it of this CTA: batch-head and key tile; a segment is a run of items
  // of one batch-head
  auto item_bh = [&](int it) { return static_cast<int>((i0 + it) / n_kt); };
  auto item_kt = [&](int it) { return static_cast<int>((i0 + it) % n_kt); };
  auto seg_start = [&](int it) { return it == 0 || item_bh(it) != item_bh(it - 1); };
  auto seg_end = [&](int it) { return it == n - 1 || item_bh(it) != item_bh(it + 1); };

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t q_full = bar0, q_empty = bar0 + 8, tab_free = bar0 + 16;
  auto k_full = [&](int s) { return bar0 + 24u + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 24u + 8u * (L::STAGES + s); };
  const uint32_t t_full = bar0 + 24u + 16u * L::STAGES;
  const uint32_t t_free = t_full + 8, ds_full = t_full + 16, ds_free = t_full + 24;
  const uint32_t dk_full = t_full + 32, dk_free = t_full + 40;
  const uint32_t dq_full = t_full + 48, dq_free = t_full + 56, drain = t_full + 64;
  // staging tile written by the softmax warps / read by the store warp's TMA stores
  const uint32_t st_full = t_full + 72, st_empty = t_full + 80;
  static_assert(3 + 2 * L::STAGES + 11 == L::NBAR, "barrier region holds every barrier");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);
  // per query column: -LSE1 log2e, -LSE2 log2e, g scale, -(LSE1 - LSE2 + KL)
  float* tab = reinterpret_cast<float*>(gb + L::OFF_TAB);

  CheckCtx ck{sb, sb + L::OFF_TAB, sb + L::OFF_BAR, sb + L::OFF_BAR + L::NBAR * 8, 0, 0,
              abort_flag, dev_status};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    bool lay_ok = true;
    if (kDeviceChecks) {  // every barrier address inside the barrier region
      lay_ok = check_bar(ck, q_full, __LINE__) && check_bar(ck, q_empty, __LINE__) &&
               check_bar(ck, tab_free, __LINE__) && check_bar(ck, t_full, __LINE__) &&
               check_bar(ck, drain, __LINE__) && check_bar(ck, st_full, __LINE__) &&
               check_bar(ck, st_empty, __LINE__);
      for (int s = 0; s < L::STAGES; ++s)
        lay_ok = lay_ok && check_bar(ck, k_full(s), __LINE__) && check_bar(ck, k_empty(s), __LINE__);
    }
    if (lay_ok) {
      mbar_init(q_full, 1);
      mbar_init(q_empty, 1);
      mbar_init(tab_free, kShSoftmaxWarps);
      for (int s = 0; s < L::STAGES; ++s) {
        mbar_init(k_full(s), 1);
        mbar_init(k_empty(s), 1);
      }
      mbar_init(t_full, 1);
      mbar_init(t_free, kShSoftmaxWarps);
      mbar_init(ds_full, kShSoftmaxWarps);
      mbar_init(ds_free, 1);
      mbar_init(dk_full, 1);
      mbar_init(dk_free, kShSoftmaxWarps);
      mbar_init(dq_full, 1);
      mbar_init(dq_free, kShSoftmaxWarps);
      mbar_init(drain, 1);
      mbar_init(st_full, kShSoftmaxWarps);
      mbar_init(st_empty, 1);
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
  if (warp == kShStoreWarp && lane == 0) {
    if (HAS2) tma_prefetch_desc(&tm_dk2);
    if (HAS1) tma_prefetch_desc(&tm_dk1);
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
    int seg = -1, it = 0, n_q = 0;
    for (; ok && it < n; ++it) {
      const int bh = item_bh(it), kt = item_kt(it);
      if (seg_start(it)) {
        ++seg;
        // the previous batch-head's Q (MMAs) and table (softmax) are no longer read
        bool good = true;
        if (lane == 0 && seg > 0)
          good = wait_bounded(q_empty, (seg - 1) & 1, wc) && wait_bounded(tab_free, (seg - 1) & 1, wc);
        if (!(ok = __shfl_sync(0xffffffffu, good, 0))) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = lane + 32 * h;
          float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
          if (q < NQ) {
            const size_t o = static_cast<size_t>(bh) * NQ + q;
            const float l1 = lse1_in[o], l2 = lse2_in[o];
            c = make_float4(-l1 * kLog2e, -l2 * kLog2e, g_in[o] * scale, -(l1 - l2 + kl_in[o]));
          }
          tab[q] = c.x;
          tab[kShQ + q] = c.y;
          tab[2 * kShQ + q] = c.z;
          tab[3 * kShQ + q] = c.w;
        }
        __syncwarp();  // the arrive below publishes the whole warp's entries
        if (lane == 0) {
          if (kDeviceChecks)
            for (int t = 0; t < 2; ++t)
              for (int b = 0; b < 2; ++b)
                ok = ok && check_tma(ck, sb + L::OFF_Q + t * L::QT + b * 8192, 8192, q_full, b * 64,
                                     D, 0, NQ, kShQ, bh, BH, __LINE__);
          if (ok) {
            mbar_arrive_expect_tx(q_full, 2 * L::QT);
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
              for (int b = 0; b < 2; ++b)
                tma_load_3d(sb + L::OFF_Q + t * L::QT + b * 8192, t == 0 ? &tm_q1 : &tm_q2, q_full,
                            b * 64, 0, bh);
            ++n_q;
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
      }
      if (lane == 0) {
        const int s = it % L::STAGES;
        ok = wait_bounded(k_empty(s), ((it / L::STAGES) & 1) ^ 1, wc);
        const uint32_t dst = sb + L::OFF_K + s * 2 * L::KT;
        if (kDeviceChecks)
          for (int t = 0; t < 2; ++t)
            for (int b = 0; b < 2; ++b)
              for (int h = 0; h < 2; ++h)
                ok = ok && check_tma(ck, dst + t * L::KT + b * 16384 + h * 8192, 8192, k_full(s),
                                     b * 64, D, kt * kBlockN + h * 64, NK, 64, bh, BH, __LINE__);
        if (ok) {
          mbar_arrive_expect_tx(k_full(s), 2 * L::KT);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d(dst + t * L::KT + b * 16384 + h * 8192, t == 0 ? &tm_k1 : &tm_k2,
                            k_full(s), b * 64, kt * kBlockN + h * 64, bh);
        }
      }
      if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;  // this item's copies were not issued
    }
    // let every copy this thread issued land before the CTA can exit
    if (lane == 0) {
      if (n_q > 0) wait_drain(q_full, (n_q - 1) & 1, timeout_ns);
      for (int j = max(0, it - L::STAGES); j < it; ++j)
        wait_drain(k_full(j % L::STAGES), (j / L::STAGES) & 1, timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t id_t = idesc_bf16(kBlockN, kShQ, 0, 0);   // T = K Q^T
      constexpr uint32_t id_dk = idesc_bf16(kBlockN, D, 0, 1);     // dK = dS Q
      constexpr uint32_t id_dq = idesc_bf16(D, kShQ, 1, 1);        // dQ^T = K^T dS
      bool ok = check_tmem(ck, tmem + L::COL_T, 128, 128, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DK, 128, L::NSETS * D, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DQ, 128, L::NSETS * kShQ, __LINE__);
      const uint64_t dq1 = smem_desc_sw128(sb + L::OFF_Q, 16, 1024);
      const uint64_t dq2 = smem_desc_sw128(sb + L::OFF_Q + L::QT, 16, 1024);
      // T of item it: K-major A (K tile) and B (Q), two GEMMs' k-steps interleaved
      auto issue_t = [&](int it) {
        const uint32_t ks = sb + L::OFF_K + (it % L::STAGES) * 2 * L::KT;
        const uint64_t dk1 = smem_desc_sw128(ks, 16, 1024), dk2d = smem_desc_sw128(ks + L::KT, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32, qo = (k >> 2) * 8192 + (k & 3) * 32;
          mma_bf16(tmem + L::COL_T, desc_advance(dk1, ko), desc_advance(dq1, qo), id_t, k > 0);
          mma_bf16(tmem + L::COL_T + 64, desc_advance(dk2d, ko), desc_advance(dq2, qo), id_t, k > 0);
        }
        mma_commit(t_full);
      };
      int seg = -1;
      bool t_issued_next = false;  // T of the current item already issued
      for (int it = 0; ok && it < n; ++it) {
        const int s = it % L::STAGES;
        const bool first = seg_start(it);
        if (first) ++seg;
        if (!t_issued_next) {
          if (first && !(ok = wait_bounded(q_full, seg & 1, wc))) break;
          if (!(ok = wait_bounded(k_full(s), (it / L::STAGES) & 1, wc))) break;
          if (it > 0 && !(ok = wait_bounded(t_free, (it - 1) & 1, wc))) break;
          tc_fence_after();
          issue_t(it);
        }
        // gradient GEMMs of this item as soon as its dS is in shared memory
        // (slot t holds the t-th computed set: set 2 first when present).
        // While the softmax warps still compute that dS, T of the next item of
        // the same batch-head goes in if it can (its K tile has landed in the
        // other stage and the softmax warps have loaded this T); otherwise it
        // waits for the next round, so a late K tile never holds up this
        // item's dK, which the softmax warps read next.
        t_issued_next = false;
        const bool can_next = it + 1 < n && !seg_start(it + 1);
        const int sn = (it + 1) % L::STAGES;
        const uint32_t phn = ((it + 1) / L::STAGES) & 1;
        auto try_next = [&]() {
          if (can_next && !t_issued_next && mbar_test_wait(k_full(sn), phn) &&
              mbar_test_wait(t_free, it & 1)) {
            tc_fence_after();
            issue_t(it + 1);
            t_issued_next = true;
          }
        };
        if (!(ok = wait_bounded_idle(ds_full, it & 1, wc, try_next))) break;
        if (it > 0 && !(ok = wait_bounded(dk_free, (it - 1) & 1, wc))) break;
        tc_fence_after();
        const uint32_t ks = sb + L::OFF_K + s * 2 * L::KT;
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          const bool set2 = HAS2 && t == 0;
          const uint32_t ds = sb + L::OFF_DS + t * L::DST;
          const uint64_t a = smem_desc_sw128(ds, 16, 1024);
          const uint64_t b = smem_desc_sw128(sb + L::OFF_Q + (set2 ? L::QT : 0), 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < kShQ / 16; ++kk)
            mma_bf16(tmem + L::COL_DK + t * D, desc_advance(a, kk * 32), desc_advance(b, kk * 2048),
                     id_dk, kk > 0);
        }
        mma_commit(dk_full);
        if (first && seg > 0 && !(ok = wait_bounded(dq_free, (seg - 1) & 1, wc))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          const bool set2 = HAS2 && t == 0;
          const uint64_t a = smem_desc_sw128(ks + (set2 ? L::KT : 0), 16384, 1024);  // K^T, MN-major
          const uint64_t b = smem_desc_sw128(sb + L::OFF_DS + t * L::DST, 8192, 1024);  // dS, MN-major
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_bf16(tmem + L::COL_DQ + t * kShQ, desc_advance(a, kk * 2048),
                     desc_advance(b, kk * 2048), id_dq, (!first || kk > 0));
        }
        mma_commit(ds_free);
        mma_commit(k_empty(s));
        if (seg_end(it)) {
          mma_commit(dq_full);
          mma_commit(q_empty);
        }
      }
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    }
  } else if (warp == kShStoreWarp) {
    // ------------------------------------------------------------ dK stores
    if (lane == 0 && n > 0) {
      bool ok = true;
      int u = 0;  // staging uses so far
      for (int it = 0; ok && it < n; ++it) {
        const int bh = item_bh(it), kt = item_kt(it);
        for (int t = 0; t < L::NSETS; ++t, ++u) {
          if (!(ok = wait_bounded(st_full, u & 1, wc))) break;
          // rows past N_K (the last tile's tail) are not written by the store
          if (!(ok = dcheck(ck, kt * kBlockN < NK && bh < BH, __LINE__))) break;
          const CUtensorMap* m = (HAS2 && t == 0) ? &tm_dk2 : &tm_dk1;
          tma_store_3d(m, sb + L::OFF_STG, 0, kt * kBlockN, bh);
          tma_store_3d(m, sb + L::OFF_STG + L::STG / 2, 64, kt * kBlockN, bh);
          bulk_commit_group();
          bulk_wait_read_all();  // the tile may be written again
          mbar_arrive(st_empty);
        }
      }
      bulk_wait_all();  // every dK tile is in global memory before the CTA exits
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogues
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row of the tile (TMEM lane); d column for dQ^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const int q0 = grp * 16;  // this thread's first query column
    bool ok = true;
    int seg = -1;
    for (int it = 0; ok && it < n; ++it) {
      const int bh = item_bh(it), kt = item_kt(it);
      const int key = kt * kBlockN + r;
      const bool first = seg_start(it);
      if (first) {
        ++seg;
        // the table of this batch-head is published by the Q barrier
        if (!(ok = __all_sync(0xffffffffu, wait_bounded(q_full, seg & 1, wc)))) break;
      }
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(t_full, it & 1, wc)))) break;
      if (!(ok = check_tmem(ck, tmem + lane_off + L::COL_T + q0, 32, 16, __LINE__) &&
                 check_tmem(ck, tmem + lane_off + L::COL_T + 64 + q0, 32, 16, __LINE__)))
        break;
      tc_fence_after();
      float a[16], b[16];
      tmem_ld16(tmem + lane_off + L::COL_T + q0, a);
      tmem_ld16(tmem + lane_off + L::COL_T + 64 + q0, b);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(t_free);
      // visible (key, query) pairs of this thread's 16 columns
      const int qlo = causal ? max(0, key - off) : 0;  // queries >= qlo see this key
      const bool full = key < NK && q0 >= qlo && q0 + 16 <= NQ;
      uint32_t d2p[8], d1p[8];
      const float2 c2 = make_float2(c, c), sc2 = make_float2(scale, scale);
      const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
      for (int k = 0; k < 16; k += 2) {
        const float2 nb1 = *reinterpret_cast<const float2*>(tab + q0 + k);
        const float2 nb2 = *reinterpret_cast<const float2*>(tab + kShQ + q0 + k);
        const float2 gs = *reinterpret_cast<const float2*>(tab + 2 * kShQ + q0 + k);
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
          const float2 ne = *reinterpret_cast<const float2*>(tab + 3 * kShQ + q0 + k);
          // g P1 (log(P1/P2) - KL), log(P1/P2) - KL = scale (s1 - s2) - e
          const float2 lr = __ffma2_rn(__ffma2_rn(s2, m1, s1), sc2, ne);
          const float2 d1 = __fmul2_rn(__fmul2_rn(p1, gs), lr);
          d1p[k >> 1] = pack_bf16x2(d1.x, d1.y);
        }
      }
      // the table is not read again in this batch-head: the producer may
      // write the next one
      if (seg_end(it)) {
        __syncwarp();
        if (lane == 0) mbar_arrive(tab_free);
      }
      // the previous item's gradient GEMMs have read the dS tiles
      if (it > 0 && !(ok = __all_sync(0xffffffffu, wait_bounded(ds_free, (it - 1) & 1, wc)))) break;
      // row r of each dS tile: 128 bytes = 64 queries; this thread's 32 bytes
      // are 16-byte chunks 2 grp and 2 grp + 1, swizzled by the row
      const uint32_t row = static_cast<uint32_t>(r * 128);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        const uint32_t* v = (HAS2 && t == 0) ? d2p : d1p;
        const uint32_t base = sb + L::OFF_DS + t * L::DST + row;
#pragma unroll
        for (int j = 0; j < 2; ++j)
          st_shared_v4(base + ((((2 * grp + j) ^ (r & 7))) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                       v[4 * j + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      // dK of this key row: d columns [32 grp, 32 grp + 32) of each set, to
      // the staging tile (box grp/2, 16-byte chunks 4 (grp%2) .. +4 of the
      // row, swizzled by the row); the store warp writes the tile out
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(dk_full, it & 1, wc)))) break;
      tc_fence_after();
      const uint32_t srow = sb + L::OFF_STG + (grp >> 1) * (L::STG / 2) + static_cast<uint32_t>(r * 128);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        float v[32];
        if (!(ok = check_tmem(ck, tmem + lane_off + L::COL_DK + t * D + grp * 32, 32, 32, __LINE__))) break;
        tmem_ld32(tmem + lane_off + L::COL_DK + t * D + grp * 32, v);
        tmem_wait_ld();
        // the store warp has read the tile's previous contents
        const int u = it * L::NSETS + t;
        if (!(ok = __all_sync(0xffffffffu, wait_bounded(st_empty, (u & 1) ^ 1, wc)))) break;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_v4(srow + ((((grp & 1) * 4 + j) ^ (r & 7)) << 4), pack_bf16x2(v[8 * j], v[8 * j + 1]),
                       pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                       pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(st_full);
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dk_free);
      // end of a batch-head: add this CTA's dQ^T partial to the fp32 accumulator
      // (thread = d column r, queries [16 grp, 16 grp + 16))
      if (seg_end(it)) {
        if (!(ok = __all_sync(0xffffffffu, wait_bounded(dq_full, seg & 1, wc)))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < L::NSETS; ++t) {
          float* acc = (HAS2 && t == 0) ? dq2acc : dq1acc;
          float v[16];
          if (!check_tmem(ck, tmem + lane_off + L::COL_DQ + t * kShQ + q0, 32, 16, __LINE__)) break;
          tmem_ld16(tmem + lane_off + L::COL_DQ + t * kShQ + q0, v);
          tmem_wait_ld();
          float* dst = acc + (static_cast<size_t>(bh) * NQ + q0) * D + r;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (q0 + k < NQ) red_add_f32(dst + static_cast<size_t>(k) * D, v[k]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dq_free);
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
cudaError_t launch_short_t(const BwdShortArgs& a, cudaStream_t stream) {
  using L = ShortLayout<SETS>;
  auto kern = streamkl_bwd_short_kernel<SETS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const long long n_items = static_cast<long long>(a.BH) * ((a.NK + kBlockN - 1) / kBlockN);
  const int ctas = static_cast<int>(a.ctas < n_items ? a.ctas : n_items);
  const int per = static_cast<int>((n_items + ctas - 1) / ctas);
  const int grid = static_cast<int>((n_items + per - 1) / per);
  kern<<<grid, kShThreads, L::ALLOC, stream>>>(
      *a.tm_q1, *a.tm_k1, *a.tm_q2, *a.tm_k2, a.NQ, a.NK, a.causal, a.scale, a.BH, per, a.kl,
      a.lse1, a.lse2, a.g, *a.tm_dk2, *a.tm_dk1, a.dq2acc, a.dq1acc, a.dev_status, a.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_short_smem_bytes(int grad1, int grad2) {
  if (grad1 && grad2) return ShortLayout<kSet1 | kSet2>::ALLOC;
  return ShortLayout<kSet2>::ALLOC;
}

cudaError_t launch_bwd_short(const BwdShortArgs& a, cudaStream_t stream) {
  if (a.grad1 && a.grad2) return launch_short_t<kSet1 | kSet2>(a, stream);
  return a.grad1 ? launch_short_t<kSet1>(a, stream) : launch_short_t<kSet2>(a, stream);
}

}  // namespace skl

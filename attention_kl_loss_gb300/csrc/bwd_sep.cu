// Backward pass as two separate kernels without atomics (gist.science
// technical summary, "Metodologia" section 2, kernel fusion paragraph: when
// dQ accumulation across key tiles contends too much, dK and dQ are computed
// by separate kernels). Probabilities are regenerated tile by tile from Q, K
// and the saved LSEs, P_t = exp(S_t - LSE_t).
//
// One template serves both kernels. A CTA keeps 128 rows of a "stationary"
// tensor pair X1, X2 in shared memory and streams 128-row tiles of the other
// pair Y1, Y2 through a 2-stage ring:
//   dQ kernel: X = Q (query block), Y = K tiles;   acc_t += dS_t K_t
//   dK kernel: X = K (key block),   Y = Q tiles;   acc_t += dS_t^T Q_t
// Per Y tile, S1 = Q1 K1^T and S2 = Q2 K2^T (M = 128 query rows, N = 128 keys)
// are recomputed into TMEM with the two GEMMs' k-steps interleaved (two
// independent accumulators keep the tensor pipe busy), the softmax warps turn
// them into dS (bf16, 128-byte-swizzled shared memory), and one GEMM per
// gradient set adds into an fp32 accumulator that stays in TMEM for the whole
// sweep and is written out once:
//   TMEM: S1 [0,128) | S2 [128,256) | acc set 2 [256, 256+d) | acc set 1
// The softmax warps release S as soon as they have loaded it, so the S GEMMs
// of tile i+1 run while they compute dS of tile i.
//
// Gradients of L = sum_i g_i KL_i, with s = scale * q.k (g and scale folded
// into dS):
//   configuration 1 (teacher P1 fixed):  dS2 = g * (P2 - P1)
//   configuration 2 (student P2 fixed):  dS1 = g * P1 * (log(P1/P2) - KL)
// with log(P1/P2) = (s1 - LSE1) - (s2 - LSE2) from logits and the saved LSEs
// (section 3, numerical stability).
//
// Shared memory at d = 128 holds X (64 KB), the Y ring (128 KB) and one dS
// tile (32 KB); with both gradient sets the two dS tiles take turns in that
// buffer (set 2 first). At d = 64, or with one set, each set has its own.
//
// Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2..17 = softmax and
// epilogue. Warp w reads TMEM lanes [32 (w%4), +32) (its quarter) and serves
// column group g = (w-2)/4: thread = query row of the S tile (TMEM lane),
// owning keys [32g, 32g+32) of every tile; at the end it writes accumulator
// row r, d columns [g d/4, (g+1) d/4). Four warps per scheduler hide the
// latency of the exp2 / FMA chains; pairs of columns go through the packed
// f32x2 FMA path.
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kSepThreads = 576;  // 18 warps
constexpr int kSoftmaxWarps = 16;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool GRAD1>
struct SepLayout {
  static constexpr int KB = D / 64;              // 128-byte boxes per row
  static constexpr int TILE = kBlockM * D * 2;   // 128 rows of one tensor
  static constexpr int NSETS = GRAD1 ? 2 : 1;
  static constexpr int NDS = (D == 128 && GRAD1) ? 1 : NSETS;  // dS buffers
  static constexpr bool SHARED_DS = NDS < NSETS;                // sets take turns
  static constexpr int DS_TILE = kBlockM * kBlockN * 2;         // 32 KB
  static constexpr int OFF_X1 = 0;
  static constexpr int OFF_X2 = TILE;
  static constexpr int OFF_Y = 2 * TILE;  // stage s: Y1 at +2s*TILE, Y2 at +(2s+1)*TILE
  static constexpr int OFF_DS = OFF_Y + 4 * TILE;
  static constexpr int OFF_BAR = OFF_DS + NDS * DS_TILE;
  // x_full, y_full[2], y2_empty[2], s_full, s_free, ds_full[4], ds_free[2],
  // acc_full, drain, y1_empty[2]. With a shared dS buffer, ds_full is per
  // (set, half) and ds_free per half; otherwise per set/buffer. Each streamed
  // tensor's slot is released as soon as its own gradient GEMM is done.
  static constexpr int NBAR = 17;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr uint32_t COL_S1 = 0, COL_S2 = 128, COL_ACC = 256;
  static_assert(COL_ACC + NSETS * D <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

struct RowConst {
  float b1, b2, gs, e;  // LSE1*log2e, LSE2*log2e, g*scale, LSE1 - LSE2 + KL
};

__device__ __forceinline__ RowConst load_row_const(const float* lse1, const float* lse2,
                                                   const float* g, const float* kl, size_t o,
                                                   float scale, bool valid) {
  RowConst q{0.f, 0.f, 0.f, 0.f};
  if (valid) {
    const float l1 = lse1[o], l2 = lse2[o];
    q.b1 = l1 * kLog2e;
    q.b2 = l2 * kLog2e;
    q.gs = g[o] * scale;
    q.e = l1 - l2 + kl[o];
  }
  return q;
}

template <int D, bool DQ, bool GRAD1>
__global__ void __launch_bounds__(kSepThreads, 1)
    streamkl_bwd_sep_kernel(const __grid_constant__ CUtensorMap tm_x1,
                            const __grid_constant__ CUtensorMap tm_x2,
                            const __grid_constant__ CUtensorMap tm_y1,
                            const __grid_constant__ CUtensorMap tm_y2, int NQ, int NK,
                            int causal, float scale, const float* __restrict__ kl_in,
                            const float* __restrict__ lse1_in, const float* __restrict__ lse2_in,
                            const float* __restrict__ g_in, __nv_bfloat16* __restrict__ out2,
                            __nv_bfloat16* __restrict__ out1, int* dev_status,
                            uint64_t timeout_ns) {
  using L = SepLayout<D, GRAD1>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int NX = DQ ? NQ : NK;
  const int nxb = (NX + kBlockM - 1) / kBlockM;
  const int off = NK - NQ;  // key j is visible to query i iff j <= i + off (causal)
  // causal: the dQ kernel's heavy blocks are the last query blocks, the dK
  // kernel's the first key blocks; launch the heavy ones first
  const int xb = (DQ && causal) ? nxb - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  const int bh = static_cast<int>(blockIdx.y);
  const int x0 = xb * kBlockM;
  int y_begin, y_end;
  if (DQ) {  // key tiles visible to some row of this query block
    const int klim = causal ? min(NK, min(NQ, x0 + kBlockM) + off) : NK;
    y_begin = 0;
    y_end = (klim + kBlockN - 1) / kBlockN;
  } else {  // query tiles with a row that sees some key of this block
    y_begin = causal ? max(0, x0 - off) / kBlockM : 0;
    y_end = (NQ + kBlockM - 1) / kBlockM;
  }
  int n_iter = y_end - y_begin;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t x_full = bar0;
  auto y_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto y2_empty = [&](int s) { return bar0 + 8u * (3 + s); };
  auto y1_empty = [&](int s) { return bar0 + 8u * (15 + s); };
  const uint32_t s_full = bar0 + 8u * 5;
  const uint32_t s_free = bar0 + 8u * 6;
  auto ds_full = [&](int t) { return bar0 + 8u * (7 + t); };
  auto ds_free = [&](int b) { return bar0 + 8u * (11 + b); };
  const uint32_t acc_full = bar0 + 8u * 13;
  const uint32_t drain = bar0 + 8u * 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);

  if (threadIdx.x == 0) {
    mbar_init(x_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(y_full(s), 1);
      mbar_init(y1_empty(s), 1);
      mbar_init(y2_empty(s), 1);
      mbar_init(ds_free(s), 1);
    }
    // one arrival per softmax warp writing the (set, half) or set
    for (int t = 0; t < 4; ++t) mbar_init(ds_full(t), L::SHARED_DS ? kSoftmaxWarps / 2 : kSoftmaxWarps);
    mbar_init(s_full, 1);
    mbar_init(s_free, kSoftmaxWarps);
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    // a failure recorded earlier (this launch or a previous one) skips the work
    *skip_flag = *reinterpret_cast<volatile int*>(dev_status) != 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x1);
    tma_prefetch_desc(&tm_x2);
    tma_prefetch_desc(&tm_y1);
    tma_prefetch_desc(&tm_y2);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_iter > 0) {
      mbar_arrive_expect_tx(x_full, 2 * L::TILE);
#pragma unroll
      for (int b = 0; b < L::KB; ++b) {
        tma_load_3d(sb + L::OFF_X1 + b * 16384, &tm_x1, x_full, b * 64, x0, bh);
        tma_load_3d(sb + L::OFF_X2 + b * 16384, &tm_x2, x_full, b * 64, x0, bh);
      }
      int it = 0;
      for (; it < n_iter; ++it) {
        const int s = it & 1;
        const uint32_t ph = ((it >> 1) & 1) ^ 1;
        const int yrow = (y_begin + it) * kBlockM;
        const uint32_t dst = sb + L::OFF_Y + s * 2 * L::TILE;
        // Y2's slot frees first (set 2's GEMM runs first): load it as soon as it does
        if (!wait_bounded(y2_empty(s), ph, wc)) break;
        mbar_arrive_expect_tx(y_full(s), 2 * L::TILE);
#pragma unroll
        for (int b = 0; b < L::KB; ++b)
          tma_load_3d(dst + L::TILE + b * 16384, &tm_y2, y_full(s), b * 64, yrow, bh);
        const bool y1_ok = wait_bounded(y1_empty(s), ph, wc);
        if (y1_ok) {
#pragma unroll
          for (int b = 0; b < L::KB; ++b)
            tma_load_3d(dst + b * 16384, &tm_y1, y_full(s), b * 64, yrow, bh);
        }
        if (!y1_ok) {
          ++it;  // Y2 of this tile is in flight: count it for the drain below
          break;
        }
      }
      // let every copy this thread issued land before the CTA can exit
      wait_drain(x_full, 0, timeout_ns);
      for (int j = max(0, it - 2); j < it; ++j) wait_drain(y_full(j & 1), (j >> 1) & 1, timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t id_s = idesc_bf16(kBlockM, kBlockN, 0, 0);
      // dQ: A = dS (K-major, keys contiguous), B = K (MN-major)
      // dK: A = dS^T (dS viewed MN-major), B = Q (MN-major)
      constexpr uint32_t id_g = DQ ? idesc_bf16(kBlockM, D, 0, 1) : idesc_bf16(kBlockN, D, 1, 1);
      auto a_desc = [&](uint32_t ds, int k) {
        return DQ ? smem_desc_sw128(ds + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024)
                  : smem_desc_sw128(ds + k * 2048, 16384, 1024);
      };
      bool ok = wait_bounded(x_full, 0, wc);
      for (int it = 0; ok && it <= n_iter; ++it) {
        if (it < n_iter) {
          const int s = it & 1;
          if (!(ok = wait_bounded(y_full(s), (it >> 1) & 1, wc))) break;
          if (!(ok = wait_bounded(s_free, (it & 1) ^ 1, wc))) break;  // S(it-1) loaded
          tc_fence_after();
          const uint32_t y1 = sb + L::OFF_Y + s * 2 * L::TILE, y2 = y1 + L::TILE;
          const uint32_t q1 = DQ ? sb + L::OFF_X1 : y1, q2 = DQ ? sb + L::OFF_X2 : y2;
          const uint32_t k1 = DQ ? y1 : sb + L::OFF_X1, k2 = DQ ? y2 : sb + L::OFF_X2;
          // S_t = Q_t K_t^T, both K-major; the two GEMMs' k-steps interleaved
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            mma_bf16(tmem + L::COL_S1, smem_desc_sw128(q1 + ko, 16, 1024),
                     smem_desc_sw128(k1 + ko, 16, 1024), id_s, k > 0);
            mma_bf16(tmem + L::COL_S2, smem_desc_sw128(q2 + ko, 16, 1024),
                     smem_desc_sw128(k2 + ko, 16, 1024), id_s, k > 0);
          }
          mma_commit(s_full);
        }
        if (it > 0) {
          // gradient GEMMs of tile j = it - 1: acc_t += dS_t (x) Y_t, 8 k-steps
          const int j = it - 1;
          const uint32_t y1 = sb + L::OFF_Y + (j & 1) * 2 * L::TILE, y2 = y1 + L::TILE;
          const uint32_t acc2 = tmem + L::COL_ACC, acc1 = acc2 + D;
          const uint32_t ds0 = sb + L::OFF_DS;
          if (L::SHARED_DS) {
            // The two sets take turns in one dS buffer (set 2, then set 1), half
            // by half: k-steps 0-3 read half 0 (keys 0-63 in the dQ kernel,
            // query rows 0-63 in the dK kernel), 4-7 half 1, and each half is
            // handed back as soon as its k-steps are done.
            for (int t = 0; ok && t < 2; ++t) {
              const uint32_t acc = t == 0 ? acc2 : acc1;
              const uint32_t yt = t == 0 ? y2 : y1;
              for (int h = 0; h < 2; ++h) {
                if (!(ok = wait_bounded(ds_full(t * 2 + h), j & 1, wc))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 4 * h; k < 4 * h + 4; ++k)
                  mma_bf16(acc, a_desc(ds0, k), smem_desc_sw128(yt + k * 2048, 16384, 1024), id_g,
                           (j > 0 || k > 0));
                mma_commit(ds_free(h));
              }
              mma_commit(t == 0 ? y2_empty(j & 1) : y1_empty(j & 1));
            }
            if (!ok) break;
          } else {
            if (!(ok = wait_bounded(ds_full(0), j & 1, wc))) break;
            if (GRAD1 && !(ok = wait_bounded(ds_full(1), j & 1, wc))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              mma_bf16(acc2, a_desc(ds0, k), smem_desc_sw128(y2 + k * 2048, 16384, 1024), id_g,
                       (j > 0 || k > 0));
              if (GRAD1)
                mma_bf16(acc1, a_desc(ds0 + L::DS_TILE, k),
                         smem_desc_sw128(y1 + k * 2048, 16384, 1024), id_g, (j > 0 || k > 0));
            }
            mma_commit(ds_free(0));
            if (GRAD1) mma_commit(ds_free(1));
            mma_commit(y2_empty(j & 1));
            mma_commit(y1_empty(j & 1));
          }
        }
      }
      mma_commit(acc_full);
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ dS / epilogue
    const int grp = (warp - 2) >> 2;  // column group
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row of the S tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const size_t rowbase = static_cast<size_t>(bh) * NQ;
    bool ok = true;

    auto qrow_of = [&](int it) { return DQ ? x0 + r : (y_begin + it) * kBlockM + r; };
    auto load_const = [&](int it) {
      const int q = qrow_of(it);
      return load_row_const(lse1_in, lse2_in, g_in, kl_in, rowbase + q, scale,
                            it < n_iter && q < NQ);
    };
    // dK kernel: raw per-row values of the next tile, loaded a whole tile ahead
    // and only turned into constants when that tile starts
    auto load_raw = [&](int it, float4& v) {
      const int q = qrow_of(it);
      v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (it < n_iter && q < NQ) {
        const size_t o = rowbase + q;
        v = make_float4(lse1_in[o], lse2_in[o], g_in[o], kl_in[o]);
      }
    };
    // half of the shared dS buffer this thread's values land in
    const int half = DQ ? (grp >> 1) : (quarter >> 1);
    // write this thread's 32 bf16 dS values (keys [32 grp, +32) of row r)
    // into buffer `buf`: half grp/2 of the tile, 16-byte chunks 4 (grp%2) + j
    auto write_ds = [&](int buf, const float (&v)[32]) {
      const uint32_t row_base =
          sb + L::OFF_DS + buf * L::DS_TILE + (grp >> 1) * 16384 + r * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_shared_v4(row_base + static_cast<uint32_t>((((grp & 1) * 4 + j) ^ (r & 7)) << 4),
                     pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                     pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
      fence_proxy_async_smem();
    };

    RowConst rc = load_const(0);
    for (int it = 0; it < n_iter; ++it) {
      float4 nraw;
      if (!DQ) load_raw(it + 1, nraw);
      const int qrow = qrow_of(it);
      const int key0 = (DQ ? (y_begin + it) * kBlockN : x0) + grp * 32;
      const int lim = causal ? min(NK, qrow + 1 + off) : NK;  // keys < lim visible
      if (!(ok = wait_bounded(s_full, it & 1, wc))) break;
      tc_fence_after();
      float a[32], b[32];
      tmem_ld32(tmem + lane_off + L::COL_S1 + grp * 32, a);
      tmem_ld32(tmem + lane_off + L::COL_S2 + grp * 32, b);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);  // the next S GEMMs may overwrite
      const bool full = key0 + 32 <= lim;
      const float2 c2 = make_float2(c, c), sc2 = make_float2(scale, scale);
      const float2 m1 = make_float2(-1.f, -1.f), gs2 = make_float2(rc.gs, rc.gs);
      const float2 nb1 = make_float2(-rc.b1, -rc.b1), nb2 = make_float2(-rc.b2, -rc.b2);
      const float2 ne = make_float2(-rc.e, -rc.e);
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float2 s1 = make_float2(a[k], a[k + 1]), s2 = make_float2(b[k], b[k + 1]);
        const float2 x1 = __ffma2_rn(s1, c2, nb1), x2 = __ffma2_rn(s2, c2, nb2);
        float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
        float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
        if (!full) {
          if (key0 + k >= lim) p1.x = p2.x = 0.f;
          if (key0 + k + 1 >= lim) p1.y = p2.y = 0.f;
        }
        const float2 d2 = __fmul2_rn(__ffma2_rn(p1, m1, p2), gs2);  // g (P2 - P1)
        if (GRAD1) {
          // g P1 (log(P1/P2) - KL), log(P1/P2) - KL = scale (s1 - s2) - e
          const float2 lr = __ffma2_rn(__ffma2_rn(s2, m1, s1), sc2, ne);
          const float2 d1 = __fmul2_rn(__fmul2_rn(p1, gs2), lr);
          a[k] = d1.x;
          a[k + 1] = d1.y;
        }
        b[k] = d2.x;
        b[k + 1] = d2.y;
      }
      const uint32_t par = it & 1;
      if (L::SHARED_DS) {
        // per half: set 2 waits for the set-1 GEMM of the previous tile, set 1
        // for the set-2 GEMM of this tile (the half's completions alternate)
        if (!(ok = wait_bounded(ds_free(half), 1, wc))) break;
        write_ds(0, b);
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full(half));
        if (!(ok = wait_bounded(ds_free(half), 0, wc))) break;
        write_ds(0, a);
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full(2 + half));
      } else {
        if (!(ok = wait_bounded(ds_free(0), par ^ 1, wc))) break;
        write_ds(0, b);
        if (GRAD1) {
          if (!(ok = wait_bounded(ds_free(1), par ^ 1, wc))) break;
          write_ds(1, a);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(ds_full(0));
          if (GRAD1) mbar_arrive(ds_full(1));
        }
      }
      if (!DQ) {
        rc.b1 = nraw.x * kLog2e;
        rc.b2 = nraw.y * kLog2e;
        rc.gs = nraw.z * scale;
        rc.e = nraw.x - nraw.y + nraw.w;
      }
    }
    // epilogue: accumulator row r -> bf16 dQ (dQ kernel) or dK (dK kernel) row
    if (ok && n_iter > 0 && wait_bounded(acc_full, 0, wc)) {
      tc_fence_after();
      const int xrow = x0 + r;
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        __nv_bfloat16* out = t == 0 ? out2 : out1;
        // group grp writes d columns [32 grp, 32 grp + 32) (d = 64: groups 0, 1)
        if (grp * 32 < D) {
          float v[32];
          tmem_ld32(tmem + lane_off + L::COL_ACC + t * D + grp * 32, v);
          tmem_wait_ld();
          if (xrow < NX) {
            uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * NX + xrow) * D +
                                                  grp * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                  pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                  pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                  pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
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

template <int D, bool DQ, bool GRAD1>
cudaError_t launch_sep_t(const BwdSepArgs& a, cudaStream_t stream) {
  using L = SepLayout<D, GRAD1>;
  auto kern = streamkl_bwd_sep_kernel<D, DQ, GRAD1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const int NX = DQ ? a.NQ : a.NK;
  dim3 grid((NX + kBlockM - 1) / kBlockM, a.BH, 1);
  const CUtensorMap* x1 = DQ ? a.tm_q1 : a.tm_k1;
  const CUtensorMap* x2 = DQ ? a.tm_q2 : a.tm_k2;
  const CUtensorMap* y1 = DQ ? a.tm_k1 : a.tm_q1;
  const CUtensorMap* y2 = DQ ? a.tm_k2 : a.tm_q2;
  kern<<<grid, kSepThreads, L::ALLOC, stream>>>(
      *x1, *x2, *y1, *y2, a.NQ, a.NK, a.causal, a.scale, a.kl, a.lse1, a.lse2, a.g,
      static_cast<__nv_bfloat16*>(DQ ? a.dq2 : a.dk2),
      static_cast<__nv_bfloat16*>(DQ ? a.dq1 : a.dk1), a.dev_status, a.timeout_ns);
  return cudaGetLastError();
}

template <int D, bool DQ>
cudaError_t launch_sep_g(const BwdSepArgs& a, cudaStream_t stream) {
  return a.grad1 ? launch_sep_t<D, DQ, true>(a, stream) : launch_sep_t<D, DQ, false>(a, stream);
}

}  // namespace

size_t bwd_sep_smem_bytes(int d, int grad1) {
  if (d == 128) return grad1 ? SepLayout<128, true>::ALLOC : SepLayout<128, false>::ALLOC;
  return grad1 ? SepLayout<64, true>::ALLOC : SepLayout<64, false>::ALLOC;
}

cudaError_t launch_bwd_separate(const BwdSepArgs& a, cudaStream_t stream) {
  cudaError_t e = a.d == 128 ? launch_sep_g<128, false>(a, stream) : launch_sep_g<64, false>(a, stream);
  if (e != cudaSuccess) return e;
  return a.d == 128 ? launch_sep_g<128, true>(a, stream) : launch_sep_g<64, true>(a, stream);
}

}  // namespace skl

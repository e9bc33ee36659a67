// Forward pass of the attention-KL primitive: one streaming pass over key
// tiles that keeps, per query row, the coupled online state of the pages'
// online formulation (gist.science technical summary, "Metodologia" section 1):
// running maxima m1, m2, exponential sums l1, l2 and the rescaled running sum
// acc = sum_j exp(s1_j - m1) (s1_j - s2_j). At the end
//     LSE_t = m_t + log l_t,   KL = acc / l1 + LSE2 - LSE1.
// S1 and S2 never leave the SM: they are produced by tcgen05 MMAs into TMEM
// and read back by the softmax warps. Key tiles past a row block's causal
// frontier are never loaded (same section: masked tiles are skipped).
//
// CTA layout (576 threads, one CTA per SM because of shared memory):
//   warp 0       TMA producer: Q1/Q2 tile once, K1/K2 tiles through a ring
//   warp 1       TMEM owner + MMA issuer: S1 = Q1 K1^T, S2 = Q2 K2^T per tile,
//                double-buffered in TMEM (2 x 256 columns)
//   warps 2..17  four softmax warpgroups; thread = one query row (TMEM lane
//                of its warp's quarter); group g owns key columns
//                [32g, 32g+32) of every tile and keeps its own five-scalar
//                state; the four states are merged at the end exactly like
//                split-K partials. Four warps per scheduler hide the exp2/FMA
//                latency, and column pairs use the packed f32x2 FMA path.
//
// Numerics: exponentials are base 2 with a reference kept in log2 units
// (r = m * scale * log2 e). A row's first chunk sets it to that chunk's
// maximum. Later chunks are folded against it directly, with no maximum
// taken: when a chunk's terms sum to F > 2^kTau (=2^8) the reference moves up
// by log2 F, which brings that sum to 1, so no accumulated term exceeds 2^8.
// A term that leaves the fp32 range (a logit more than 128 log2 units above
// the reference) leaves NaN in the row's state; a CTA with such a row sweeps
// its key tiles a second time, folding every chunk from its maximum (moved
// only when that exceeds the reference by more than kTau). Moving the
// reference rescales l and acc, so the result is the same for any reference.
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kFwdThreads = 576;  // 18 warps
constexpr int kGroups = 4;        // softmax column groups (warpgroups)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTau = 8.0f;
constexpr float kSumMax = 256.0f;  // 2^kTau

// CTA-wide barrier 0 that the threads of one warp may reach from different
// code paths (the roles end their first sweep in different branches); the
// non-aligned form of the instruction allows that, __syncthreads does not.
__device__ __forceinline__ void cta_barrier_divergent() { asm volatile("barrier.sync 0;" ::: "memory"); }

template <int D>
struct FwdLayout {
  static constexpr int KB = D / 64;          // 64-column (128-byte) boxes per row
  static constexpr int TILE = kBlockM * D * 2;  // one 128-row bf16 tile
  static constexpr int STAGES = D == 128 ? 2 : 4;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = TILE;
  static constexpr int OFF_K = 2 * TILE;  // stage s: K1 at +2s*TILE, K2 at +(2s+1)*TILE
  static constexpr int OFF_BAR = OFF_K + STAGES * 2 * TILE;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], s_empty[2], drain
  static constexpr int NBAR = 1 + 2 * STAGES + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
  static constexpr int OFF_XCH = OFF_MISC + 16;        // [groups-1][5][128] floats
  static constexpr int BYTES = OFF_XCH + (kGroups - 1) * 5 * kBlockM * 4;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024
};

struct RowState {
  float r1, l1, r2, l2, acc;  // r_t in log2 units; acc in raw dot-product units
};

// Fold one 32-column chunk of a row into the state. a = S1 row values, b = S2
// (raw dot products). With MASK, keys >= lim are excluded. Unless from_max,
// a row with finite references folds the chunk against them; a term that
// overflows there leaves NaN in l1 or l2 (inf times the 1/inf rescale), for
// the sweep from the maxima to rebuild. Otherwise the chunk's maximum moves
// the references first.
template <bool MASK>
__device__ __forceinline__ void fold_chunk(float (&a)[32], float (&b)[32], int key0, int lim,
                                           float c, RowState& st, bool from_max) {
  if (MASK) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      if (key0 + k >= lim) {
        a[k] = -INFINITY;
        b[k] = -INFINITY;
      }
    }
  }
  if (!from_max && st.r1 != -INFINITY && st.r2 != -INFINITY) {
    const float2 c2 = make_float2(c, c), m1 = make_float2(-1.f, -1.f);
    const float2 nr1 = make_float2(-st.r1, -st.r1), nr2 = make_float2(-st.r2, -st.r2);
    float2 l1p[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 l2p[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 ap[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      const float2 s1 = make_float2(a[k], a[k + 1]), s2 = make_float2(b[k], b[k + 1]);
      const float2 x1 = __ffma2_rn(s1, c2, nr1), x2 = __ffma2_rn(s2, c2, nr2);
      const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
      const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
      const int h = (k >> 1) & 1;
      l1p[h] = __fadd2_rn(l1p[h], p1);
      l2p[h] = __fadd2_rn(l2p[h], p2);
      float2 dd = __ffma2_rn(s2, m1, s1);  // s1 - s2
      if (MASK) {
        if (a[k] == -INFINITY) dd.x = 0.f;
        if (a[k + 1] == -INFINITY) dd.y = 0.f;
      }
      ap[h] = __ffma2_rn(p1, dd, ap[h]);
    }
    const float2 l1s = __fadd2_rn(l1p[0], l1p[1]), l2s = __fadd2_rn(l2p[0], l2p[1]);
    const float2 as = __fadd2_rn(ap[0], ap[1]);
    const float f1 = l1s.x + l1s.y, f2 = l2s.x + l2s.y, fa = as.x + as.y;
    if (f1 > kSumMax) {  // reference up by log2 f1: the state and this chunk scale by 1/f1
      const float inv = 1.f / f1;
      st.r1 += __log2f(f1);
      st.l1 = (st.l1 + f1) * inv;
      st.acc = (st.acc + fa) * inv;
    } else {
      st.l1 += f1;
      st.acc += fa;
    }
    if (f2 > kSumMax) {
      st.r2 += __log2f(f2);
      st.l2 = (st.l2 + f2) * (1.f / f2);
    } else {
      st.l2 += f2;
    }
    return;
  }
  float x1[11], x2[11];
#pragma unroll
  for (int k = 0; k < 10; ++k) {
    x1[k] = max3(a[3 * k], a[3 * k + 1], a[3 * k + 2]);
    x2[k] = max3(b[3 * k], b[3 * k + 1], b[3 * k + 2]);
  }
  x1[10] = fmaxf(a[30], a[31]);
  x2[10] = fmaxf(b[30], b[31]);
  const float cm1 = max3(max3(x1[0], x1[1], x1[2]), max3(x1[3], x1[4], x1[5]),
                         max3(max3(x1[6], x1[7], x1[8]), x1[9], x1[10]));
  const float cm2 = max3(max3(x2[0], x2[1], x2[2]), max3(x2[3], x2[4], x2[5]),
                         max3(max3(x2[6], x2[7], x2[8]), x2[9], x2[10]));
  if (MASK && cm1 == -INFINITY) return;  // no allowed key in this chunk
  const float t1 = cm1 * c, t2 = cm2 * c;
  if (t1 > st.r1 + kTau) {
    const float al = ex2(st.r1 - t1);
    st.l1 *= al;
    st.acc *= al;
    st.r1 = t1;
  }
  if (t2 > st.r2 + kTau) {
    st.l2 *= ex2(st.r2 - t2);
    st.r2 = t2;
  }
  const float2 c2 = make_float2(c, c), m1 = make_float2(-1.f, -1.f);
  const float2 nr1 = make_float2(-st.r1, -st.r1), nr2 = make_float2(-st.r2, -st.r2);
  float2 l1p[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 l2p[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 ap[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    const float2 s1 = make_float2(a[k], a[k + 1]), s2 = make_float2(b[k], b[k + 1]);
    const float2 x1 = __ffma2_rn(s1, c2, nr1), x2 = __ffma2_rn(s2, c2, nr2);
    const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
    const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
    const int h = (k >> 1) & 1;
    l1p[h] = __fadd2_rn(l1p[h], p1);
    l2p[h] = __fadd2_rn(l2p[h], p2);
    float2 dd = __ffma2_rn(s2, m1, s1);  // s1 - s2
    if (MASK) {
      if (a[k] == -INFINITY) dd.x = 0.f;
      if (a[k + 1] == -INFINITY) dd.y = 0.f;
    }
    ap[h] = __ffma2_rn(p1, dd, ap[h]);
  }
  const float2 l1s = __fadd2_rn(l1p[0], l1p[1]), l2s = __fadd2_rn(l2p[0], l2p[1]);
  const float2 as = __fadd2_rn(ap[0], ap[1]);
  st.l1 += l1s.x + l1s.y;
  st.l2 += l2s.x + l2s.y;
  st.acc += as.x + as.y;
}

// Merge state y into x (same row, disjoint key sets).
__device__ __forceinline__ void merge_state(RowState& x, const RowState& y) {
  const float R1 = fmaxf(x.r1, y.r1), R2 = fmaxf(x.r2, y.r2);
  if (R1 == -INFINITY) return;  // neither side saw an allowed key
  const float wx1 = ex2(x.r1 - R1), wy1 = ex2(y.r1 - R1);
  const float wx2 = ex2(x.r2 - R2), wy2 = ex2(y.r2 - R2);
  x.l1 = x.l1 * wx1 + y.l1 * wy1;
  x.acc = x.acc * wx1 + y.acc * wy1;
  x.l2 = x.l2 * wx2 + y.l2 * wy2;
  x.r1 = R1;
  x.r2 = R2;
}

__device__ __forceinline__ void finish_row(const RowState& s, float scale, float& kl, float& lse1,
                                           float& lse2) {
  lse1 = (s.r1 + log2f(s.l1)) * kLn2;
  lse2 = (s.r2 + log2f(s.l2)) * kLn2;
  kl = scale * (s.acc / s.l1) - lse1 + lse2;
}

// PACKED: a variable-length batch of packed sequences (no split-K) instead of
// dense [B, H, N, d] tensors; a template parameter so that the dense kernel
// keeps its sizes as kernel parameters.
template <int D, bool SPLIT, bool PACKED>
__global__ void __launch_bounds__(kFwdThreads, 1)
    streamkl_fwd_kernel(const __grid_constant__ CUtensorMap tm_q1,
                        const __grid_constant__ CUtensorMap tm_k1,
                        const __grid_constant__ CUtensorMap tm_q2,
                        const __grid_constant__ CUtensorMap tm_k2, int NQ, int NK, int causal,
                        float scale, float* __restrict__ kl_out, float* __restrict__ lse1_out,
                        float* __restrict__ lse2_out, float* __restrict__ part, int splits,
                        int tiles_per_split, long long plane, const int* __restrict__ cu_q,
                        const int* __restrict__ cu_k, int H, int total_q, int total_k,
                        int* dev_status, uint64_t timeout_ns) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int split = static_cast<int>(blockIdx.y);
  const int bh = static_cast<int>(blockIdx.z);
  // this (batch, head) slice: the whole tensor's sizes, or one sequence of a
  // packed variable-length batch (the grid covers the longest one)
  const SeqView sv = PACKED ? seq_view_packed(bh, H, NQ, NK, D, cu_q, cu_k, total_q, total_k)
                            : seq_view_dense(bh, NQ, NK, D);
  const int nq = sv.nq, nk = sv.nk;
  const int nqb = (nq + kBlockM - 1) / kBlockM;
  const bool active = sv.ok && static_cast<int>(blockIdx.x) < nqb && !(causal && nq > nk);
  const int qb = causal ? (nqb - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int off = nk - nq;
  const int row_hi = min(nq, (qb + 1) * kBlockM);  // exclusive
  const int klim_blk = causal ? min(nk, row_hi + off) : nk;
  const int n_tiles = (klim_blk + kBlockN - 1) / kBlockN;
  const int t_begin = SPLIT ? split * tiles_per_split : 0;
  const int t_end = SPLIT ? min(n_tiles, t_begin + tiles_per_split) : n_tiles;
  int n_iter = active ? max(0, t_end - t_begin) : 0;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t q_full = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + L::STAGES + s); };
  auto s_full = [&](int k) { return bar0 + 8u * (1 + 2 * L::STAGES + k); };
  auto s_empty = [&](int k) { return bar0 + 8u * (3 + 2 * L::STAGES + k); };
  const uint32_t drain = bar0 + 8u * (5 + 2 * L::STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);
  volatile int* redo_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 12);

  // debug build: the layout's regions (TMEM fields are set once allocated)
  CheckCtx ck{sb, sb + L::OFF_BAR, sb + L::OFF_BAR, sb + L::OFF_BAR + L::NBAR * 8, 0, 0,
              abort_flag, dev_status};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *redo_flag = 0;
    bool lay_ok = true;
    if (kDeviceChecks) {  // every barrier address inside the barrier region
      lay_ok = check_bar(ck, q_full, __LINE__) && check_bar(ck, drain, __LINE__);
      for (int s = 0; s < L::STAGES; ++s)
        lay_ok = lay_ok && check_bar(ck, kv_full(s), __LINE__) && check_bar(ck, kv_empty(s), __LINE__);
      for (int k = 0; k < 2; ++k)
        lay_ok = lay_ok && check_bar(ck, s_full(k), __LINE__) && check_bar(ck, s_empty(k), __LINE__);
    }
    if (lay_ok) {
      mbar_init(q_full, 1);
      for (int s = 0; s < L::STAGES; ++s) {
        mbar_init(kv_full(s), 1);
        mbar_init(kv_empty(s), 1);
      }
      for (int k = 0; k < 2; ++k) {
        mbar_init(s_full(k), 1);
        mbar_init(s_empty(k), 4 * kGroups);  // one arrival per softmax warp
      }
      mbar_init(drain, 1);
    }
    // a failure recorded earlier (this launch or a previous one), or a
    // failed layout check, skips the work
    *skip_flag = !lay_ok || *reinterpret_cast<volatile int*>(dev_status) != 0;
    // malformed sequence offsets, or a causal sequence with more query rows
    // than keys (its first rows would see no key): reported, never computed
    if (!sv.ok || (causal && nq > nk)) atomicCAS(dev_status, 0, kStatusInvalidArg);
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
  // TMA coordinate extents: rows of the Q and K maps, their third dimension
  const int q_rows = PACKED ? total_q : NQ, k_rows = PACKED ? total_k : NK;
  const int z_hi = PACKED ? H : static_cast<int>(gridDim.z);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool q_ok = true;
    if (kDeviceChecks && lane == 0 && n_iter > 0)
      for (int kb = 0; kb < L::KB; ++kb)
        q_ok = q_ok &&
               check_tma(ck, sb + L::OFF_Q1 + kb * 16384, 16384, q_full, kb * 64, D,
                         sv.q_row0 + qb * kBlockM, q_rows, kBlockM, sv.z, z_hi, __LINE__) &&
               check_tma(ck, sb + L::OFF_Q2 + kb * 16384, 16384, q_full, kb * 64, D,
                         sv.q_row0 + qb * kBlockM, q_rows, kBlockM, sv.z, z_hi, __LINE__);
    if (lane == 0 && n_iter > 0 && q_ok) {
      mbar_arrive_expect_tx(q_full, 2 * L::TILE);
#pragma unroll
      for (int kb = 0; kb < L::KB; ++kb) {
        tma_load_3d(sb + L::OFF_Q1 + kb * 16384, &tm_q1, q_full, kb * 64, sv.q_row0 + qb * kBlockM,
                    sv.z);
        tma_load_3d(sb + L::OFF_Q2 + kb * 16384, &tm_q2, q_full, kb * 64, sv.q_row0 + qb * kBlockM,
                    sv.z);
      }
      int g = 0;  // key tiles loaded so far, over both sweeps
      for (int pass = 0; pass < 2; ++pass) {
      if (pass == 1) {
        // a second sweep when a chunk overflowed against its reference
        cta_barrier_divergent();
        if (!*redo_flag) break;
      }
      for (int it = 0; it < n_iter; ++it, ++g) {
        const int s = g % L::STAGES;
        const uint32_t ph = (g / L::STAGES) & 1;
        if (!wait_bounded(kv_empty(s), ph ^ 1, wc)) break;
        const int krow = sv.k_row0 + (t_begin + it) * kBlockN;
        const uint32_t dst = sb + L::OFF_K + s * 2 * L::TILE;
        bool k_ok = true;
        if (kDeviceChecks)
          for (int kb = 0; kb < L::KB; ++kb)
            k_ok = k_ok &&
                   check_tma(ck, dst + kb * 16384, 16384, kv_full(s), kb * 64, D, krow, k_rows,
                             kBlockN, sv.z, z_hi, __LINE__) &&
                   check_tma(ck, dst + L::TILE + kb * 16384, 16384, kv_full(s), kb * 64, D, krow,
                             k_rows, kBlockN, sv.z, z_hi, __LINE__);
        if (!k_ok) break;
        mbar_arrive_expect_tx(kv_full(s), 2 * L::TILE);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
          tma_load_3d(dst + kb * 16384, &tm_k1, kv_full(s), kb * 64, krow, sv.z);
          tma_load_3d(dst + L::TILE + kb * 16384, &tm_k2, kv_full(s), kb * 64, krow, sv.z);
        }
      }
      }
      // Let every copy this thread issued land before the CTA can exit.
      wait_drain(q_full, 0, timeout_ns);
      for (int j = max(0, g - L::STAGES); j < g; ++j)
        wait_drain(kv_full(j % L::STAGES), (j / L::STAGES) & 1, timeout_ns);
    } else {
      cta_barrier_divergent();  // the first sweep's end (every thread takes part once)
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idesc = idesc_bf16(kBlockM, kBlockN, 0, 0);
      bool ok = wait_bounded(q_full, 0, wc);
      tc_fence_after();
      int g = 0;  // key tiles so far, over both sweeps
      for (int pass = 0; pass < 2; ++pass) {
      if (pass == 1) {
        cta_barrier_divergent();  // the first sweep's end
        if (!*redo_flag) break;
      }
      for (int it = 0; ok && it < n_iter; ++it, ++g) {
        const int s = g % L::STAGES;
        const uint32_t ph = (g / L::STAGES) & 1;
        const int slot = g & 1;
        const uint32_t sph = (g >> 1) & 1;
        if (!(ok = wait_bounded(kv_full(s), ph, wc))) break;
        if (!(ok = wait_bounded(s_empty(slot), sph ^ 1, wc))) break;
        tc_fence_after();
        const uint32_t kbase = sb + L::OFF_K + s * 2 * L::TILE;
        const uint32_t d1 = tmem + slot * 256, d2 = d1 + 128;
        if (!(ok = check_tmem(ck, d1, 128, 256, __LINE__))) break;
        // the two GEMMs' k-steps interleaved: independent accumulators keep
        // the tensor pipe busy where one dependent chain would stall it
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
          mma_bf16(d1, smem_desc_sw128(sb + L::OFF_Q1 + koff, 16, 1024),
                   smem_desc_sw128(kbase + koff, 16, 1024), idesc, k > 0);
          mma_bf16(d2, smem_desc_sw128(sb + L::OFF_Q2 + koff, 16, 1024),
                   smem_desc_sw128(kbase + L::TILE + koff, 16, 1024), idesc, k > 0);
        }
        mma_commit(s_full(slot));
      }
      }
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    } else {
      cta_barrier_divergent();  // the first sweep's end (every thread takes part once)
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax / KL
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qrow = qb * kBlockM + r;
    const float c = scale * kLog2e;
    const int lim = causal ? min(nk, qrow + 1 + off) : nk;  // keys < lim visible
    RowState st;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + grp * 32;
    int g = 0;  // key tiles so far, over both sweeps
    for (int pass = 0; pass < 2; ++pass) {
      if (pass == 1) {
        cta_barrier_divergent();  // the first sweep's end: did any chunk overflow?
        if (!*redo_flag) break;
      }
      st = RowState{-INFINITY, 0.f, -INFINITY, 0.f, 0.f};
      for (int it = 0; it < n_iter; ++it, ++g) {
        const int slot = g & 1;
        const uint32_t sph = (g >> 1) & 1;
        if (!wait_bounded(s_full(slot), sph, wc)) break;
        // the S GEMMs were the K stage's only readers
        if (warp == 2 && lane == 0) mbar_arrive(kv_empty(g % L::STAGES));
        tc_fence_after();
        float a[32], b[32];
        const uint32_t ta = lane_base + slot * 256;
        if (!(check_tmem(ck, ta, 32, 32, __LINE__) && check_tmem(ck, ta + 128, 32, 32, __LINE__)))
          break;
        tmem_ld32(ta, a);
        tmem_ld32(ta + 128, b);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(slot));
        const int key0 = (t_begin + it) * kBlockN + grp * 32;
        if (key0 + 32 <= lim)
          fold_chunk<false>(a, b, key0, lim, c, st, pass > 0);
        else
          fold_chunk<true>(a, b, key0, lim, c, st, pass > 0);
      }
      // an overflowed chunk left NaN in l1 or l2 (inf times the 1/inf rescale)
      if (pass == 0 && !(st.l1 == st.l1 && st.l2 == st.l2)) *redo_flag = 1;
    }
    // merge the column groups' states of each row into group 0
    float* xch = reinterpret_cast<float*>(gb + L::OFF_XCH);
    if (grp > 0) {
      float* x = xch + (grp - 1) * 5 * kBlockM;
      x[0 * kBlockM + r] = st.r1;
      x[1 * kBlockM + r] = st.l1;
      x[2 * kBlockM + r] = st.r2;
      x[3 * kBlockM + r] = st.l2;
      x[4 * kBlockM + r] = st.acc;
    }
    named_bar_sync(1, 32 * 4 * kGroups);
    if (grp == 0) {
#pragma unroll
      for (int gq = 0; gq < kGroups - 1; ++gq) {
        const float* x = xch + gq * 5 * kBlockM;
        const RowState other{x[0 * kBlockM + r], x[1 * kBlockM + r], x[2 * kBlockM + r],
                             x[3 * kBlockM + r], x[4 * kBlockM + r]};
        merge_state(st, other);
      }
      if (active && qrow < nq) {
        const size_t o = static_cast<size_t>(sv.v_off + static_cast<long long>(qrow) * sv.v_stride);
        // (the debug build skips an out-of-range row's writes)
        if (!dcheck(ck, o < static_cast<size_t>(plane), __LINE__)) {
        } else if (SPLIT) {
          const size_t base = static_cast<size_t>(split) * plane + o;
          const size_t fstride = static_cast<size_t>(splits) * plane;
          part[0 * fstride + base] = st.r1;
          part[1 * fstride + base] = st.l1;
          part[2 * fstride + base] = st.r2;
          part[3 * fstride + base] = st.l2;
          part[4 * fstride + base] = st.acc;
        } else {
          float kl, l1, l2;
          finish_row(st, scale, kl, l1, l2);
          kl_out[o] = kl;
          lse1_out[o] = l1;
          lse2_out[o] = l2;
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

// ---------------------------------------------------------------------------
// The same forward as CTA pairs (dense batches, no split, an even number of
// query blocks). A cluster of two CTAs takes two query blocks of one
// (batch, head) slice and runs S1, S2 as tcgen05 MMAs with M = 256 over both
// (cta_group::2): each CTA keeps its own Q tile and loads only half of every
// key tile (64 keys), and the MMAs read the other half from the peer's shared
// memory. Per CTA that halves the key bytes loaded and the B-operand bytes
// the MMAs read, the shared-memory traffic the single-CTA kernel's MMAs are
// bound by. The even CTA issues the MMAs; the odd CTA's warp 1 relays the
// arrival of its Q tile and key halves to the even CTA's barriers; both
// CTAs' softmax warps free an S buffer on the even CTA's barrier; the even
// CTA's commits arrive on both CTAs' barriers. Each CTA reads its own rows of
// S from its own TMEM, so the softmax / KL part is the single-CTA kernel's.
// The pair sweeps the key tiles of its later query block; the earlier block
// masks the keys past its frontier.
template <int D>
struct PairLayout {
  static constexpr int KB = D / 64;
  static constexpr int TILE = kBlockM * D * 2;     // one 128-row Q tile
  static constexpr int HALF = 64 * D * 2;          // 64 rows of one K tensor
  static constexpr int STAGES = D == 128 ? 4 : 8;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = TILE;
  static constexpr int OFF_K = 2 * TILE;           // stage s: K1 half at +2s HALF, K2 half at +(2s+1) HALF
  static constexpr int OFF_BAR = OFF_K + STAGES * 2 * HALF;
  // q_full, q_peer, kv_full[S], kv_peer[S], kv_empty[S], s_full[2], s_empty[2], drain
  static constexpr int NBAR = 2 + 3 * STAGES + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_XCH = OFF_MISC + 16;
  static constexpr int BYTES = OFF_XCH + (kGroups - 1) * 5 * kBlockM * 4;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    streamkl_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q1,
                             const __grid_constant__ CUtensorMap tm_k1,
                             const __grid_constant__ CUtensorMap tm_q2,
                             const __grid_constant__ CUtensorMap tm_k2, int NQ, int NK, int causal,
                             float scale, float* __restrict__ kl_out, float* __restrict__ lse1_out,
                             float* __restrict__ lse2_out, int* dev_status, uint64_t timeout_ns) {
  using L = PairLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int bh = static_cast<int>(blockIdx.z);
  const int nqb = (NQ + kBlockM - 1) / kBlockM;  // even
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  // causal: heavy pairs first; the even CTA takes the later block of the pair
  const int qb_hi = causal ? nqb - 1 - 2 * pair : 2 * pair + 1;
  const int qb = rank == 0 ? qb_hi : qb_hi - 1;
  const int off = NK - NQ;
  const int klim_pair = causal ? min(NK, min(NQ, (qb_hi + 1) * kBlockM) + off) : NK;
  int n_iter = (klim_pair + kBlockN - 1) / kBlockN;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t q_full = bar0, q_peer = bar0 + 8;
  auto kv_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto kv_peer = [&](int s) { return bar0 + 8u * (2 + L::STAGES + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (2 + 2 * L::STAGES + s); };
  auto s_full = [&](int k) { return bar0 + 8u * (2 + 3 * L::STAGES + k); };
  auto s_empty = [&](int k) { return bar0 + 8u * (4 + 3 * L::STAGES + k); };
  const uint32_t drain = bar0 + 8u * (6 + 3 * L::STAGES);
  static_assert(2 + 3 * L::STAGES + 4 + 1 == L::NBAR, "barrier region holds every barrier");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);

  CheckCtx ck{sb, sb + L::OFF_BAR, sb + L::OFF_BAR, sb + L::OFF_BAR + L::NBAR * 8, 0, 0,
              abort_flag, dev_status};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    bool lay_ok = true;
    if (kDeviceChecks) {  // every barrier address inside the barrier region
      lay_ok = check_bar(ck, q_full, __LINE__) && check_bar(ck, q_peer, __LINE__) &&
               check_bar(ck, drain, __LINE__);
      for (int s = 0; s < L::STAGES; ++s)
        lay_ok = lay_ok && check_bar(ck, kv_full(s), __LINE__) && check_bar(ck, kv_peer(s), __LINE__) &&
                 check_bar(ck, kv_empty(s), __LINE__);
      for (int k = 0; k < 2; ++k)
        lay_ok = lay_ok && check_bar(ck, s_full(k), __LINE__) && check_bar(ck, s_empty(k), __LINE__);
    }
    if (lay_ok) {
      mbar_init(q_full, 1);
      mbar_init(q_peer, 1);
      for (int s = 0; s < L::STAGES; ++s) {
        mbar_init(kv_full(s), 1);
        mbar_init(kv_peer(s), 1);
        mbar_init(kv_empty(s), 1);
      }
      for (int k = 0; k < 2; ++k) {
        mbar_init(s_full(k), 1);
        mbar_init(s_empty(k), 2 * 4 * kGroups);  // one arrival per softmax warp of both CTAs
      }
      mbar_init(drain, 1);
    }
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
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before either arrives on the other's
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (*skip_flag) n_iter = 0;
  const WaitCtx wc{abort_flag, dev_status, timeout_ns};
  ck.tmem = tmem;
  ck.tmem_cols = 512;
  const int z_hi = static_cast<int>(gridDim.z);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // this CTA's Q tile once, then its half (keys [64 rank, 64 rank + 64)) of
    // every key tile through its own ring
    if (lane == 0 && n_iter > 0) {
      bool ok = true;
      if (kDeviceChecks)
        for (int kb = 0; kb < L::KB; ++kb)
          ok = ok &&
               check_tma(ck, sb + L::OFF_Q1 + kb * 16384, 16384, q_full, kb * 64, D, qb * kBlockM,
                         NQ, kBlockM, bh, z_hi, __LINE__) &&
               check_tma(ck, sb + L::OFF_Q2 + kb * 16384, 16384, q_full, kb * 64, D, qb * kBlockM,
                         NQ, kBlockM, bh, z_hi, __LINE__);
      int it = 0;
      if (ok) {
        mbar_arrive_expect_tx(q_full, 2 * L::TILE);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
          tma_load_3d(sb + L::OFF_Q1 + kb * 16384, &tm_q1, q_full, kb * 64, qb * kBlockM, bh);
          tma_load_3d(sb + L::OFF_Q2 + kb * 16384, &tm_q2, q_full, kb * 64, qb * kBlockM, bh);
        }
        for (; it < n_iter; ++it) {
          const int s = it % L::STAGES;
          if (!wait_bounded(kv_empty(s), ((it / L::STAGES) & 1) ^ 1, wc)) break;
          const int krow = it * kBlockN + 64 * static_cast<int>(rank);
          const uint32_t dst = sb + L::OFF_K + s * 2 * L::HALF;
          bool k_ok = true;
          if (kDeviceChecks)
            for (int kb = 0; kb < L::KB; ++kb)
              k_ok = k_ok &&
                     check_tma(ck, dst + kb * 8192, 8192, kv_full(s), kb * 64, D, krow, NK, 64, bh,
                               z_hi, __LINE__) &&
                     check_tma(ck, dst + L::HALF + kb * 8192, 8192, kv_full(s), kb * 64, D, krow, NK,
                               64, bh, z_hi, __LINE__);
          if (!k_ok) break;
          mbar_arrive_expect_tx(kv_full(s), 2 * L::HALF);
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb) {
            tma_load_3d(dst + kb * 8192, &tm_k1, kv_full(s), kb * 64, krow, bh);
            tma_load_3d(dst + L::HALF + kb * 8192, &tm_k2, kv_full(s), kb * 64, krow, bh);
          }
        }
        // let every copy this thread issued land before the CTA can exit
        wait_drain(q_full, 0, timeout_ns);
        for (int j = max(0, it - L::STAGES); j < it; ++j)
          wait_drain(kv_full(j % L::STAGES), (j / L::STAGES) & 1, timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && n_iter > 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      constexpr uint32_t idesc = idesc_bf16(2 * kBlockM, kBlockN, 0, 0);
      bool ok = check_tmem(ck, tmem, 128, 512, __LINE__) && wait_bounded(q_full, 0, wc) &&
                wait_bounded(q_peer, 0, wc);
      tc_fence_after();
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % L::STAGES;
        const uint32_t ph = (it / L::STAGES) & 1;
        const int slot = it & 1;
        const uint32_t sph = (it >> 1) & 1;
        if (!(ok = wait_bounded(kv_full(s), ph, wc) && wait_bounded(kv_peer(s), ph, wc))) break;
        if (!(ok = wait_bounded(s_empty(slot), sph ^ 1, wc))) break;
        tc_fence_after();
        const uint32_t kbase = sb + L::OFF_K + s * 2 * L::HALF;
        const uint32_t d1 = tmem + slot * 256, d2 = d1 + 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qoff = (k >> 2) * 16384 + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * 8192 + (k & 3) * 32;
          mma_bf16_pair(d1, smem_desc_sw128(sb + L::OFF_Q1 + qoff, 16, 1024),
                        smem_desc_sw128(kbase + koff, 16, 1024), idesc, k > 0);
          mma_bf16_pair(d2, smem_desc_sw128(sb + L::OFF_Q2 + qoff, 16, 1024),
                        smem_desc_sw128(kbase + L::HALF + koff, 16, 1024), idesc, k > 0);
        }
        mma_commit_pair(s_full(slot));
        mma_commit_pair(kv_empty(s));
      }
      mma_commit_pair(drain);
      wait_drain(drain, 0, timeout_ns);
    } else if (lane == 0 && n_iter > 0) {
      // ---------------------------------------------------------- relay (odd CTA)
      // this CTA's Q tile and key halves have landed: tell the even CTA
      bool ok = wait_bounded(q_full, 0, wc);
      if (ok) mbar_arrive_cluster(mapa_shared(q_peer, 0));
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % L::STAGES;
        if (!(ok = wait_bounded(kv_full(s), (it / L::STAGES) & 1, wc))) break;
        mbar_arrive_cluster(mapa_shared(kv_peer(s), 0));
      }
      // the even CTA's MMAs (which read this CTA's shared memory and write
      // its TMEM) have ended
      wait_drain(drain, 0, timeout_ns);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax / KL
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qrow = qb * kBlockM + r;
    const float c = scale * kLog2e;
    const int lim = causal ? min(NK, qrow + 1 + off) : NK;  // keys < lim visible
    RowState st{-INFINITY, 0.f, -INFINITY, 0.f, 0.f};
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + grp * 32;
    for (int it = 0; it < n_iter; ++it) {
      const int slot = it & 1;
      const uint32_t sph = (it >> 1) & 1;
      if (!wait_bounded(s_full(slot), sph, wc)) break;
      tc_fence_after();
      float a[32], b[32];
      const uint32_t ta = lane_base + slot * 256;
      if (!(check_tmem(ck, ta, 32, 32, __LINE__) && check_tmem(ck, ta + 128, 32, 32, __LINE__)))
        break;
      tmem_ld32(ta, a);
      tmem_ld32(ta + 128, b);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      // S of this slot is in registers (tcgen05.wait::ld above): free it on
      // the even CTA's barrier; the arrival publishes no memory, so relaxed
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(s_empty(slot), 0));
      const int key0 = it * kBlockN + grp * 32;
      // (the pair kernel folds every chunk from its maximum)
      if (key0 + 32 <= lim)
        fold_chunk<false>(a, b, key0, lim, c, st, true);
      else
        fold_chunk<true>(a, b, key0, lim, c, st, true);
    }
    float* xch = reinterpret_cast<float*>(gb + L::OFF_XCH);
    if (grp > 0) {
      float* x = xch + (grp - 1) * 5 * kBlockM;
      x[0 * kBlockM + r] = st.r1;
      x[1 * kBlockM + r] = st.l1;
      x[2 * kBlockM + r] = st.r2;
      x[3 * kBlockM + r] = st.l2;
      x[4 * kBlockM + r] = st.acc;
    }
    named_bar_sync(1, 32 * 4 * kGroups);
    if (grp == 0) {
#pragma unroll
      for (int gq = 0; gq < kGroups - 1; ++gq) {
        const float* x = xch + gq * 5 * kBlockM;
        const RowState other{x[0 * kBlockM + r], x[1 * kBlockM + r], x[2 * kBlockM + r],
                             x[3 * kBlockM + r], x[4 * kBlockM + r]};
        merge_state(st, other);
      }
      if (n_iter > 0 && qrow < NQ) {
        const size_t o = static_cast<size_t>(bh) * NQ + qrow;
        float kl, l1, l2;
        finish_row(st, scale, kl, l1, l2);
        kl_out[o] = kl;
        lse1_out[o] = l1;
        lse2_out[o] = l2;
      }
    }
  }

  // neither CTA releases TMEM or leaves while the pair still works on it
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
  cluster_sync();
}

// One thread per (bh, row): merge the split partial states and finish.
__global__ void streamkl_fwd_combine_kernel(const float* __restrict__ part, int splits,
                                            long long plane, float scale,
                                            float* __restrict__ kl_out,
                                            float* __restrict__ lse1_out,
                                            float* __restrict__ lse2_out) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= plane) return;
  const long long fstride = static_cast<long long>(splits) * plane;
  RowState st{-INFINITY, 0.f, -INFINITY, 0.f, 0.f};
  for (int s = 0; s < splits; ++s) {
    const long long b = s * plane + i;
    const RowState y{part[b], part[fstride + b], part[2 * fstride + b], part[3 * fstride + b],
                     part[4 * fstride + b]};
    merge_state(st, y);
  }
  float kl, l1, l2;
  finish_row(st, scale, kl, l1, l2);
  kl_out[i] = kl;
  lse1_out[i] = l1;
  lse2_out[i] = l2;
}

template <int D>
cudaError_t launch_fwd_pair_t(const FwdArgs& a, cudaStream_t stream) {
  using L = PairLayout<D>;
  auto kern = streamkl_fwd_pair_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const int nqb = (a.NQ + kBlockM - 1) / kBlockM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nqb, 1, a.BH);
  cfg.blockDim = dim3(kFwdThreads, 1, 1);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *a.tm_q1, *a.tm_k1, *a.tm_q2, *a.tm_k2, a.NQ, a.NK, a.causal,
                            a.scale, a.kl, a.lse1, a.lse2, a.dev_status, a.timeout_ns);
}

template <int D, bool SPLIT, bool PACKED>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = streamkl_fwd_kernel<D, SPLIT, PACKED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const int nqb = (a.NQ + kBlockM - 1) / kBlockM;
  dim3 grid(nqb, SPLIT ? a.splits : 1, a.BH);
  kern<<<grid, kFwdThreads, L::ALLOC, stream>>>(*a.tm_q1, *a.tm_k1, *a.tm_q2, *a.tm_k2, a.NQ, a.NK,
                                                a.causal, a.scale, a.kl, a.lse1, a.lse2, a.part,
                                                a.splits, a.tiles_per_split, a.plane, a.cu_q, a.cu_k,
                                                a.H, a.total_q, a.total_k, a.dev_status,
                                                a.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int d) {
  return d == 128 ? FwdLayout<128>::ALLOC : FwdLayout<64>::ALLOC;
}

bool fwd_pair_eligible(int NQ, int splits, bool packed) {
  const int nqb = (NQ + kBlockM - 1) / kBlockM;
  return !packed && splits <= 1 && nqb % 2 == 0;
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.pairs) return a.d == 128 ? launch_fwd_pair_t<128>(a, stream) : launch_fwd_pair_t<64>(a, stream);
  const bool split = a.splits > 1;
  if (a.cu_q != nullptr)  // packed batches never split
    return a.d == 128 ? launch_fwd_t<128, false, true>(a, stream) : launch_fwd_t<64, false, true>(a, stream);
  if (a.d == 128)
    return split ? launch_fwd_t<128, true, false>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
  return split ? launch_fwd_t<64, true, false>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
}

cudaError_t launch_fwd_combine(const FwdArgs& a, cudaStream_t stream) {
  const long long plane = a.plane;
  const int threads = 256;
  const long long blocks = (plane + threads - 1) / threads;
  streamkl_fwd_combine_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      a.part, a.splits, plane, a.scale, a.kl, a.lse1, a.lse2);
  return cudaGetLastError();
}

}  // namespace skl

// Backward pass as two separate kernels without atomics (gist.science
// technical summary, "Metodologia" section 2, kernel fusion paragraph: when
// dQ accumulation across key tiles contends too much, dK and dQ are computed
// by separate kernels). Probabilities are regenerated tile by tile from Q, K
// and the saved LSEs, P_t = exp(S_t - LSE_t).
//
// One template serves both kernels. A CTA keeps 128 rows of a "stationary"
// tensor pair X1, X2 in shared memory and streams steps of STEP rows of the
// other pair Y1, Y2 through a ring of 4-8 stages (STEP = 64; 128 in the dQ
// kernel with one gradient set at d = 64):
//   dQ kernel: X = Q (query block), Y = K steps;  acc_t += dS_t   K_t
//   dK kernel: X = K (key block),   Y = Q steps;  acc_t += dS_t^T Q_t
// In both, T_t = X_t Y_t^T (M = 128 X rows, N = STEP Y rows) is the score
// tile seen from the X side (S_t in the dQ kernel, S_t^T in the dK kernel),
// the softmax warps turn T1, T2 into the matching dS tiles and the gradient
// GEMM is acc_t += dT_t Y_t (M = 128, N = d, K = STEP), accumulated in TMEM
// over the whole sweep and written out once. With few query blocks the dQ kernel
// also splits its keys across CTAs (grid z): each split writes its
// accumulator as an fp32 partial and a combine kernel sums the partials.
//
// dS never goes through shared memory: each softmax thread owns one X row,
// which is one TMEM lane, so it stores its bf16 dS values straight into TMEM
// and the gradient GEMMs read their A operand from there. TMEM columns (64-row
// steps): T [0,128) (T1 low 64, T2 high 64) | dS buffer 0 [128,192) | dS
// buffer 1 [192,256) (set 2 low 32, set 1 high 32) | acc set 2 [256, 256+d) |
// acc set 1; 128-row steps (one set): T1, T2 128 each | two 64-column dS
// buffers | acc.
// Shared memory holds only X (64 KB at d = 128), the Y ring and, in the dK
// kernel, a per-stage table of per-query constants. The T GEMMs of step j+1
// are issued as soon as the softmax warps have loaded T of step j, and run
// while those warps compute dS of step j; the gradient GEMMs of step j follow
// once that dS is in TMEM. With double-buffered dS the softmax warps never
// wait on a gradient GEMM, and the deep Y ring keeps each tile's load well
// ahead of its first use.
//
// Gradients of L = sum_i g_i KL_i, with s = scale * q.k (g and scale folded
// into dS):
//   configuration 1 (teacher P1 fixed):  dS2 = g * (P2 - P1)
//   configuration 2 (student P2 fixed):  dS1 = g * P1 * (log(P1/P2) - KL)
// with log(P1/P2) - KL = scale (s1 - s2) - (LSE1 - LSE2 + KL) from logits and
// the saved LSEs (section 3, numerical stability); the logit difference comes
// first, so equal inputs give exactly zero.
//
// Warps: 0 = TMA producer (lane 0) and, in the dK kernel, the per-query
// constant table of each Y stage (all lanes); 1 = TMEM owner + T-GEMM issuer;
// 18 = gradient-GEMM issuer; 2..17 = softmax and epilogue. Warp w reads TMEM lanes [32 (w%4), +32) (its
// quarter) and serves column group g = (w-2)/4: thread = X row (TMEM lane),
// owning Y columns [g STEP/4, (g+1) STEP/4) of every step and, at the end, d columns
// [g d/4, (g+1) d/4) of its output row. Per-query constants (LSE1, LSE2, g,
// KL) are per row in the dQ kernel (registers) and per column in the dK kernel
// (the table, written next to each Y stage and published by its barrier).
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kSepThreads = 608;  // 19 warps
constexpr int kGradWarp = 18;     // issues the gradient GEMMs
constexpr int kSoftmaxWarps = 16;
constexpr int kBoxRows = 64;      // rows of one TMA box
constexpr float kLog2e = 1.4426950408889634f;

// Gradient sets a launch computes (bit mask): configuration 1 (P1 fixed)
// gives dQ2/dK2 from dS2, configuration 2 (P2 fixed) gives dQ1/dK1 from dS1.
constexpr int kSet2 = 1, kSet1 = 2;

template <int D, bool DQ, int SETS>
struct SepLayout {
  static constexpr int KB = D / 64;                   // 128-byte boxes per row
  static constexpr int XT = kBlockM * D * 2;          // 128 rows of one X tensor
  static constexpr int NSETS = SETS == (kSet1 | kSet2) ? 2 : 1;
  // Y rows per step: 128 in the dQ kernel with one gradient set at d = 64
  // (T1, T2 at N = 128, where the T GEMMs run at the tensor pipe's full rate
  // against two thirds of it at N = 64, and two dS buffers fit TMEM next to
  // one accumulator; five 32 KB Y stages fit shared memory); 64 otherwise:
  // two accumulators leave TMEM room for N = 64 only, the dK kernel's
  // per-column constants and 32 columns per thread spill its registers, and
  // at d = 128 only two 64 KB stages fit, which exposes the tile loads
  // (measured: mid and split-K backward 14-17 % slower than with 64-row steps)
  static constexpr int STEP = (NSETS == 1 && DQ && D == 64) ? 128 : 64;
  static constexpr int YT = STEP * D * 2;             // one Y tensor of a step
  static constexpr int YBOX = STEP * 128;             // one 64-column box of it
  static constexpr int NCOL = STEP / 4;               // Y columns per softmax thread
  // as many Y stages as fit next to X (and the dK kernel's tables)
  static constexpr int STAGES = STEP == 128 ? (D == 64 ? 5 : 2) : (D == 64 ? 8 : (DQ ? 5 : 4));
  static constexpr int OFF_X = 0;                     // X1, X2
  static constexpr int OFF_Y = 2 * XT;                // stage s: Y1 at +2s YT, Y2 at +(2s+1) YT
  static constexpr int OFF_TAB = OFF_Y + STAGES * 2 * YT;  // dK: [stage][4][STEP] float
  static constexpr int TAB_BYTES = DQ ? 0 : STAGES * 4 * STEP * 4;
  static constexpr int OFF_BAR = OFF_TAB + TAB_BYTES;
  // x_full, y_full[S], y_empty[S], s_full, s_free, ds_full[2], ds_free[2],
  // acc_full, drain, x_free, acc_empty (these two: persistent kernel), ep_full,
  // ep_empty (output staging)
  static constexpr int NBAR = 1 + 2 * STAGES + 12;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  // TMEM: T1 [0, STEP), T2 [STEP, 2 STEP) | dS buffers 0, 1 (DSW columns
  // each: STEP/2 packed columns per set) | accumulators (D columns per set)
  static constexpr uint32_t COL_T = 0, COL_DS = 2 * STEP, DSW = NSETS * STEP / 2;
  static constexpr uint32_t COL_ACC = COL_DS + 2 * DSW;
  static_assert(COL_ACC + NSETS * D <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Per-query constants: LSE1 log2e, LSE2 log2e, g scale, LSE1 - LSE2 + KL.
// Rows past N_Q get all zeros (g = 0: no gradient).
__device__ __forceinline__ float4 query_const(const float* lse1, const float* lse2, const float* g,
                                              const float* kl, size_t o, float scale, bool valid) {
  float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) {
    const float l1 = lse1[o], l2 = lse2[o];
    q = make_float4(l1 * kLog2e, l2 * kLog2e, g[o] * scale, l1 - l2 + kl[o]);
  }
  return q;
}

// PACKED: a variable-length batch of packed sequences instead of dense
// [B, H, N, d] tensors; a template parameter so that the dense kernel keeps
// its sizes as kernel parameters. PERSIST (dK kernel, dense batches): each
// CTA takes (key block, batch-head) items round-robin, heavy key blocks
// first, and loads the next item's X as soon as the last T GEMMs of the
// current one have read X; for short query sweeps, where a CTA's fixed start
// and end would otherwise weigh.
template <int D, bool DQ, int SETS, bool PACKED, bool PERSIST>
__global__ void __launch_bounds__(kSepThreads, 1)
    streamkl_bwd_sep_kernel(const __grid_constant__ CUtensorMap tm_x1,
                            const __grid_constant__ CUtensorMap tm_x2,
                            const __grid_constant__ CUtensorMap tm_y1,
                            const __grid_constant__ CUtensorMap tm_y2,
                            const __grid_constant__ CUtensorMap tm_o2,
                            const __grid_constant__ CUtensorMap tm_o1, int NQ, int NK,
                            int causal, float scale, const float* __restrict__ kl_in,
                            const float* __restrict__ lse1_in, const float* __restrict__ lse2_in,
                            const float* __restrict__ g_in, __nv_bfloat16* __restrict__ out2,
                            __nv_bfloat16* __restrict__ out1, float* __restrict__ part,
                            int splits, int split_steps, int n_bh, const int* __restrict__ cu_q,
                            const int* __restrict__ cu_k, int H, int total_q, int total_k,
                            int* dev_status, uint64_t timeout_ns) {
  using L = SepLayout<D, DQ, SETS>;
  constexpr bool HAS2 = SETS & kSet2, HAS1 = SETS & kSet1;
  static_assert(!PERSIST || (!DQ && !PACKED), "persistent: dense dK kernel only");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One work item: an X block of one (batch, head) slice (and, dQ kernel with
  // a key split, one range of key steps).
  struct Item {
    SeqView sv;
    int nq, nk, NX, off, x0, x_row0, y_row0, y_begin, n_iter;
    bool active;
  };
  auto make_item = [&](int bx, int bh, int bz) {
    Item I;
    // this (batch, head) slice: the whole tensor's sizes, or one sequence of a
    // packed variable-length batch (the grid covers the longest one)
    I.sv = PACKED ? seq_view_packed(bh, H, NQ, NK, D, cu_q, cu_k, total_q, total_k)
                  : seq_view_dense(bh, NQ, NK, D);
    I.nq = I.sv.nq;
    I.nk = I.sv.nk;
    I.NX = DQ ? I.nq : I.nk;
    const int nxb = (I.NX + kBlockM - 1) / kBlockM;
    I.active = I.sv.ok && bx < nxb && !(causal && I.nq > I.nk);
    I.off = I.nk - I.nq;  // key j is visible to query i iff j <= i + off (causal)
    // causal: the dQ kernel's heavy blocks are the last query blocks, the dK
    // kernel's the first key blocks; launch the heavy ones first
    const int xb = (DQ && causal) ? nxb - 1 - bx : bx;
    I.x0 = xb * kBlockM;
    I.x_row0 = DQ ? I.sv.q_row0 : I.sv.k_row0;
    I.y_row0 = DQ ? I.sv.k_row0 : I.sv.q_row0;
    int y_end;  // in steps of STEP Y rows
    if (DQ) {  // key steps visible to some row of this query block
      const int klim = causal ? min(I.nk, min(I.nq, I.x0 + kBlockM) + I.off) : I.nk;
      I.y_begin = 0;
      y_end = (klim + L::STEP - 1) / L::STEP;
    } else {  // query steps with a row that sees some key of this block
      I.y_begin = causal ? max(0, I.x0 - I.off) / L::STEP : 0;
      y_end = (I.nq + L::STEP - 1) / L::STEP;
    }
    // dQ kernel with a key split: this CTA takes key steps [z S, z S + S) of
    // them (S = split_steps, z = blockIdx.z) and writes an fp32 partial dQ
    if (DQ && splits > 1) {
      I.y_begin = bz * split_steps;
      y_end = min(y_end, I.y_begin + split_steps);
    }
    I.n_iter = I.active ? max(0, y_end - I.y_begin) : 0;
    return I;
  };
  const bool split_out = DQ && splits > 1;
  // items: one per CTA, or (persistent) item i = key block i / n_bh of slice
  // i % n_bh for i = blockIdx.x, blockIdx.x + gridDim.x, ...
  const int n_items = PERSIST ? ((NK + kBlockM - 1) / kBlockM) * n_bh : 1;
  const int item_stride = PERSIST ? static_cast<int>(gridDim.x) : 1;
  const int item_first = PERSIST ? static_cast<int>(blockIdx.x) : 0;
  auto item_at = [&](int i) {
    return PERSIST ? make_item(i / n_bh, i % n_bh, 0)
                   : make_item(static_cast<int>(blockIdx.x), static_cast<int>(blockIdx.y),
                               static_cast<int>(blockIdx.z));
  };
  const Item I0 = item_at(item_first);

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t x_full = bar0;
  constexpr int kStages = L::STAGES;
  auto y_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto y_empty = [&](int s) { return bar0 + 8u * (1 + kStages + s); };
  const uint32_t s_full = bar0 + 8u * (1 + 2 * kStages);
  const uint32_t s_free = s_full + 8;
  // per dS buffer: a warp that runs a step ahead arrives on the other one
  auto ds_full = [&](int b) { return s_full + 16 + 8u * b; };
  auto ds_free = [&](int b) { return s_full + 32 + 8u * b; };
  // With both gradient sets the dS buffer of step G is known free from the
  // release of step G-2's Y stage (the same gradient GEMMs end both), which
  // saves the gradient issuer one commit per step (a commit costs the tensor
  // pipe about as much as an MMA): 1.5-2.4 % faster with both sets, while
  // with one set the separate dS-free barrier measured ~2 % faster (and the
  // persistent and packed kernels keep it: their registers are tighter). The
  // Y stage of step G-2 cannot be reused (phase G-2+S) before dS of step G+1
  // is stored, so its phase is not overtaken while the softmax warps wait.
  constexpr bool kYFreesDs = L::NSETS == 2 && !PERSIST && !PACKED;
  static_assert(!kYFreesDs || kStages >= 3, "Y ring deep enough to stand for the dS buffers");
  auto ds_free_test = [&](int G) {
    if constexpr (kYFreesDs)
      return G < 2 || mbar_test_wait(y_empty((G - 2) % kStages), ((G - 2) / kStages) & 1);
    else
      return mbar_test_wait(ds_free(G & 1), ((G >> 1) & 1) ^ 1);
  };
  auto ds_free_wait = [&](int G, const WaitCtx& w) {
    if constexpr (kYFreesDs)
      return G < 2 || wait_bounded(y_empty((G - 2) % kStages), ((G - 2) / kStages) & 1, w);
    else
      return wait_bounded(ds_free(G & 1), ((G >> 1) & 1) ^ 1, w);
  };
  const uint32_t acc_full = s_full + 48;
  const uint32_t drain = s_full + 56;
  // persistent: X of the next item may be loaded; the accumulators were read
  const uint32_t x_free = s_full + 64;
  const uint32_t acc_empty = s_full + 72;
  // dense non-persistent kernels: the output tile is staged in the X region
  // (free once the last T GEMMs have run) and written by TMA stores that the
  // producer lane issues; one round holds both sets' bf16 rows, or one set's
  // fp32 partial rows
  const uint32_t ep_full = s_full + 80, ep_empty = s_full + 88;
  static_assert(1 + 2 * kStages + 12 <= L::NBAR, "barrier region holds every barrier");
  constexpr bool kTmaOut = !PACKED && !PERSIST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 8);
  // number of T steps whose GEMMs the T issuer has queued
  volatile int* t_queued = reinterpret_cast<volatile int*>(gb + L::OFF_MISC + 12);
  // dK kernel, per stage: -LSE1 log2e, -LSE2 log2e, g scale, -(LSE1 - LSE2 + KL),
  // 64 entries each, so that a column pair's values are one 8-byte load
  float* tab = reinterpret_cast<float*>(gb + L::OFF_TAB);

  // debug build: the layout's regions (TMEM fields are set once allocated)
  CheckCtx ck{sb + L::OFF_X, sb + L::OFF_TAB, sb + L::OFF_BAR, sb + L::OFF_BAR + L::NBAR * 8, 0, 0,
              abort_flag, dev_status};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    bool lay_ok = true;
    if (kDeviceChecks) {  // every barrier address inside the barrier region
      lay_ok = check_bar(ck, x_full, __LINE__) && check_bar(ck, s_full, __LINE__) &&
               check_bar(ck, s_free, __LINE__) && check_bar(ck, acc_full, __LINE__) &&
               check_bar(ck, drain, __LINE__) && check_bar(ck, x_free, __LINE__) &&
               check_bar(ck, acc_empty, __LINE__) && check_bar(ck, ep_full, __LINE__) &&
               check_bar(ck, ep_empty, __LINE__);
      for (int s = 0; s < kStages; ++s)
        lay_ok = lay_ok && check_bar(ck, y_full(s), __LINE__) && check_bar(ck, y_empty(s), __LINE__);
      for (int b = 0; b < 2; ++b)
        lay_ok = lay_ok && check_bar(ck, ds_full(b), __LINE__) && check_bar(ck, ds_free(b), __LINE__);
    }
    if (lay_ok) {
      mbar_init(x_full, 1);
      for (int s = 0; s < kStages; ++s) {
        mbar_init(y_full(s), 1);
        mbar_init(y_empty(s), 1);
      }
      mbar_init(s_full, 1);
      mbar_init(s_free, kSoftmaxWarps);   // one arrival per softmax warp
      for (int b = 0; b < 2; ++b) {
        mbar_init(ds_full(b), kSoftmaxWarps);
        mbar_init(ds_free(b), 1);
      }
      mbar_init(acc_full, 1);
      mbar_init(drain, 2);  // one commit per MMA-issuing thread
      mbar_init(x_free, 1);
      mbar_init(acc_empty, kSoftmaxWarps);
      mbar_init(ep_full, kSoftmaxWarps);
      mbar_init(ep_empty, 1);
    }
    // a failure recorded earlier (this launch or a previous one), or a
    // failed layout check, skips the work
    *skip_flag = !lay_ok || *reinterpret_cast<volatile int*>(dev_status) != 0;
    // malformed sequence offsets, or a causal sequence with more query rows
    // than keys: reported, never computed
    if (!I0.sv.ok || (causal && I0.nq > I0.nk)) atomicCAS(dev_status, 0, kStatusInvalidArg);
    *t_queued = 0;
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
  const bool skip = *skip_flag;
  const WaitCtx wc{abort_flag, dev_status, timeout_ns};
  ck.tmem = tmem;
  ck.tmem_cols = 512;
  // TMA coordinate extents: rows of the X and Y maps, their third dimension
  const int q_rows = PACKED ? total_q : NQ, k_rows = PACKED ? total_k : NK;
  const int x_rows = DQ ? q_rows : k_rows, y_rows = DQ ? k_rows : q_rows;
  const int z_hi = PACKED ? H : n_bh;
  // the items of this CTA in order; steps are numbered globally across them
  // (g = steps of the earlier items) for the Y ring and the per-step barriers
  auto item_steps = [&](const Item& I) { return skip ? 0 : I.n_iter; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int g = 0, ic = 0, n_x = 0;  // steps so far, items so far, X loads issued
    for (int item = item_first; ok && item < n_items; item += item_stride) {
      const Item I = item == item_first ? I0 : item_at(item);
      const int n = item_steps(I);
      if (n == 0) continue;
      if (lane == 0) {
        // persistent: the previous item's T GEMMs have read X
        if (ic > 0) ok = wait_bounded(x_free, (ic - 1) & 1, wc);
        if (kDeviceChecks)
          for (int t = 0; t < 2; ++t)
            for (int b = 0; b < L::KB; ++b)
              for (int h = 0; h < 2; ++h)
                ok = ok && check_tma(ck, sb + L::OFF_X + t * L::XT + b * 16384 + h * 8192, 8192,
                                     x_full, b * 64, D, I.x_row0 + I.x0 + h * kBoxRows, x_rows,
                                     kBoxRows, I.sv.z, z_hi, __LINE__);
        if (ok) {
          mbar_arrive_expect_tx(x_full, 2 * L::XT);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int b = 0; b < L::KB; ++b)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d(sb + L::OFF_X + t * L::XT + b * 16384 + h * 8192,
                            t == 0 ? &tm_x1 : &tm_x2, x_full, b * 64,
                            I.x_row0 + I.x0 + h * kBoxRows, I.sv.z);
          ++n_x;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      auto qv = [&](int q) {  // per-row vector element of query row q
        return static_cast<size_t>(I.sv.v_off + static_cast<long long>(q) * I.sv.v_stride);
      };
      int it = 0;
      for (; it < n; ++it) {
        const int G = g + it;
        const int s = G % kStages;
        const int yrow = (I.y_begin + it) * L::STEP;
        // dK kernel: this lane's table entries (rows yrow + lane + 32 e),
        // loaded before the wait
        constexpr int NE = L::STEP / 32;
        float4 ce[NE];
        if (!DQ) {
#pragma unroll
          for (int e = 0; e < NE; ++e)
            ce[e] = query_const(lse1_in, lse2_in, g_in, kl_in, qv(yrow + lane + 32 * e), scale,
                                yrow + lane + 32 * e < I.nq);
        }
        bool good = true;
        if (lane == 0) good = wait_bounded(y_empty(s), ((G / kStages) & 1) ^ 1, wc);
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
        if (!DQ) {
          float* ts = tab + s * 4 * L::STEP;
#pragma unroll
          for (int e = 0; e < NE; ++e) {
            const int j = lane + 32 * e;
            ts[j] = -ce[e].x, ts[L::STEP + j] = -ce[e].y;
            ts[2 * L::STEP + j] = ce[e].z, ts[3 * L::STEP + j] = -ce[e].w;
          }
          __syncwarp();  // the arrive below publishes the whole warp's entries
        }
        // a step's Y tile: per tensor, 64-column boxes of STEP rows, each
        // loaded as 64-row TMA boxes
        const uint32_t dst = sb + L::OFF_Y + s * 2 * L::YT;
        if (kDeviceChecks && lane == 0)
          for (int t = 0; t < 2; ++t)
            for (int b = 0; b < L::KB; ++b)
              for (int h = 0; h < L::STEP / kBoxRows; ++h)
                good = good && check_tma(ck, dst + t * L::YT + b * L::YBOX + h * 8192, 8192, y_full(s),
                                         b * 64, D, I.y_row0 + yrow + h * kBoxRows, y_rows, kBoxRows,
                                         I.sv.z, z_hi, __LINE__);
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(y_full(s), 2 * L::YT);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int b = 0; b < L::KB; ++b)
#pragma unroll
              for (int h = 0; h < L::STEP / kBoxRows; ++h)
                tma_load_3d(dst + t * L::YT + b * L::YBOX + h * 8192, t == 0 ? &tm_y1 : &tm_y2,
                            y_full(s), b * 64, I.y_row0 + yrow + h * kBoxRows, I.sv.z);
        }
      }
      g += it;
      ++ic;
      if (it < n) ok = false;
    }
    // let every copy this thread issued land before the CTA can exit
    if (lane == 0) {
      if (n_x > 0) wait_drain(x_full, (n_x - 1) & 1, timeout_ns);
      for (int j = max(0, g - kStages); j < g; ++j)
        wait_drain(y_full(j % kStages), (j / kStages) & 1, timeout_ns);
    }
    // output tiles staged by the softmax warps -> global memory
    if (kTmaOut && lane == 0 && ok && item_steps(I0) > 0) {
      const int rounds = split_out ? L::NSETS : 1;
      for (int rd = 0; rd < rounds; ++rd) {
        if (!wait_bounded(ep_full, rd & 1, wc)) break;
        if (!dcheck(ck, I0.x0 < I0.NX && I0.sv.z < n_bh, __LINE__)) break;
        if (split_out) {  // one set's fp32 rows: D/32 boxes of 16 KB
#pragma unroll
          for (int b = 0; b < D / 32; ++b)
            tma_store_4d(&tm_o2, sb + L::OFF_X + b * 16384, b * 32, I0.x0, I0.sv.z,
                         rd * splits + static_cast<int>(blockIdx.z));
        } else {  // both sets' bf16 rows: D/64 boxes of 16 KB per set
#pragma unroll
          for (int t = 0; t < L::NSETS; ++t)
#pragma unroll
            for (int b = 0; b < D / 64; ++b)
              tma_store_3d((HAS2 && t == 0) ? &tm_o2 : &tm_o1,
                           sb + L::OFF_X + t * L::XT + b * 16384, b * 64, I0.x0, I0.sv.z);
        }
        bulk_commit_group();
        if (rd + 1 < rounds) {
          bulk_wait_read_all();  // the staging may be written again
          mbar_arrive(ep_empty);
        }
      }
      bulk_wait_all();  // the outputs are in global memory before the CTA exits
    }
  } else if (warp == 1 || warp == kGradWarp) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the T GEMMs, warp 18 the gradient GEMMs: each one's waits
    // overlap the other's MMAs in the tensor pipe. A thread's commit tracks
    // only the MMAs that thread issued.
    if (lane == 0 && (PERSIST || item_steps(I0) > 0)) {
      constexpr uint32_t id_t = idesc_bf16(kBlockM, L::STEP, 0, 0);
      constexpr uint32_t id_g = idesc_bf16(kBlockM, D, 0, 1);
      const uint32_t x1 = sb + L::OFF_X, x2 = x1 + L::XT;
      // Descriptors are built once per stage and advanced by compile-time
      // offsets, so issuing an MMA costs two adds.
      const uint64_t dx1 = smem_desc_sw128(x1, 16, 1024), dx2 = smem_desc_sw128(x2, 16, 1024);
      // T = X Y^T of global step G (two K-major GEMMs, k-steps interleaved)
      auto issue_t = [&](int G) {
        const uint64_t dy = smem_desc_sw128(sb + L::OFF_Y + (G % kStages) * 2 * L::YT, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t xo = (k >> 2) * 16384 + (k & 3) * 32, yo = (k >> 2) * L::YBOX + (k & 3) * 32;
          mma_bf16(tmem + L::COL_T, desc_advance(dx1, xo), desc_advance(dy, yo), id_t, k > 0);
          mma_bf16(tmem + L::COL_T + L::STEP, desc_advance(dx2, xo), desc_advance(dy, L::YT + yo),
                   id_t, k > 0);
        }
        mma_commit(s_full);
      };
      // gradient GEMMs of global step G (step j of its item): A = dS from TMEM
      // buffer G&1 (slot t of a buffer holds the t-th computed set), B = the
      // set's Y (set 2: Y2, set 1: Y1) MN-major; with two sets their k-steps
      // interleave; the item's first step starts the accumulators
      auto issue_g = [&](int G, int j) {
        const uint64_t dy = smem_desc_sw128(sb + L::OFF_Y + (G % kStages) * 2 * L::YT, L::YBOX, 1024);
        const uint32_t dsb = tmem + L::COL_DS + (G & 1) * L::DSW;
#pragma unroll
        for (int kg = 0; kg < L::STEP / 16; ++kg)
#pragma unroll
          for (int t = 0; t < L::NSETS; ++t) {
            const bool set2 = HAS2 && t == 0;
            mma_bf16_ts(tmem + L::COL_ACC + t * D, dsb + (L::STEP / 2) * t + 8 * kg,
                        desc_advance(dy, (set2 ? L::YT : 0) + kg * 2048), id_g, (j > 0 || kg > 0));
          }
        if constexpr (!kYFreesDs) mma_commit(ds_free(G & 1));
        mma_commit(y_empty(G % kStages));
      };
      // the T tiles, the two dS buffers and the accumulators inside the allocation
      bool ok = check_tmem(ck, tmem + L::COL_T, 128, 2 * L::STEP, __LINE__) &&
                check_tmem(ck, tmem + L::COL_DS, 128, 2 * L::DSW, __LINE__) &&
                check_tmem(ck, tmem + L::COL_ACC, 128, L::NSETS * D, __LINE__);
      int g = 0, ic = 0;
      if (warp == 1) {
        // T of step G goes in as soon as the softmax warps have loaded T of
        // step G-1, and runs while they compute dS of step G-1
        for (int item = item_first; ok && item < n_items; item += item_stride) {
          const Item I = item == item_first ? I0 : item_at(item);
          const int n = item_steps(I);
          if (n == 0) continue;
          if (!(ok = wait_bounded(x_full, ic & 1, wc))) break;
          for (int st = 0; st < n; ++st) {
            const int G = g + st;
            if (!(ok = wait_bounded(y_full(G % kStages), (G / kStages) & 1, wc))) break;
            if (G > 0 && !(ok = wait_bounded(s_free, (G - 1) & 1, wc))) break;
            tc_fence_after();
            issue_t(G);
            *t_queued = G + 1;
          }
          if (!ok) break;
          if (PERSIST) mma_commit(x_free);  // X is read by this item's T GEMMs only
          g += n;
          ++ic;
        }
      } else {
        // gradient GEMMs of step G once its dS is in TMEM, queued behind the T
        // GEMMs of step G+kGradLag of the same item: the next T is on the
        // softmax warps' critical path, these GEMMs are not (their dS buffer is
        // next written two steps on). The dQ kernel, bound by the tensor pipe,
        // lags by 2; the dK kernel, whose shallower Y ring must be released
        // sooner, by 1. The lag stays below the ring's depth: the T GEMMs of
        // step G + lag need the Y stage that step G's gradient GEMMs release
        // once the ring has wrapped.
        constexpr int kGradLag = (DQ && kStages >= 3) ? 2 : 1;
        static_assert(kGradLag < kStages, "gradient GEMM lag below the Y ring's depth");
        for (int item = item_first; ok && item < n_items; item += item_stride) {
          const Item I = item == item_first ? I0 : item_at(item);
          const int n = item_steps(I);
          if (n == 0) continue;
          for (int j = 0; j < n; ++j) {
            const int G = g + j;
            if (!(ok = wait_bounded(ds_full(G & 1), (G >> 1) & 1, wc))) break;
            const int need = min(G + kGradLag + 1, g + n);
            const uint64_t t0 = global_timer_ns();
            while (*t_queued < need && !*abort_flag && global_timer_ns() - t0 < timeout_ns) {
            }
            // persistent: the previous item's accumulators have been read out
            if (PERSIST && j == 0 && ic > 0 && !(ok = wait_bounded(acc_empty, (ic - 1) & 1, wc)))
              break;
            tc_fence_after();
            issue_g(G, j);
          }
          if (!ok) break;
          mma_commit(acc_full);
          g += n;
          ++ic;
        }
      }
      mma_commit(drain);
      wait_drain(drain, 0, timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int grp = (warp - 2) >> 2;   // column group
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // X row within the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = scale * kLog2e;
    bool ok = true;
    int g = 0, ic = 0;
    for (int item = item_first; ok && item < n_items; item += item_stride) {
    const Item I = item == item_first ? I0 : item_at(item);
    const int n_iter = item_steps(I);
    // an item without steps still runs its epilogue when no step reaches
    // its X block at all (zero rows, below)
    if (n_iter == 0 && !(I.active && I.n_iter == 0)) continue;
    const int xrow = I.x0 + r;

    // dQ kernel: constants of this thread's query row
    float4 rc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (DQ)
      rc = query_const(lse1_in, lse2_in, g_in, kl_in,
                       static_cast<size_t>(I.sv.v_off + static_cast<long long>(xrow) * I.sv.v_stride),
                       scale, xrow < I.nq);

    // T of global step G into a, b (all lanes agree on every wait's outcome,
    // so the warp-wide TMEM loads and the __syncwarp below are never reached
    // by part of a warp); then the T GEMMs of step G+1 may overwrite T
    constexpr int NC = L::NCOL;  // this thread's Y columns per step
    float a[NC], b[NC];
    auto load_t = [&](int G) {
      // dK kernel: the stage's barrier also publishes its constant table; its
      // phase completed before these T GEMMs were issued, so test it first
      // and let the round trip overlap the T wait
      const bool tab = DQ || mbar_test_wait(y_full(G % kStages), (G / kStages) & 1);
      if (!__all_sync(0xffffffffu, wait_bounded(s_full, G & 1, wc))) return false;
      const uint32_t ta = tmem + lane_off + L::COL_T + grp * NC;
      if (!(check_tmem(ck, ta, 32, NC, __LINE__) && check_tmem(ck, ta + L::STEP, 32, NC, __LINE__)))
        return false;
      tc_fence_after();
      if constexpr (NC == 32) {
        tmem_ld32(ta, a);
        tmem_ld32(ta + L::STEP, b);
      } else {
        tmem_ld16(ta, a);
        tmem_ld16(ta + L::STEP, b);
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      return DQ || __all_sync(0xffffffffu, tab) ||
             __all_sync(0xffffffffu, wait_bounded(y_full(G % kStages), (G / kStages) & 1, wc));
    };
    // The next step's T is loaded right after this step's dS is computed and
    // before it is stored, so the next T GEMMs can start as early as possible.
    bool good = n_iter > 0 && load_t(g);
    for (int it = 0; it < n_iter; ++it) {
      if (!good) {
        ok = false;
        break;
      }
      const int G = g + it;
      const int y0 = (I.y_begin + it) * L::STEP + grp * NC;  // first Y row of this thread's columns
      // the gradient GEMMs of step G-2 have read this step's dS buffer: nearly
      // always done by now; test early, block only if not
      const bool ds_ready = ds_free_test(G);
      uint32_t d2p[NC / 2], d1p[NC / 2];
      {
        // visibility of (query, key) over this thread's NC columns
        bool full;
        int lim = 0;
        if (DQ) {
          lim = causal ? min(I.nk, xrow + 1 + I.off) : I.nk;  // keys < lim visible
          full = y0 + NC <= lim;
        } else {
          lim = causal ? xrow - I.off : 0;  // queries >= lim (and < N_Q) see this key
          full = y0 + NC <= I.nq && y0 >= lim;
        }
        auto visible = [&](int y) { return DQ ? y < lim : (y < I.nq && y >= lim); };
        const float* tq = tab + (G % kStages) * 4 * L::STEP + grp * NC;
        const float2 c2 = make_float2(c, c), sc2 = make_float2(scale, scale);
        const float2 m1 = make_float2(-1.f, -1.f);
        float4 q1c, q2c, qgc, qec;  // dK kernel: 4 columns of each constant, one 16-byte load each
#pragma unroll
        for (int k = 0; k < NC; k += 2) {
          float2 nb1, nb2, gs, ne;
          if (DQ) {
            nb1 = make_float2(-rc.x, -rc.x);
            nb2 = make_float2(-rc.y, -rc.y);
            gs = make_float2(rc.z, rc.z);
            ne = make_float2(-rc.w, -rc.w);
          } else {
            if ((k & 3) == 0) {
              q1c = *reinterpret_cast<const float4*>(tq + k);
              q2c = *reinterpret_cast<const float4*>(tq + L::STEP + k);
              qgc = *reinterpret_cast<const float4*>(tq + 2 * L::STEP + k);
              if (HAS1) qec = *reinterpret_cast<const float4*>(tq + 3 * L::STEP + k);
            }
            const bool lo = (k & 3) == 0;
            nb1 = lo ? make_float2(q1c.x, q1c.y) : make_float2(q1c.z, q1c.w);
            nb2 = lo ? make_float2(q2c.x, q2c.y) : make_float2(q2c.z, q2c.w);
            gs = lo ? make_float2(qgc.x, qgc.y) : make_float2(qgc.z, qgc.w);
            if (HAS1) ne = lo ? make_float2(qec.x, qec.y) : make_float2(qec.z, qec.w);
          }
          const float2 s1 = make_float2(a[k], a[k + 1]), s2 = make_float2(b[k], b[k + 1]);
          const float2 x1 = __ffma2_rn(s1, c2, nb1);
          float2 p1 = make_float2(ex2(x1.x), ex2(x1.y)), p2 = p1;
          if constexpr (HAS2) {  // P2 only for configuration 1
            const float2 x2 = __ffma2_rn(s2, c2, nb2);
            p2 = make_float2(ex2(x2.x), ex2(x2.y));
          }
          if (!full) {
            if (!visible(y0 + k)) p1.x = p2.x = 0.f;
            if (!visible(y0 + k + 1)) p1.y = p2.y = 0.f;
          }
          if constexpr (HAS2) {
            const float2 d2 = __fmul2_rn(__ffma2_rn(p1, m1, p2), gs);  // g (P2 - P1)
            d2p[k >> 1] = pack_bf16x2(d2.x, d2.y);
          }
          if constexpr (HAS1) {
            // g P1 (log(P1/P2) - KL), log(P1/P2) - KL = scale (s1 - s2) - e
            const float2 lr = __ffma2_rn(__ffma2_rn(s2, m1, s1), sc2, ne);
            const float2 d1 = __fmul2_rn(__fmul2_rn(p1, gs), lr);
            d1p[k >> 1] = pack_bf16x2(d1.x, d1.y);
          }
        }
      }
      // 64-row steps: load the next T before storing this dS (the next T GEMMs
      // start earlier); 128-row steps store first, which keeps this step's
      // packed dS out of the registers the next T lands in
      constexpr bool kLoadFirst = L::STEP == 64;
      if (kLoadFirst && it + 1 < n_iter) good = load_t(G + 1);
      if (!__all_sync(0xffffffffu, ds_ready) &&
          !__all_sync(0xffffffffu, ds_free_wait(G, wc))) {
        ok = false;
        break;
      }
      // this thread's NC values of row r: NC/2 packed columns per set at
      // [NC/2 grp, NC/2 (grp + 1)) of the set's STEP/2-column slot of buffer G&1
      const uint32_t dsb = tmem + lane_off + L::COL_DS + (G & 1) * L::DSW + grp * (NC / 2);
      if (!check_tmem(ck, dsb, 32, (HAS2 && HAS1) ? L::STEP / 2 + NC / 2 : NC / 2, __LINE__)) {
        ok = false;
        break;
      }
      tc_fence_after();  // the stores below follow the MMAs that read this buffer
      if (HAS2) tmem_st_cols<NC / 2>(dsb, d2p);
      if (HAS1) tmem_st_cols<NC / 2>(dsb + (HAS2 ? L::STEP / 2 : 0), d1p);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full(G & 1));
      if (!kLoadFirst && it + 1 < n_iter) good = load_t(G + 1);
    }
    // epilogue: accumulator row r -> bf16 dQ (dQ kernel) or dK (dK kernel)
    // row, d columns [grp d/4, (grp+1) d/4); with a key split, the fp32 row
    // of this split's partial dQ instead ([set][split][B H N_Q][d], dense
    // batches only), zero when the split holds no key this block sees
    constexpr int EC = D / 4;
    auto part_row = [&](int t) {
      const size_t plane = static_cast<size_t>(gridDim.y) * NQ;
      dcheck(ck, t < L::NSETS && static_cast<int>(blockIdx.z) < splits &&
                     static_cast<size_t>(I.sv.v_off + xrow) < plane, __LINE__);
      return reinterpret_cast<float4*>(
          part + ((static_cast<size_t>(t) * splits + blockIdx.z) * plane +
                  static_cast<size_t>(I.sv.v_off + xrow)) * D + grp * EC);
    };
    // an X block no Y step reaches has zero gradient: a packed sequence
    // without query rows (its keys' dK), or, with a key split, a split that
    // holds no key of this query block (a zero partial)
    if (ok && I.active && I.n_iter == 0 && xrow < I.NX) {
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        if (split_out) {
          float4* dst = part_row(t);
#pragma unroll
          for (int i = 0; i < EC / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          __nv_bfloat16* out = (HAS2 && t == 0) ? out2 : out1;
          uint4* dst = reinterpret_cast<uint4*>(
              out + (DQ ? I.sv.q_off : I.sv.k_off) + static_cast<long long>(xrow) * I.sv.row_stride +
              grp * EC);
#pragma unroll
          for (int i = 0; i < EC / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    if (kTmaOut && ok && n_iter > 0 && __all_sync(0xffffffffu, wait_bounded(acc_full, ic & 1, wc))) {
      tc_fence_after();
      // row r's piece of EC columns into the staging tile: bf16 rows of set t
      // at t XT, or (key split) one set's fp32 rows per round; 128-byte rows
      // per 16 KB box, 16-byte chunks swizzled by the row
      const bool f32 = split_out;
      const int pb = EC * (f32 ? 4 : 2);        // bytes of this thread's piece
      const int ppb = 128 / pb;                 // pieces per 128-byte box row
      const uint32_t rowoff = static_cast<uint32_t>((grp / ppb) * 16384 + r * 128);
      const int c0 = (grp % ppb) * (pb / 16);
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        float v[EC];
        if (!(ok = check_tmem(ck, tmem + lane_off + L::COL_ACC + t * D + grp * EC, 32, EC, __LINE__)))
          break;
        if constexpr (EC == 32)
          tmem_ld32(tmem + lane_off + L::COL_ACC + t * D + grp * EC, v);
        else
          tmem_ld16(tmem + lane_off + L::COL_ACC + t * D + grp * EC, v);
        tmem_wait_ld();
        if (f32) {
          // round t: the producer has sent round t-1 out
          if (t > 0 && !(ok = __all_sync(0xffffffffu, wait_bounded(ep_empty, (t - 1) & 1, wc)))) break;
          const uint32_t base = sb + L::OFF_X + rowoff;
#pragma unroll
          for (int j = 0; j < EC / 4; ++j)
            st_shared_v4(base + (((c0 + j) ^ (r & 7)) << 4), __float_as_uint(v[4 * j]),
                         __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                         __float_as_uint(v[4 * j + 3]));
        } else {
          const uint32_t base = sb + L::OFF_X + t * L::XT + rowoff;
#pragma unroll
          for (int j = 0; j < EC / 8; ++j)
            st_shared_v4(base + (((c0 + j) ^ (r & 7)) << 4), pack_bf16x2(v[8 * j], v[8 * j + 1]),
                         pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                         pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        }
        if (f32 || t + 1 == L::NSETS) {  // a round is complete
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(ep_full);
        }
      }
    } else if (!kTmaOut && ok && n_iter > 0 &&
               __all_sync(0xffffffffu, wait_bounded(acc_full, ic & 1, wc))) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < L::NSETS; ++t) {
        __nv_bfloat16* out = (HAS2 && t == 0) ? out2 : out1;
        float v[EC];
        if (!check_tmem(ck, tmem + lane_off + L::COL_ACC + t * D + grp * EC, 32, EC, __LINE__))
          break;
        if constexpr (EC == 32)
          tmem_ld32(tmem + lane_off + L::COL_ACC + t * D + grp * EC, v);
        else
          tmem_ld16(tmem + lane_off + L::COL_ACC + t * D + grp * EC, v);
        tmem_wait_ld();
        if (xrow < I.NX) {
          if (split_out) {
            float4* dst = part_row(t);
#pragma unroll
            for (int i = 0; i < EC / 4; ++i)
              dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(
                out + (DQ ? I.sv.q_off : I.sv.k_off) + static_cast<long long>(xrow) * I.sv.row_stride +
                grp * EC);
#pragma unroll
            for (int i = 0; i < EC / 8; ++i)
              dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                  pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                  pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                  pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
          }
        }
      }
      if (PERSIST) {  // the next item's gradient GEMMs may overwrite the accumulators
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      }
    } else {
      ok = false;
    }
    g += n_iter;
    ++ic;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Sum of the key splits' fp32 partial dQ rows -> bf16 dQ: one thread per 8
// columns of one row of one gradient set; out_a is the first computed set's
// output (dQ2 when present), out_b the second's.
__global__ void streamkl_dq_split_combine_kernel(const float* __restrict__ part, int splits,
                                                 long long rows, int d, int nsets,
                                                 __nv_bfloat16* __restrict__ out_a,
                                                 __nv_bfloat16* __restrict__ out_b) {
  const long long per_set = rows * (d / 8);
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= per_set * nsets) return;
  const int t = static_cast<int>(i / per_set);
  const long long j = i - t * per_set;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < splits; ++s) {
    const float4* p = reinterpret_cast<const float4*>(
        part + (static_cast<size_t>(t) * splits + s) * static_cast<size_t>(rows) * d) + 2 * j;
    const float4 a = p[0], b = p[1];
    acc[0] += a.x, acc[1] += a.y, acc[2] += a.z, acc[3] += a.w;
    acc[4] += b.x, acc[5] += b.y, acc[6] += b.z, acc[7] += b.w;
  }
  uint4* dst = reinterpret_cast<uint4*>(t == 0 ? out_a : out_b) + j;
  *dst = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                    pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

template <int D, bool DQ, int SETS, bool PACKED, bool PERSIST>
cudaError_t launch_sep_p(const BwdSepArgs& a, cudaStream_t stream) {
  using L = SepLayout<D, DQ, SETS>;
  auto kern = streamkl_bwd_sep_kernel<D, DQ, SETS, PACKED, PERSIST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const int NX = DQ ? a.NQ : a.NK;  // the longest sequence for packed batches
  const int splits = (DQ && !PACKED) ? a.dq_splits : 1;
  dim3 grid((NX + kBlockM - 1) / kBlockM, a.BH, splits);
  if (PERSIST) grid = dim3(a.dk_persist_ctas, 1, 1);
  const CUtensorMap* x1 = DQ ? a.tm_q1 : a.tm_k1;
  const CUtensorMap* x2 = DQ ? a.tm_q2 : a.tm_k2;
  const CUtensorMap* y1 = DQ ? a.tm_k1 : a.tm_q1;
  const CUtensorMap* y2 = DQ ? a.tm_k2 : a.tm_q2;
  // output maps of the dense non-persistent kernels (the others store rows
  // directly and get the input maps as placeholders)
  const CUtensorMap* o2 = x1;
  const CUtensorMap* o1 = x1;
  if (!PACKED && !PERSIST) {
    o2 = splits > 1 ? a.tm_part : (DQ ? a.tm_dq2 : a.tm_dk2);
    o1 = splits > 1 ? a.tm_part : (DQ ? a.tm_dq1 : a.tm_dk1);
    if (o2 == nullptr || o1 == nullptr) return cudaErrorInvalidValue;
  }
  kern<<<grid, kSepThreads, L::ALLOC, stream>>>(
      *x1, *x2, *y1, *y2, *o2, *o1, a.NQ, a.NK, a.causal, a.scale, a.kl, a.lse1, a.lse2, a.g,
      static_cast<__nv_bfloat16*>(DQ ? a.dq2 : a.dk2),
      static_cast<__nv_bfloat16*>(DQ ? a.dq1 : a.dk1), splits > 1 ? a.dq_part : nullptr, splits,
      a.dq_split_steps, a.BH, a.cu_q, a.cu_k, a.H, a.total_q, a.total_k, a.dev_status,
      a.timeout_ns);
  return cudaGetLastError();
}

template <int D, bool DQ, int SETS>
cudaError_t launch_sep_t(const BwdSepArgs& a, cudaStream_t stream) {
  if (a.cu_q != nullptr) return launch_sep_p<D, DQ, SETS, true, false>(a, stream);
  if (!DQ && a.dk_persist_ctas > 0) return launch_sep_p<D, DQ, SETS, false, !DQ>(a, stream);
  return launch_sep_p<D, DQ, SETS, false, false>(a, stream);
}

template <int D, bool DQ>
cudaError_t launch_sep_g(const BwdSepArgs& a, cudaStream_t stream) {
  if (a.grad1 && a.grad2) return launch_sep_t<D, DQ, kSet1 | kSet2>(a, stream);
  return a.grad1 ? launch_sep_t<D, DQ, kSet1>(a, stream) : launch_sep_t<D, DQ, kSet2>(a, stream);
}

}  // namespace

size_t bwd_sep_smem_bytes(int d, int grad1) {
  constexpr int both = kSet1 | kSet2;
  if (d == 128) return grad1 ? SepLayout<128, false, both>::ALLOC : SepLayout<128, false, kSet2>::ALLOC;
  return grad1 ? SepLayout<64, false, both>::ALLOC : SepLayout<64, false, kSet2>::ALLOC;
}

cudaError_t launch_bwd_separate(const BwdSepArgs& a, cudaStream_t stream) {
  cudaError_t e = a.d == 128 ? launch_sep_g<128, false>(a, stream) : launch_sep_g<64, false>(a, stream);
  if (e != cudaSuccess) return e;
  e = a.d == 128 ? launch_sep_g<128, true>(a, stream) : launch_sep_g<64, true>(a, stream);
  if (e != cudaSuccess || a.dq_splits <= 1 || a.cu_q != nullptr) return e;
  const int nsets = (a.grad1 ? 1 : 0) + (a.grad2 ? 1 : 0);
  const long long rows = static_cast<long long>(a.BH) * a.NQ;
  const long long threads = rows * (a.d / 8) * nsets;
  const int block = 256;
  streamkl_dq_split_combine_kernel<<<static_cast<unsigned>((threads + block - 1) / block), block, 0,
                                     stream>>>(
      a.dq_part, a.dq_splits, rows, a.d, nsets,
      static_cast<__nv_bfloat16*>(a.grad2 ? a.dq2 : a.dq1), static_cast<__nv_bfloat16*>(a.dq1));
  return cudaGetLastError();
}

}  // namespace skl

// C-ABI layer: argument checks, TMA tensor maps, split choice, launches.
// No allocation, no synchronisation; everything is enqueued on the caller's
// stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "streamkl.h"
#include "kernels.h"

namespace {

thread_local char g_err[512] = "";

streamkl_status fail(streamkl_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

streamkl_status cuda_fail(cudaError_t e, const char* what) {
  return fail(STREAMKL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

uint64_t wait_timeout_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("STREAMKL_WAIT_TIMEOUT_MS");
    long long ms = s ? std::atoll(s) : 2000;
    if (ms < 1) ms = 1;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return v;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 152;
  }
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

streamkl_status check_sizes(int B, int H, int NQ, int NK, int d, int causal) {
  if (B < 1 || H < 1 || NQ < 1 || NK < 1)
    return fail(STREAMKL_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d H=%d NQ=%d NK=%d)", B, H, NQ, NK);
  if (d != 64 && d != 128) return fail(STREAMKL_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
  if (static_cast<long long>(B) * H > 65535)
    return fail(STREAMKL_ERR_UNSUPPORTED, "B*H=%lld exceeds 65535", static_cast<long long>(B) * H);
  if (NQ > (1 << 30) || NK > (1 << 30)) return fail(STREAMKL_ERR_UNSUPPORTED, "sequence length above 2^30");
  if (causal != 0 && causal != 1) return fail(STREAMKL_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (causal && NQ > NK)
    return fail(STREAMKL_ERR_INVALID_ARG, "causal needs NQ <= NK (bottom-right alignment), got NQ=%d NK=%d", NQ, NK);
  return STREAMKL_OK;
}

int key_tiles(int NK) { return (NK + skl::kBlockN - 1) / skl::kBlockN; }

// Choose the split count with a two-part model of the forward's time:
//   compute: waves of CTAs, each costing its key tiles plus a fixed start and
//            end (Q load, TMEM set-up, partial-state write), one CTA per SM;
//   memory:  the K1/K2 (and Q1/Q2) bytes over the HBM bandwidth, which one
//            SM cannot reach alone: a few CTAs stream at ~100 GB/s each.
// Splitting the keys adds CTAs (better SM fill, more streams) but cannot
// beat the chip's bandwidth; with few query rows against many keys the
// forward is memory-bound and splits only add partial-state traffic. The
// constants are GB300 measurements: ~1 us per 128x128 tile pair at d = 128
// (0.6 us at d = 64), ~3 us of fixed cost per CTA, ~7 TB/s of HBM bandwidth.
int choose_splits_impl(int B, int H, int NQ, int NK, int d) {
  const long long ctas = static_cast<long long>((NQ + skl::kBlockM - 1) / skl::kBlockM) * B * H;
  const int tiles = key_tiles(NK);
  const int sms = num_sms();
  if (ctas >= 8LL * sms) return 1;
  const double tile_us = d == 128 ? 1.0 : 0.6, cta_us = 3.0;
  const double bytes = static_cast<double>(B) * H * (static_cast<double>(NK) + NQ) * d * 4.0;
  const int smax = std::max(1, std::min(32, tiles / 4));
  auto cost = [&](int s) {
    const long long units = ctas * s;
    const long long waves = (units + sms - 1) / sms;
    const long long tps = (tiles + s - 1) / s;
    const double t_mma = static_cast<double>(waves) * (static_cast<double>(tps) * tile_us + cta_us);
    const double streams = static_cast<double>(std::min<long long>(units, sms));
    const double t_mem = bytes / std::min(7.0e12, streams * 1.0e11) * 1e6;
    return std::max(t_mma, t_mem);
  };
  int best = 1;
  double best_t = cost(1);
  for (int s = 2; s <= smax; ++s) {
    const double t = cost(s);
    if (t < best_t) {
      best_t = t;
      best = s;
    }
  }
  if (best > 1 && best_t > 0.95 * cost(1)) return 1;
  return best;
}

// Forward as CTA pairs (cta_group::2 MMAs over two query blocks), for dense
// batches without a key split and with an even number of query blocks, when
// switched on (streamkl_set_fwd_pairs(1)). Off by default: measured on
// GB300 it matches the one-CTA kernel at 64K causal (27.6 against 28.0 ms)
// and is 3-8 % slower on the smaller workloads.
std::atomic<int> g_fwd_pairs{0};  // 0: never, 1: when eligible

bool fwd_pairs_impl(int NQ, int splits) {
  return g_fwd_pairs.load() == 1 && skl::fwd_pair_eligible(NQ, splits, false);
}

// Effective split count and tiles per split for a requested count.
void split_plan(int requested, int NK, int* splits, int* tps) {
  const int tiles = key_tiles(NK);
  int s = std::max(1, std::min(requested, tiles));
  const int per = (tiles + s - 1) / s;
  *tps = per;
  *splits = (tiles + per - 1) / per;
}

// Backward algorithm: 0 = separate dK and dQ kernels (accumulators stay on
// chip, no atomics, no workspace), 1 = one fused kernel per key tile with dQ
// reduced through fp32 atomics. STREAMKL_BWD_ALGO=separate|fused sets the
// initial override; streamkl_set_bwd_algorithm changes it.
std::atomic<int> g_forced_algo{-2};  // -2: environment not read yet, -1: automatic

int forced_algo() {
  int v = g_forced_algo.load();
  if (v == -2) {
    const char* s = std::getenv("STREAMKL_BWD_ALGO");
    int e = -1;
    if (s && s[0] == 'f') e = 1;
    if (s && s[0] == 's') e = 0;
    g_forced_algo.compare_exchange_strong(v, e);
    v = g_forced_algo.load();
  }
  return v;
}

// The fused algorithm runs the short-sweep kernel (persistent grid, dQ kept
// on chip per batch-head) when the query rows fit one 64-row tile at d = 128;
// otherwise one CTA per key tile, with per-tile dQ reductions (at d = 64
// through TMA bulk reductions of staged tiles).
bool short_sweep(int NQ, int d) { return d == 128 && NQ <= skl::kShortMaxQ; }

// Automatic choice, from the fused-vs-separate sweep on GB300: the fused
// short-sweep kernel for decode-like shapes (at most 64 query rows at
// d = 128, where it reads the keys once against the separate kernels'
// twice); the fused d = 64 kernel with one gradient set from 512 query rows
// on (1.09-1.38x: the separate kernels each pay the exponentials and dS that
// bound d = 64, the fused kernel once; below 512 rows a CTA has only one to
// three query blocks and the persistent dK kernel wins); the fused d = 128
// kernel with one gradient set from 512 query rows on without a mask and from
// 1,024 with the causal one (non-causal 1.03-1.11x, causal 1.02-1.03x; at 512
// causal rows, the split-K shape, the two are level, and at 256 rows the
// separate kernels are faster); the separate kernels everywhere else, both
// gradient sets included.
int bwd_algo_impl(int B, int H, int NQ, int NK, int d, int causal, int grad1) {
  const int forced = forced_algo();
  if (forced >= 0) return forced;
  (void)B, (void)H, (void)NK;
  if (short_sweep(NQ, d)) return 1;
  if (grad1) return 0;
  if (d == 64) return NQ >= 512 ? 1 : 0;
  return NQ >= (causal ? 1024 : 512) ? 1 : 0;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t fwd_ws(int B, int H, int NQ, int splits) {
  if (splits <= 1) return 0;
  return align256(static_cast<size_t>(5) * splits * B * H * NQ * sizeof(float));
}

size_t bwd_ws(int B, int H, int NQ, int NK, int d, int causal, int grad1) {
  if (bwd_algo_impl(B, H, NQ, NK, d, causal, grad1) == 0) return 0;
  const size_t one = align256(static_cast<size_t>(B) * H * NQ * d * sizeof(float));
  return grad1 ? 2 * one : one;
}

// Key split of the separate backward's dQ kernel. Like the forward's key
// split (gist.science technical summary, section 3 "Variante Split-K") it fills the GPU
// when there are few query blocks: each split sweeps a contiguous range of
// key steps into an fp32 partial dQ, and a combine kernel sums the
// partials. Same wave model as the forward's choice, with the dQ kernel's
// per-step cost (~1 us per 64 keys at d = 128, 0.6 us at d = 64; a 128-key
// step of the one-set d = 64 kernel ~1.6 times a 64-key one) and the
// partials' extra bytes.
std::atomic<int> g_forced_dq_splits{0};  // 0: automatic

// Key rows per step of the separate backward's dQ kernel: 128 with one
// gradient set at d = 64, 64 otherwise (the kernel's layout).
int sep_step_rows(int nsets, int d) { return (nsets == 1 && d == 64) ? 128 : 64; }

int dq_steps(int NK, int nsets, int d) {
  const int step = sep_step_rows(nsets, d);
  return (NK + step - 1) / step;
}

int dq_splits_auto(int B, int H, int NQ, int NK, int d, int nsets) {
  const long long ctas = static_cast<long long>((NQ + skl::kBlockM - 1) / skl::kBlockM) * B * H;
  const int steps = dq_steps(NK, nsets, d);
  const int sms = num_sms();
  if (ctas >= 8LL * sms) return 1;
  const double step_us = (d == 128 ? 1.0 : 0.6) * (sep_step_rows(nsets, d) == 128 ? 1.6 : 1.0);
  const double cta_us = 4.0;
  const double in_bytes = static_cast<double>(B) * H * (static_cast<double>(NK) + NQ) * d * 4.0;
  const double part_bytes = static_cast<double>(B) * H * NQ * d * 4.0 * nsets;
  // at least 512 keys per split
  const int smax = std::max(1, std::min(32, steps * sep_step_rows(nsets, d) / 512));
  auto cost = [&](int s) {
    const long long units = ctas * s;
    const long long waves = (units + sms - 1) / sms;
    const long long per = (steps + s - 1) / s;
    const double t_mma = static_cast<double>(waves) * (static_cast<double>(per) * step_us + cta_us);
    const double streams = static_cast<double>(std::min<long long>(units, sms));
    const double t_mem = in_bytes / std::min(7.0e12, streams * 1.0e11) * 1e6;
    // partials written once and read once by the combine
    const double t_comb = s > 1 ? 2.0 * s * part_bytes / 6.0e12 * 1e6 + 3.0 : 0.0;
    return std::max(t_mma, t_mem) + t_comb;
  };
  int best = 1;
  double best_t = cost(1);
  for (int s = 2; s <= smax; ++s) {
    const double t = cost(s);
    if (t < best_t) {
      best_t = t;
      best = s;
    }
  }
  if (best > 1 && best_t > 0.95 * cost(1)) return 1;
  return best;
}

// Effective split count and key steps per split (dense batches).
void dq_split_plan(int B, int H, int NQ, int NK, int d, int nsets, int* splits, int* per) {
  const int forced = g_forced_dq_splits.load();
  const int steps = dq_steps(NK, nsets, d);
  const int req = forced > 0 ? forced : dq_splits_auto(B, H, NQ, NK, d, nsets);
  const int s = std::max(1, std::min(req, steps));
  *per = (steps + s - 1) / s;
  *splits = (steps + *per - 1) / *per;
}

// Persistent dK kernel for short query sweeps: with at most 6 steps of 64
// query rows per key block (N_Q <= 384) a CTA's fixed start and end (X load,
// barrier and TMEM set-up, accumulator read-out) weigh against its few steps,
// so one CTA per SM takes (key block, batch-head) items in turn and loads the
// next item's X while the current one finishes. Measured on GB300 (64K-131K
// keys, against one CTA per key block writing its rows with TMA stores):
// 1.11-1.18x at 128 query rows, 1.04x at 256, 1.01x at 384, 0.98-0.99x at 512.
std::atomic<int> g_forced_dk_persist{0};  // 0: automatic, -1: never, n > 0: n CTAs

int dk_persist_ctas(int B, int H, int NQ, int NK) {
  const int forced = g_forced_dk_persist.load();
  if (forced < 0) return 0;
  if (forced > 0) return forced;
  const long long items = static_cast<long long>((NK + skl::kBlockM - 1) / skl::kBlockM) * B * H;
  const int sms = num_sms();
  return (NQ <= 384 && items > sms) ? sms : 0;
}

size_t dq_split_ws(int B, int H, int NQ, int NK, int d, int nsets) {
  int splits, per;
  dq_split_plan(B, H, NQ, NK, d, nsets, &splits, &per);
  if (splits <= 1) return 0;
  return align256(static_cast<size_t>(nsets) * splits * B * H * NQ * d * sizeof(float));
}

// 3-D map {d, N, B*H} of one bf16 tensor, 64-column x box_rows boxes, 128-byte swizzle.
streamkl_status make_map(CUtensorMap* m, const void* ptr, int BH, int N, int d, const char* name,
                         int box_rows = skl::kBlockM) {
  auto enc = encode_fn();
  if (!enc) return fail(STREAMKL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), gdim, gstride, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(STREAMKL_ERR_CUDA, "tensor map for %s failed (CUresult %d)", name, static_cast<int>(r));
  return STREAMKL_OK;
}

// 3-D map {d, N, BH} of an fp32 [BH][N][d] accumulator: 32-column (128-byte)
// x box_rows boxes, 128-byte swizzle (the fused kernels' TMA reductions).
streamkl_status make_map_acc(CUtensorMap* m, void* ptr, int BH, int N, int d,
                             int box_rows = skl::kBlockM) {
  auto enc = encode_fn();
  if (!enc) return fail(STREAMKL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(STREAMKL_ERR_CUDA, "tensor map for the dQ accumulator failed (CUresult %d)", static_cast<int>(r));
  return STREAMKL_OK;
}

// 4-D map {d, N, BH, planes} of fp32 [planes][BH][N][d] rows (the dQ split's
// partials): 32-column (128-byte) x 128-row boxes, 128-byte swizzle, so a
// store of a 128-row tile stops at the end of its own (plane, batch-head).
streamkl_status make_map_part(CUtensorMap* m, void* ptr, int planes, int BH, int N, int d) {
  auto enc = encode_fn();
  if (!enc) return fail(STREAMKL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH), static_cast<cuuint64_t>(planes)};
  const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4,
                                 static_cast<cuuint64_t>(BH) * N * d * 4};
  const cuuint32_t box[4] = {32, static_cast<cuuint32_t>(skl::kBlockM), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(STREAMKL_ERR_CUDA, "tensor map for the dQ partials failed (CUresult %d)", static_cast<int>(r));
  return STREAMKL_OK;
}

// 3-D map {d, total, H} of a packed [total, H, d] bf16 tensor: rows of one
// head are H d elements apart. 64-column x box_rows boxes, 128-byte swizzle.
streamkl_status make_map_packed(CUtensorMap* m, const void* ptr, int total, int H, int d,
                                const char* name, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return fail(STREAMKL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(total),
                              static_cast<cuuint64_t>(H)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(H) * d * 2, static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), gdim, gstride, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(STREAMKL_ERR_CUDA, "tensor map for %s failed (CUresult %d)", name, static_cast<int>(r));
  return STREAMKL_OK;
}

// Host checks shared by the packed entry points (the offsets themselves are
// device data: the kernels check them and report STREAMKL_ERR_INVALID_ARG
// through the status word).
streamkl_status check_packed(const int* cu_q, const int* cu_k, int B, int H, int total_q, int total_k,
                             int max_q, int max_k, int d, int causal) {
  if (!cu_q || !cu_k) return fail(STREAMKL_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(cu_q) | reinterpret_cast<uintptr_t>(cu_k)) & 3)
    return fail(STREAMKL_ERR_INVALID_ARG, "cu_seqlens arrays must be 4-byte aligned");
  if (total_q < 1 || total_k < 1) return fail(STREAMKL_ERR_INVALID_ARG, "total_q and total_k must be >= 1");
  if (max_q > total_q || max_k > total_k)
    return fail(STREAMKL_ERR_INVALID_ARG, "max_seqlen above the packed total (%d > %d or %d > %d)",
                max_q, total_q, max_k, total_k);
  if (static_cast<long long>(total_q) * H > (1LL << 31) || static_cast<long long>(total_k) * H > (1LL << 31))
    return fail(STREAMKL_ERR_UNSUPPORTED, "total rows x heads above 2^31");
  // the per-sequence causal condition (N_Q <= N_K) is checked on the device
  return check_sizes(B, H, max_q, max_k, d, 0);
}

streamkl_status check_inputs(const void* q1, const void* k1, const void* q2, const void* k2) {
  const void* ps[4] = {q1, k1, q2, k2};
  const char* names[4] = {"q1", "k1", "q2", "k2"};
  for (int i = 0; i < 4; ++i) {
    if (!ps[i]) return fail(STREAMKL_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ps[i])) return fail(STREAMKL_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  return STREAMKL_OK;
}

}  // namespace

extern "C" {

const char* streamkl_status_string(streamkl_status s) {
  switch (s) {
    case STREAMKL_OK: return "STREAMKL_OK";
    case STREAMKL_ERR_INVALID_ARG: return "STREAMKL_ERR_INVALID_ARG";
    case STREAMKL_ERR_UNSUPPORTED: return "STREAMKL_ERR_UNSUPPORTED";
    case STREAMKL_ERR_CUDA: return "STREAMKL_ERR_CUDA";
    case STREAMKL_ERR_TIMEOUT: return "STREAMKL_ERR_TIMEOUT";
    case STREAMKL_ERR_DEVICE_CHECK: return "STREAMKL_ERR_DEVICE_CHECK";
  }
  return "STREAMKL_ERR_UNKNOWN";
}

const char* streamkl_last_error(void) { return g_err; }

int streamkl_choose_splits(int B, int H, int NQ, int NK, int d, int causal) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK) return 0;
  int s, tps;
  split_plan(choose_splits_impl(B, H, NQ, NK, d), NK, &s, &tps);
  return s;
}

size_t streamkl_fwd_workspace_size(int B, int H, int NQ, int NK, int d, int causal, int num_splits) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK || num_splits < 0) return 0;
  int s, tps;
  split_plan(num_splits > 0 ? num_splits : choose_splits_impl(B, H, NQ, NK, d), NK, &s, &tps);
  return fwd_ws(B, H, NQ, s);
}

size_t streamkl_bwd_workspace_size(int B, int H, int NQ, int NK, int d, int causal, int want_grad1) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK) return 0;
  const int g1 = want_grad1 ? 1 : 0;
  const size_t sep = dq_split_ws(B, H, NQ, NK, d, 1 + g1);
  if (bwd_algo_impl(B, H, NQ, NK, d, causal, g1) == 0) return sep;
  const size_t fused = bwd_ws(B, H, NQ, NK, d, causal, g1);
  // one set under the per-key-tile fused algorithm may be configuration 2
  // alone, which that kernel hands to the separate kernels
  if (!g1 && !short_sweep(NQ, d)) return fused > sep ? fused : sep;
  return fused;
}

int streamkl_bwd_dq_splits(int B, int H, int NQ, int NK, int d, int causal, int want_grad1) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK) return -1;
  int splits, per;
  dq_split_plan(B, H, NQ, NK, d, want_grad1 ? 2 : 1, &splits, &per);
  return splits;
}

int streamkl_bwd_dk_persist(int B, int H, int NQ, int NK, int d, int causal) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK) return -1;
  return dk_persist_ctas(B, H, NQ, NK);
}

int streamkl_set_bwd_dk_persist(int ctas) {
  if (ctas < -1) {
    fail(STREAMKL_ERR_INVALID_ARG, "persistent dK CTA count must be >= -1 (0: automatic, -1: off)");
    return -1;
  }
  g_forced_dk_persist.store(ctas);
  return 0;
}

int streamkl_set_bwd_dq_splits(int splits) {
  if (splits < 0) {
    fail(STREAMKL_ERR_INVALID_ARG, "dQ split count must be >= 0 (0: automatic)");
    return -1;
  }
  g_forced_dq_splits.store(splits);
  return 0;
}

int streamkl_fwd_pairs(int B, int H, int NQ, int NK, int d, int causal, int num_splits) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK || num_splits < 0) return -1;
  int s, tps;
  split_plan(num_splits > 0 ? num_splits : choose_splits_impl(B, H, NQ, NK, d), NK, &s, &tps);
  return fwd_pairs_impl(NQ, s) ? 1 : 0;
}

int streamkl_set_fwd_pairs(int mode) {
  if (mode != 0 && mode != 1) {
    fail(STREAMKL_ERR_INVALID_ARG, "mode must be 0 (never, the default) or 1 (when eligible)");
    return -1;
  }
  g_fwd_pairs.store(mode);
  return 0;
}

int streamkl_bwd_algorithm(int B, int H, int NQ, int NK, int d, int causal, int want_grad1) {
  if (check_sizes(B, H, NQ, NK, d, causal) != STREAMKL_OK) return -1;
  return bwd_algo_impl(B, H, NQ, NK, d, causal, want_grad1 ? 1 : 0);
}

int streamkl_set_bwd_algorithm(int algo) {
  if (algo < -1 || algo > 1) {
    fail(STREAMKL_ERR_INVALID_ARG, "algorithm must be -1, 0 or 1");
    return -1;
  }
  forced_algo();  // settle the environment's initial value first
  g_forced_algo.store(algo);
  return 0;
}

size_t streamkl_workspace_size(int B, int H, int NQ, int NK, int d, int causal, int want_grad1) {
  const size_t a = streamkl_fwd_workspace_size(B, H, NQ, NK, d, causal, 0);
  const size_t b = streamkl_bwd_workspace_size(B, H, NQ, NK, d, causal, want_grad1);
  return a > b ? a : b;
}

streamkl_status streamkl_fwd(const void* q1, const void* k1, const void* q2, const void* k2, int B,
                             int H, int NQ, int NK, int d, float scale, int causal, int num_splits,
                             float* kl, float* lse1, float* lse2, void* workspace, size_t ws_bytes,
                             int* dev_status, void* stream) {
  g_err[0] = '\0';
  streamkl_status st = check_sizes(B, H, NQ, NK, d, causal);
  if (st != STREAMKL_OK) return st;
  if ((st = check_inputs(q1, k1, q2, k2)) != STREAMKL_OK) return st;
  if (!kl || !lse1 || !lse2) return fail(STREAMKL_ERR_INVALID_ARG, "kl/lse1/lse2 must be non-NULL");
  if (!dev_status) return fail(STREAMKL_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(STREAMKL_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (num_splits < 0) return fail(STREAMKL_ERR_INVALID_ARG, "num_splits must be >= 0");
  int splits, tps;
  split_plan(num_splits > 0 ? num_splits : choose_splits_impl(B, H, NQ, NK, d), NK, &splits, &tps);
  const size_t need = fwd_ws(B, H, NQ, splits);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace)))
    return fail(STREAMKL_ERR_INVALID_ARG, "forward workspace too small: need %zu bytes, got %zu", need, ws_bytes);

  const int BH = B * H;
  // CTA pairs: each CTA loads 64-row halves of the key tiles
  const bool pairs = fwd_pairs_impl(NQ, splits);
  const int k_box = pairs ? 64 : skl::kBlockM;
  CUtensorMap mq1, mk1, mq2, mk2;
  if ((st = make_map(&mq1, q1, BH, NQ, d, "q1")) != STREAMKL_OK) return st;
  if ((st = make_map(&mk1, k1, BH, NK, d, "k1", k_box)) != STREAMKL_OK) return st;
  if ((st = make_map(&mq2, q2, BH, NQ, d, "q2")) != STREAMKL_OK) return st;
  if ((st = make_map(&mk2, k2, BH, NK, d, "k2", k_box)) != STREAMKL_OK) return st;

  skl::FwdArgs a{};
  a.pairs = pairs;
  a.tm_q1 = &mq1;
  a.tm_k1 = &mk1;
  a.tm_q2 = &mq2;
  a.tm_k2 = &mk2;
  a.BH = BH;
  a.plane = static_cast<long long>(BH) * NQ;
  a.NQ = NQ;
  a.NK = NK;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.kl = kl;
  a.lse1 = lse1;
  a.lse2 = lse2;
  a.part = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  a.splits = splits;
  a.tiles_per_split = tps;
  a.dev_status = dev_status;
  a.timeout_ns = wait_timeout_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = skl::launch_fwd(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (splits > 1) {
    e = skl::launch_fwd_combine(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "split combine launch");
  }
  return STREAMKL_OK;
}

// ---------------------------------------------------------------------------
// Forward pass without any caller-provided workspace.
//
// Split partial states go to a fixed scratch array compiled into the library
// instead of a buffer the caller allocates. Every GPU that loads the library
// holds this array until the process exits, and every call on that GPU shares
// it, so calls whose kernels overlap on the GPU (other streams, other host
// threads) race on it. Nothing in it has to start at zero: each call writes
// every partial state it later reads.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

constexpr size_t kFwdScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_fwd_scratch[kFwdScratchBytes];

// Device address of g_fwd_scratch, per device, and the driver context it was
// looked up in. The library's module (and with it the array) is loaded anew
// in every context: after cudaDeviceReset, or while the caller has another
// driver context current, the array lives at another address.
struct ScratchAddr {
  CUcontext ctx;
  void* ptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[256] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_current_once;

PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
  std::call_once(g_ctx_current_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  return g_ctx_current;
}

// Device address of the scratch array in the current device's current
// context. The host-side name of the array is only a stand-in, so the address
// is looked up with that device current, cached, and looked up again whenever
// the current context differs from the one the cached address came from.
streamkl_status fwd_scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 256) return fail(STREAMKL_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  auto get_ctx = ctx_current_fn();
  if (!get_ctx) return fail(STREAMKL_ERR_CUDA, "cuCtxGetCurrent unavailable from the driver");
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return fail(STREAMKL_ERR_CUDA, "cuCtxGetCurrent failed");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& c = g_scratch_addr[dev];
  if (!c.ptr || ctx == nullptr || c.ctx != ctx) {
    void* p = nullptr;
    // a runtime call: it also creates the device's primary context when no
    // context is current yet, so the context is read again afterwards
    e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return fail(STREAMKL_ERR_CUDA, "no current CUDA context");
    c.ctx = ctx;
    c.ptr = p;
  }
  *out = c.ptr;
  return STREAMKL_OK;
}

}  // namespace

extern "C" {

streamkl_status streamkl_fwd_noalloc(const void* q1, const void* k1, const void* q2,
                                     const void* k2, int B, int H, int NQ, int NK, int d,
                                     float scale, int causal, int num_splits, float* kl,
                                     float* lse1, float* lse2, int* dev_status, void* stream) {
  g_err[0] = '\0';
  streamkl_status st = check_sizes(B, H, NQ, NK, d, causal);
  if (st != STREAMKL_OK) return st;
  if (num_splits < 0) return fail(STREAMKL_ERR_INVALID_ARG, "num_splits must be >= 0");
  int splits, tps;
  split_plan(num_splits > 0 ? num_splits : choose_splits_impl(B, H, NQ, NK, d), NK, &splits, &tps);
  const size_t need = fwd_ws(B, H, NQ, splits);
  if (need > kFwdScratchBytes)
    return fail(STREAMKL_ERR_INVALID_ARG,
                "this call needs %zu bytes of split scratch but the built-in scratch holds %zu; "
                "request fewer splits or use streamkl_fwd with a workspace",
                need, kFwdScratchBytes);
  void* scratch = nullptr;
  if (need > 0 && (st = fwd_scratch_ptr(&scratch)) != STREAMKL_OK) return st;
  return streamkl_fwd(q1, k1, q2, k2, B, H, NQ, NK, d, scale, causal, splits, kl, lse1, lse2,
                      scratch, need > 0 ? kFwdScratchBytes : 0, dev_status, stream);
}

streamkl_status streamkl_bwd(const void* q1, const void* k1, const void* q2, const void* k2, int B,
                             int H, int NQ, int NK, int d, float scale, int causal, const float* kl,
                             const float* lse1, const float* lse2, const float* dkl, void* dq2,
                             void* dk2, void* dq1, void* dk1, void* workspace, size_t ws_bytes,
                             int* dev_status, void* stream) {
  g_err[0] = '\0';
  streamkl_status st = check_sizes(B, H, NQ, NK, d, causal);
  if (st != STREAMKL_OK) return st;
  if ((st = check_inputs(q1, k1, q2, k2)) != STREAMKL_OK) return st;
  if (!kl || !lse1 || !lse2 || !dkl) return fail(STREAMKL_ERR_INVALID_ARG, "kl/lse1/lse2/dkl must be non-NULL");
  if ((dq2 == nullptr) != (dk2 == nullptr))
    return fail(STREAMKL_ERR_INVALID_ARG, "dq2 and dk2 must be both NULL or both non-NULL");
  if ((dq1 == nullptr) != (dk1 == nullptr))
    return fail(STREAMKL_ERR_INVALID_ARG, "dq1 and dk1 must be both NULL or both non-NULL");
  if (!dq2 && !dq1) return fail(STREAMKL_ERR_INVALID_ARG, "no gradient requested: dq2/dk2 and dq1/dk1 are all NULL");
  if ((dq2 && (!aligned16(dq2) || !aligned16(dk2))) || (dq1 && (!aligned16(dq1) || !aligned16(dk1))))
    return fail(STREAMKL_ERR_INVALID_ARG, "gradient outputs must be 16-byte aligned");
  if (!dev_status) return fail(STREAMKL_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(STREAMKL_ERR_INVALID_ARG, "scale must be finite and > 0");
  const int grad1 = dq1 != nullptr, grad2 = dq2 != nullptr;
  // configuration 2 alone runs the separate kernels unless the fused
  // algorithm's short-sweep kernel takes the shape (the per-key-tile fused
  // kernel always produces dQ2/dK2)
  int algo = bwd_algo_impl(B, H, NQ, NK, d, causal, grad1);
  if (!grad2 && !(algo == 1 && short_sweep(NQ, d))) algo = 0;
  // separate kernels: the dQ kernel's key split keeps its fp32 partials in
  // the workspace; fused kernels: one fp32 dQ accumulator per gradient set
  int dq_splits = 1, dq_per = 0;
  if (algo == 0) dq_split_plan(B, H, NQ, NK, d, grad1 + grad2, &dq_splits, &dq_per);
  const size_t need = algo == 0 ? dq_split_ws(B, H, NQ, NK, d, grad1 + grad2)
                                : bwd_ws(B, H, NQ, NK, d, causal, grad1 && grad2);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace)))
    return fail(STREAMKL_ERR_INVALID_ARG, "backward workspace too small: need %zu bytes, got %zu", need, ws_bytes);

  const int BH = B * H;
  const bool short_kernel = algo == 1 && short_sweep(NQ, d);
  // the separate and short-sweep kernels move 64-row boxes, the per-key-tile
  // fused one 128-row boxes
  const int box_rows = (algo == 0 || short_kernel) ? 64 : skl::kBlockM;
  CUtensorMap mq1, mk1, mq2, mk2;
  if ((st = make_map(&mq1, q1, BH, NQ, d, "q1", box_rows)) != STREAMKL_OK) return st;
  if ((st = make_map(&mk1, k1, BH, NK, d, "k1", box_rows)) != STREAMKL_OK) return st;
  if ((st = make_map(&mq2, q2, BH, NQ, d, "q2", box_rows)) != STREAMKL_OK) return st;
  if ((st = make_map(&mk2, k2, BH, NK, d, "k2", box_rows)) != STREAMKL_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (algo == 0) {
    skl::BwdSepArgs a{};
    a.tm_q1 = &mq1;
    a.tm_k1 = &mk1;
    a.tm_q2 = &mq2;
    a.tm_k2 = &mk2;
    a.BH = BH;
    a.NQ = NQ;
    a.NK = NK;
    a.d = d;
    a.causal = causal;
    a.grad1 = grad1;
    a.grad2 = grad2;
    a.dq_splits = dq_splits;
    a.dq_split_steps = dq_per;
    a.dq_part = dq_splits > 1 ? static_cast<float*>(workspace) : nullptr;
    a.dk_persist_ctas = dk_persist_ctas(B, H, NQ, NK);
    a.scale = scale;
    a.kl = kl;
    a.lse1 = lse1;
    a.lse2 = lse2;
    a.g = dkl;
    a.dq2 = dq2;
    a.dk2 = dk2;
    a.dq1 = dq1;
    a.dk1 = dk1;
    // the outputs leave the kernels through TMA stores of 128-row tiles
    CUtensorMap mdk2, mdk1, mdq2, mdq1, mpart;
    if (grad2) {
      if ((st = make_map(&mdk2, dk2, BH, NK, d, "dk2", skl::kBlockM)) != STREAMKL_OK) return st;
      if ((st = make_map(&mdq2, dq2, BH, NQ, d, "dq2", skl::kBlockM)) != STREAMKL_OK) return st;
    }
    if (grad1) {
      if ((st = make_map(&mdk1, dk1, BH, NK, d, "dk1", skl::kBlockM)) != STREAMKL_OK) return st;
      if ((st = make_map(&mdq1, dq1, BH, NQ, d, "dq1", skl::kBlockM)) != STREAMKL_OK) return st;
    }
    a.tm_dk2 = grad2 ? &mdk2 : &mdk1;
    a.tm_dk1 = grad1 ? &mdk1 : &mdk2;
    a.tm_dq2 = grad2 ? &mdq2 : &mdq1;
    a.tm_dq1 = grad1 ? &mdq1 : &mdq2;
    if (dq_splits > 1) {
      if ((st = make_map_part(&mpart, workspace, (grad1 + grad2) * dq_splits, BH, NQ, d)) != STREAMKL_OK)
        return st;
      a.tm_part = &mpart;
    }
    a.dev_status = dev_status;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = skl::launch_bwd_separate(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return STREAMKL_OK;
  }
  cudaError_t e = cudaMemsetAsync(workspace, 0, need, s);
  if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
  const size_t one = need / (grad1 + grad2);
  const long long n = static_cast<long long>(BH) * NQ * d;
  if (short_kernel) {
    skl::BwdShortArgs a{};
    a.tm_q1 = &mq1;
    a.tm_k1 = &mk1;
    a.tm_q2 = &mq2;
    a.tm_k2 = &mk2;
    a.BH = BH;
    a.NQ = NQ;
    a.NK = NK;
    a.causal = causal;
    a.grad1 = grad1;
    a.grad2 = grad2;
    a.scale = scale;
    a.kl = kl;
    a.lse1 = lse1;
    a.lse2 = lse2;
    a.g = dkl;
    a.dk2 = dk2;
    a.dk1 = dk1;
    // dK leaves through TMA stores of 128-row tiles
    CUtensorMap mdk2, mdk1;
    if (grad2 && (st = make_map(&mdk2, dk2, BH, NK, d, "dk2", skl::kBlockN)) != STREAMKL_OK) return st;
    if (grad1 && (st = make_map(&mdk1, dk1, BH, NK, d, "dk1", skl::kBlockN)) != STREAMKL_OK) return st;
    a.tm_dk2 = grad2 ? &mdk2 : &mdk1;
    a.tm_dk1 = grad1 ? &mdk1 : &mdk2;
    // the accumulators of the sets computed, set 2's first
    a.dq2acc = grad2 ? static_cast<float*>(workspace) : nullptr;
    a.dq1acc = grad1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + (grad2 ? one : 0))
                     : nullptr;
    a.ctas = num_sms();
    a.dev_status = dev_status;
    a.timeout_ns = wait_timeout_ns();
    e = skl::launch_bwd_short(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    if (grad2) {
      e = skl::launch_dq_convert(a.dq2acc, dq2, n, s);
      if (e != cudaSuccess) return cuda_fail(e, "dq2 convert launch");
    }
    if (grad1) {
      e = skl::launch_dq_convert(a.dq1acc, dq1, n, s);
      if (e != cudaSuccess) return cuda_fail(e, "dq1 convert launch");
    }
    return STREAMKL_OK;
  }
  skl::BwdArgs a{};
  a.tm_q1 = &mq1;
  a.tm_k1 = &mk1;
  a.tm_q2 = &mq2;
  a.tm_k2 = &mk2;
  a.BH = BH;
  a.NQ = NQ;
  a.NK = NK;
  a.d = d;
  a.causal = causal;
  a.grad1 = grad1;
  a.scale = scale;
  a.kl = kl;
  a.lse1 = lse1;
  a.lse2 = lse2;
  a.g = dkl;
  a.dq2acc = static_cast<float*>(workspace);
  a.dq1acc = grad1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + one) : nullptr;
  a.dk2 = dk2;
  a.dk1 = dk1;
  a.dev_status = dev_status;
  a.timeout_ns = wait_timeout_ns();
  if (d == 64) {
    // one CTA per key tile; dQ through TMA reductions, dK through TMA stores
    CUtensorMap mq2acc, mq1acc, mdk2, mdk1;
    if ((st = make_map_acc(&mq2acc, a.dq2acc, BH, NQ, d)) != STREAMKL_OK) return st;
    if ((st = make_map(&mdk2, dk2, BH, NK, d, "dk2", skl::kBlockN)) != STREAMKL_OK) return st;
    if (grad1) {
      if ((st = make_map_acc(&mq1acc, a.dq1acc, BH, NQ, d)) != STREAMKL_OK) return st;
      if ((st = make_map(&mdk1, dk1, BH, NK, d, "dk1", skl::kBlockN)) != STREAMKL_OK) return st;
    }
    a.tm_dq2 = &mq2acc;
    a.tm_dq1 = grad1 ? &mq1acc : &mq2acc;
    a.tm_dk2 = &mdk2;
    a.tm_dk1 = grad1 ? &mdk1 : &mdk2;
    e = skl::launch_bwd_fused64(a, s);
  } else {
    // 64-row query steps: Q maps with 64-row boxes; dQ^T through TMA reductions
    CUtensorMap mq1s, mq2s, mq2acc, mq1acc, mdk2, mdk1;
    if ((st = make_map(&mq1s, q1, BH, NQ, d, "q1", 64)) != STREAMKL_OK) return st;
    if ((st = make_map(&mq2s, q2, BH, NQ, d, "q2", 64)) != STREAMKL_OK) return st;
    if ((st = make_map_acc(&mq2acc, a.dq2acc, BH, NQ, d, 64)) != STREAMKL_OK) return st;
    if ((st = make_map(&mdk2, dk2, BH, NK, d, "dk2", skl::kBlockN)) != STREAMKL_OK) return st;
    if (grad1) {
      if ((st = make_map_acc(&mq1acc, a.dq1acc, BH, NQ, d, 64)) != STREAMKL_OK) return st;
      if ((st = make_map(&mdk1, dk1, BH, NK, d, "dk1", skl::kBlockN)) != STREAMKL_OK) return st;
    }
    a.tm_q1 = &mq1s;
    a.tm_q2 = &mq2s;
    a.tm_dq2 = &mq2acc;
    a.tm_dq1 = grad1 ? &mq1acc : &mq2acc;
    a.tm_dk2 = &mdk2;
    a.tm_dk1 = grad1 ? &mdk1 : &mdk2;
    e = skl::launch_bwd_fused128(a, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  e = skl::launch_dq_convert(a.dq2acc, dq2, n, s);
  if (e != cudaSuccess) return cuda_fail(e, "dq2 convert launch");
  if (grad1) {
    e = skl::launch_dq_convert(a.dq1acc, dq1, n, s);
    if (e != cudaSuccess) return cuda_fail(e, "dq1 convert launch");
  }
  return STREAMKL_OK;
}

// ---------------------------------------------------------------------------
// Reverse direction KL(P2 || P1): the teacher-first computation with the two
// distributions exchanged. Only the argument slots move.
streamkl_status streamkl_fwd_reverse(const void* q1, const void* k1, const void* q2, const void* k2,
                                     int B, int H, int NQ, int NK, int d, float scale, int causal,
                                     int num_splits, float* kl, float* lse1, float* lse2,
                                     void* workspace, size_t ws_bytes, int* dev_status,
                                     void* stream) {
  return streamkl_fwd(q2, k2, q1, k1, B, H, NQ, NK, d, scale, causal, num_splits, kl, lse2, lse1,
                      workspace, ws_bytes, dev_status, stream);
}

streamkl_status streamkl_bwd_reverse(const void* q1, const void* k1, const void* q2, const void* k2,
                                     int B, int H, int NQ, int NK, int d, float scale, int causal,
                                     const float* kl, const float* lse1, const float* lse2,
                                     const float* dkl, void* dq2, void* dk2, void* dq1, void* dk1,
                                     void* workspace, size_t ws_bytes, int* dev_status,
                                     void* stream) {
  g_err[0] = '\0';
  if ((dq2 == nullptr) != (dk2 == nullptr))
    return fail(STREAMKL_ERR_INVALID_ARG, "dq2 and dk2 must be both NULL or both non-NULL");
  if ((dq1 == nullptr) != (dk1 == nullptr))
    return fail(STREAMKL_ERR_INVALID_ARG, "dq1 and dk1 must be both NULL or both non-NULL");
  // In the exchanged call the student is the first distribution: its
  // gradients are that call's configuration-2 outputs (dq1/dk1 slots), the
  // teacher's its configuration-1 outputs (dq2/dk2 slots).
  return streamkl_bwd(q2, k2, q1, k1, B, H, NQ, NK, d, scale, causal, kl, lse2, lse1, dkl, dq1, dk1,
                      dq2, dk2, workspace, ws_bytes, dev_status, stream);
}

streamkl_status streamkl_fwd_varlen(const void* q1, const void* k1, const void* q2, const void* k2,
                                    const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                                    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                    int d, float scale, int causal, float* kl, float* lse1,
                                    float* lse2, int* dev_status, void* stream) {
  g_err[0] = '\0';
  streamkl_status st = check_packed(cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                                    max_seqlen_q, max_seqlen_k, d, causal);
  if (st != STREAMKL_OK) return st;
  if (causal != 0 && causal != 1) return fail(STREAMKL_ERR_INVALID_ARG, "causal must be 0 or 1");
  if ((st = check_inputs(q1, k1, q2, k2)) != STREAMKL_OK) return st;
  if (!kl || !lse1 || !lse2) return fail(STREAMKL_ERR_INVALID_ARG, "kl, lse1, lse2 must be non-NULL");
  if (!dev_status) return fail(STREAMKL_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(STREAMKL_ERR_INVALID_ARG, "scale must be finite and > 0");
  CUtensorMap mq1, mk1, mq2, mk2;
  if ((st = make_map_packed(&mq1, q1, total_q, H, d, "q1", skl::kBlockM)) != STREAMKL_OK) return st;
  if ((st = make_map_packed(&mk1, k1, total_k, H, d, "k1", skl::kBlockM)) != STREAMKL_OK) return st;
  if ((st = make_map_packed(&mq2, q2, total_q, H, d, "q2", skl::kBlockM)) != STREAMKL_OK) return st;
  if ((st = make_map_packed(&mk2, k2, total_k, H, d, "k2", skl::kBlockM)) != STREAMKL_OK) return st;
  skl::FwdArgs a{};
  a.tm_q1 = &mq1;
  a.tm_k1 = &mk1;
  a.tm_q2 = &mq2;
  a.tm_k2 = &mk2;
  a.BH = B * H;
  a.NQ = max_seqlen_q;
  a.NK = max_seqlen_k;
  a.d = d;
  a.causal = causal;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.H = H;
  a.total_q = total_q;
  a.total_k = total_k;
  a.plane = static_cast<long long>(total_q) * H;
  a.scale = scale;
  a.kl = kl;
  a.lse1 = lse1;
  a.lse2 = lse2;
  a.part = nullptr;
  a.splits = 1;
  a.tiles_per_split = key_tiles(max_seqlen_k);
  a.dev_status = dev_status;
  a.timeout_ns = wait_timeout_ns();
  cudaError_t e = skl::launch_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return STREAMKL_OK;
}

streamkl_status streamkl_bwd_varlen(const void* q1, const void* k1, const void* q2, const void* k2,
                                    const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                                    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                    int d, float scale, int causal, const float* kl,
                                    const float* lse1, const float* lse2, const float* dkl,
                                    void* dq2, void* dk2, void* dq1, void* dk1, int* dev_status,
                                    void* stream) {
  g_err[0] = '\0';
  streamkl_status st = check_packed(cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                                    max_seqlen_q, max_seqlen_k, d, causal);
  if (st != STREAMKL_OK) return st;
  if (causal != 0 && causal != 1) return fail(STREAMKL_ERR_INVALID_ARG, "causal must be 0 or 1");
  if ((st = check_inputs(q1, k1, q2, k2)) != STREAMKL_OK) return st;
  if (!kl || !lse1 || !lse2 || !dkl) return fail(STREAMKL_ERR_INVALID_ARG, "kl/lse1/lse2/dkl must be non-NULL");
  if ((dq2 == nullptr) != (dk2 == nullptr))
    return fail(STREAMKL_ERR_INVALID_ARG, "dq2 and dk2 must be both NULL or both non-NULL");
  if ((dq1 == nullptr) != (dk1 == nullptr))
    return fail(STREAMKL_ERR_INVALID_ARG, "dq1 and dk1 must be both NULL or both non-NULL");
  if (!dq2 && !dq1) return fail(STREAMKL_ERR_INVALID_ARG, "no gradient requested: dq2/dk2 and dq1/dk1 are all NULL");
  if ((dq2 && (!aligned16(dq2) || !aligned16(dk2))) || (dq1 && (!aligned16(dq1) || !aligned16(dk1))))
    return fail(STREAMKL_ERR_INVALID_ARG, "gradient outputs must be 16-byte aligned");
  if (!dev_status) return fail(STREAMKL_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(STREAMKL_ERR_INVALID_ARG, "scale must be finite and > 0");
  CUtensorMap mq1, mk1, mq2, mk2;  // the separate kernels move 64-row boxes
  if ((st = make_map_packed(&mq1, q1, total_q, H, d, "q1", 64)) != STREAMKL_OK) return st;
  if ((st = make_map_packed(&mk1, k1, total_k, H, d, "k1", 64)) != STREAMKL_OK) return st;
  if ((st = make_map_packed(&mq2, q2, total_q, H, d, "q2", 64)) != STREAMKL_OK) return st;
  if ((st = make_map_packed(&mk2, k2, total_k, H, d, "k2", 64)) != STREAMKL_OK) return st;
  skl::BwdSepArgs a{};
  a.tm_q1 = &mq1;
  a.tm_k1 = &mk1;
  a.tm_q2 = &mq2;
  a.tm_k2 = &mk2;
  a.BH = B * H;
  a.NQ = max_seqlen_q;
  a.NK = max_seqlen_k;
  a.d = d;
  a.causal = causal;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.H = H;
  a.total_q = total_q;
  a.total_k = total_k;
  a.grad1 = dq1 != nullptr;
  a.grad2 = dq2 != nullptr;
  a.scale = scale;
  a.kl = kl;
  a.lse1 = lse1;
  a.lse2 = lse2;
  a.g = dkl;
  a.dq2 = dq2;
  a.dk2 = dk2;
  a.dq1 = dq1;
  a.dk1 = dk1;
  a.dev_status = dev_status;
  a.timeout_ns = wait_timeout_ns();
  cudaError_t e = skl::launch_bwd_separate(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return STREAMKL_OK;
}

streamkl_status streamkl_selftest_device_check(int* dev_status, void* stream) {
  g_err[0] = '\0';
  if (!dev_status) return fail(STREAMKL_ERR_INVALID_ARG, "dev_status must be non-NULL");
  cudaError_t e = skl::launch_check_selftest(dev_status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return STREAMKL_OK;
}

streamkl_status streamkl_selftest_wait_timeout(int* dev_status, unsigned timeout_us, void* stream) {
  g_err[0] = '\0';
  if (!dev_status) return fail(STREAMKL_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if (timeout_us < 1 || timeout_us > 5000000u)
    return fail(STREAMKL_ERR_INVALID_ARG, "timeout_us must be in [1, 5e6]");
  cudaError_t e = skl::launch_wait_selftest(dev_status, static_cast<uint64_t>(timeout_us) * 1000ull,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return STREAMKL_OK;
}

}  // extern "C"

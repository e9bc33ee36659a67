// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace skl {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per tile

// Where one (batch, head) slice of the inputs lives.
//   dense  [B, H, N, d]:     rows of a head are contiguous (d apart)
//   packed [total, H, d]:    variable-length batch, sequence b owning rows
//                            cu[b] .. cu[b+1]; rows of one head are H d apart
// TMA maps see the dense tensors as {d, N, B H} and the packed ones as
// {d, total, H}; per-row fp32 vectors (KL, LSE, g) are [B, H, N_Q] or
// [total_q, H] accordingly.
struct SeqView {
  int nq, nk;               // this slice's query and key rows
  int q_row0, k_row0;       // TMA row coordinate of its row 0
  int z;                    // TMA third coordinate
  long long v_off;          // per-row vectors: element of query row 0
  int v_stride;             // ... and between consecutive query rows
  long long q_off, k_off;   // bf16 tensors: element (row 0, column 0)
  long long row_stride;     // elements between consecutive rows
  bool ok;                  // offsets well formed (packed batches only can fail)
};

// Dense [B, H, N, d] slice bh (sizes NQ, NK).
__device__ __forceinline__ SeqView seq_view_dense(int bh, int NQ, int NK, int d) {
  SeqView v;
  v.nq = NQ;
  v.nk = NK;
  v.q_row0 = v.k_row0 = 0;
  v.z = bh;
  v.v_off = static_cast<long long>(bh) * NQ;
  v.v_stride = 1;
  v.q_off = static_cast<long long>(bh) * NQ * d;
  v.k_off = static_cast<long long>(bh) * NK * d;
  v.row_stride = d;
  v.ok = true;
  return v;
}

// Packed [total, H, d] slice bh = b H + h: sequence b's offsets from cu_q,
// cu_k (device); max_q, max_k are the lengths the grid was sized for.
__device__ __forceinline__ SeqView seq_view_packed(int bh, int H, int max_q, int max_k, int d,
                                                   const int* cu_q, const int* cu_k, int total_q,
                                                   int total_k) {
  SeqView v;
  const int b = bh / H, h = bh - b * H;
  const int q0 = cu_q[b], q1 = cu_q[b + 1], k0 = cu_k[b], k1 = cu_k[b + 1];
  v.nq = q1 - q0;
  v.nk = k1 - k0;
  v.q_row0 = q0;
  v.k_row0 = k0;
  v.z = h;
  v.v_off = static_cast<long long>(q0) * H + h;
  v.v_stride = H;
  v.q_off = (static_cast<long long>(q0) * H + h) * d;
  v.k_off = (static_cast<long long>(k0) * H + h) * d;
  v.row_stride = static_cast<long long>(H) * d;
  // query rows need at least one key (a softmax over no key is undefined)
  v.ok = q0 >= 0 && k0 >= 0 && v.nq >= 0 && v.nk >= 0 && v.nq <= max_q && v.nk <= max_k &&
         q1 <= total_q && k1 <= total_k && !(v.nq > 0 && v.nk == 0);
  return v;
}

struct FwdArgs {
  const CUtensorMap* tm_q1;
  const CUtensorMap* tm_k1;
  const CUtensorMap* tm_q2;
  const CUtensorMap* tm_k2;
  int BH, NQ, NK, d, causal;
  const int* cu_q = nullptr;  // packed variable-length batch (device offsets), else null
  const int* cu_k = nullptr;
  int H = 1, total_q = 0, total_k = 0;
  long long plane = 0;        // per-row vector entries (B H N_Q, or total_q H)
  float scale;
  float* kl;
  float* lse1;
  float* lse2;
  float* part;  // split partial states, [5][splits][BH][NQ]; null when splits == 1
  int splits;
  int tiles_per_split;
  // CTA pairs (cta_group::2 MMAs over two query blocks; needs
  // fwd_pair_eligible): the K maps then have 64-row boxes
  bool pairs = false;
  int* dev_status;
  uint64_t timeout_ns;
};

// Fused algorithm beyond the short-sweep shapes (one CTA per key tile, each
// (query, key) pair visited once, dQ added into fp32 accumulators).
struct BwdArgs {
  const CUtensorMap* tm_q1;
  const CUtensorMap* tm_k1;
  const CUtensorMap* tm_q2;
  const CUtensorMap* tm_k2;
  int BH, NQ, NK, d, causal, grad1;
  float scale;
  const float* kl;
  const float* lse1;
  const float* lse2;
  const float* g;
  float* dq2acc;  // [BH][NQ][d] fp32, zeroed by the caller
  float* dq1acc;  // same, grad1 only
  void* dk2;      // bf16 [BH][NK][d]
  void* dk1;      // bf16, grad1 only
  // d = 64 kernel: the fp32 dQ accumulators as {d, N_Q, BH} maps with
  // 32-column x 128-row boxes (TMA reductions) and the bf16 dK outputs as
  // {d, N_K, BH} maps with 64-column x 128-row boxes (TMA stores); a set not
  // computed may repeat the other's map
  const CUtensorMap* tm_dq2 = nullptr;
  const CUtensorMap* tm_dq1 = nullptr;
  const CUtensorMap* tm_dk2 = nullptr;
  const CUtensorMap* tm_dk1 = nullptr;
  int* dev_status;
  uint64_t timeout_ns;
};

struct BwdSepArgs {
  const CUtensorMap* tm_q1;  // 64-column x 64-row boxes
  const CUtensorMap* tm_k1;
  const CUtensorMap* tm_q2;
  const CUtensorMap* tm_k2;
  int BH, NQ, NK, d, causal;
  const int* cu_q = nullptr;  // packed variable-length batch (device offsets), else null
  const int* cu_k = nullptr;
  int H = 1, total_q = 0, total_k = 0;
  int grad1, grad2;  // gradient sets wanted: dQ1/dK1 (configuration 2), dQ2/dK2 (configuration 1)
  float scale;
  const float* kl;
  const float* lse1;
  const float* lse2;
  const float* g;
  void* dq2;  // bf16 outputs (NULL when grad2 == 0)
  void* dk2;
  void* dq1;  // grad1 only
  void* dk1;
  // dQ kernel key split (dense batches): dq_splits > 1 splits the key steps
  // into chunks of dq_split_steps; partial dQ rows go to dq_part (fp32
  // [sets][dq_splits][BH NQ][d]) and a combine kernel sums them
  int dq_splits = 1, dq_split_steps = 0;
  // dK kernel as a persistent grid of this many CTAs over (key block, batch-head)
  // items (dense batches; 0: one CTA per key block)
  int dk_persist_ctas = 0;
  float* dq_part = nullptr;
  // output tensor maps (dense batches; packed batches and the persistent dK
  // kernel store rows directly): bf16 dK / dQ as {d, N, BH} with 64-column x
  // 128-row boxes, the dQ split's fp32 partials as {d, N_Q, BH, set x split}
  // with 32-column x 128-row boxes; a set not computed may repeat another map
  const CUtensorMap* tm_dk2 = nullptr;
  const CUtensorMap* tm_dk1 = nullptr;
  const CUtensorMap* tm_dq2 = nullptr;
  const CUtensorMap* tm_dq1 = nullptr;
  const CUtensorMap* tm_part = nullptr;
  int* dev_status;
  uint64_t timeout_ns;
};

// Fused backward for short query sweeps (N_Q <= 64, d = 128, dense batches):
// a persistent grid over (batch-head, 128-key tile) items; dK written per
// item, dQ kept in TMEM per batch-head and added to the fp32 accumulators
// (zeroed by the caller) when a CTA's batch-head changes.
struct BwdShortArgs {
  const CUtensorMap* tm_q1;  // 64-column x 64-row boxes
  const CUtensorMap* tm_k1;
  const CUtensorMap* tm_q2;
  const CUtensorMap* tm_k2;
  int BH, NQ, NK, causal;
  int grad1, grad2;  // gradient sets: configuration 2 (dQ1/dK1), configuration 1 (dQ2/dK2)
  float scale;
  const float* kl;
  const float* lse1;
  const float* lse2;
  const float* g;
  void* dk2;       // bf16 [BH][NK][d]
  void* dk1;
  const CUtensorMap* tm_dk2;  // the dK outputs, 64-column x 128-row boxes (a
  const CUtensorMap* tm_dk1;  // set not computed: any valid map, never used)
  float* dq2acc;   // fp32 [BH][NQ][d]
  float* dq1acc;
  int ctas;        // persistent grid size (one CTA per SM)
  int* dev_status;
  uint64_t timeout_ns;
};
constexpr int kShortMaxQ = 64;  // query rows the short-sweep kernel handles

// Each returns the launch error (cudaSuccess when queued).
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
bool fwd_pair_eligible(int NQ, int splits, bool packed);
cudaError_t launch_fwd_combine(const FwdArgs& a, cudaStream_t stream);
// fused algorithm at d = 64 (one CTA per key tile, dQ through TMA reductions)
cudaError_t launch_bwd_fused64(const BwdArgs& a, cudaStream_t stream);
// fused algorithm at d = 128: one CTA per key tile, 64-row query steps, dQ^T
// through TMA reductions; the Q maps with 64-row boxes, the dQ accumulator
// maps with 32-column x 64-row boxes
cudaError_t launch_bwd_fused128(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_separate(const BwdSepArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_short(const BwdShortArgs& a, cudaStream_t stream);
cudaError_t launch_dq_convert(const float* acc, void* out_bf16, long long n, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* dev_status, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_check_selftest(int* dev_status, cudaStream_t stream);

size_t fwd_smem_bytes(int d);
size_t bwd_sep_smem_bytes(int d, int grad1);
size_t bwd_short_smem_bytes(int grad1, int grad2);

}  // namespace skl

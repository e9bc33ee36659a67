// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace skl {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per tile

struct FwdArgs {
  const CUtensorMap* tm_q1;
  const CUtensorMap* tm_k1;
  const CUtensorMap* tm_q2;
  const CUtensorMap* tm_k2;
  int BH, NQ, NK, d, causal;
  float scale;
  float* kl;
  float* lse1;
  float* lse2;
  float* part;  // split partial states, [5][splits][BH][NQ]; null when splits == 1
  int splits;
  int tiles_per_split;
  int* dev_status;
  uint64_t timeout_ns;
};

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
  float* dq2acc;  // [BH][NQ][d] fp32, zeroed by the caller of launch_bwd
  float* dq1acc;  // same, grad1 only
  void* dk2;      // bf16 [BH][NK][d]
  void* dk1;      // bf16, grad1 only
  int* dev_status;
  uint64_t timeout_ns;
};

struct BwdSepArgs {
  const CUtensorMap* tm_q1;  // 64-column x 64-row boxes
  const CUtensorMap* tm_k1;
  const CUtensorMap* tm_q2;
  const CUtensorMap* tm_k2;
  int BH, NQ, NK, d, causal;
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
  int* dev_status;
  uint64_t timeout_ns;
};

// Each returns the launch error (cudaSuccess when queued).
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_combine(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_separate(const BwdSepArgs& a, cudaStream_t stream);
cudaError_t launch_dq_convert(const float* acc, void* out_bf16, long long n, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* dev_status, uint64_t timeout_ns, cudaStream_t stream);

size_t fwd_smem_bytes(int d);
size_t bwd_smem_bytes(int d, int grad1);
size_t bwd_sep_smem_bytes(int d, int grad1);

}  // namespace skl

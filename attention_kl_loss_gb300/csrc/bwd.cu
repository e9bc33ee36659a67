// Helpers of the backward: the fused algorithm's fp32 -> bf16 dQ conversion
// and the self-test kernels of the bounded waits and of the debug build's
// range checks.
#include "kernels.h"
#include "ptx.cuh"

namespace skl {

namespace {

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

}  // namespace

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

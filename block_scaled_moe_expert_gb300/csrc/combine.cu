// Deterministic gather-combine of the weighted per-pair rows.
//
// fp8_grouped_mm_experts_forward (source excerpt on the error page
// "grouped_mm experts dispatch does not support activation_scheme='static'")
// zeroes the
// sentinel rows and then reduces the top-k rows of each token with
// view(T, K, H).sum(1) instead of index_add_, because atomicAdd with
// duplicate indices is non-deterministic; the result is cast back to the
// input dtype. Here each token reads the fp32 rows of its valid slots in
// ascending k (a skipped slot is never read, which is the zeroing), sums them
// in fp32 in that fixed order and rounds once to bf16. One thread owns 8
// output columns; there are no atomics.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace bsmoe {

namespace {

constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv, int H, int K,
               __nv_bfloat16* __restrict__ out) {
  const int t = blockIdx.x;
  __shared__ int rows[kMaxTopK];
  pdl_wait();  // y comes from GEMM2
  pdl_launch_dependents();
  if (threadIdx.x < K) rows[threadIdx.x] = __ldg(inv + static_cast<size_t>(t) * K + threadIdx.x);
  __syncthreads();
  for (int c = (blockIdx.y * kCombineThreads + threadIdx.x) * 8; c < H; c += gridDim.y * kCombineThreads * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < K; ++k) {
      const int r = rows[k];
      if (r < 0) continue;
      const float4* p = reinterpret_cast<const float4*>(y + static_cast<size_t>(r) * H + c);
      const float4 a = __ldg(p), b = __ldg(p + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    __nv_bfloat162 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + c) = *reinterpret_cast<uint4*>(o);
  }
}

}  // namespace

cudaError_t launch_combine(const float* y, const int32_t* inv, int T, int H, int K, void* out, cudaStream_t st) {
  const int ygrid = ceil_div(H, kCombineThreads * 8);
  return launch_kernel(true, combine_kernel, dim3(T, ygrid), kCombineThreads, 0, st, y, inv, H, K,
                       reinterpret_cast<__nv_bfloat16*>(out));
}

}  // namespace bsmoe

// Dynamic activation quantization fused with the padded permute, and the
// host-side arguments of the small-batch routing + quantization device code
// that the single-launch decode forward runs.
//
// The grouped experts dispatch quantizes activations dynamically per block
// (error page "grouped_mm experts dispatch does not support
// activation_scheme='static'", section "What it means"); rows are then
// gathered by slot // K into the grouped layout (fp8_grouped_mm_experts_forward,
// the source excerpt on the same page). The rule and the shared device code
// are in route_quant.cuh.
#include <cuda_bf16.h>

#include "route_quant.cuh"

namespace bsmoe {

namespace {

constexpr int kQuantWarps = 8;

// One CTA per token: gathers the token's valid slots from inv (in ascending
// k) and quantizes the row into each of their padded rows (kFp4: the e2m1
// 1x32 rule of the FP4-activation variant). With the combine in GEMM2's
// epilogue (comb_cnt non-null) it also sets up the token's arrival counters
// and, for a token whose slots are all skipped, its +0 output row.
template <bool kFp4>
__global__ void __launch_bounds__(kQuantWarps * 32)
quant_permute_kernel(const __nv_bfloat16* __restrict__ hidden, const float* __restrict__ topk_w, int H, int K, int Kp,
                     const int32_t* __restrict__ inv, uint8_t* __restrict__ xq, uint32_t* __restrict__ xsf,
                     float* __restrict__ row_w, int32_t* __restrict__ comb_cnt, int comb_stride,
                     __nv_bfloat16* __restrict__ out) {
  const int t = blockIdx.x;
  __shared__ int rows[kMaxTopK];
  __shared__ int nrows;
  __shared__ __align__(128) uint8_t qrow[kMaxRowBytes];
  __shared__ uint32_t qsf[kMaxRowBytes / 128];
  pdl_wait();  // inv comes from the routing kernel
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    int n = 0;
    for (int k = 0; k < K; ++k) {
      const int r = __ldg(inv + static_cast<size_t>(t) * K + k);
      if (r >= 0) {
        rows[n++] = r;
        row_w[r] = __ldg(topk_w + static_cast<size_t>(t) * K + k);
      }
    }
    nrows = n;
  }
  __syncthreads();
  if (comb_cnt != nullptr) setup_combine(t, nrows, comb_cnt, comb_stride, out, H);
  if (nrows == 0) return;
  quantize_token<kQuantWarps, false, kFp4>(hidden + static_cast<size_t>(t) * H, H, Kp, rows, nrows, xq, xsf, qrow,
                                           qsf);
}

}  // namespace

cudaError_t launch_quant(int fmt, const void* hidden, const float* topk_w, int T, int H, int K, const WsLayout& L,
                         uint8_t* ws, void* out, cudaStream_t st) {
  const moe_workspace_layout& p = L.pub;
  return launch_kernel(true, fmt == MOE_W_FP4_ACT_FP4 ? quant_permute_kernel<true> : quant_permute_kernel<false>, T,
                       kQuantWarps * 32, 0, st,
                       reinterpret_cast<const __nv_bfloat16*>(hidden), topk_w, H, K, p.xq_cols,
                       reinterpret_cast<const int32_t*>(ws + p.inv), ws + p.xq, reinterpret_cast<uint32_t*>(ws + p.xsf),
                       reinterpret_cast<float*>(ws + L.row_w),
                       L.combine_cnt ? reinterpret_cast<int32_t*>(ws + L.combine_cnt) : nullptr, L.combine_stride,
                       reinterpret_cast<__nv_bfloat16*>(out));
}

RqArgs make_rq_args(const int32_t* topk_idx, const void* hidden, const float* topk_w, int T, int H, int E, int K,
                    const WsLayout& L, uint8_t* ws, void* out) {
  const moe_workspace_layout& p = L.pub;
  RqArgs a;
  a.idx = topk_idx;
  a.topk_w = topk_w;
  a.row_w = reinterpret_cast<float*>(ws + L.row_w);
  a.hidden = reinterpret_cast<const __nv_bfloat16*>(hidden);
  a.T = T;
  a.S = T * K;
  a.E = E;
  a.K = K;
  a.H = H;
  a.Kp = p.xq_cols;
  a.M = L.M;
  a.counts = reinterpret_cast<int32_t*>(ws + p.counts);
  a.offsets = reinterpret_cast<int32_t*>(ws + p.offsets);
  a.padded_offsets = reinterpret_cast<int32_t*>(ws + p.padded_offsets);
  a.perm = reinterpret_cast<int32_t*>(ws + p.perm);
  a.inv = reinterpret_cast<int32_t*>(ws + p.inv);
  a.row_slot = reinterpret_cast<int32_t*>(ws + p.row_slot);
  a.tiles = reinterpret_cast<int32_t*>(ws + p.tiles);
  a.status = reinterpret_cast<uint32_t*>(ws + p.status);
  a.xq = ws + p.xq;
  a.xsf = reinterpret_cast<uint32_t*>(ws + p.xsf);
  a.comb_cnt = L.combine_cnt ? reinterpret_cast<int32_t*>(ws + L.combine_cnt) : nullptr;
  a.comb_stride = L.combine_stride;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.ready = L.chunk_ready ? reinterpret_cast<int32_t*>(ws + L.chunk_ready) : nullptr;
  a.ready_n = L.M / kChunkRows;
  return a;
}

}  // namespace bsmoe

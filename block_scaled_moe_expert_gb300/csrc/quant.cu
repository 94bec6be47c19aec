// Dynamic 1x128 activation quantization fused with the padded permute.
//
// The grouped experts dispatch quantizes activations dynamically per block
// (finegrained_fp8.py error page, "What it means"); rows are then gathered by
// slot // K into the grouped layout ("fp8_grouped_mm_experts_forward",
// finegrained_fp8.py excerpt). Each token is quantized once and its bytes are
// copied to the padded row of every valid slot of that token, which equals
// quantizing the gathered rows.
//
// Rule per 128-wide block of a row (last block partial when H % 128 != 0):
//   e = min{n : amax <= 448 * 2^n} (0 if amax == 0, clamped to [-127, 127]),
//   q = e4m3(x * 2^-e), round to nearest even with saturation.
// x * 2^-e is exact (power-of-two scaling of a bf16 value), so the byte only
// depends on the hardware conversion's rounding. Columns [H, Kp) of every
// written row are zero so that K padding contributes nothing.
#include <cuda_bf16.h>

#include "act_quant.cuh"
#include "moe_internal.cuh"

namespace bsmoe {

namespace {

constexpr int kQuantWarps = 8;

// One CTA per token. A warp covers 256 columns (two 128-column blocks) per
// step: each lane loads 8 bf16 (16 bytes), the 16 lanes of a half-warp reduce
// the block's amax, and each lane stores 8 code bytes per destination row, so
// a warp writes 256 contiguous bytes of every row it copies to.
__global__ void __launch_bounds__(kQuantWarps * 32)
quant_permute_kernel(const __nv_bfloat16* __restrict__ hidden, int H, int K, int Kp,
                     const int32_t* __restrict__ inv, uint8_t* __restrict__ xq, uint32_t* __restrict__ xsf) {
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = Kp / 128;
  __shared__ int rows[kMaxTopK];
  __shared__ int nrows;
  if (threadIdx.x == 0) {
    int n = 0;
    for (int k = 0; k < K; ++k) {
      const int r = __ldg(inv + static_cast<size_t>(t) * K + k);
      if (r >= 0) rows[n++] = r;
    }
    nrows = n;
  }
  __syncthreads();
  const int n = nrows;
  if (n == 0) return;
  const __nv_bfloat16* xr = hidden + static_cast<size_t>(t) * H;
  for (int c0w = warp * 256; c0w < Kp; c0w += kQuantWarps * 256) {
    const int c0 = c0w + lane * 8;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (c0 < H) {  // H % 64 == 0: a lane's 8 columns are all in or all out
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(xr + c0));
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __low2float(p2[i]);
        v[2 * i + 1] = __high2float(p2[i]);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = act_exponent(amax);
    const float s = exp2_neg(e);
    const uint2 q = make_uint2(pack4_e4m3(v[0] * s, v[1] * s, v[2] * s, v[3] * s),
                               pack4_e4m3(v[4] * s, v[5] * s, v[6] * s, v[7] * s));
    const uint32_t word = static_cast<uint32_t>(e + 127) * 0x01010101u;
    const bool in_range = c0 < Kp;
    const int blk = c0 / 128;
    for (int i = 0; i < n; ++i) {
      const int r = rows[i];
      if (in_range) {
        *reinterpret_cast<uint2*>(xq + static_cast<size_t>(r) * Kp + c0) = q;
        if ((lane & 15) == 0) xsf[sf_word_index(r, blk, nblk)] = word;
      }
    }
  }
}

}  // namespace

cudaError_t launch_quant(const void* hidden, int T, int H, int K, const WsLayout& L, uint8_t* ws, cudaStream_t st) {
  const moe_workspace_layout& p = L.pub;
  quant_permute_kernel<<<T, kQuantWarps * 32, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(hidden), H, K, p.xq_cols, reinterpret_cast<const int32_t*>(ws + p.inv),
      ws + p.xq, reinterpret_cast<uint32_t*>(ws + p.xsf));
  return cudaGetLastError();
}

}  // namespace bsmoe

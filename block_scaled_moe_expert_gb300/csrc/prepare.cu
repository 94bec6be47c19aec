// One-shot weight transform into the kernel layout.
//
// The Mega MoE forward (source excerpt on the error pages "DeepGEMM Mega MoE
// requires a process_group for the EP group" and "... requires FP4-packed
// expert weights") packs the
// UE8M0 scale factors and interleaves the L1/L2 weights once, before the
// first forward. This is the same idea made explicit:
//   * gate_up rows are interleaved in 64-row groups so that one 256-row
//     N tile t holds gate and up rows of the same 128 intermediate columns:
//       tile rows [  0, 64) gate j = 128t + r      [ 64,128) up j = 128t + r - 64
//       tile rows [128,192) gate j = 128t + r - 64 [192,256) up j = 128t + r - 128
//     (up j is original row I + j); rows with j >= I are zero;
//   * K is padded to a multiple of 128 and N to a multiple of 256 with zeros;
//   * FP8 block scales become one fp32 per (32 prepared rows, 128-K block),
//     laid out [E][N tile][K block][8] so that the 8 scales of one tile and K
//     block are 32 contiguous bytes;
//   * FP4 UE8M0 scales become, per (expert, N tile, K block), the 1 KB image
//     of the two 128-row scale blocks that tcgen05.cp copies into tensor
//     memory: word(row r) at 4 * (r % 32) + r / 32, byte j = scale of the
//     j-th 32-wide K chunk.
// The experts dispatch picks grouped_fp8_fp4_matmul_nn when the expert
// weights are stored transposed (is_transposed: N contiguous instead of K);
// the transposed variant below reads that storage and writes the same
// prepared layout, so the forward is the same for both.
#include "moe_internal.cuh"

namespace bsmoe {

GemmGeom geom_w13(int H, int I) {
  GemmGeom g;
  g.Kp = ceil_div(H, 128) * 128;
  g.KB = g.Kp / 128;
  g.Np = 2 * ceil_div(I, 128) * 128;
  g.NT = g.Np / 256;
  g.N = 2 * I;
  return g;
}

GemmGeom geom_w2(int H, int I) {
  GemmGeom g;
  g.Kp = ceil_div(I, 128) * 128;
  g.KB = g.Kp / 128;
  g.Np = ceil_div(H, 256) * 256;
  g.NT = g.Np / 256;
  g.N = H;
  return g;
}

PrepLayout prep_layout(int fmt, int E, const GemmGeom& g) {
  PrepLayout p;
  const size_t row_bytes = (fmt == MOE_W_FP8) ? g.Kp : g.Kp / 2;
  p.codes_off = 0;
  p.codes_bytes = static_cast<size_t>(E) * g.Np * row_bytes;
  p.scale_off = align_up(p.codes_bytes, 1024);
  if (fmt == MOE_W_FP8)
    p.scale_bytes = static_cast<size_t>(E) * (g.Np / 32) * g.KB * sizeof(float);
  else
    p.scale_bytes = static_cast<size_t>(E) * g.NT * g.KB * 256 * sizeof(uint32_t);
  p.total = align_up(p.scale_off + p.scale_bytes, 1024);
  return p;
}

namespace {

// Prepared row -> original row, or -1 for a zero row.
__device__ __forceinline__ int orig_row(bool is_w13, int p, int I, int H) {
  if (!is_w13) return p < H ? p : -1;
  static_assert(kBlockN == 4 * kGroup, "an N tile holds two gate and two up groups");
  const int t = p / kBlockN, r = p % kBlockN;
  const int q = r / kGroup;
  const int j = (kBlockN / 2) * t + kGroup * (q / 2) + (r % kGroup);
  if (j >= I) return -1;
  return (q & 1) ? I + j : j;
}

// Copy one prepared row of codes (row_bytes = Kp or Kp/2), zero padded.
__global__ void prep_codes_kernel(bool is_w13, const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int Np,
                                  int src_row_bytes, int dst_row_bytes, int src_rows, int I, int H) {
  const int p = blockIdx.x, e = blockIdx.y;
  const int o = orig_row(is_w13, p, I, H);
  uint8_t* d = dst + (static_cast<size_t>(e) * Np + p) * dst_row_bytes;
  const uint8_t* s = (o >= 0) ? src + (static_cast<size_t>(e) * src_rows + o) * src_row_bytes : nullptr;
  for (int c = threadIdx.x * 16; c < dst_row_bytes; c += blockDim.x * 16) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (s != nullptr && c < src_row_bytes) {
      if (c + 16 <= src_row_bytes && (src_row_bytes % 16) == 0) {
        v = *reinterpret_cast<const uint4*>(s + c);
      } else {
        uint8_t tmp[16];
        for (int i = 0; i < 16; ++i) tmp[i] = (c + i < src_row_bytes) ? s[c + i] : 0;
        v = *reinterpret_cast<uint4*>(tmp);
      }
    }
    *reinterpret_cast<uint4*>(d + c) = v;
  }
}

// FP8 scales: out[e][nt][kb][j] = scale[e][orig(256 nt + 32 j) / 128][kb]
// (0 for zero rows).
__global__ void prep_scale_fp8_kernel(bool is_w13, bool transposed, const float* __restrict__ src,
                                      float* __restrict__ dst, int Np, int KB, int src_rb, int src_kb, int I, int H) {
  const int e = blockIdx.y;
  const int NT = Np / 256;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < NT * KB * 8; i += gridDim.x * blockDim.x) {
    const int j = i % 8, kb = (i / 8) % KB, nt = i / (8 * KB);
    const int o = orig_row(is_w13, nt * 256 + j * 32, I, H);
    float v = 0.f;
    if (o >= 0 && kb < src_kb)
      v = transposed ? src[(static_cast<size_t>(e) * src_kb + kb) * src_rb + o / 128]
                     : src[(static_cast<size_t>(e) * src_rb + o / 128) * src_kb + kb];
    dst[static_cast<size_t>(e) * NT * KB * 8 + i] = v;
  }
}

// FP4 scales into the tensor-memory staging image (see the file comment).
__global__ void prep_scale_fp4_kernel(bool is_w13, bool transposed, const uint8_t* __restrict__ src,
                                      uint32_t* __restrict__ dst, int NT, int KB, int src_cols, int I, int H) {
  const int e = blockIdx.y;
  const int total = NT * KB * 256;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int w = i % 256;
    const int kb = (i / 256) % KB;
    const int nt = i / (256 * KB);
    const int half = w / 128, wi = w % 128;
    const int rr = 32 * (wi % 4) + wi / 4;  // inverse of word(r) = 4 (r % 32) + r / 32
    const int p = nt * 256 + half * 128 + rr;
    const int o = orig_row(is_w13, p, I, H);
    uint32_t word = 0;
    for (int j = 0; j < 4; ++j) {
      const int c = kb * 4 + j;
      uint32_t b = 127;
      if (o >= 0 && c < src_cols) {
        const int src_rows = is_w13 ? 2 * I : H;
        b = transposed ? src[(static_cast<size_t>(e) * src_cols + c) * src_rows + o]
                       : src[(static_cast<size_t>(e) * src_rows + o) * src_cols + c];
      }
      word |= b << (8 * j);
    }
    dst[static_cast<size_t>(e) * total + i] = word;
  }
}

// Codes from transposed storage: src[e][k][n] (FP8 bytes; FP4 two codes per
// byte along n, low nibble = even n). One CTA transposes a tile of 32
// prepared rows x one 128-K block through shared memory. The 32 prepared
// rows of a tile come from 32 consecutive original rows (the interleave
// moves 64-row groups) that are either all real or all zero rows, because
// I and H are multiples of 64.
constexpr int kTRows = 32;
__global__ void __launch_bounds__(256)
prep_codes_t_kernel(bool is_w13, bool fp4, const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int Np,
                    int K, int N, int dst_row_bytes, int I, int H) {
  __shared__ __align__(16) uint8_t tile[kBlockK][kTRows];  // [k][row] codes, one byte each
  const int p0 = blockIdx.x * kTRows, kb = blockIdx.y, e = blockIdx.z;
  const int o0 = orig_row(is_w13, p0, I, H);
  const int k0 = kb * kBlockK;
  const int t = threadIdx.x;
  if (!fp4) {
    // 128 k rows x 32 bytes: two 16-byte loads per k row
    const int k = t / 2, half = t % 2;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (o0 >= 0 && k0 + k < K)
      v = *reinterpret_cast<const uint4*>(src + (static_cast<size_t>(e) * K + k0 + k) * N + o0 + 16 * half);
    *reinterpret_cast<uint4*>(&tile[k][16 * half]) = v;
  } else if (t < kBlockK) {
    // 128 k rows x 16 bytes (32 codes): unpack the nibbles
    const int k = t;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (o0 >= 0 && k0 + k < K)
      v = *reinterpret_cast<const uint4*>(src + (static_cast<size_t>(e) * K + k0 + k) * (N / 2) + o0 / 2);
    const uint8_t* b = reinterpret_cast<const uint8_t*>(&v);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      tile[k][2 * i] = b[i] & 0xF;
      tile[k][2 * i + 1] = b[i] >> 4;
    }
  }
  __syncthreads();
  // Write 32 prepared rows x this K block: FP8 128 bytes per row (8 threads x
  // 16 bytes), FP4 64 bytes per row (8 threads x 8 bytes, two codes per byte
  // along k, low nibble = even k).
  const int r = t / 8, c = t % 8;
  uint8_t* d = dst + (static_cast<size_t>(e) * Np + p0 + r) * dst_row_bytes;
  if (!fp4) {
    uint8_t out[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = tile[16 * c + i][r];
    *reinterpret_cast<uint4*>(d + k0 + 16 * c) = *reinterpret_cast<uint4*>(out);
  } else {
    uint8_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = tile[16 * c + 2 * i][r] | (tile[16 * c + 2 * i + 1][r] << 4);
    *reinterpret_cast<uint2*>(d + k0 / 2 + 8 * c) = *reinterpret_cast<uint2*>(out);
  }
}

cudaError_t prep_one(int fmt, bool is_w13, bool transposed, int E, int H, int I, const void* w, const void* ws,
                     uint8_t* out, cudaStream_t st) {
  const GemmGeom g = is_w13 ? geom_w13(H, I) : geom_w2(H, I);
  const PrepLayout L = prep_layout(fmt, E, g);
  const bool fp4 = (fmt != MOE_W_FP8);  // MOE_W_FP4 and MOE_W_FP4_ACT_FP4 share the weights
  const int src_rows = is_w13 ? 2 * I : H;  // N of the original weight
  const int src_k = is_w13 ? H : I;
  const int dst_row_bytes = fp4 ? g.Kp / 2 : g.Kp;
  // The alignment gaps are zeroed too: the prepared bytes are a function of
  // the weights alone.
  cudaError_t err = cudaMemsetAsync(out + L.codes_off + L.codes_bytes, 0, L.scale_off - L.codes_bytes, st);
  if (err == cudaSuccess)
    err = cudaMemsetAsync(out + L.scale_off + L.scale_bytes, 0, L.total - (L.scale_off + L.scale_bytes), st);
  if (err != cudaSuccess) return err;
  if (transposed) {
    prep_codes_t_kernel<<<dim3(g.Np / kTRows, g.KB, E), 256, 0, st>>>(
        is_w13, fp4, static_cast<const uint8_t*>(w), out + L.codes_off, g.Np, src_k, src_rows, dst_row_bytes, I, H);
  } else {
    const int src_row_bytes = fp4 ? src_k / 2 : src_k;
    prep_codes_kernel<<<dim3(g.Np, E), 128, 0, st>>>(is_w13, static_cast<const uint8_t*>(w), out + L.codes_off,
                                                     g.Np, src_row_bytes, dst_row_bytes, src_rows, I, H);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (!fp4) {
    prep_scale_fp8_kernel<<<dim3(64, E), 256, 0, st>>>(is_w13, transposed, static_cast<const float*>(ws),
                                                       reinterpret_cast<float*>(out + L.scale_off), g.Np, g.KB,
                                                       ceil_div(src_rows, 128), ceil_div(src_k, 128), I, H);
  } else {
    prep_scale_fp4_kernel<<<dim3(64, E), 256, 0, st>>>(is_w13, transposed, static_cast<const uint8_t*>(ws),
                                                       reinterpret_cast<uint32_t*>(out + L.scale_off), g.NT, g.KB,
                                                       src_k / 32, I, H);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare(int fmt, bool transposed, int E, int H, int I, const void* w13, const void* w13s,
                           const void* w2, const void* w2s, uint8_t* p13, uint8_t* p2, cudaStream_t st) {
  cudaError_t e = prep_one(fmt, true, transposed, E, H, I, w13, w13s, p13, st);
  if (e != cudaSuccess) return e;
  return prep_one(fmt, false, transposed, E, H, I, w2, w2s, p2, st);
}

}  // namespace bsmoe

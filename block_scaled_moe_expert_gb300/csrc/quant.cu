// Dynamic 1x128 activation quantization fused with the padded permute.
//
// The grouped experts dispatch quantizes activations dynamically per block
// (error page "grouped_mm experts dispatch does not support
// activation_scheme='static'", section "What it means"); rows are then
// gathered by slot // K into the grouped layout (fp8_grouped_mm_experts_forward,
// the source excerpt on the same page). Each token is quantized once and its bytes are
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
#include "ptx.cuh"

namespace bsmoe {

namespace {

constexpr int kQuantWarps = 8;

constexpr int kMaxRowBytes = 32768;  // the largest hidden size the library accepts

// Shared -> global bulk copy (both addresses 16-byte aligned, size a
// multiple of 16), tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_store_commit_and_wait() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// Quantizes one token row and copies its bytes to the n padded rows listed
// in `rows`. A warp covers 256 columns (two 128-column blocks) per step: each
// lane loads 8 bf16 (16 bytes) and the 16 lanes of a half-warp reduce the
// block's amax. The loads of kLoadBatch steps are issued together, so a row
// (up to 8 x 256 x kLoadBatch columns) costs one memory latency instead of
// one per step. The codes and exponent words are assembled in shared memory
// (`qrow`, `qsf`) and each destination row is written by one bulk copy:
// writing them with per-lane stores, eight rows of a token took 3-4 µs of
// store issue alone.
constexpr int kLoadBatch = 4;
__device__ __forceinline__ void quantize_token(const __nv_bfloat16* __restrict__ xr, int H, int Kp,
                                               const int* rows, int n, uint8_t* __restrict__ xq,
                                               uint32_t* __restrict__ xsf, uint8_t* qrow, uint32_t* qsf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = Kp / 128;
  constexpr int kStep = kQuantWarps * 256;
  for (int base = warp * 256; base < Kp; base += kStep * kLoadBatch) {
    uint4 raw[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int c0 = base + u * kStep + lane * 8;
      // H % 64 == 0: a lane's 8 columns are all in or all out
      raw[u] = (c0 < H) ? __ldg(reinterpret_cast<const uint4*>(xr + c0)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int c0w = base + u * kStep;
      if (c0w >= Kp) break;
      const int c0 = c0w + lane * 8;
      float v[8];
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __low2float(p2[i]);
        v[2 * i + 1] = __high2float(p2[i]);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int e = act_exponent(amax);
      const float s = exp2_neg(e);
      if (c0 < Kp) {
        *reinterpret_cast<uint2*>(qrow + c0) = make_uint2(pack4_e4m3(v[0] * s, v[1] * s, v[2] * s, v[3] * s),
                                                          pack4_e4m3(v[4] * s, v[5] * s, v[6] * s, v[7] * s));
        if ((lane & 15) == 0) qsf[c0 / 128] = static_cast<uint32_t>(e + 127) * 0x01010101u;
      }
    }
  }
  fence_proxy_async_smem();  // the bulk copies read qrow through the async proxy
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < n; ++i) bulk_store(xq + static_cast<size_t>(rows[i]) * Kp, qrow, Kp);
  }
  // exponent words: scattered in the MMA scale layout, plain stores
  for (int j = threadIdx.x; j < n * nblk; j += blockDim.x) {
    const int i = j / nblk, b = j - i * nblk;
    xsf[sf_word_index(rows[i], b, nblk)] = qsf[b];
  }
  // the copies read shared memory until they complete
  if (threadIdx.x == 0) bulk_store_commit_and_wait();
}

// Per-token setup of the top-k combine fused into GEMM2's epilogue. The number of valid slots, zeroed arrival counters, and the +0
// output row of a token whose slots are all skipped (no GEMM2 tile reaches it).
__device__ __forceinline__ void setup_combine(int t, int n, int32_t* __restrict__ cnt, int stride,
                                              __nv_bfloat16* __restrict__ out, int H) {
  int32_t* c = cnt + static_cast<size_t>(t) * stride;
  for (int i = threadIdx.x; i < stride; i += blockDim.x) c[i] = (i == 0) ? n : 0;
  if (n == 0) {
    uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
  }
}

// One CTA per token: gathers the token's valid slots from inv (in ascending
// k) and quantizes the row into each of their padded rows.
__global__ void __launch_bounds__(kQuantWarps * 32)
quant_permute_kernel(const __nv_bfloat16* __restrict__ hidden, int H, int K, int Kp,
                     const int32_t* __restrict__ inv, uint8_t* __restrict__ xq, uint32_t* __restrict__ xsf) {
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
      if (r >= 0) rows[n++] = r;
    }
    nrows = n;
  }
  __syncthreads();
  if (nrows == 0) return;
  quantize_token(hidden + static_cast<size_t>(t) * H, H, Kp, rows, nrows, xq, xsf, qrow, qsf);
}

// ---------------------------------------------------------------------------
// Small batches (T * K <= kFusedRouteQuantSlots): routing and quantization in
// one launch. Every CTA (one per token) reads all S expert ids and computes
// the complete routing in shared memory: the per-expert counts, their
// exclusive scans (offsets, padded group starts, m-tile offsets) and each
// slot's stable rank (the number of earlier slots with the same key), which
// gives exactly the counting sort of the routing kernel. CTA 0 writes the
// routing arrays; every CTA quantizes its own token into its rows.

constexpr int kScanPer = 4;  // entries per thread in the (E + 1)-entry scans: 256 x 4 >= kMaxExperts + 1

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__global__ void __launch_bounds__(kQuantWarps * 32)
route_quant_small_kernel(const int32_t* __restrict__ idx, const __nv_bfloat16* __restrict__ hidden, int S, int E,
                         int K, int H, int Kp, int M, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ padded_offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                         int32_t* __restrict__ row_slot, int32_t* __restrict__ tiles, uint32_t* __restrict__ status,
                         uint8_t* __restrict__ xq, uint32_t* __restrict__ xsf, int32_t* __restrict__ comb_cnt,
                         int comb_stride, __nv_bfloat16* __restrict__ out) {
  constexpr int kThreads = kQuantWarps * 32;
  __shared__ int key[kFusedRouteQuantSlots];
  __shared__ int rank[kFusedRouteQuantSlots];
  __shared__ int cnt[kMaxExperts + 1];
  __shared__ int off[kMaxExperts + 1];
  __shared__ int pad[kMaxExperts + 1];
  __shared__ int mts[kMaxExperts + 1];
  __shared__ int chs[kMaxExperts + 1];
  __shared__ int wsum[4][kQuantWarps];
  __shared__ int rows[kMaxTopK];
  __shared__ int nrows;
  __shared__ int bad;
  __shared__ __align__(128) uint8_t qrow[kMaxRowBytes];
  __shared__ uint32_t qsf[kMaxRowBytes / 128];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, t = blockIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) bad = 0;
  for (int e = tid; e <= E; e += kThreads) cnt[e] = 0;
  __syncthreads();
  for (int s = tid; s < S; s += kThreads) {
    const int v = __ldg(idx + s);
    const int k = (v >= 0 && v < E) ? v : E;
    if (v != -1 && k == E) bad = 1;
    key[s] = k;
    atomicAdd(&cnt[k], 1);
  }
  __syncthreads();

  // Exclusive scans over the E + 1 keys of: counts, counts padded to the
  // group alignment, 128-row m-tiles, 32-row chunks. Thread i owns entries
  // [kScanPer i, kScanPer i + kScanPer).
  {
    int v[kScanPer][4], a[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int e = tid * kScanPer + j;
      const int c = (e < E) ? cnt[e] : 0;  // the skipped key E takes no rows
      v[j][0] = c;
      v[j][1] = (c + kRowAlign - 1) / kRowAlign * kRowAlign;
      v[j][2] = (c + kBlockM - 1) / kBlockM;
      v[j][3] = (c + kChunkRows - 1) / kChunkRows;
#pragma unroll
      for (int q = 0; q < 4; ++q) a[q] += v[j][q];
    }
    int inc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      inc[q] = warp_incl_scan(a[q]);
      if (lane == 31) wsum[q][warp] = inc[q];
    }
    __syncthreads();
    int base[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int b = 0;
      for (int w = 0; w < warp; ++w) b += wsum[q][w];
      base[q] = b + inc[q] - a[q];
    }
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int e = tid * kScanPer + j;
      if (e <= E) {
        off[e] = base[0];
        pad[e] = base[1];
        mts[e] = base[2];
        chs[e] = base[3];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) base[q] += v[j][q];
    }
  }
  // Stable rank of every slot among the slots with the same key.
  for (int s = warp; s < S; s += kQuantWarps) {
    const int k = key[s];
    int c = 0;
    for (int j = lane; j < s; j += 32) c += (key[j] == k);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) rank[s] = c;
  }
  __syncthreads();

  if (t == 0) {
    if (tid == 0) {
      *status = bad ? MOE_DEV_BAD_EXPERT_ID : 0u;
      offsets[E] = off[E];
      padded_offsets[E] = pad[E];
      tiles[0] = mts[E];
      tiles[1] = chs[E];
      tiles[kTilesHdr + E] = mts[E];
      tiles[tiles_chunk_off(E) + E] = chs[E];
    }
    for (int e = tid; e < E; e += kThreads) {
      counts[e] = cnt[e];
      offsets[e] = off[e];
      padded_offsets[e] = pad[e];
      tiles[kTilesHdr + e] = mts[e];
      tiles[tiles_chunk_off(E) + e] = chs[e];
    }
    for (int s = tid; s < S; s += kThreads) {
      const int k = key[s];
      perm[off[k] + rank[s]] = s;  // skipped slots: key E, after every group
      if (k < E) {
        const int row = pad[k] + rank[s];
        inv[s] = row;
        row_slot[row] = s;
      } else {
        inv[s] = -1;
      }
    }
    // Work lists and padding rows, one warp per touched expert (at most 256
    // slots, so few experts have any), its lanes writing consecutive entries.
    int32_t* expert_of = tiles + tiles_expert_of(E);
    int32_t* chunk_expert = tiles + tiles_chunk_expert(E, M);
    for (int e = warp; e < E; e += kQuantWarps) {
      const int c = cnt[e];
      if (c == 0) continue;
      for (int g = mts[e] + lane; g < mts[e + 1]; g += 32) expert_of[g] = e;
      for (int g = chs[e] + lane; g < chs[e + 1]; g += 32) chunk_expert[g] = e;
      for (int r = pad[e] + c + lane; r < pad[e + 1]; r += 32) row_slot[r] = -1;  // padding rows
    }
  }

  if (tid == 0) {
    int n = 0;
    for (int k = 0; k < K; ++k) {
      const int s = t * K + k;
      if (key[s] < E) rows[n++] = pad[key[s]] + rank[s];
    }
    nrows = n;
  }
  __syncthreads();
  if (comb_cnt != nullptr) setup_combine(t, nrows, comb_cnt, comb_stride, out, H);
  if (nrows == 0) return;
  quantize_token(hidden + static_cast<size_t>(t) * H, H, Kp, rows, nrows, xq, xsf, qrow, qsf);
}

}  // namespace

cudaError_t launch_quant(const void* hidden, int T, int H, int K, const WsLayout& L, uint8_t* ws, cudaStream_t st) {
  const moe_workspace_layout& p = L.pub;
  return launch_kernel(true, quant_permute_kernel, T, kQuantWarps * 32, 0, st,
                       reinterpret_cast<const __nv_bfloat16*>(hidden), H, K, p.xq_cols,
                       reinterpret_cast<const int32_t*>(ws + p.inv), ws + p.xq, reinterpret_cast<uint32_t*>(ws + p.xsf));
}

cudaError_t launch_route_quant_small(const int32_t* topk_idx, const void* hidden, int T, int H, int E, int K,
                                     const WsLayout& L, uint8_t* ws, void* out, cudaStream_t st) {
  const moe_workspace_layout& p = L.pub;
  // The first kernel of the forward is an ordinary launch: it follows
  // whatever the caller queued on the stream.
  return launch_kernel(false, route_quant_small_kernel, T, kQuantWarps * 32, 0, st, topk_idx,
                       reinterpret_cast<const __nv_bfloat16*>(hidden), T * K, E, K, H, p.xq_cols, L.M,
                       reinterpret_cast<int32_t*>(ws + p.counts), reinterpret_cast<int32_t*>(ws + p.offsets),
                       reinterpret_cast<int32_t*>(ws + p.padded_offsets), reinterpret_cast<int32_t*>(ws + p.perm),
                       reinterpret_cast<int32_t*>(ws + p.inv), reinterpret_cast<int32_t*>(ws + p.row_slot),
                       reinterpret_cast<int32_t*>(ws + p.tiles), reinterpret_cast<uint32_t*>(ws + p.status),
                       ws + p.xq, reinterpret_cast<uint32_t*>(ws + p.xsf),
                       L.combine_cnt ? reinterpret_cast<int32_t*>(ws + L.combine_cnt) : nullptr, L.combine_stride,
                       reinterpret_cast<__nv_bfloat16*>(out));
}

}  // namespace bsmoe

// Routing + dynamic 1x128 activation quantization of a small batch in one
// kernel, as device code of the single-launch decode forward (T * K <= 32;
// sized for kFusedCombineSlots), and the per-token quantization shared with
// the separate quantization kernel.
//
// Routing follows fp8_grouped_mm_experts_forward (source excerpt on the error
// page "grouped_mm experts dispatch does not support
// activation_scheme='static'"): flatten the slots s = t*K + k, sort them by
// expert id (stable: equal ids keep ascending slot order; a skipped slot, -1
// or an id outside [-1, E) which also raises MOE_DEV_BAD_EXPERT_ID, takes key
// E and sorts after every group), place the groups in the padded grouped
// layout (sorted_to_padded of the deepgemm_fp8_fp4_experts_forward excerpt).
// Every CTA computes the whole routing of the small batch in shared memory;
// CTA 0 writes the routing arrays; each CTA quantizes its own tokens.
//
// Quantization ("quantizes activations dynamically per block", section "What
// it means" of the same error page), per 128-wide block of a row (last block
// partial when H % 128 != 0):
//   e = min{n : amax <= 448 * 2^n} (0 if amax == 0, clamped to [-127, 127]),
//   q = e4m3(x * 2^-e), round to nearest even with saturation.
// x * 2^-e is exact (power-of-two scaling of a bf16 value), so the byte only
// depends on the hardware conversion's rounding. Columns [H, Kp) of every
// written row are zero so that K padding contributes nothing. A token is
// quantized once and its bytes are copied to the padded row of every valid
// slot of that token, which equals quantizing the gathered rows.
#pragma once
#include <cuda_bf16.h>

#include "act_quant.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace bsmoe {

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
// Only until the copies have read their shared-memory source; the global
// writes finish on their own and are complete when the grid is.
__device__ __forceinline__ void bulk_store_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Quantizes one token row and copies its bytes to the n padded rows listed
// in `rows`, with all kNW warps of the CTA. A warp covers 256 columns (two
// 128-column blocks) per step: each lane loads 8 bf16 (16 bytes) and the 16
// lanes of a half-warp reduce the block's amax. The loads of kLoadBatch
// steps are issued together, so a row costs one memory latency instead of
// one per step. The codes and exponent words are assembled in shared memory
// (`qrow`, `qsf`) and each destination row is written by one bulk copy:
// writing them with per-lane stores, eight rows of a token took 3-4 µs of
// store issue alone.
constexpr int kLoadBatch = 4;
// kComplete: wait for the rows' global writes to complete (they are read in
// the same grid after a grid-wide barrier); otherwise only until the copies
// have read shared memory (a later kernel reads the rows).
// kFp4: the FP4-activation variant's rule instead (1x32 blocks of four lanes,
// n = min{n : amax <= 6 * 2^n}, e2m1 codes two per byte, so a row is Kp / 2
// bytes; byte j of a block's scale word is the exponent of its 1x32
// sub-block j).
template <int kNW, bool kComplete, bool kFp4 = false>
__device__ __forceinline__ void quantize_token(const __nv_bfloat16* __restrict__ xr, int H, int Kp,
                                               const int* rows, int n, uint8_t* __restrict__ xq,
                                               uint32_t* __restrict__ xsf, uint8_t* qrow, uint32_t* qsf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = Kp / 128;
  const int row_bytes = kFp4 ? Kp / 2 : Kp;
  constexpr int kStep = kNW * 256;
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
      if constexpr (kFp4) {
#pragma unroll
        for (int o = 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int e = act_exponent_e2m1(amax);
        const float s = exp2_neg(e);
        if (c0 < Kp) {
          *reinterpret_cast<uint32_t*>(qrow + c0 / 2) =
              pack8_e2m1(v[0] * s, v[1] * s, v[2] * s, v[3] * s, v[4] * s, v[5] * s, v[6] * s, v[7] * s);
          if ((lane & 3) == 0) reinterpret_cast<uint8_t*>(qsf)[c0 / 32] = static_cast<uint8_t>(e + 127);
        }
      } else {
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
  }
  fence_proxy_async_smem();  // the bulk copies read qrow through the async proxy
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < n; ++i) bulk_store(xq + static_cast<size_t>(rows[i]) * row_bytes, qrow, row_bytes);
  }
  // exponent words: scattered in the MMA scale layout, plain stores
  for (int j = threadIdx.x; j < n * nblk; j += blockDim.x) {
    const int i = j / nblk, b = j - i * nblk;
    xsf[sf_word_index(rows[i], b, nblk)] = qsf[b];
  }
  // the copies read shared memory until then
  if (threadIdx.x == 0) {
    if constexpr (kComplete) {
      bulk_store_commit_and_wait();
    } else {
      bulk_store_commit_and_wait_read();
    }
  }
  __syncthreads();
}

// Per-token setup of the top-k combine fused into GEMM2's epilogue: the
// number of valid slots, zeroed arrival counters, and the +0 output row of a
// token whose slots are all skipped (no GEMM2 tile reaches it).
__device__ __forceinline__ void setup_combine(int t, int n, int32_t* __restrict__ cnt, int stride,
                                              __nv_bfloat16* __restrict__ out, int H) {
  int32_t* c = cnt + static_cast<size_t>(t) * stride;
  for (int i = threadIdx.x; i < stride; i += blockDim.x) c[i] = (i == 0) ? n : 0;
  if (n == 0) {
    uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Arguments of the small-batch routing + quantization.
struct RqArgs {
  const int32_t* idx;          // [T, K] expert ids
  const __nv_bfloat16* hidden; // [T, H]
  const float* topk_w;         // [T, K] routing weights
  float* row_w;                // [M] routing weight per padded row (written for valid rows)
  int T, S, E, K, H, Kp, M;
  int32_t* counts;
  int32_t* offsets;
  int32_t* padded_offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* row_slot;
  int32_t* tiles;
  uint32_t* status;
  uint8_t* xq;
  uint32_t* xsf;
  int32_t* comb_cnt;           // null: no fused combine
  int comb_stride;
  __nv_bfloat16* out;
  int32_t* ready;              // single-launch forward: per 32-row chunk, GEMM1 units done (zeroed here)
  int ready_n;
};

// Shared memory of the small-batch routing + quantization.
template <int kNW>
struct RqSmem {
  int key[kFusedCombineSlots];
  int rank[kFusedCombineSlots];
  int cnt[kMaxExperts + 1];
  int off[kMaxExperts + 1];
  int pad[kMaxExperts + 1];
  int mts[kMaxExperts + 1];
  int chs[kMaxExperts + 1];
  int wsum[4][kNW];
  int rows[kMaxTopK];
  int nrows;
  int bad;
  alignas(128) uint8_t qrow[kMaxRowBytes];
  uint32_t qsf[kMaxRowBytes / 128];
};

// The routing of all S slots computed in this CTA's shared memory: counts,
// the exclusive scans (offsets, padded group starts, m-tile and chunk
// offsets) and each slot's stable rank among the slots with the same key,
// which is exactly the counting sort of the routing kernel. Every thread of
// the CTA takes part.
template <int kNW>
__device__ __forceinline__ void route_small_in_smem(RqSmem<kNW>& sm, const RqArgs& a) {
  constexpr int kThreads = kNW * 32;
  constexpr int kScanPer = (kMaxExperts + 1 + kThreads - 1) / kThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, S = a.S;
  if (tid == 0) sm.bad = 0;
  for (int e = tid; e <= E; e += kThreads) sm.cnt[e] = 0;
  __syncthreads();
  for (int s = tid; s < S; s += kThreads) {
    const int v = __ldg(a.idx + s);
    const int k = (v >= 0 && v < E) ? v : E;
    if (v != -1 && k == E) sm.bad = 1;
    sm.key[s] = k;
    atomicAdd(&sm.cnt[k], 1);
  }
  __syncthreads();

  // Exclusive scans over the E + 1 keys of: counts, counts padded to the
  // group alignment, 128-row m-tiles, 32-row chunks. Thread i owns entries
  // [kScanPer i, kScanPer i + kScanPer).
  {
    int v[kScanPer][4], acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int e = tid * kScanPer + j;
      const int c = (e < E) ? sm.cnt[e] : 0;  // the skipped key E takes no rows
      v[j][0] = c;
      v[j][1] = (c + kRowAlign - 1) / kRowAlign * kRowAlign;
      v[j][2] = (c + kBlockM - 1) / kBlockM;
      v[j][3] = (c + kChunkRows - 1) / kChunkRows;
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] += v[j][q];
    }
    int inc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      inc[q] = warp_incl_scan(acc[q]);
      if (lane == 31) sm.wsum[q][warp] = inc[q];
    }
    __syncthreads();
    int base[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int b = 0;
      for (int w = 0; w < warp; ++w) b += sm.wsum[q][w];
      base[q] = b + inc[q] - acc[q];
    }
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int e = tid * kScanPer + j;
      if (e <= E) {
        sm.off[e] = base[0];
        sm.pad[e] = base[1];
        sm.mts[e] = base[2];
        sm.chs[e] = base[3];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) base[q] += v[j][q];
    }
  }
  // Stable rank of every slot among the slots with the same key.
  for (int s = warp; s < S; s += kNW) {
    const int k = sm.key[s];
    int c = 0;
    for (int j = lane; j < s; j += 32) c += (sm.key[j] == k);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) sm.rank[s] = c;
  }
  __syncthreads();
}

// CTA 0's part: the routing arrays, work lists and padding rows in global
// memory (and, for the single-launch forward, the zeroed chunk counters).
template <int kNW>
__device__ __forceinline__ void write_routing(RqSmem<kNW>& sm, const RqArgs& a) {
  constexpr int kThreads = kNW * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, S = a.S;
  if (tid == 0) {
    *a.status = sm.bad ? MOE_DEV_BAD_EXPERT_ID : 0u;
    a.offsets[E] = sm.off[E];
    a.padded_offsets[E] = sm.pad[E];
    a.tiles[0] = sm.mts[E];
    a.tiles[1] = sm.chs[E];
    a.tiles[kTilesHdr + E] = sm.mts[E];
    a.tiles[tiles_chunk_off(E) + E] = sm.chs[E];
  }
  for (int e = tid; e < E; e += kThreads) {
    a.counts[e] = sm.cnt[e];
    a.offsets[e] = sm.off[e];
    a.padded_offsets[e] = sm.pad[e];
    a.tiles[kTilesHdr + e] = sm.mts[e];
    a.tiles[tiles_chunk_off(E) + e] = sm.chs[e];
  }
  for (int s = tid; s < S; s += kThreads) {
    const int k = sm.key[s];
    a.perm[sm.off[k] + sm.rank[s]] = s;  // skipped slots: key E, after every group
    if (k < E) {
      const int row = sm.pad[k] + sm.rank[s];
      a.inv[s] = row;
      a.row_slot[row] = s;
    } else {
      a.inv[s] = -1;
    }
  }
  // Work lists and padding rows, one warp per touched expert (at most 256
  // slots, so few experts have any), its lanes writing consecutive entries.
  int32_t* expert_of = a.tiles + tiles_expert_of(E);
  int32_t* chunk_expert = a.tiles + tiles_chunk_expert(E, a.M);
  for (int e = warp; e < E; e += kNW) {
    const int c = sm.cnt[e];
    if (c == 0) continue;
    for (int g = sm.mts[e] + lane; g < sm.mts[e + 1]; g += 32) expert_of[g] = e;
    for (int g = sm.chs[e] + lane; g < sm.chs[e + 1]; g += 32) chunk_expert[g] = e;
    for (int r = sm.pad[e] + c + lane; r < sm.pad[e + 1]; r += 32) a.row_slot[r] = -1;  // padding rows
  }
  if (a.ready != nullptr)
    for (int i = tid; i < a.ready_n; i += kThreads) a.ready[i] = 0;
}

// Tokens t0, t0 + stride, ... : the valid slots' padded rows (ascending k),
// the fused-combine setup, and the quantization into those rows (kFp4: the
// e2m1 1x32 rule of the FP4-activation variant).
template <int kNW, bool kComplete, bool kFp4>
__device__ __forceinline__ void quantize_tokens(RqSmem<kNW>& sm, const RqArgs& a, int t0, int stride) {
  for (int t = t0; t < a.T; t += stride) {
    if (threadIdx.x == 0) {
      int n = 0;
      for (int k = 0; k < a.K; ++k) {
        const int s = t * a.K + k;
        if (sm.key[s] < a.E) {
          const int r = sm.pad[sm.key[s]] + sm.rank[s];
          sm.rows[n++] = r;
          a.row_w[r] = __ldg(a.topk_w + s);
        }
      }
      sm.nrows = n;
    }
    __syncthreads();
    const int n = sm.nrows;
    if (a.comb_cnt != nullptr) setup_combine(t, n, a.comb_cnt, a.comb_stride, a.out, a.H);
    if (n > 0)
      quantize_token<kNW, kComplete, kFp4>(a.hidden + static_cast<size_t>(t) * a.H, a.H, a.Kp, sm.rows, n, a.xq, a.xsf,
                                           sm.qrow, sm.qsf);
    __syncthreads();  // rows / nrows are rewritten for the next token
  }
}

// Host: the arguments for a forward on workspace `ws` with layout L.
RqArgs make_rq_args(const int32_t* topk_idx, const void* hidden, const float* topk_w, int T, int H, int E, int K,
                    const WsLayout& L, uint8_t* ws, void* out);

}  // namespace bsmoe

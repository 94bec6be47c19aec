// Routing: flatten the top-k pairs, count them per expert and place them in a
// padded grouped layout with a stable counting sort.
//
// Follows fp8_grouped_mm_experts_forward (source excerpt on the error page
// "grouped_mm experts dispatch does not support activation_scheme='static'"):
// flatten (slot s = t*K + k), sort by expert id, gather rows by s // K; and
// the sorted_to_padded map of the deepgemm_fp8_fp4_experts_forward source
// excerpt (error record "DeepGEMM experts selected on a model spanning
// multiple CUDA devices"). The sort
// is stable (equal ids keep ascending slot order) and a skipped slot (-1, or
// an id outside [-1, E), which also raises MOE_DEV_BAD_EXPERT_ID) takes key E
// so it sorts after every group.
//
// Up to 8192 slots: one CTA of 32 warps. Warp w owns a contiguous range of slots and walks it
// 32 slots at a time; __match_any_sync groups equal keys inside a step, so a
// slot's rank is (#equal keys in earlier warps) + (#equal keys earlier in its
// own warp), which is exactly the stable order. No data atomics are used:
// the result is deterministic.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace bsmoe {

namespace {

constexpr int kWarps = 32;
constexpr int kThreads = kWarps * 32;
constexpr int kSingleCtaSlots = 8192;  // up to this many slots one CTA routes everything

__device__ __forceinline__ int slot_key(const int32_t* idx, int s, int E, uint32_t* status) {
  int v = __ldg(idx + s);
  if (v >= 0 && v < E) return v;
  if (v != -1 && status != nullptr) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
  return E;
}

// expert_of[g] = e for every m-tile g of expert e (m-tile offsets in s_mt,
// E + 1 entries): lets the GEMMs find a tile's expert with one load.
__device__ __forceinline__ void write_expert_of(int E, const int* s_mt, int32_t* expert_of) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int e = warp; e < E; e += nwarps)
    for (int g = s_mt[e] + lane; g < s_mt[e + 1]; g += 32) expert_of[g] = e;
}

// Block-wide exclusive scan of one int per thread (1024 threads).
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int ws = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    warp_sums[lane] = ws - w;  // exclusive
    if (lane == 31) *total = ws;
  }
  __syncthreads();
  int r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

// From the slot count c_e of expert tid (tid < E, 0 otherwise; 1024
// threads): the exclusive scans of the counts, of the counts padded to the
// group alignment, of the 128-row m-tiles and of the 32-row chunks; writes
// counts, offsets, padded_offsets and the GEMM work lists of the tiles
// region, and leaves the offsets and group starts in s_off / s_pad.
__device__ void scan_counts_and_tables(int E, int M, int c_e, int32_t* __restrict__ counts,
                                       int32_t* __restrict__ offsets, int32_t* __restrict__ padded_offsets,
                                       int32_t* __restrict__ tiles, int* s_off, int* s_pad, int* s_mt, int* s_ch,
                                       int* warp_sums, int* tot) {
  const int tid = threadIdx.x;
  const int off = block_excl_scan(c_e, warp_sums, &tot[0]);
  const int pad = block_excl_scan((c_e + kRowAlign - 1) / kRowAlign * kRowAlign, warp_sums, &tot[1]);
  const int mts = block_excl_scan((c_e + kBlockM - 1) / kBlockM, warp_sums, &tot[2]);
  const int chs = block_excl_scan((c_e + kChunkRows - 1) / kChunkRows, warp_sums, &tot[3]);
  if (tid < E) {
    counts[tid] = c_e;
    offsets[tid] = off;
    padded_offsets[tid] = pad;
    tiles[kTilesHdr + tid] = mts;
    tiles[tiles_chunk_off(E) + tid] = chs;
    s_off[tid] = off;
    s_pad[tid] = pad;
    s_mt[tid] = mts;
    s_ch[tid] = chs;
  }
  if (tid == 0) {
    offsets[E] = tot[0];
    padded_offsets[E] = tot[1];
    tiles[0] = tot[2];
    tiles[1] = tot[3];
    tiles[kTilesHdr + E] = tot[2];
    tiles[tiles_chunk_off(E) + E] = tot[3];
    s_off[E] = tot[0];
    s_pad[E] = tot[1];
    s_mt[E] = tot[2];
    s_ch[E] = tot[3];
  }
  __syncthreads();
  write_expert_of(E, s_mt, tiles + tiles_expert_of(E));
  write_expert_of(E, s_ch, tiles + tiles_chunk_expert(E, M));
}

__global__ void __launch_bounds__(kThreads, 1)
route_kernel(const int32_t* __restrict__ idx, int S, int E, int M, int32_t* __restrict__ counts,
             int32_t* __restrict__ offsets, int32_t* __restrict__ padded_offsets, int32_t* __restrict__ perm,
             int32_t* __restrict__ inv, int32_t* __restrict__ row_slot, int32_t* __restrict__ tiles,
             uint32_t* __restrict__ status) {
  extern __shared__ int hist[];  // [kWarps][E + 1]
  __shared__ int warp_sums[32];
  __shared__ int tot[4];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pad[kMaxExperts + 1];
  __shared__ int s_mt[kMaxExperts + 1];
  __shared__ int s_ch[kMaxExperts + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int stride = E + 1;
  pdl_wait();
  pdl_launch_dependents();
  // The status word reflects the most recent forward on this workspace.
  if (tid == 0) *status = 0u;
  for (int i = tid; i < kWarps * stride; i += kThreads) hist[i] = 0;
  __syncthreads();

  const int chunk = ((S + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int beg = warp * chunk;
  const int end = min(S, beg + chunk);
  int* h = hist + warp * stride;

  // Pass 1: per-warp histogram.
  for (int base = beg; base < end; base += 32) {
    const int s = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, s < end);
    if (s < end) {
      const int key = slot_key(idx, s, E, status);
      const unsigned peers = __match_any_sync(active, key);
      if (lane == __ffs(peers) - 1) h[key] += __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();

  // Exclusive prefix over warps for each key; totals per key.
  int cnt = 0;
  if (tid <= E) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = hist[w * stride + tid];
      hist[w * stride + tid] = run;
      run += c;
    }
    cnt = run;
  }
  const int c_e = (tid < E) ? cnt : 0;
  scan_counts_and_tables(E, M, c_e, counts, offsets, padded_offsets, tiles, s_off, s_pad, s_mt, s_ch, warp_sums, tot);

  // Pass 2: scatter.
  for (int base = beg; base < end; base += 32) {
    const int s = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, s < end);
    if (s < end) {
      const int key = slot_key(idx, s, E, status);
      const unsigned peers = __match_any_sync(active, key);
      const int leader = __ffs(peers) - 1;
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = h[key] + rank;
      __syncwarp(active);
      if (lane == leader) h[key] += __popc(peers);
      perm[s_off[key] + pos] = s;
      if (key < E) {
        const int row = s_pad[key] + pos;
        inv[s] = row;
        row_slot[row] = s;
      } else {
        inv[s] = -1;
      }
    }
    __syncwarp();
  }

  // Padding rows of every group belong to no slot.
  for (int e = warp; e < E; e += kWarps) {
    const int lo = s_pad[e] + (s_off[e + 1] - s_off[e]);
    const int hi = s_pad[e + 1];
    for (int r = lo + lane; r < hi; r += 32) row_slot[r] = -1;
  }
}

// ---------------------------------------------------------------------------
// Multi-CTA path for large S: the slots are split into chunks of
// kChunk consecutive slots. (1) every chunk counts its keys; (2) one CTA
// turns the per-chunk counts into, for each key, the number of equal keys in
// earlier chunks, and computes the per-expert totals and offsets; (3) every
// chunk places its slots with the same per-warp stable ranking as above.
// The placement is identical to the single-CTA kernel's.

constexpr int kChunk = 1024;
constexpr int kChunkWarps = 8;

__global__ void __launch_bounds__(kChunkWarps * 32)
route_hist_kernel(const int32_t* __restrict__ idx, int S, int E, int32_t* __restrict__ chunk_hist) {
  extern __shared__ int h[];  // [E + 1]
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int beg = blockIdx.x * kChunk, end = min(S, beg + kChunk);
  for (int s = beg + threadIdx.x; s < end; s += blockDim.x) atomicAdd(&h[slot_key(idx, s, E, nullptr)], 1);
  __syncthreads();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) chunk_hist[static_cast<size_t>(blockIdx.x) * (E + 1) + i] = h[i];
}

__global__ void __launch_bounds__(kThreads, 1)
route_scan_kernel(int E, int M, int G, int32_t* __restrict__ chunk_hist, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ padded_offsets,
                  int32_t* __restrict__ row_slot, int32_t* __restrict__ tiles, uint32_t* __restrict__ status) {
  __shared__ int warp_sums[32];
  __shared__ int tot[4];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pad[kMaxExperts + 1];
  __shared__ int s_mt[kMaxExperts + 1];
  __shared__ int s_ch[kMaxExperts + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  // The status word reflects the most recent forward; the scatter kernel
  // raises the invalid-id flag after this.
  if (tid == 0) *status = 0u;
  int cnt = 0;
  if (tid <= E) {  // exclusive prefix over chunks, in place
    // eight chunks' counts are loaded before any of them is overwritten, so
    // the loads of a batch are in flight together
    constexpr int kBatch = 8;
    int run = 0;
    for (int g0 = 0; g0 < G; g0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        v[j] = (g0 + j < G) ? chunk_hist[static_cast<size_t>(g0 + j) * (E + 1) + tid] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (g0 + j < G) {
          chunk_hist[static_cast<size_t>(g0 + j) * (E + 1) + tid] = run;
          run += v[j];
        }
      }
    }
    cnt = run;
  }
  const int c_e = (tid < E) ? cnt : 0;
  scan_counts_and_tables(E, M, c_e, counts, offsets, padded_offsets, tiles, s_off, s_pad, s_mt, s_ch, warp_sums, tot);
  for (int e = warp; e < E; e += kWarps) {
    const int lo = s_pad[e] + (s_off[e + 1] - s_off[e]);
    const int hi = s_pad[e + 1];
    for (int r = lo + lane; r < hi; r += 32) row_slot[r] = -1;
  }
}

__global__ void __launch_bounds__(kChunkWarps * 32)
route_scatter_kernel(const int32_t* __restrict__ idx, int S, int E, const int32_t* __restrict__ chunk_base,
                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ padded_offsets,
                     int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* __restrict__ row_slot,
                     uint32_t* __restrict__ status) {
  extern __shared__ int smem[];
  const int stride = E + 1;
  int* hist = smem;                       // [kChunkWarps][E + 1]
  int* s_off = smem + kChunkWarps * stride;  // [E + 1]
  int* s_pad = s_off + stride;               // [E + 1]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  for (int i = tid; i < kChunkWarps * stride; i += blockDim.x) hist[i] = 0;
  for (int i = tid; i <= E; i += blockDim.x) {
    s_off[i] = offsets[i];
    s_pad[i] = padded_offsets[i];
  }
  __syncthreads();
  const int cbeg = blockIdx.x * kChunk, cend = min(S, cbeg + kChunk);
  const int per = kChunk / kChunkWarps;
  const int beg = cbeg + warp * per, end = min(cend, beg + per);
  int* h = hist + warp * stride;
  for (int base = beg; base < end; base += 32) {
    const int s = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, s < end);
    if (s < end) {
      const int key = slot_key(idx, s, E, status);
      const unsigned peers = __match_any_sync(active, key);
      if (lane == __ffs(peers) - 1) h[key] += __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();
  // per key: chunk base (equal keys in earlier chunks) + equal keys in earlier warps
  const int32_t* cb = chunk_base + static_cast<size_t>(blockIdx.x) * stride;
  for (int k = tid; k <= E; k += blockDim.x) {
    int run = cb[k];
    for (int w = 0; w < kChunkWarps; ++w) {
      const int c = hist[w * stride + k];
      hist[w * stride + k] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = beg; base < end; base += 32) {
    const int s = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, s < end);
    if (s < end) {
      const int key = slot_key(idx, s, E, nullptr);
      const unsigned peers = __match_any_sync(active, key);
      const int leader = __ffs(peers) - 1;
      const int pos = h[key] + __popc(peers & ((1u << lane) - 1u));
      __syncwarp(active);
      if (lane == leader) h[key] += __popc(peers);
      perm[s_off[key] + pos] = s;
      if (key < E) {
        const int row = s_pad[key] + pos;
        inv[s] = row;
        row_slot[row] = s;
      } else {
        inv[s] = -1;
      }
    }
    __syncwarp();
  }
}

}  // namespace

int route_chunks(int S) { return S <= kSingleCtaSlots ? 0 : (S + kChunk - 1) / kChunk; }

cudaError_t launch_route(const int32_t* topk_idx, int S, int E, const WsLayout& L, uint8_t* ws, cudaStream_t st) {
  const moe_workspace_layout& p = L.pub;
  const int G = route_chunks(S);
  if (G > 0) {
    int32_t* chunk_hist = reinterpret_cast<int32_t*>(ws + L.route_scratch);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + p.status);
    cudaError_t e = launch_kernel(false, route_hist_kernel, G, kChunkWarps * 32, sizeof(int) * (E + 1), st,
                                  topk_idx, S, E, chunk_hist);
    if (e != cudaSuccess) return e;
    e = launch_kernel(true, route_scan_kernel, 1, kThreads, 0, st, E, L.M, G, chunk_hist,
                      reinterpret_cast<int32_t*>(ws + p.counts), reinterpret_cast<int32_t*>(ws + p.offsets),
                      reinterpret_cast<int32_t*>(ws + p.padded_offsets), reinterpret_cast<int32_t*>(ws + p.row_slot),
                      reinterpret_cast<int32_t*>(ws + p.tiles), status);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(int) * (kChunkWarps + 2) * (E + 1);
    return launch_kernel(true, route_scatter_kernel, G, kChunkWarps * 32, smem, st, topk_idx, S, E,
                         static_cast<const int32_t*>(chunk_hist), reinterpret_cast<const int32_t*>(ws + p.offsets),
                         reinterpret_cast<const int32_t*>(ws + p.padded_offsets),
                         reinterpret_cast<int32_t*>(ws + p.perm), reinterpret_cast<int32_t*>(ws + p.inv),
                         reinterpret_cast<int32_t*>(ws + p.row_slot), status);
  }
  const size_t smem = sizeof(int) * kWarps * (E + 1);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // The first kernel of the forward is an ordinary launch: it follows
  // whatever the caller queued on the stream.
  return launch_kernel(false, route_kernel, 1, kThreads, smem, st, topk_idx, S, E, L.M,
                       reinterpret_cast<int32_t*>(ws + p.counts), reinterpret_cast<int32_t*>(ws + p.offsets),
                       reinterpret_cast<int32_t*>(ws + p.padded_offsets), reinterpret_cast<int32_t*>(ws + p.perm),
                       reinterpret_cast<int32_t*>(ws + p.inv), reinterpret_cast<int32_t*>(ws + p.row_slot),
                       reinterpret_cast<int32_t*>(ws + p.tiles), reinterpret_cast<uint32_t*>(ws + p.status));
}

}  // namespace bsmoe

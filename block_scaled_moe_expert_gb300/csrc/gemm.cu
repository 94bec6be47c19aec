// Grouped block-scaled GEMMs of the experts forward on tcgen05 tensor cores.
//
// The error record "DeepGEMM experts selected on a model spanning multiple
// CUDA devices" (source excerpt of deepgemm_fp8_fp4_experts_forward) runs the
// experts as two grouped matmuls with FP8 activations and FP8 or FP4 expert
// weights (grouped_fp8_fp4_matmul_nt: both operands K-major). This kernel computes,
// for every expert e and every 128-row tile of its group in the padded
// grouped layout, one 128 x 256 output tile:
//
//   D[r, n] = sum_k deq(A)[r, k] * deq(W_e)[n, k]
//
// GEMM1 (A = quantized hidden rows, W = interleaved gate_up) ends with the
// SwiGLU epilogue: optional clamp (swiglu_limit, "absent -> unclamped" in the
// Mega MoE docstring), act = silu(gate) * up in fp32, requantization of act
// in 1x128 blocks with the same power-of-two e4m3 rule as the input.
// GEMM2 (A = act, W = down_proj) multiplies each row by the routing weight of
// its slot and stores fp32 rows for the deterministic combine (in the FP4
// decode mode with at most 256 slots it also performs that combine).
//
// Pipeline (one persistent CTA per SM, 12 warps):
//   warp 0      TMA producer: A tile 128x128 B (decode mode: a 32-row chunk),
//               W tile 256x128 B (+ FP4 scale blocks) per 128-K stage into a
//               4-deep (decode mode: 5-deep) shared-memory ring;
//   warp 1      allocates tensor memory and issues tcgen05.mma (one thread;
//               the whole warp in decode mode);
//   warp 2      FP8: producer of the promotion scales; FP4: idle;
//   warp 3      idle;
//   warps 4..11 two epilogue warpgroups, each owning 128 of the 256 columns.
// The first warpgroup hands registers to the epilogue warpgroups with
// setmaxnreg (launch: 384 x 168; after: 128 x 56 + 256 x 224 = 64512).
// FP8 weights carry an fp32 scale per 128x128 block, which the block-scaled
// MMA cannot apply (it takes power-of-two scale bytes), so each 128-K block
// is multiplied without scaling into one of two TMEM partial buffers and the
// epilogue warps promote it into fp32 registers with 2^e_act * s_w.
// FP4 weights use the hardware block-scaled MMA (kind::mxf8f6f4, one UE8M0
// byte per 32 K for both operands); the activation's 1x128 exponent is
// replicated into four bytes, and the scale blocks are copied shared ->
// tensor memory with tcgen05.cp before the stage's MMAs.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "act_quant.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route_quant.cuh"

namespace bsmoe {

namespace {

constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;  // warps 4..11 are the two epilogue warpgroups
constexpr int kEpiThreads = 256;
constexpr uint32_t kTileABytes = kBlockM * kBlockK;  // 16 KB: the 128 activation rows an MMA reads
constexpr uint32_t kTileBBytes = kBlockN * kBlockK;  // 32 KB (FP4 is unpacked to 1 B/elem in smem)
constexpr uint32_t kSfaBytes = 512;
constexpr uint32_t kSfbBytes = 1024;
constexpr int kScaleSlots = 4;          // FP8: slots of the promotion-scale ring
constexpr int kScaleGroup = 4;          // FP8: K blocks per slot
constexpr uint32_t kSwBytes = 32;       // FP8: 8 weight scales (one per 32 columns) per K block
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemCol = 256;  // FP4: per stage 4 SFA + 8 SFB columns from here
// FP4 x FP4 (FP4 activations): a stage spans K = 256 (128 bytes of packed
// codes a row, the SWIZZLE_128B row, like an FP8 stage), i.e. two 128-K
// scale chunks: 8 SFA + 16 SFB TMEM columns per stage.
constexpr int kMx = MOE_W_FP4_ACT_FP4;
template <int FMT>
constexpr uint32_t kSfColsPerStage = FMT == kMx ? 24 : 12;

// Pipeline shape. Tile mode: a work unit is a 128-row token tile; a stage
// holds its 16 KB of activation rows and a 32 KB weight tile (4 stages).
// Decode mode (FP4 weights, few pairs per expert): a work unit is a 32-row
// token chunk and a stage loads only its 4 KB of activation rows into an
// overlapping window: the MMA reads 128 rows from the window start, rows
// 32-127 being whatever follows in shared memory; they only reach output
// rows that are never stored. The 12 KB saved per stage buy a fifth weight
// stage, i.e. 80 KB instead of 64 KB of FP4 weights in flight per SM.
template <bool DEC>
struct Pipe {
  static constexpr int kStages = DEC ? 5 : 4;
  static constexpr int kRows = DEC ? kChunkRows : kBlockM;  // activation rows loaded per stage
  static constexpr uint32_t kAStride = kRows * kBlockK;
  static constexpr uint32_t kARegion = kStages * kAStride + (kTileABytes - kAStride);
};

constexpr uint32_t kYBoxBytes = 32 * 16 * 4;

template <bool DEC, int FMT>
struct __align__(1024) SmemT {
  static constexpr int kSfChunks = FMT == kMx ? 2 : 1;  // 128-K scale chunks a stage
  // slots of the FP8 promotion-scale ring below: unused by the FP4 formats,
  // and shrunk for FP4 activations, whose larger scale stages need the room
  static constexpr int kSlots = FMT == kMx ? 1 : kScaleSlots;
  uint8_t b[Pipe<DEC>::kStages][kTileBBytes];
  uint8_t a[Pipe<DEC>::kARegion];  // stage s at s * kAStride (1024-byte aligned)
  // GEMM2 in tile mode: per epilogue warp, a 32-row x 16-column fp32 box
  // through which its row stores are transposed (tile mode only).
  uint8_t ystage[DEC ? 16 : kEpiThreads / 32 * kYBoxBytes];
  uint8_t sfa[Pipe<DEC>::kStages][kSfChunks * kSfaBytes];
  uint8_t sfb[Pipe<DEC>::kStages][kSfChunks * kSfbBytes];
  uint64_t full[Pipe<DEC>::kStages];
  uint64_t empty[Pipe<DEC>::kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  float amax_x[2][2][kBlockM];
  // FP8 promotion scales, filled by the producer and released by the
  // epilogue (its own ring: the MMA frees the operand stages before the
  // epilogue reads the scales of that K block).
  uint32_t sfa_w[kSlots][kScaleGroup][kBlockM];
  float sw[kSlots][kScaleGroup][8];
  uint64_t sfull[kScaleSlots];
  uint64_t sempty[kScaleSlots];
  uint32_t tmem_base;
  int abort_flag;
  __device__ uint8_t* a_stage(int s) { return a + s * Pipe<DEC>::kAStride; }
};

template <bool DEC, int FMT>
constexpr bool smem_layout_ok() {
  using S = SmemT<DEC, FMT>;
  return offsetof(S, a) % 1024 == 0 && Pipe<DEC>::kAStride % 1024 == 0 && offsetof(S, sfa) % 16 == 0 &&
         offsetof(S, sfb) % 16 == 0 && offsetof(S, sfa_w) % 16 == 0 && offsetof(S, sw) % 16 == 0 &&
         sizeof(S) + 1024 <= 227 * 1024 && kSfTmemCol + Pipe<DEC>::kStages * kSfColsPerStage<FMT> <= kTmemCols;
}
static_assert(smem_layout_ok<false, MOE_W_FP8>() && smem_layout_ok<false, MOE_W_FP4>() &&
                  smem_layout_ok<true, MOE_W_FP4>() && smem_layout_ok<false, kMx>() && smem_layout_ok<true, kMx>(),
              "shared / tensor memory layout");

struct TileCoord {
  int e, mt, nt, row0, valid;
};

// Work unit idx -> (expert, token unit, n tile). A token unit is a 128-row
// m-tile (tile mode) or a 32-row chunk (decode mode) of the expert's group.
// Units are ordered expert-major, then by n tile, with the expert's token
// units fastest, so CTAs running at the same time share weight tiles
// through L2. Expert e owns idx in [NT * off[e], NT * off[e + 1]), so
// idx / NT is one of e's token units and the routing kernel's owner table
// gives e in one load.
template <bool DEC>
__device__ __forceinline__ TileCoord decode_tile(int idx, int E, int M, int NT, const int32_t* __restrict__ tiles,
                                                 const int32_t* __restrict__ counts,
                                                 const int32_t* __restrict__ padded_offsets) {
  constexpr int kRows = Pipe<DEC>::kRows;
  const int32_t* off = tiles + (DEC ? tiles_chunk_off(E) : kTilesHdr);
  const int32_t* owner = tiles + (DEC ? tiles_chunk_expert(E, M) : tiles_expert_of(E));
  const int e = __ldg(owner + idx / NT);
  const int u0 = __ldg(off + e);
  const int m_e = __ldg(off + e + 1) - u0;
  const int local = idx - NT * u0;
  TileCoord c;
  c.e = e;
  c.nt = local / m_e;
  c.mt = local % m_e;
  c.row0 = __ldg(padded_offsets + e) + kRows * c.mt;
  c.valid = min(kRows, __ldg(counts + e) - kRows * c.mt);
  return c;
}

// Barrier over the two epilogue warpgroups that also ORs a flag across them,
// so that both take the same decision to stop after a failed wait.
__device__ __forceinline__ bool epi_barrier_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}

// silu(g) * u with the fast exponential and division (relative error a few
// ulp of fp32; the result is requantized to e4m3 right after).
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

// 2^(b - 127) for a UE8M0 byte b in [0, 254], built from the bits.
__device__ __forceinline__ float ue8m0_to_float(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Element i of the thread's 128 accumulators, held as 64 fp32 pairs so the
// promotion can use packed fp32x2 FMAs without re-pairing registers.
#define ACC(i) (((i) & 1) ? acc2[(i) >> 1].y : acc2[(i) >> 1].x)

// What one launch of the kernel body runs: GEMM1 alone, GEMM2 alone, or
// (single-launch decode forward) routing + quantization, then GEMM1 and
// GEMM2 units of one work list, GEMM2 units waiting on their chunk's GEMM1
// units.
enum : int { kG1 = 0, kG2 = 1, kBoth = 2 };

// The kernel body. Side 1 (ta1, tb1, a1) is the only GEMM for KIND kG1 /
// kG2; for kBoth work units [0, U1) are GEMM1's and [U1, total) GEMM2's
// (side 2), U1 and total taken from the routing tables after the grid-wide
// barrier that ends the routing + quantization phase (rq).
template <int FMT, int KIND, bool DEC>
__device__ __forceinline__ void gemm_body(const CUtensorMap* ta1, const CUtensorMap* tb1, const GemmArgs& a1,
                                          const CUtensorMap* ta2, const CUtensorMap* tb2, const GemmArgs& a2,
                                          const RqArgs* rq) {
  static_assert(!DEC || FMT != MOE_W_FP8, "decode mode is built for FP4 weights");
  static_assert(KIND != kBoth || DEC, "the single-launch forward runs the decode mode");
  using Smem = SmemT<DEC, FMT>;
  constexpr int kStages = Pipe<DEC>::kStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned (SWIZZLE_128B atoms). The offset is applied to the
  // __shared__ array itself so the compiler keeps shared-space addressing.
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;
  int U1 = 0;  // kBoth: number of GEMM1 units
  // Per work unit: which GEMM (side 1 or 2), its arguments and index.
  auto on_side1 = [&](int idx) { return KIND != kBoth || idx < U1; };
  auto is_gemm1 = [&](int idx) { return KIND == kG1 || (KIND == kBoth && idx < U1); };
  auto tile_at = [&](int idx) {
    const bool s1 = on_side1(idx);
    const GemmArgs& A = s1 ? a1 : a2;
    return decode_tile<DEC>(s1 ? idx : idx - U1, A.E, A.M, A.g.NT, A.tiles, A.counts, A.padded_offsets);
  };

  if (tid == 0) {
    sm.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], kEpiThreads / 32);
    }
    for (int b = 0; b < kScaleSlots; ++b) {
      mbar_init(&sm.sfull[b], 1);
      mbar_init(&sm.sempty[b], kEpiThreads / 32);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  // FP4 stage bytes: the tile lands unpacked (16 codes per 16 bytes) but the
  // copy's transaction count is the packed global size.
  constexpr uint32_t kStageBytes = (FMT == MOE_W_FP4)
                                       ? Pipe<DEC>::kAStride + kTileBBytes / 2 + kSfaBytes + kSfbBytes
                                       : Pipe<DEC>::kAStride + kTileBBytes;
  // Decode-mode GEMM2: the weight tiles (and their scale blocks) of the first
  // stages of this CTA's first unit are loaded before the dependency wait,
  // while GEMM1 drains; only the activation side waits. The unit comes from
  // the routing tables, which are complete: this grid cannot start before
  // every GEMM1 CTA has passed its own wait, i.e. before the routing kernel
  // has finished.
  int pre_unit = -1, pre_n = 0;
  int total_tiles = 0;
  if constexpr (KIND == kBoth) {
    // Routing + quantization of the small batch (every CTA routes the whole
    // batch in shared memory, borrowing the weight ring; CTA 0 writes the
    // routing arrays and zeroes the chunk counters; each CTA quantizes its
    // tokens), then a grid-wide barrier: every unit below may read any of it.
    RqSmem<kThreads / 32>& rs = *reinterpret_cast<RqSmem<kThreads / 32>*>(&sm.b[0][0]);
    route_small_in_smem<kThreads / 32>(rs, *rq);
    if (blockIdx.x == 0) write_routing<kThreads / 32>(rs, *rq);
    quantize_tokens<kThreads / 32, true, FMT == kMx>(rs, *rq, blockIdx.x, gridDim.x);
    const int nchunks = rs.chs[rq->E];
    // the generic-proxy writes above (global: routing arrays, counters;
    // shared: the borrowed ring) are ordered before the TMA traffic below
    __threadfence();
    fence_proxy_async_global();
    fence_proxy_async_smem();
    cooperative_groups::this_grid().sync();
    fence_proxy_async_global();
    U1 = nchunks * a1.g.NT;
    total_tiles = U1 + nchunks * a2.g.NT;
  } else {
    if constexpr (DEC && KIND == kG2) {
      const GemmGeom& g = a1.g;
      if (tid == 0 && static_cast<int>(blockIdx.x) < __ldg(a1.tiles + 1) * g.NT) {
        const TileCoord c = tile_at(blockIdx.x);
        pre_unit = blockIdx.x;
        // FP4 activations: stages of two 128-K blocks (see the producer)
        const int KS = (FMT == kMx) ? (g.KB + 1) / 2 : g.KB;
        pre_n = min(kStages, KS);
        const int wrow = c.e * g.Np + c.nt * kBlockN;
        for (int s = 0; s < pre_n; ++s) {
          if constexpr (FMT == kMx) {
            const int nch = min(2, g.KB - 2 * s);
            mbar_arrive_expect_tx(&sm.full[s], Pipe<DEC>::kAStride + kTileBBytes + nch * (kSfaBytes + kSfbBytes));
            tma_load_2d(sm.b[s], tb1, &sm.full[s], s * 128, wrow);
            bulk_load(sm.sfb[s], a1.w_scale + ((static_cast<size_t>(c.e) * g.NT + c.nt) * g.KB + 2 * s) * kSfbBytes,
                      nch * kSfbBytes, &sm.full[s]);
          } else {
            mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
            tma_load_2d(sm.b[s], tb1, &sm.full[s], s * kBlockK, wrow);
            bulk_load(sm.sfb[s], a1.w_scale + ((static_cast<size_t>(c.e) * g.NT + c.nt) * g.KB + s) * kSfbBytes,
                      kSfbBytes, &sm.full[s]);
          }
        }
      }
    }
    // Everything above overlaps the previous kernel's tail; the tile list and
    // the activations are written by the kernels before this one.
    pdl_wait();
    pdl_launch_dependents();
    total_tiles = __ldg(a1.tiles + (DEC ? 1 : 0)) * a1.g.NT;
  }

  if (warp < kEpiWarp0) {
   regs_dec<56>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(ta1);
      tma_prefetch_desc(tb1);
      if constexpr (KIND == kBoth) {
        tma_prefetch_desc(ta2);
        tma_prefetch_desc(tb2);
      }
      int stage = 0;
      uint32_t phase = 0;
      int pf_idx = -1, pf_seen = 0;  // single launch: next GEMM2 unit's counter, read ahead
      for (int idx = blockIdx.x; idx < total_tiles && !*abort_flag; idx += gridDim.x) {
        const bool s1 = on_side1(idx);
        const GemmArgs& A = s1 ? a1 : a2;
        const CUtensorMap* TA = s1 ? ta1 : ta2;
        const CUtensorMap* TB = s1 ? tb1 : tb2;
        const int KB = A.g.KB, NT = A.g.NT;
        const TileCoord c = tile_at(idx);
        const int wrow = c.e * A.g.Np + c.nt * kBlockN;
        int kb0 = 0;
        if (KIND == kBoth && !s1) {
          // GEMM2 unit of the single-launch forward. Its chunk's counter was
          // read (relaxed) while the previous unit was being issued; if the
          // chunk was complete then, an acquire fence makes its rows visible
          // and the unit takes the ordinary path. Otherwise the weight side
          // of the first stages goes out now and the activation side once
          // every GEMM1 unit of the chunk has stored its rows (bounded wait).
          const int32_t* ready = A.chunk_ready + c.row0 / kChunkRows;
          int seen = 0;
          if (pf_idx == idx) {
            seen = pf_seen;
          } else {
            asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(ready) : "memory");
          }
          if (seen >= A.ready_target) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");  // the relaxed read + fence acquire
            fence_proxy_async_global();
          } else {
            // (FP4 activations: a stage is two 128-K blocks, as below)
            const int npre = min(kStages, (FMT == kMx) ? (KB + 1) / 2 : KB);
            const int st0 = stage;
            bool ok = true;
            for (int kb = 0; kb < npre; ++kb) {
              if (!mbar_wait(&sm.empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
              if constexpr (FMT == kMx) {
                const int nch = min(2, KB - 2 * kb);
                mbar_arrive_expect_tx(&sm.full[stage],
                                      Pipe<DEC>::kAStride + kTileBBytes + nch * (kSfaBytes + kSfbBytes));
                tma_load_2d(sm.b[stage], TB, &sm.full[stage], kb * 128, wrow);
                bulk_load(sm.sfb[stage],
                          A.w_scale + ((static_cast<size_t>(c.e) * NT + c.nt) * KB + 2 * kb) * kSfbBytes,
                          nch * kSfbBytes, &sm.full[stage]);
              } else {
                mbar_arrive_expect_tx(&sm.full[stage], kStageBytes);
                tma_load_2d(sm.b[stage], TB, &sm.full[stage], kb * kBlockK, wrow);
                bulk_load(sm.sfb[stage], A.w_scale + ((static_cast<size_t>(c.e) * NT + c.nt) * KB + kb) * kSfbBytes,
                          kSfbBytes, &sm.full[stage]);
              }
              if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok || !wait_counter(ready, A.ready_target, abort_flag)) break;
            fence_proxy_async_global();
            for (int kb = 0; kb < npre; ++kb) {
              const int s = (st0 + kb) % kStages;
              if constexpr (FMT == kMx) {
                const int nch = min(2, KB - 2 * kb);
                tma_load_2d(sm.a_stage(s), TA, &sm.full[s], kb * 128, c.row0);
                bulk_load(sm.sfa[s], A.a_sf + (static_cast<size_t>(c.row0 / kBlockM) * KB + 2 * kb) * kSfaBytes,
                          nch * kSfaBytes, &sm.full[s]);
              } else {
                tma_load_2d(sm.a_stage(s), TA, &sm.full[s], kb * kBlockK, c.row0);
                bulk_load(sm.sfa[s], A.a_sf + (static_cast<size_t>(c.row0 / kBlockM) * KB + kb) * kSfaBytes,
                          kSfaBytes, &sm.full[s]);
              }
            }
            kb0 = npre;
          }
        }
        // FP4 activations: a stage covers two 128-K blocks (the last one may
        // hold one: its TMA boxes run past K and read zeros)
        const int KS = (FMT == kMx) ? (KB + 1) / 2 : KB;
        for (int kb = kb0; kb < KS; ++kb) {
          if constexpr (KIND == kBoth) {
            // read the next unit's chunk counter ahead (its value is used at
            // that unit's start); placed a few stages in, so that the table
            // loads it needs do not delay this unit's first copies
            if (kb == kb0 + 2 || (kb == kb0 && KS - kb0 <= 2)) {
              const int nidx = idx + static_cast<int>(gridDim.x);
              if (nidx >= U1 && nidx < total_tiles) {
                const TileCoord nc = tile_at(nidx);
                asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];"
                             : "=r"(pf_seen)
                             : "l"(a2.chunk_ready + nc.row0 / kChunkRows)
                             : "memory");
                pf_idx = nidx;
              }
            }
          }
          if (!mbar_wait(&sm.empty[stage], phase ^ 1, abort_flag)) break;
          if constexpr (FMT == kMx) {
            const int ch0 = 2 * kb, nch = min(2, KB - ch0);
            // decode mode: weight side already in flight from before the dependency wait
            const bool pre = idx == pre_unit && kb < pre_n;
            if (!pre)
              mbar_arrive_expect_tx(&sm.full[stage],
                                    Pipe<DEC>::kAStride + kTileBBytes + nch * (kSfaBytes + kSfbBytes));
            tma_load_2d(sm.a_stage(stage), TA, &sm.full[stage], kb * 128, c.row0);  // x in bytes
            if (!pre) tma_load_2d(sm.b[stage], TB, &sm.full[stage], kb * 128, wrow);
            bulk_load(sm.sfa[stage], A.a_sf + (static_cast<size_t>(c.row0 / kBlockM) * KB + ch0) * kSfaBytes,
                      nch * kSfaBytes, &sm.full[stage]);
            if (!pre)
              bulk_load(sm.sfb[stage], A.w_scale + ((static_cast<size_t>(c.e) * NT + c.nt) * KB + ch0) * kSfbBytes,
                        nch * kSfbBytes, &sm.full[stage]);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
            continue;
          }
          // weights already in flight from before the dependency wait
          const bool pre = idx == pre_unit && kb < pre_n;
          if (!pre) mbar_arrive_expect_tx(&sm.full[stage], kStageBytes);
          tma_load_2d(sm.a_stage(stage), TA, &sm.full[stage], kb * kBlockK, c.row0);
          if (!pre) tma_load_2d(sm.b[stage], TB, &sm.full[stage], kb * kBlockK, wrow);
          if constexpr (FMT == MOE_W_FP4) {
            bulk_load(sm.sfa[stage], A.a_sf + (static_cast<size_t>(c.row0 / kBlockM) * KB + kb) * kSfaBytes,
                      kSfaBytes, &sm.full[stage]);
            if (!pre)
              bulk_load(sm.sfb[stage],
                        A.w_scale + ((static_cast<size_t>(c.e) * NT + c.nt) * KB + kb) * kSfbBytes, kSfbBytes,
                        &sm.full[stage]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues; in decode mode the whole warp walks the stages (it
    // moves the chunk's activation scale words before each copy).
    if (DEC || lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t bphase = 0;
      // (decode mode: the whole warp walks the stages, so it leaves together)
      for (int idx = blockIdx.x; idx < total_tiles && !(DEC ? __any_sync(0xffffffffu, *abort_flag != 0) : *abort_flag);
           idx += gridDim.x) {
        const int KB = (on_side1(idx) ? a1 : a2).g.KB;
        if constexpr (FMT == MOE_W_FP8) {
          constexpr uint32_t idesc = idesc_f8f6f4(0, 0, kBlockM, kBlockN);
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait_spin(&sm.full[stage], phase, abort_flag)) break;
            if (!mbar_wait_spin(&sm.tempty[buf], bphase ^ 1, abort_flag)) break;
            tc_fence_after();
            const uint64_t ad = smem_desc(smem_u32(sm.a_stage(stage)), 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(smem_u32(sm.b[stage]), 16, 1024, kSwizzle128B);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_f8f6f4(tbase + buf * kBlockN, ad + 2 * j, bd + 2 * j, idesc, j > 0 ? 1u : 0u);
            mma_commit(&sm.empty[stage]);
            mma_commit(&sm.tfull[buf]);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
            buf ^= 1;
            if (buf == 0) bphase ^= 1;
          }
        } else if constexpr (FMT == kMx) {
          // one issuing thread (tile mode); in decode mode the warp walks the
          // stages as for FP4 weights and moves the chunk's scale words
          bool ok = mbar_wait(&sm.tempty[0], bphase ^ 1, abort_flag);
          if constexpr (DEC) ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          int q = 0;
          if constexpr (DEC) q = (tile_at(idx).row0 % kBlockM) / kChunkRows;
          const int KS = (KB + 1) / 2;
          for (int ks = 0; ks < KS; ++ks) {
            bool okf = mbar_wait(&sm.full[stage], phase, abort_flag);
            if constexpr (DEC) okf = __all_sync(0xffffffffu, okf);
            if (!okf) { ok = false; break; }
            const int nch = min(2, KB - 2 * ks);
            if constexpr (DEC) {
              if (q != 0) {
                // the chunk's words are column q of each 128-row block image
                for (int ch = 0; ch < nch; ++ch) {
                  uint32_t* w = reinterpret_cast<uint32_t*>(sm.sfa[stage] + ch * kSfaBytes);
                  const uint32_t v = w[4 * lane + q];
                  __syncwarp();
                  w[4 * lane] = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
              }
            }
            if (lane == 0) {
              tc_fence_after();
              const uint32_t sfa_col = kSfTmemCol + stage * kSfColsPerStage<FMT>;
              const uint32_t sfb_col = sfa_col + 8;
              for (int ch = 0; ch < nch; ++ch) {
                tmem_cp_32x128b_warpx4(tbase + sfa_col + 4 * ch,
                                       smem_desc(smem_u32(sm.sfa[stage] + ch * kSfaBytes), 0, 128, kSwizzleNone));
                tmem_cp_32x128b_warpx4(tbase + sfb_col + 8 * ch,
                                       smem_desc(smem_u32(sm.sfb[stage] + ch * kSfbBytes), 0, 128, kSwizzleNone));
                tmem_cp_32x128b_warpx4(
                    tbase + sfb_col + 8 * ch + 4,
                    smem_desc(smem_u32(sm.sfb[stage] + ch * kSfbBytes + 512), 0, 128, kSwizzleNone));
              }
              const uint64_t ad = smem_desc(smem_u32(sm.a_stage(stage)), 16, 1024, kSwizzle128B);
              const uint64_t bd = smem_desc(smem_u32(sm.b[stage]), 16, 1024, kSwizzle128B);
              // four K = 64 steps of 32 bytes; step j takes scale bytes 2 (j % 2)
              // and 2 (j % 2) + 1 of chunk j / 2
              for (int j = 0; j < 2 * nch; ++j)
                mma_mxf4(tbase, ad + 2 * j, bd + 2 * j, idesc_mxf4(kBlockM, kBlockN, 2 * (j & 1), 2 * (j & 1)),
                         tbase + sfa_col + 4 * (j >> 1), tbase + sfb_col + 8 * (j >> 1),
                         (ks > 0 || j > 0) ? 1u : 0u);
              mma_commit(&sm.empty[stage]);
            }
            if constexpr (DEC) __syncwarp();
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          if (lane == 0) mma_commit(&sm.tfull[0]);
          bphase ^= 1;
        } else {
          bool ok = mbar_wait(&sm.tempty[0], bphase ^ 1, abort_flag);
          if constexpr (DEC) ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          // Decode mode: the chunk's activation scale words are column q of
          // its 128-row block's image; the MMA reads A rows 0-31 (the chunk)
          // from the first column.
          int q = 0;
          if constexpr (DEC) q = (tile_at(idx).row0 % kBlockM) / kChunkRows;
          for (int kb = 0; kb < KB; ++kb) {
            bool okf = mbar_wait(&sm.full[stage], phase, abort_flag);
            if constexpr (DEC) okf = __all_sync(0xffffffffu, okf);
            if (!okf) { ok = false; break; }
            if constexpr (DEC) {
              if (q != 0) {
                uint32_t* w = reinterpret_cast<uint32_t*>(sm.sfa[stage]);
                const uint32_t v = w[4 * lane + q];
                __syncwarp();
                w[4 * lane] = v;
                fence_proxy_async_smem();
                __syncwarp();
              }
            }
            if (lane == 0) {
              tc_fence_after();
              const uint32_t sfa_col = kSfTmemCol + stage * 12;
              const uint32_t sfb_col = sfa_col + 4;
              tmem_cp_32x128b_warpx4(tbase + sfa_col, smem_desc(smem_u32(sm.sfa[stage]), 0, 128, kSwizzleNone));
              tmem_cp_32x128b_warpx4(tbase + sfb_col, smem_desc(smem_u32(sm.sfb[stage]), 0, 128, kSwizzleNone));
              tmem_cp_32x128b_warpx4(tbase + sfb_col + 4,
                                     smem_desc(smem_u32(sm.sfb[stage] + 512), 0, 128, kSwizzleNone));
              const uint64_t ad = smem_desc(smem_u32(sm.a_stage(stage)), 16, 1024, kSwizzle128B);
              const uint64_t bd = smem_desc(smem_u32(sm.b[stage]), 16, 1024, kSwizzle128B);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_mxf8f6f4(tbase, ad + 2 * j, bd + 2 * j, idesc_mxf8f6f4(0, 5, kBlockM, kBlockN, j, j),
                             tbase + sfa_col, tbase + sfb_col, (kb > 0 || j > 0) ? 1u : 0u);
              mma_commit(&sm.empty[stage]);
            }
            if constexpr (DEC) __syncwarp();
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          if (lane == 0) mma_commit(&sm.tfull[0]);
          bphase ^= 1;
        }
      }
    }
   } else if (warp == 2 && FMT == MOE_W_FP8) {
    // ------------------------------------------------------ scale producer
    // Promotion scales for kScaleGroup consecutive K blocks per slot: the
    // activation exponent words of the 128 rows and the 8 weight scales.
    // Both are contiguous in K for a tile, so a slot is two bulk copies.
    if (lane == 0) {
      int slot = 0;
      uint32_t sphase = 0;
      const GemmArgs& args = a1;
      const int KB = args.g.KB, NT = args.g.NT;
      for (int idx = blockIdx.x; idx < total_tiles && !*abort_flag; idx += gridDim.x) {
        const TileCoord c = tile_at(idx);
        for (int kb0 = 0; kb0 < KB; kb0 += kScaleGroup) {
          const int n = min(kScaleGroup, KB - kb0);
          if (!mbar_wait(&sm.sempty[slot], sphase ^ 1, abort_flag)) break;
          mbar_arrive_expect_tx(&sm.sfull[slot], n * (kSfaBytes + kSwBytes));
          bulk_load(sm.sfa_w[slot], args.a_sf + (static_cast<size_t>(c.row0 / kBlockM) * KB + kb0) * kSfaBytes,
                    n * kSfaBytes, &sm.sfull[slot]);
          bulk_load(sm.sw[slot], args.w_scale + ((static_cast<size_t>(c.e) * NT + c.nt) * KB + kb0) * kSwBytes,
                    n * kSwBytes, &sm.sfull[slot]);
          if (++slot == kScaleSlots) { slot = 0; sphase ^= 1; }
        }
      }
    }
   }
  } else {
    regs_inc<224>();
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - kEpiWarp0) / 4;  // column half of the tile
    const int quarter = warp & 3;           // TMEM lane quarter this warp may access
    const int m = quarter * 32 + lane;      // tile row owned by this thread
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int buf = 0;
    uint32_t bphase = 0;
    int sslot = 0;
    uint32_t ssphase = 0;
    int tile_parity = 0;
    const float limit = a1.swiglu_limit;
    const bool clamp = limit > 0.f && limit < INFINITY;
    // (no abort test in the loop condition: a thread that saw the flag
    // early would leave while the others wait at the epilogue barrier; after
    // an abort every wait fails and the reducing barrier stops them together)
    for (int idx = blockIdx.x; idx < total_tiles; idx += gridDim.x) {
      const bool GEMM1 = is_gemm1(idx);
      const GemmArgs& args = on_side1(idx) ? a1 : a2;
      const int KB = args.g.KB;
      const TileCoord c = tile_at(idx);
      float2 acc2[64];
      bool ok = true;
      if constexpr (FMT == MOE_W_FP8) {
#pragma unroll
        for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.f, 0.f);
        const int wi = 4 * (m % 32) + m / 32;  // this row's scale word in a 128-row block
        for (int kb = 0; kb < KB; ++kb) {
          const int gi = kb % kScaleGroup;
          if (gi == 0 && !mbar_wait_spin(&sm.sfull[sslot], ssphase, abort_flag)) { ok = false; break; }
          const float sa = ue8m0_to_float(sm.sfa_w[sslot][gi][wi] & 0xFF);
          float2 sc2[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float v = sa * sm.sw[sslot][gi][wg * 4 + q];
            sc2[q] = make_float2(v, v);
          }
          if (gi == kScaleGroup - 1 || kb == KB - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sempty[sslot]);
            if (++sslot == kScaleSlots) { sslot = 0; ssphase ^= 1; }
          }
          if (!mbar_wait_spin(&sm.tfull[buf], bphase, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(tbase + lane_base + buf * kBlockN + wg * 128 + h * 64, r0);
            tmem_ld_32x32b_x32(tbase + lane_base + buf * kBlockN + wg * 128 + h * 64 + 32, r1);
            tmem_wait_ld();
            if (h == 1) {
              // The partial is in registers: hand the buffer back to the MMA
              // before the last FMAs.
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[buf]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc2[h * 32 + j] = __ffma2_rn(make_float2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1])),
                                            sc2[2 * h], acc2[h * 32 + j]);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc2[h * 32 + 16 + j] =
                  __ffma2_rn(make_float2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1])), sc2[2 * h + 1],
                             acc2[h * 32 + 16 + j]);
          }
          buf ^= 1;
          if (buf == 0) bphase ^= 1;
        }
      } else {
        // warp-uniform: the drain below is made of warp-collective loads
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[0], bphase, abort_flag));
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // a warp whose 32 rows are all padding (light experts' last
            // tiles) reads nothing; it still takes part in the hand-off
            if (quarter * 32 >= c.valid) break;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + lane_base + wg * 128 + q * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc2[q * 16 + j] = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.tempty[0]);
          bphase ^= 1;
        }
      }
      const int row = c.row0 + m;
      if (FMT == kMx && GEMM1) {
        // FP4 activations: SwiGLU, then the 1x32 e2m1 rule; a thread's 64
        // intermediate columns j = 128 nt + 64 wg + i are two whole blocks,
        // so no exchange between the warpgroups is needed. In the single
        // launch every epilogue thread meets the release barrier below, so
        // all of them stop together if any wait failed.
        if constexpr (KIND == kBoth) {
          if (epi_barrier_any(!ok)) break;
        } else {
          if (!ok) break;  // warp-uniform
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float gt = ACC(i), up = ACC(64 + i);
          if (clamp) {
            gt = fminf(gt, limit);
            up = fminf(fmaxf(up, -limit), limit);
          }
          ACC(i) = silu_mul(gt, up);
        }
        if (m < c.valid) {
          if (args.act_f32 != nullptr) {
            // debug tap: the fp32 values requantized below (row stride in elements)
            float* dst = args.act_f32 + static_cast<size_t>(row) * (2 * args.out_cols) + c.nt * 128 + wg * 64;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              st_global_v8(dst + 8 * v, __float_as_uint(ACC(8 * v)), __float_as_uint(ACC(8 * v + 1)),
                           __float_as_uint(ACC(8 * v + 2)), __float_as_uint(ACC(8 * v + 3)),
                           __float_as_uint(ACC(8 * v + 4)), __float_as_uint(ACC(8 * v + 5)),
                           __float_as_uint(ACC(8 * v + 6)), __float_as_uint(ACC(8 * v + 7)));
          }
          uint32_t pk[8];
          uint32_t ex = 0;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(ACC(32 * b + i)));
            const int e = act_exponent_e2m1(amax);
            const float s = exp2_neg(e);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i0 = 32 * b + 8 * u;
              pk[4 * b + u] = pack8_e2m1(ACC(i0) * s, ACC(i0 + 1) * s, ACC(i0 + 2) * s, ACC(i0 + 3) * s,
                                         ACC(i0 + 4) * s, ACC(i0 + 5) * s, ACC(i0 + 6) * s, ACC(i0 + 7) * s);
            }
            ex |= static_cast<uint32_t>(e + 127) << (8 * b);
          }
          st_global_v8(args.out_q + static_cast<size_t>(row) * args.out_cols + c.nt * 64 + wg * 32, pk[0], pk[1],
                       pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          // bytes 2 wg and 2 wg + 1 of the (row, 128-column block nt) scale word
          reinterpret_cast<uint16_t*>(args.out_sf)[2 * sf_word_index(row, c.nt, args.out_blocks) + wg] =
              static_cast<uint16_t>(ex);
        }
        if constexpr (KIND == kBoth) {
          // release this unit's rows to the GEMM2 units of the chunk, as below
          __threadfence();
          fence_proxy_async_global();
          epi_barrier_any(false);
          if (tid == kEpiWarp0 * 32) atomicAdd(args.chunk_ready + c.row0 / kChunkRows, 1);
        }
      } else if (GEMM1) {
        // ACC(0..63) = gate, ACC(64..127) = up of intermediate columns
        // j = 128 nt + 64 wg + i.
        float amax = 0.f;
        if (ok) {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            float gt = ACC(i), up = ACC(64 + i);
            if (clamp) {
              gt = fminf(gt, limit);
              up = fminf(fmaxf(up, -limit), limit);
            }
            const float a = silu_mul(gt, up);
            ACC(i) = a;
            amax = fmaxf(amax, fabsf(a));
          }
        }
        sm.amax_x[tile_parity][wg][m] = amax;
        // Every epilogue thread reaches this barrier once per tile, failed
        // wait or not; all of them stop together if any wait failed.
        if (epi_barrier_any(!ok)) break;
        amax = fmaxf(sm.amax_x[tile_parity][0][m], sm.amax_x[tile_parity][1][m]);
        tile_parity ^= 1;
        const int e = act_exponent(amax);
        const float s = exp2_neg(e);
        if (args.act_f32 != nullptr && m < c.valid) {
          // debug tap: the fp32 values requantized below
          float* dst = args.act_f32 + static_cast<size_t>(row) * args.out_cols + c.nt * 128 + wg * 64;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st_global_v8(dst + 8 * v, __float_as_uint(ACC(8 * v)), __float_as_uint(ACC(8 * v + 1)),
                         __float_as_uint(ACC(8 * v + 2)), __float_as_uint(ACC(8 * v + 3)),
                         __float_as_uint(ACC(8 * v + 4)), __float_as_uint(ACC(8 * v + 5)),
                         __float_as_uint(ACC(8 * v + 6)), __float_as_uint(ACC(8 * v + 7)));
        }
        if (m < c.valid) {
          uint8_t* dst = args.out_q + static_cast<size_t>(row) * args.out_cols + c.nt * 128 + wg * 64;
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            uint32_t pk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int i0 = 32 * v + 4 * u;
              pk[u] = pack4_e4m3(ACC(i0) * s, ACC(i0 + 1) * s, ACC(i0 + 2) * s, ACC(i0 + 3) * s);
            }
            st_global_v8(dst + 32 * v, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          }
          if (wg == 0)
            reinterpret_cast<uint32_t*>(args.out_sf)[sf_word_index(row, c.nt, args.out_blocks)] =
                static_cast<uint32_t>(e + 127) * 0x01010101u;
        }
        if constexpr (KIND == kBoth) {
          // Release this unit's rows to the GEMM2 units of the chunk: every
          // thread's stores, a fence, the epilogue barrier, then one count.
          __threadfence();
          fence_proxy_async_global();
          epi_barrier_any(false);
          if (tid == kEpiWarp0 * 32) atomicAdd(args.chunk_ready + c.row0 / kChunkRows, 1);
        }
      } else {
        // warp-uniform: the stores and the fused combine below use warp
        // barriers and shuffles
        if (!__all_sync(0xffffffffu, ok)) break;
        bool last = false;
        int t_last = 0;
        if (!DEC) {
          // Tile mode: the warp's 32 rows leave in 16-column boxes transposed
          // through shared memory, so that each store instruction writes 64
          // contiguous bytes of 8 rows instead of 32 bytes of 32 rows (a
          // lane per row): the per-SM store rate of the fp32 rows bounds this
          // phase. The lane of row r writes 16-byte piece p of its box row at
          // r * 64 + (p ^ ((r / 2) % 4)) * 16, conflict-free on both sides.
          float wgt = 0.f;
          if (m < c.valid) wgt = __ldg(args.row_w + row);
          const float2 w2 = make_float2(wgt, wgt);
          const int col0 = c.nt * kBlockN + wg * 128;
          const uint32_t stg = smem_u32(sm.ystage) + (warp - kEpiWarp0) * kYBoxBytes;
          const int rr = lane >> 2, pp = lane & 3;  // read-back: row rr + 8 i, piece pp
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (col0 + 16 * j < args.H) {  // warp-uniform (an if: a break here spills)
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const float2 lo = __fmul2_rn(acc2[8 * j + 2 * p], w2), hi = __fmul2_rn(acc2[8 * j + 2 * p + 1], w2);
                st_shared_v4(stg + lane * 64 + ((p ^ ((lane >> 1) & 3)) << 4), lo.x, lo.y, hi.x, hi.y);
              }
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int r = 8 * i + rr;
                const float4 v = ld_shared_v4(stg + r * 64 + ((pp ^ ((r >> 1) & 3)) << 4));
                if (quarter * 32 + r < c.valid)
                  *reinterpret_cast<float4*>(args.out_y + static_cast<size_t>(c.row0 + quarter * 32 + r) * args.H +
                                             col0 + 16 * j + 4 * pp) = v;
              }
              __syncwarp();
            }
          }
        } else if (m < c.valid) {
          const float wgt = __ldg(args.row_w + row);
          const int slot = (DEC && args.combine_cnt != nullptr) ? __ldg(args.row_slot + row) : 0;
          const int col0 = c.nt * kBlockN + wg * 128;
          float* dst = args.out_y + static_cast<size_t>(row) * args.H + col0;
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            if (col0 + 8 * v < args.H) {
              const float2 w2 = make_float2(wgt, wgt);
              const float2 p0 = __fmul2_rn(acc2[4 * v], w2), p1 = __fmul2_rn(acc2[4 * v + 1], w2);
              const float2 p2 = __fmul2_rn(acc2[4 * v + 2], w2), p3 = __fmul2_rn(acc2[4 * v + 3], w2);
              st_global_v8(dst + 8 * v, __float_as_uint(p0.x), __float_as_uint(p0.y), __float_as_uint(p1.x),
                           __float_as_uint(p1.y), __float_as_uint(p2.x), __float_as_uint(p2.y), __float_as_uint(p3.x),
                           __float_as_uint(p3.y));
            }
          }
          if (DEC && args.combine_cnt != nullptr) {
            // Fused combine: count this row's arrival for its token and these
            // 128 columns (the combine itself runs warp-wide below).
            t_last = slot / args.K;
            __threadfence();  // this row is visible before it is counted
            int32_t* cnt = args.combine_cnt + static_cast<size_t>(t_last) * args.combine_stride;
            last = (atomicAdd(cnt + 1 + kCombineSplits * c.nt + wg, 1) + 1) == __ldg(cnt);
          }
        }
        if (DEC && args.combine_cnt != nullptr) {
          // Fused combine (decode mode, small batches): the top-k combine. The last of a token's rows to
          // arrive for these 128 columns triggers the sum of all of them in
          // ascending k, in fp32, rounded once to bf16 - the deterministic
          // reduction of the pages (view(T, K, H).sum(1), no atomics on data),
          // whatever the order in which the tiles finish. The warp serves its
          // last arrivers one by one, each lane summing 4 of the 128 columns
          // with all K row loads in flight together.
          unsigned todo = __ballot_sync(0xffffffffu, last);
          if (todo) {
            // the counting thread's fence, then the warp barrier, order the
            // other rows' stores before every lane's loads
            __threadfence();
            __syncwarp();
          }
          const int col0 = c.nt * kBlockN + wg * 128 + 4 * lane;
          while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int t = __shfl_sync(0xffffffffu, t_last, src);
            const int my_row = (lane < args.K) ? __ldg(args.inv + static_cast<size_t>(t) * args.K + lane) : -1;
            // H may end halfway through these 128 columns: lanes past it load
            // nothing, but every lane stays in the shuffles
            const bool in_h = col0 < args.H;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0 = 0; k0 < args.K; k0 += 8) {
              int r[8];
              float4 v[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                r[u] = __shfl_sync(0xffffffffu, my_row, (k0 + u) & 31);
                if (k0 + u >= args.K) r[u] = -1;
                v[u] = (in_h && r[u] >= 0)
                           ? __ldcg(reinterpret_cast<const float4*>(args.out_y + static_cast<size_t>(r[u]) * args.H + col0))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                if (r[u] >= 0) {
                  acc.x += v[u].x;
                  acc.y += v[u].y;
                  acc.z += v[u].z;
                  acc.w += v[u].w;
                }
              }
            }
            if (in_h) {
              const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
              uint2 pk;
              pk.x = *reinterpret_cast<const uint32_t*>(&lo);
              pk.y = *reinterpret_cast<const uint32_t*>(&hi);
              *reinterpret_cast<uint2*>(args.out + static_cast<size_t>(t) * args.H + col0) = pk;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
  if (tid == 0 && sm.abort_flag) atomicOr(a1.status, MOE_DEV_TIMEOUT);
}

template <int FMT, bool GEMM1, bool DEC>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ GemmArgs args) {
  gemm_body<FMT, GEMM1 ? kG1 : kG2, DEC>(&tmap_a, &tmap_b, args, &tmap_a, &tmap_b, args, nullptr);
}

// The single-launch decode forward (FP4 weights, e4m3 or e2m1 activations;
// sized for T * K <= 256, run for T * K <= 32): routing, quantization, GEMM1
// + SwiGLU + requantization, GEMM2 + routing weight + the top-k combine, in
// one cooperative launch of one CTA per SM.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
single_launch_decode_kernel(const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1,
                            const __grid_constant__ CUtensorMap ta2, const __grid_constant__ CUtensorMap tb2,
                            const __grid_constant__ GemmArgs a1, const __grid_constant__ GemmArgs a2,
                            const __grid_constant__ RqArgs rq) {
  gemm_body<FMT, kBoth, true>(&ta1, &tb1, a1, &ta2, &tb2, a2, &rq);
}

template <int FMT, bool GEMM1, bool DEC>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args, int num_sms,
                       cudaStream_t st) {
  auto kern = grouped_gemm_kernel<FMT, GEMM1, DEC>;
  const int smem = static_cast<int>(sizeof(SmemT<DEC, FMT>)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, kern, num_sms, kThreads, smem, st, ta, tb, args);
}

static_assert(sizeof(RqSmem<kThreads / 32>) <= sizeof(SmemT<true, MOE_W_FP4>::b) &&
                  sizeof(RqSmem<kThreads / 32>) <= sizeof(SmemT<true, kMx>::b),
              "the routing + quantization phase borrows the weight ring");

template <int FMT>
cudaError_t launch_single(const CUtensorMap& ta1, const CUtensorMap& tb1, const CUtensorMap& ta2,
                          const CUtensorMap& tb2, const GemmArgs& a1, const GemmArgs& a2, const RqArgs& rq,
                          int num_sms, cudaStream_t st) {
  auto kern = single_launch_decode_kernel<FMT>;
  const int smem = static_cast<int>(sizeof(SmemT<true, FMT>)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  // Cooperative: every CTA is resident at once (the grid-wide barrier after
  // routing and the GEMM2 units' waits on GEMM1 units rely on it). The first
  // kernel of the forward: an ordinary (not programmatic) dependency on what
  // the caller queued before.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta1, tb1, ta2, tb2, a1, a2, rq);
}

}  // namespace

cudaError_t launch_single_decode(int fmt, const CUtensorMap& ta1, const CUtensorMap& tb1, const CUtensorMap& ta2,
                                 const CUtensorMap& tb2, const GemmArgs& a1, const GemmArgs& a2, const RqArgs& rq,
                                 int num_sms, cudaStream_t st) {
  return fmt == kMx ? launch_single<kMx>(ta1, tb1, ta2, tb2, a1, a2, rq, num_sms, st)
                    : launch_single<MOE_W_FP4>(ta1, tb1, ta2, tb2, a1, a2, rq, num_sms, st);
}

cudaError_t launch_gemm(int fmt, bool is_gemm1, bool decode, const CUtensorMap& ta, const CUtensorMap& tb,
                        const GemmArgs& args, int num_sms, cudaStream_t st) {
  if (fmt == MOE_W_FP8)
    return is_gemm1 ? launch_one<MOE_W_FP8, true, false>(ta, tb, args, num_sms, st)
                    : launch_one<MOE_W_FP8, false, false>(ta, tb, args, num_sms, st);
  if (fmt == kMx) {
    if (decode)
      return is_gemm1 ? launch_one<kMx, true, true>(ta, tb, args, num_sms, st)
                      : launch_one<kMx, false, true>(ta, tb, args, num_sms, st);
    return is_gemm1 ? launch_one<kMx, true, false>(ta, tb, args, num_sms, st)
                    : launch_one<kMx, false, false>(ta, tb, args, num_sms, st);
  }
  if (decode)
    return is_gemm1 ? launch_one<MOE_W_FP4, true, true>(ta, tb, args, num_sms, st)
                    : launch_one<MOE_W_FP4, false, true>(ta, tb, args, num_sms, st);
  return is_gemm1 ? launch_one<MOE_W_FP4, true, false>(ta, tb, args, num_sms, st)
                  : launch_one<MOE_W_FP4, false, false>(ta, tb, args, num_sms, st);
}

}  // namespace bsmoe

// Internal declarations shared by the kernels and the C-ABI host layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_experts.h"

namespace bsmoe {

constexpr int kBlockM = 128;     // token rows per tile (tcgen05 M)
constexpr int kBlockN = 256;     // weight rows per tile (tcgen05 N)
constexpr int kBlockK = 128;     // K per pipeline stage (= activation block)
constexpr int kRowAlign = 128;   // group alignment of the padded layout
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
constexpr int kGroup = 64;       // gate/up interleave granularity
constexpr int kSfChunkBytes = 512;  // scale words of 128 rows x one K block

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Geometry of one GEMM operand set, shared by host and device.
struct GemmGeom {
  int Kp;      // padded K (multiple of 128)
  int KB;      // Kp / 128
  int Np;      // padded N of the prepared weights per expert (multiple of 256)
  int NT;      // Np / 256
  int N;       // logical N (2I for GEMM1, H for GEMM2)
};

// Prepared weight layout (one of w13 / w2).
struct PrepLayout {
  size_t codes_off, codes_bytes;  // u8 [E][Np][Kp] (FP8) or [E][Np][Kp/2] (FP4)
  size_t scale_off, scale_bytes;  // FP8: f32 [E][NT][KB][8]; FP4: u32 chunks [E][NT][KB][256]
  size_t total;
};

PrepLayout prep_layout(int fmt, int E, const GemmGeom& g);
GemmGeom geom_w13(int H, int I);
GemmGeom geom_w2(int H, int I);

// Decode mode (FP4 weights, with e4m3 or e2m1 activations, at most
// kDecodePairsPerExpert pairs per expert on average): 32-row token chunks in
// the GEMMs.
constexpr int kDecodePairsPerExpert = 8;
constexpr int kCombineSplits = 2;  // column halves of a GEMM2 tile row, finished by separate warpgroups
inline bool decode_mode(int fmt, long long S, int E) {
  return (fmt == MOE_W_FP4 || fmt == MOE_W_FP4_ACT_FP4) && S <= static_cast<long long>(kDecodePairsPerExpert) * E;
}

struct WsLayout {
  moe_workspace_layout pub;
  int S, M, max_m_tiles;
  size_t route_scratch;  // int32 [chunks][E + 1] for the multi-CTA routing
  // With the combine fused into GEMM2 only (0 otherwise): int32
  // [T][combine_stride], per token the number of valid slots, then one
  // arrival counter per (GEMM2 n tile, column half).
  size_t combine_cnt;
  int combine_stride;
  // Single-launch decode forward only (0 otherwise): int32 [M / 32], per
  // 32-row chunk the number of GEMM1 units that have stored their rows.
  size_t chunk_ready;
  // fp32 [M]: the routing weight of the slot in each padded row, written by
  // the quantization next to the row's codes (padding rows are not written
  // and never read), so that GEMM2's epilogue needs one load per row.
  size_t row_w;
};

// Number of routing chunks for S slots (0: the single-CTA kernel is used).
int route_chunks(int S);
bool ws_layout(int fmt, int T, int H, int I, int E, int K, WsLayout* out);

// The int32 "tiles" region (GEMM work lists; M = padded row capacity):
//   [0] number of 128-row m-tiles, [1] number of 32-row chunks;
//   [kTilesHdr + e]                 first m-tile of expert e (E + 1 entries);
//   [tiles_chunk_off(E) + e]        first chunk of expert e (E + 1 entries);
//   [tiles_expert_of(E) + g]        expert owning m-tile g (M / 128 entries);
//   [tiles_chunk_expert(E, M) + c]  expert owning chunk c (M / 32 entries).
constexpr int kTilesHdr = 16;
constexpr int kChunkRows = 32;  // token rows per work unit of the decode-mode GEMMs
__host__ __device__ constexpr int tiles_chunk_off(int E) { return kTilesHdr + E + 1; }
__host__ __device__ constexpr int tiles_expert_of(int E) { return kTilesHdr + 2 * (E + 1); }
__host__ __device__ constexpr int tiles_chunk_expert(int E, int M) { return tiles_expert_of(E) + M / kBlockM; }
__host__ __device__ constexpr int tiles_ints(int E, int M) { return tiles_chunk_expert(E, M) + M / kChunkRows; }

// Launches `kern` on `st`. With `dependent`, the launch may begin while the
// preceding kernel in the stream is still running (programmatic stream
// serialization); every kernel of the forward therefore calls pdl_wait()
// before it touches memory that an earlier kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool dependent, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- launches
cudaError_t launch_route(const int32_t* topk_idx, int S, int E, const WsLayout& L, uint8_t* ws, cudaStream_t st);
// With the combine in GEMM2's epilogue (fused_combine) the quantization
// kernel also sets that up: per-token valid-slot counts, zeroed arrival
// counters, and the +0 output rows of tokens whose slots are all skipped.
cudaError_t launch_quant(int fmt, const void* hidden, const float* topk_w, int T, int H, int K, const WsLayout& L,
                         uint8_t* ws, void* out, cudaStream_t st);
// The top-k combine fused into GEMM2's epilogue: decode batches of at most
// kFusedCombineSlots slots. At larger decode batches the separate combine
// kernel is faster (the epilogue's combines then hold up the accumulator
// hand-back). The small-batch routing + quantization device code of the
// single-launch forward is sized for the same batches. With FP4 activations
// GEMM2 itself is faster and the threshold lower (DeepSeek-V3 shape, same
// box: T=32, 256 slots, 0.397 ms with the fused combine against 0.390 in
// tile mode with the combine kernel; T=8 0.185 against 0.189).
constexpr int kFusedCombineSlots = 256;
constexpr int kFusedCombineSlotsFp4Act = 64;
inline bool fused_combine(int fmt, long long S, int E) {
  return decode_mode(fmt, S, E) && S <= (fmt == MOE_W_FP4_ACT_FP4 ? kFusedCombineSlotsFp4Act : kFusedCombineSlots);
}
// The whole forward as one cooperative launch (routing + quantization, then
// the GEMM1 and GEMM2 units of one work list, GEMM2 units waiting on device
// counters for their chunk's GEMM1 units; the combine in GEMM2's epilogue),
// for FP4-weight fused-combine batches of at most kSingleLaunchSlots slots
// (either activation format). Measured at
// the DeepSeek-V3 shape (FP4, K = 8), one launch against the kernel
// sequence: T=1 0.0652 vs 0.0706 ms, T=2 0.0942 vs 0.0971, T=4 0.1372 vs
// 0.1380, T=8 0.2161 vs 0.2088, T=16 0.3549 vs 0.3263.
constexpr int kSingleLaunchSlots = 32;
inline bool single_launch(int fmt, long long S, int E) {
  return fused_combine(fmt, S, E) && S <= kSingleLaunchSlots;
}
cudaError_t launch_combine(const float* y, const int32_t* inv, int T, int H, int K, void* out, cudaStream_t st);
// transposed: the weights are stored [E][K][N] (N contiguous) instead of [E][N][K].
cudaError_t launch_prepare(int fmt, bool transposed, int E, int H, int I, const void* w13, const void* w13s,
                           const void* w2, const void* w2s, uint8_t* p13, uint8_t* p2, cudaStream_t st);

struct GemmArgs {
  // operands
  const uint8_t* a_sf;        // activation scale words (chunk layout)
  const uint8_t* w_scale;     // prepared weight scales
  const int32_t* counts;
  const int32_t* padded_offsets;
  const int32_t* tiles;
  const int32_t* row_slot;
  const float* row_w;         // GEMM2: routing weight per padded row
  uint32_t* status;
  // outputs
  uint8_t* out_q;             // GEMM1: e4m3 act [M][act_cols] (FP4 activations: e2m1, act_cols / 2 bytes a row)
  uint8_t* out_sf;            // GEMM1: act scale words
  float* out_y;               // GEMM2: f32 [M][H]
  int out_cols;               // GEMM1: bytes of an act row (Kp of GEMM2, halved for FP4 activations); GEMM2: H
  int out_blocks;             // GEMM1: act_blocks
  int E, I, H;
  int M;                      // padded row capacity (locates the chunk work list)
  // GEMM2 in decode mode with the fused combine (combine_cnt non-null): the
  // last arriving row of a token sums the token's rows in ascending k and
  // writes the bf16 output row
  const int32_t* inv;         // [T][K] slot -> padded row, -1 skipped
  int32_t* combine_cnt;       // [T][combine_stride]; null: no fused combine
  int combine_stride;
  int K;
  __nv_bfloat16* out;         // bf16 [T][H]
  float swiglu_limit;         // > 0 and finite: clamp
  // GEMM1 debug tap (null in every timed path): the epilogue also stores
  // the fp32 SwiGLU values it requantizes, [M][out_cols] row-major.
  float* act_f32;
  // Single-launch decode forward: per 32-row chunk, the number of GEMM1
  // units that have stored their rows; a GEMM2 unit waits for ready_target.
  int32_t* chunk_ready;
  int ready_target;
  GemmGeom g;
};

// The whole forward on a caller-provided workspace; events (6 entries or
// null) are recorded at the stage boundaries; act_f32 (null or
// [M][act_cols] fp32) receives GEMM1's fp32 SwiGLU values and selects the
// multi-kernel sequence (the single-launch forward has no tap).
moe_status forward_impl(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T, int H, int I,
                        int E, int K, int fmt, const void* w13_prep, const void* w2_prep, float swiglu_limit,
                        void* workspace, size_t workspace_bytes, void* out, void* stream, void* const* events,
                        float* act_f32 = nullptr, bool allow_single_launch = true);

// decode: FP4 only; 32-row token chunks, activation tensor maps with a
// 32-row box (tile mode: 128-row m-tiles, 128-row box); see decode_mode().
cudaError_t launch_gemm(int fmt, bool is_gemm1, bool decode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                        const GemmArgs& args, int num_sms, cudaStream_t st);

struct RqArgs;
// The single-launch decode forward: one cooperative launch of num_sms CTAs.
cudaError_t launch_single_decode(int fmt, const CUtensorMap& ta1, const CUtensorMap& tb1, const CUtensorMap& ta2,
                                 const CUtensorMap& tb2, const GemmArgs& a1, const GemmArgs& a2, const RqArgs& rq,
                                 int num_sms, cudaStream_t st);

}  // namespace bsmoe

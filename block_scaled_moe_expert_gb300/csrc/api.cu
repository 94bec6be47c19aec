// C-ABI host layer: argument checks, workspace layout, tensor maps and the
// launch sequence route -> quant -> GEMM1 -> GEMM2 -> combine on the caller's
// stream. No allocation, no host synchronization (except
// moe_get_device_status).
//
// The refusals mirror the ones on the transformers pages: hidden states must
// be bf16 (the API takes bf16 only, ValueError in the deepgemm excerpt); a
// model spanning several CUDA devices in one process is refused because the
// kernels are bound to one context (RuntimeError, same excerpt) -- here every
// pointer must belong to the current device; the tensor-core path needs the
// Blackwell family (the SM100 gate run before loading DeepGEMM) -- here
// compute capability 10.3 exactly, the target this library is built for.
#include <cmath>
#include <cstring>
#include <mutex>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route_quant.cuh"

namespace bsmoe {

namespace {

bool shape_ok(int fmt, int H, int I, int E) {
  if (fmt != MOE_W_FP8 && fmt != MOE_W_FP4 && fmt != MOE_W_FP4_ACT_FP4) return false;
  if (E < 1 || E > kMaxExperts) return false;
  if (H < 128 || I < 128 || H > 32768 || I > 32768) return false;
  if (H % 64 || I % 64) return false;
  if (fmt == MOE_W_FP8 && (H % 128 || I % 128)) return false;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D K-major operand: rows x k_elems; box 128 (K) x box_rows.
bool make_tmap(CUtensorMap* m, bool fp4, const void* base, uint64_t k_elems, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {k_elems, rows};
  const cuuint64_t strides[1] = {fp4 ? k_elems / 2 : k_elems};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                         const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct DevInfo {
  int id = -1, sms = 0, major = 0, minor = 0;
};

moe_status current_device(DevInfo* d) {
  if (cudaGetDevice(&d->id) != cudaSuccess) return MOE_ERR_CUDA;
  static DevInfo cache[64];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (d->id >= 0 && d->id < 64 && cache[d->id].id == d->id) {
    *d = cache[d->id];
  } else {
    if (cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&d->major, cudaDevAttrComputeCapabilityMajor, d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&d->minor, cudaDevAttrComputeCapabilityMinor, d->id) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (d->id >= 0 && d->id < 64) cache[d->id] = *d;
  }
  if (d->major != 10 || d->minor != 3) return MOE_ERR_UNSUPPORTED_ARCH;
  return MOE_OK;
}

// Every pointer must be device (or managed) memory of the current device.
moe_status check_ptr(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_DEVICE_MISMATCH;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return MOE_ERR_DEVICE_MISMATCH;
  if (a.device != dev) return MOE_ERR_DEVICE_MISMATCH;
  return MOE_OK;
}

// Self-test of the bounded-wait paths: thread 0 waits, through the helper
// the GEMM pipeline uses, on an mbarrier phase that nothing completes; thread
// 32 waits, through the helper the single-launch forward's GEMM2 units use,
// for a counter (the status word's neighbour, zeroed here) that nothing
// increments. Each wait gives up after its bound, raises the abort flag, and
// the kernel reports MOE_DEV_TIMEOUT the way the GEMMs do, then returns.
__global__ void wait_timeout_selftest_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_bar, abort_cnt;
  if (threadIdx.x == 0) {
    abort_bar = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const bool done = mbar_wait(&bar, 0, &abort_bar);
    if (!done && abort_bar) atomicOr(status, MOE_DEV_TIMEOUT);
  } else if (threadIdx.x == 32) {
    abort_cnt = 0;
    int32_t* counter = reinterpret_cast<int32_t*>(status + 1);
    *counter = 0;
    __threadfence();
    const bool done = wait_counter(counter, 1, &abort_cnt);
    if (!done && abort_cnt) atomicOr(status, MOE_DEV_TIMEOUT);
  }
}

}  // namespace

bool ws_layout(int fmt, int T, int H, int I, int E, int K, WsLayout* out) {
  if (!shape_ok(fmt, H, I, E) || T < 0 || K < 1 || K > kMaxTopK) return false;
  const long long S = static_cast<long long>(T) * K;
  if (S > (1ll << 26)) return false;
  const long long nonempty = std::min<long long>(E, S);
  long long M = S + nonempty * (kRowAlign - 1);
  M = (M + kBlockM - 1) / kBlockM * kBlockM;
  const GemmGeom g1 = geom_w13(H, I), g2 = geom_w2(H, I);
  WsLayout L;
  std::memset(&L, 0, sizeof(L));
  moe_workspace_layout& p = L.pub;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  p.status = take(256);
  p.counts = take(4ull * E);
  p.offsets = take(4ull * (E + 1));
  p.padded_offsets = take(4ull * (E + 1));
  p.tiles = take(4ull * tiles_ints(E, static_cast<int>(M)));
  p.perm = take(4ull * S);
  p.inv = take(4ull * S);
  p.row_slot = take(4ull * M);
  // e4m3 activations: a byte per element; e2m1 (FP4 activations): two per byte
  const size_t per_byte = (fmt == MOE_W_FP4_ACT_FP4) ? 2 : 1;
  p.xq = take(static_cast<size_t>(M) * g1.Kp / per_byte);
  p.xsf = take(4ull * M * g1.KB);
  p.act = take(static_cast<size_t>(M) * g2.Kp / per_byte);
  p.asf = take(4ull * M * g2.KB);
  p.y = take(4ull * M * H);
  L.row_w = take(4ull * M);
  L.route_scratch = take(4ull * (static_cast<size_t>(route_chunks(static_cast<int>(S))) + 1) * (E + 1));
  if (fused_combine(fmt, S, E)) {
    L.combine_stride = 1 + kCombineSplits * g2.NT;
    L.combine_cnt = take(4ull * static_cast<size_t>(T) * L.combine_stride);
  }
  if (single_launch(fmt, S, E)) L.chunk_ready = take(4ull * static_cast<size_t>(M / kChunkRows));
  p.total_bytes = off;
  p.row_capacity = static_cast<int32_t>(M);
  p.row_align = kRowAlign;
  p.xq_cols = g1.Kp;
  p.act_cols = g2.Kp;
  p.x_blocks = g1.KB;
  p.act_blocks = g2.KB;
  L.S = static_cast<int>(S);
  L.M = static_cast<int>(M);
  L.max_m_tiles = static_cast<int>(M / kBlockM);
  *out = L;
  return true;
}

}  // namespace bsmoe

using namespace bsmoe;

extern "C" {

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_UNSUPPORTED_ARCH: return "MOE_ERR_UNSUPPORTED_ARCH";
    case MOE_ERR_DEVICE_MISMATCH: return "MOE_ERR_DEVICE_MISMATCH";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_FAULT: return "MOE_ERR_DEVICE_FAULT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_abi_version(void) { return MOE_ABI_VERSION; }

size_t moe_prepared_w13_bytes(int fmt, int E, int H, int I) {
  if (!shape_ok(fmt, H, I, E)) return 0;
  return prep_layout(fmt, E, geom_w13(H, I)).total;
}

size_t moe_prepared_w2_bytes(int fmt, int E, int H, int I) {
  if (!shape_ok(fmt, H, I, E)) return 0;
  return prep_layout(fmt, E, geom_w2(H, I)).total;
}

size_t moe_workspace_bytes(int fmt, int T_max, int H, int I, int E, int K) {
  WsLayout L;
  if (!ws_layout(fmt, T_max, H, I, E, K, &L)) return 0;
  return L.pub.total_bytes;
}

moe_status moe_query_workspace_layout(int fmt, int T, int H, int I, int E, int K, moe_workspace_layout* layout) {
  if (layout == nullptr) return MOE_ERR_INVALID_ARG;
  WsLayout L;
  if (!ws_layout(fmt, T, H, I, E, K, &L)) return MOE_ERR_UNSUPPORTED_SHAPE;
  *layout = L.pub;
  return MOE_OK;
}

}  // extern "C"

namespace {

moe_status prepare_impl(bool transposed, int fmt, int E, int H, int I, const void* w13, const void* w13_scale,
                        const void* w2, const void* w2_scale, void* w13_prep, size_t w13_prep_bytes, void* w2_prep,
                        size_t w2_prep_bytes, void* stream) {
  if (!shape_ok(fmt, H, I, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const void* ptrs[6] = {w13, w13_scale, w2, w2_scale, w13_prep, w2_prep};
  for (const void* p : ptrs)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  for (const void* p : ptrs)
    if (!aligned(p, 256)) return MOE_ERR_ALIGNMENT;
  if (w13_prep_bytes < moe_prepared_w13_bytes(fmt, E, H, I) || w2_prep_bytes < moe_prepared_w2_bytes(fmt, E, H, I))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo d;
  moe_status s = current_device(&d);
  if (s != MOE_OK) return s;
  for (const void* p : ptrs)
    if ((s = check_ptr(p, d.id)) != MOE_OK) return s;
  if (launch_prepare(fmt, transposed, E, H, I, w13, w13_scale, w2, w2_scale, static_cast<uint8_t*>(w13_prep),
                     static_cast<uint8_t*>(w2_prep), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_prepare_weights(int fmt, int E, int H, int I, const void* w13, const void* w13_scale, const void* w2,
                               const void* w2_scale, void* w13_prep, size_t w13_prep_bytes, void* w2_prep,
                               size_t w2_prep_bytes, void* stream) {
  return prepare_impl(false, fmt, E, H, I, w13, w13_scale, w2, w2_scale, w13_prep, w13_prep_bytes, w2_prep,
                      w2_prep_bytes, stream);
}

moe_status moe_prepare_weights_transposed(int fmt, int E, int H, int I, const void* w13, const void* w13_scale,
                                          const void* w2, const void* w2_scale, void* w13_prep,
                                          size_t w13_prep_bytes, void* w2_prep, size_t w2_prep_bytes,
                                          void* stream) {
  return prepare_impl(true, fmt, E, H, I, w13, w13_scale, w2, w2_scale, w13_prep, w13_prep_bytes, w2_prep,
                      w2_prep_bytes, stream);
}

}  // extern "C"

moe_status bsmoe::forward_impl(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T, int H,
                               int I, int E, int K, int fmt, const void* w13_prep, const void* w2_prep,
                               float swiglu_limit, void* workspace, size_t workspace_bytes, void* out,
                               void* stream, void* const* events, float* act_f32, bool allow_single_launch) {
  if (T < 0 || K < 1 || K > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(fmt, H, I, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
  WsLayout L;
  if (!ws_layout(fmt, T, H, I, E, K, &L)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  const void* ptrs[7] = {hidden, topk_idx, topk_w, w13_prep, w2_prep, workspace, out};
  for (const void* p : ptrs)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(w13_prep, 256) || !aligned(w2_prep, 256) || !aligned(workspace, 256))
    return MOE_ERR_ALIGNMENT;
  if (workspace_bytes < L.pub.total_bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  {
    // out must not overlap an input.
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + static_cast<size_t>(T) * H * 2;
    const uintptr_t h0 = reinterpret_cast<uintptr_t>(hidden), h1 = h0 + static_cast<size_t>(T) * H * 2;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + L.pub.total_bytes;
    if ((o0 < h1 && h0 < o1) || (o0 < w1 && w0 < o1)) return MOE_ERR_INVALID_ARG;
  }
  DevInfo d;
  moe_status s = current_device(&d);
  if (s != MOE_OK) return s;
  for (const void* p : ptrs)
    if ((s = check_ptr(p, d.id)) != MOE_OK) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const moe_workspace_layout& p = L.pub;
  const GemmGeom g1 = geom_w13(H, I), g2 = geom_w2(H, I);
  const PrepLayout P1 = prep_layout(fmt, E, g1), P2 = prep_layout(fmt, E, g2);
  const bool fp4 = (fmt == MOE_W_FP4);
  // FP4 activations: both operands stay packed in shared memory (plain byte
  // maps over K / 2 bytes a row, 128-byte boxes = 256 codes).
  const bool mx = (fmt == MOE_W_FP4_ACT_FP4);
  // FP4 weights with few pairs per expert: the weight-streaming decode mode
  // of the grouped GEMMs (32-row token chunks, five weight stages).
  const bool decode = decode_mode(fmt, L.S, E);
  const int a_box = decode ? kChunkRows : kBlockM;
  const uint64_t k1 = mx ? g1.Kp / 2 : g1.Kp, k2 = mx ? g2.Kp / 2 : g2.Kp;

  CUtensorMap ta1, tb1, ta2, tb2;
  if (!make_tmap(&ta1, false, ws + p.xq, k1, L.M, a_box) ||
      !make_tmap(&tb1, fp4, static_cast<const uint8_t*>(w13_prep) + P1.codes_off, k1,
                 static_cast<uint64_t>(E) * g1.Np, kBlockN) ||
      !make_tmap(&ta2, false, ws + p.act, k2, L.M, a_box) ||
      !make_tmap(&tb2, fp4, static_cast<const uint8_t*>(w2_prep) + P2.codes_off, k2,
                 static_cast<uint64_t>(E) * g2.Np, kBlockN))
    return MOE_ERR_CUDA;

  auto mark = [&](int i) {
    return events == nullptr || events[i] == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.counts = reinterpret_cast<const int32_t*>(ws + p.counts);
  a.padded_offsets = reinterpret_cast<const int32_t*>(ws + p.padded_offsets);
  a.tiles = reinterpret_cast<const int32_t*>(ws + p.tiles);
  a.row_slot = reinterpret_cast<const int32_t*>(ws + p.row_slot);
  a.row_w = reinterpret_cast<const float*>(ws + L.row_w);
  a.status = reinterpret_cast<uint32_t*>(ws + p.status);
  a.E = E;
  a.I = I;
  a.H = H;
  a.M = L.M;
  a.swiglu_limit = (std::isfinite(swiglu_limit) && swiglu_limit > 0.f) ? swiglu_limit : 0.f;

  GemmArgs a1 = a;
  a1.a_sf = ws + p.xsf;
  a1.w_scale = static_cast<const uint8_t*>(w13_prep) + P1.scale_off;
  a1.out_q = ws + p.act;
  a1.out_sf = ws + p.asf;
  a1.out_cols = mx ? g2.Kp / 2 : g2.Kp;
  a1.out_blocks = g2.KB;
  a1.act_f32 = act_f32;
  a1.g = g1;

  GemmArgs a2 = a;
  a2.a_sf = ws + p.asf;
  a2.w_scale = static_cast<const uint8_t*>(w2_prep) + P2.scale_off;
  a2.out_y = reinterpret_cast<float*>(ws + p.y);
  const bool fuse_combine = fused_combine(fmt, L.S, E);
  if (fuse_combine) {
    a2.inv = reinterpret_cast<const int32_t*>(ws + p.inv);
    a2.combine_cnt = reinterpret_cast<int32_t*>(ws + L.combine_cnt);
    a2.combine_stride = L.combine_stride;
    a2.K = K;
    a2.out = static_cast<__nv_bfloat16*>(out);
  }
  a2.out_cols = H;
  a2.g = g2;

  if (!mark(0)) return MOE_ERR_CUDA;
  if (allow_single_launch && act_f32 == nullptr && single_launch(fmt, L.S, E)) {
    // Small FP4 decode batches: the whole forward in one cooperative launch
    // (the stage events after it are recorded back to back).
    a1.chunk_ready = a2.chunk_ready = reinterpret_cast<int32_t*>(ws + L.chunk_ready);
    a2.ready_target = g1.NT;
    const RqArgs rq = make_rq_args(topk_idx, hidden, topk_w, T, H, E, K, L, ws, out);
    if (launch_single_decode(fmt, ta1, tb1, ta2, tb2, a1, a2, rq, d.sms, st) != cudaSuccess) return MOE_ERR_CUDA;
    for (int i = 1; i <= 5; ++i)
      if (!mark(i)) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // Routing and quantization as two kernels (one kernel for both, which the
  // single launch runs as device code, was slower at every batch size it was
  // measured on: the quantization kernel's dependent launch hides the routing
  // kernel's tail, and each CTA of the fused kernel recomputed the routing).
  if (launch_route(topk_idx, L.S, E, L, ws, st) != cudaSuccess || !mark(1)) return MOE_ERR_CUDA;
  if (launch_quant(fmt, hidden, topk_w, T, H, K, L, ws, out, st) != cudaSuccess || !mark(2)) return MOE_ERR_CUDA;

  if (launch_gemm(fmt, true, decode, ta1, tb1, a1, d.sms, st) != cudaSuccess || !mark(3)) return MOE_ERR_CUDA;

  if (launch_gemm(fmt, false, decode, ta2, tb2, a2, d.sms, st) != cudaSuccess || !mark(4)) return MOE_ERR_CUDA;

  // With the fused combine GEMM2 already wrote the output.
  if (!fuse_combine && launch_combine(reinterpret_cast<const float*>(ws + p.y), reinterpret_cast<const int32_t*>(ws + p.inv),
                                T, H, K, out, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark(5)) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" {

moe_status moe_experts_forward(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T, int H,
                               int I, int E, int K, int fmt, const void* w13_prep, const void* w2_prep,
                               float swiglu_limit, void* workspace, size_t workspace_bytes, void* out,
                               void* stream) {
  return forward_impl(hidden, topk_idx, topk_w, T, H, I, E, K, fmt, w13_prep, w2_prep, swiglu_limit, workspace,
                      workspace_bytes, out, stream, nullptr);
}

moe_status moe_experts_forward_timed(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T,
                                     int H, int I, int E, int K, int fmt, const void* w13_prep,
                                     const void* w2_prep, float swiglu_limit, void* workspace,
                                     size_t workspace_bytes, void* out, void* stream, void* const* events) {
  return forward_impl(hidden, topk_idx, topk_w, T, H, I, E, K, fmt, w13_prep, w2_prep, swiglu_limit, workspace,
                      workspace_bytes, out, stream, events);
}

moe_status moe_debug_forward_act_f32(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T,
                                     int H, int I, int E, int K, int fmt, const void* w13_prep,
                                     const void* w2_prep, float swiglu_limit, void* workspace,
                                     size_t workspace_bytes, void* out, float* act_f32, size_t act_f32_bytes,
                                     void* stream) {
  WsLayout L;
  if (T > 0 && K >= 1 && K <= kMaxTopK && ws_layout(fmt, T, H, I, E, K, &L)) {
    if (act_f32 == nullptr) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(act_f32) % 32) return MOE_ERR_ALIGNMENT;
    if (act_f32_bytes < 4ull * L.M * L.pub.act_cols) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DevInfo d;
    moe_status s = current_device(&d);
    if (s != MOE_OK) return s;
    if ((s = check_ptr(act_f32, d.id)) != MOE_OK) return s;
  }
  return forward_impl(hidden, topk_idx, topk_w, T, H, I, E, K, fmt, w13_prep, w2_prep, swiglu_limit, workspace,
                      workspace_bytes, out, stream, nullptr, act_f32);
}

}  // extern "C"

extern "C" {

moe_status moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || workspace_bytes < 2 * sizeof(uint32_t) || reinterpret_cast<uintptr_t>(workspace) % 4)
    return MOE_ERR_INVALID_ARG;
  DevInfo d;
  moe_status s = current_device(&d);
  if (s != MOE_OK) return s;
  if ((s = check_ptr(workspace, d.id)) != MOE_OK) return s;
  wait_timeout_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(workspace));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_get_device_status(void* workspace, void* stream, uint32_t* flags) {
  if (workspace == nullptr || flags == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  *flags = v;
  return v ? MOE_ERR_DEVICE_FAULT : MOE_OK;
}

}  // extern "C"

/*
 * Block-scaled MoE experts forward for one GB300 (sm_103a): C ABI.
 *
 * The operation is the experts half of a Mixture-of-Experts layer as the
 * transformers integration pages describe it:
 *
 *   - fp8_grouped_mm_experts_forward (source excerpt on the error page
 *     "grouped_mm experts dispatch does not support activation_scheme='static'"): flatten the T*K token-expert pairs, sort them by expert,
 *     gather hidden rows by slot // K, run the grouped block-scaled matmuls
 *     with activations quantized dynamically per block, zero the sentinel
 *     rows, reduce the top-k rows of each token with a deterministic
 *     reshape+sum (no atomics) and cast back to the input dtype;
 *   - "deepgemm_fp8_fp4_experts_forward" (source excerpt of the error record
 *     "DeepGEMM experts selected on a model spanning multiple CUDA devices"):
 *     grouped FP8-activation x FP8/FP4-weight matmuls over a
 *     padded grouped layout (sorted_to_padded), bf16 hidden states only,
 *     static activation scales refused, one CUDA device per call;
 *   - the DeepGEMM Mega MoE forward docstring (source excerpt of the error
 *     record "DeepGEMM Mega MoE requires a process_group for the EP group"):
 *     top-k ids are GLOBAL expert ids and -1 marks a skipped slot;
 *     gate_up / down weights carry UE8M0 scale factors and are transformed
 *     once before the first forward (scale packing and weight interleave);
 *     swiglu_limit is an optional clamp, unclamped when absent.
 *
 * Formats (fixed here, the pages only name them):
 *   MOE_W_FP8: e4m3 weight codes with one fp32 scale per 128x128 block
 *              (weight = code * scale);
 *   MOE_W_FP4: e2m1 codes packed two per byte along K (low nibble = even K
 *              index) with one UE8M0 byte per 1x32 block along K
 *              (weight = code * 2^(byte - 127)).
 *   Activations (hidden and the SwiGLU output) are quantized per 1x128 block
 *   to e4m3 with a power-of-two scale 2^e, e = min{n : amax <= 448 * 2^n}.
 *   MOE_W_FP4_ACT_FP4: the FP4 x FP4 variant (both GEMM operands e2m1, the
 *              tensor cores' FP4 block-scaled MMA): MOE_W_FP4 weights, and
 *              activations quantized per 1x32 block to e2m1 with a UE8M0
 *              exponent n = min{n : amax <= 6 * 2^n} (round to nearest even,
 *              sign of zero kept, two codes per byte, low nibble = even
 *              column). The pages name FP4 x FP4 only as a variant; its
 *              activation rule here is the microscaling rule of the FP4
 *              weights. Results differ from MOE_W_FP4 by the coarser
 *              activation rounding.
 *   SwiGLU: rows [0, I) of w13 are gate, [I, 2I) are up; with a limit L,
 *   gate = min(gate, L) and up = clamp(up, -L, L); act = silu(gate) * up.
 *
 * Conventions for every call:
 *   - all array pointers are DEVICE pointers on the calling thread's current
 *     device unless stated otherwise; weights, prepared weights and the
 *     workspace must be 256-byte aligned, hidden and out 16-byte aligned,
 *     topk_idx and topk_w 4-byte aligned (MOE_ERR_ALIGNMENT otherwise);
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); every device
 *     call is enqueued on it and returns without synchronizing, except
 *     moe_get_device_status;
 *   - nothing is allocated: the caller owns every buffer, including the
 *     workspace, whose size comes from moe_workspace_bytes;
 *   - a non-MOE_OK status means nothing was enqueued;
 *   - element types are not checked here: every array is passed as a plain
 *     pointer, so the caller guarantees the types the calls name (bf16
 *     hidden and out, int32 ids, fp32 routing weights). The Python binding
 *     refuses other dtypes (a non-bf16 hidden state raises ValueError, as
 *     the deepgemm excerpt does) before it calls into this library.
 */
#ifndef BSMOE_MOE_EXPERTS_H_
#define BSMOE_MOE_EXPERTS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer, negative size, T > capacity */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* dimension outside what the kernels take */
  MOE_ERR_UNSUPPORTED_ARCH = 3,   /* device is not compute capability 10.3 */
  MOE_ERR_DEVICE_MISMATCH = 4,    /* a pointer is not memory of the current device */
  MOE_ERR_ALIGNMENT = 5,          /* a pointer breaks its alignment rule (see Conventions) */
  MOE_ERR_WORKSPACE_TOO_SMALL = 6,
  MOE_ERR_CUDA = 7,               /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_FAULT = 8        /* moe_get_device_status found flags set */
} moe_status;

typedef enum {
  MOE_W_FP8 = 0,         /* e4m3 + fp32 128x128 block scales */
  MOE_W_FP4 = 1,         /* e2m1 packed in bytes + UE8M0 1x32 block scales */
  MOE_W_FP4_ACT_FP4 = 2  /* MOE_W_FP4 weights with e2m1 1x32 activations */
} moe_wfmt;

/* Sticky flags in the workspace status word (moe_get_device_status). */
#define MOE_DEV_BAD_EXPERT_ID 0x1u /* an id outside [-1, E): treated as skipped */
#define MOE_DEV_TIMEOUT 0x2u       /* a pipeline wait gave up; outputs invalid */

/* Human-readable name of a status code; never NULL. */
const char* moe_status_string(int status);

/* MOE_ABI_VERSION of the loaded library. */
int moe_abi_version(void);

/*
 * Supported shapes: 1 <= E <= 512, 1 <= K <= 32, H and I multiples of 64
 * (multiples of 128 for MOE_W_FP8, whose weight blocks are 128x128; the
 * FP4 formats take multiples of 64),
 * 128 <= H, I <= 32768. T may be 0 (nothing is enqueued).
 */

/*
 * Bytes of the prepared (kernel-layout) weights made by moe_prepare_weights.
 * Returns 0 for an unsupported shape or format.
 */
size_t moe_prepared_w13_bytes(int fmt, int E, int H, int I);
size_t moe_prepared_w2_bytes(int fmt, int E, int H, int I);

/*
 * Bytes of workspace a forward with up to T_max tokens needs. A workspace of
 * this size serves every call with T <= T_max and the same (fmt, H, I, E, K).
 * Returns 0 for an unsupported shape.
 */
size_t moe_workspace_bytes(int fmt, int T_max, int H, int I, int E, int K);

/*
 * One-shot weight transform, the analogue of the Mega MoE "pack UE8M0 SFs
 * and interleave the L1/L2 weights" first-forward step (made explicit here
 * instead of lazy). Reads the checkpoint-layout weights and writes the
 * kernel layout: gate/up rows interleaved in 64-row groups, K padded to a
 * multiple of 128 and N to a multiple of 256 with zeros, scale factors
 * rearranged into the layout the tensor-core pipeline stages.
 *
 * Inputs (read only, device):
 *   MOE_W_FP8: w13 u8 [E, 2I, H], w13_scale f32 [E, 2I/128, H/128],
 *              w2  u8 [E, H, I],  w2_scale  f32 [E, H/128, I/128];
 *   MOE_W_FP4: w13 u8 [E, 2I, H/2], w13_scale u8 [E, 2I, H/32],
 *              w2  u8 [E, H, I/2],  w2_scale  u8 [E, H, I/32];
 *   MOE_W_FP4_ACT_FP4: as MOE_W_FP4 (same inputs, same prepared bytes).
 * Outputs (device, caller-owned): w13_prep of moe_prepared_w13_bytes,
 *   w2_prep of moe_prepared_w2_bytes. Their content is opaque.
 * Errors: MOE_ERR_INVALID_ARG / UNSUPPORTED_SHAPE / ALIGNMENT /
 *   DEVICE_MISMATCH / UNSUPPORTED_ARCH / WORKSPACE_TOO_SMALL (an output
 *   buffer smaller than required) / CUDA.
 */
moe_status moe_prepare_weights(int fmt, int E, int H, int I, const void* w13, const void* w13_scale,
                               const void* w2, const void* w2_scale, void* w13_prep, size_t w13_prep_bytes,
                               void* w2_prep, size_t w2_prep_bytes, void* stream);

/*
 * The same transform for expert weights stored transposed, N contiguous
 * (the `is_transposed` storage that the experts dispatch serves with
 * grouped_fp8_fp4_matmul_nn instead of _nt: the deepgemm_fp8_fp4_experts_forward
 * source excerpt). Writes exactly the bytes moe_prepare_weights writes for
 * the same weights in the K-major storage, so the forward does not change.
 *
 * Inputs (read only, device):
 *   MOE_W_FP8: w13 u8 [E, H, 2I], w13_scale f32 [E, H/128, 2I/128],
 *              w2  u8 [E, I, H],  w2_scale  f32 [E, I/128, H/128];
 *   MOE_W_FP4: w13 u8 [E, H, 2I/2] (two codes per byte along N, low nibble
 *              = even N index), w13_scale u8 [E, H/32, 2I] (UE8M0 per 32 K
 *              of one N column), w2 u8 [E, I, H/2], w2_scale u8 [E, I/32, H].
 * Outputs, ownership and errors as moe_prepare_weights.
 */
moe_status moe_prepare_weights_transposed(int fmt, int E, int H, int I, const void* w13, const void* w13_scale,
                                          const void* w2, const void* w2_scale, void* w13_prep,
                                          size_t w13_prep_bytes, void* w2_prep, size_t w2_prep_bytes,
                                          void* stream);

/*
 * The experts forward:
 *   out[t, :] = bf16( sum_{k : idx[t,k] valid} w[t,k] * FFN_{idx[t,k]}(x[t, :]) )
 * summed in ascending k in fp32 (deterministic, no atomics); a token whose
 * slots are all skipped gets +0.
 *
 *   hidden    bf16 [T, H] (row-major), device
 *   topk_idx  int32 [T, K] global expert ids, -1 = skipped slot
 *   topk_w    fp32 [T, K] routing weights (ignored for skipped slots)
 *   w13_prep, w2_prep  from moe_prepare_weights with the same (fmt, E, H, I)
 *   swiglu_limit  clamp L; NaN or <= 0 means unclamped
 *   workspace  >= moe_workspace_bytes(fmt, T, H, I, E, K) bytes, device
 *   out       bf16 [T, H], device; must not overlap any input
 *
 * Ids outside [-1, E) are treated as skipped and set MOE_DEV_BAD_EXPERT_ID.
 * Asynchronous; the workspace must not be used by another call until this
 * one has finished on `stream`.
 *
 * Launches: routing, quantization, GEMM1, GEMM2 and the combine (inside
 * GEMM2 for FP4 weights with T*K <= 256 and T*K <= 8E); for FP4
 * weights with T*K <= 8E (the weight-streaming decode batches) and
 * T*K <= 32 the whole forward is one cooperative launch of one CTA per SM
 * (GEMM2 work units wait on device counters for the GEMM1 units of their
 * rows), which needs every SM of the device free for the launch.
 * MOE_W_FP4_ACT_FP4 follows MOE_W_FP4 (decode mode, the single launch; the
 * combine in GEMM2 for T*K <= 64 with this format).
 */
moe_status moe_experts_forward(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T, int H,
                               int I, int E, int K, int fmt, const void* w13_prep, const void* w2_prep,
                               float swiglu_limit, void* workspace, size_t workspace_bytes, void* out,
                               void* stream);

/*
 * The same forward, doing the same work, that also records events[i]
 * (cudaEvent_t values created by the caller; a NULL entry is skipped) on
 * `stream` at the stage boundaries: 0 before routing, 1 after routing,
 * 2 after the input quantization, 3 after GEMM1 (+SwiGLU epilogue),
 * 4 after GEMM2, 5 after the combine. `events` points to 6 entries (host
 * memory). Where stages share a kernel the events between them are recorded
 * back to back: GEMM2 and the combine for FP4 weights with T*K <= 8E and
 * T*K <= 256 (T*K <= 64 for MOE_W_FP4_ACT_FP4) (events 4 and 5), and every stage
 * for FP4 weights with T*K <= 32 and T*K <= 8E, which run as one launch
 * (events 1 to 5 after it). Meant for
 * measuring the stages; errors as moe_experts_forward.
 */
moe_status moe_experts_forward_timed(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T,
                                     int H, int I, int E, int K, int fmt, const void* w13_prep,
                                     const void* w2_prep, float swiglu_limit, void* workspace,
                                     size_t workspace_bytes, void* out, void* stream, void* const* events);

/*
 * The forward for callers that cannot allocate device memory (for example a
 * host runtime that owns every device allocation and only lends out model
 * tensors, or code running where allocation is not allowed). It takes no
 * workspace: its scratch memory is one fixed device array inside this
 * library, moe_static_workspace_capacity() bytes (64 MiB) on every GPU that
 * loads the library, held until the process exits. The transformers pages
 * have no counterpart of this call; it exists for such callers only.
 *
 * Arguments and results are those of moe_experts_forward minus the
 * workspace. A call whose moe_workspace_bytes(fmt, T, H, I, E, K) exceeds the
 * capacity returns MOE_ERR_WORKSPACE_TOO_SMALL and enqueues nothing (at the
 * DeepSeek-V3 shape, for instance, single-token decode fits and large
 * batches do not). No cudaMalloc, cudaFree or other allocating routine is
 * called.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before capturing a stream. The address is kept per device and looked up
 * again when the device's context has changed (for example after
 * cudaDeviceReset, which reloads the library's device code). Every call
 * shares the one array, and its content is whatever the last call left
 * there: the forward writes every part it reads before reading it, so
 * nothing needs clearing, but calls that overlap on the GPU (other streams,
 * other host threads) race on it and must be serialized by the caller.
 * The flags such a call raises (MOE_DEV_BAD_EXPERT_ID, MOE_DEV_TIMEOUT) sit
 * in the array's status word: read them with moe_static_get_device_status.
 */
moe_status moe_experts_forward_static(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T,
                                      int H, int I, int E, int K, int fmt, const void* w13_prep,
                                      const void* w2_prep, float swiglu_limit, void* out, void* stream);

/* Bytes of the fixed device array used by moe_experts_forward_static. */
size_t moe_static_workspace_capacity(void);

/*
 * moe_get_device_status for the fixed array of moe_experts_forward_static on
 * the current device: synchronizes `stream`, reads the flags raised by the
 * most recent static forward into *flags (host pointer) and clears them.
 * Returns MOE_ERR_DEVICE_FAULT when a flag was set, MOE_OK otherwise,
 * MOE_ERR_INVALID_ARG for a null `flags`, MOE_ERR_CUDA if a CUDA call fails.
 * Like the forward it allocates nothing; it must not overlap a static
 * forward running on another stream.
 */
moe_status moe_static_get_device_status(void* stream, uint32_t* flags);

/*
 * Synchronizes `stream` and reads the status word of `workspace` into *flags
 * (host pointer), then clears it. The word holds the flags raised by the most
 * recent forward that used this workspace (each forward starts by clearing
 * it). Returns MOE_ERR_DEVICE_FAULT when a flag was set, MOE_OK otherwise.
 */
moe_status moe_get_device_status(void* workspace, void* stream, uint32_t* flags);

/*
 * Self-test of the failure path of the bounded waits. Enqueues on `stream`
 * one CTA in which one thread waits, through the same bounded mbarrier wait
 * the GEMMs use, on a phase that nothing completes, and another waits,
 * through the same bounded counter wait the single-launch forward's GEMM2
 * units use, for the second word of `workspace` (set to 0 first) to reach 1,
 * which nothing does. After their bound (2e9 SM clock cycles, about one
 * second) the waits give up and the kernel ORs MOE_DEV_TIMEOUT into the
 * status word of `workspace` (its first 4 bytes; 8 bytes of device memory of
 * the current device, 4-byte aligned) and returns; the context stays usable.
 * Read the result with moe_get_device_status.
 * Returns MOE_ERR_INVALID_ARG for a null, short or misaligned workspace,
 * MOE_ERR_DEVICE_MISMATCH for memory of another device or the host,
 * MOE_ERR_UNSUPPORTED_ARCH off sm_103, MOE_ERR_CUDA if the launch fails.
 */
moe_status moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Byte offsets of the forward's intermediate results inside the workspace,
 * for inspection after a forward (tests compare them with the oracle).
 * All regions are int32 unless noted; M = padded row capacity.
 *   counts [E]; offsets [E+1] (exclusive scan of counts);
 *   padded_offsets [E+1] (group starts, multiples of row_align);
 *   perm [S] (sorted position -> slot, skipped slots last);
 *   inv [S] (slot -> padded row, -1 if skipped);
 *   row_slot [M] (padded row -> slot, -1 for padding rows);
 *   tiles [16 + 2 (E+1) + M/128 + M/32] (GEMM work lists): [0] number of
 *     128-row m-tiles, [1] number of 32-row chunks, [16 + e] first m-tile
 *     and [16 + E + 1 + e] first chunk of expert e (E+1 entries each), then
 *     the expert owning each m-tile, then the expert owning each chunk;
 *   xq u8 [M, xq_cols] (e4m3 hidden rows in grouped order; for
 *     MOE_W_FP4_ACT_FP4 u8 [M, xq_cols / 2], e2m1 codes two per byte);
 *   xsf u32 (activation scale words, see below);
 *   act u8 [M, act_cols] (e4m3 SwiGLU output; for MOE_W_FP4_ACT_FP4
 *     u8 [M, act_cols / 2] e2m1), asf u32 likewise;
 *   y f32 [M, H] (weighted per-pair outputs).
 * xq_cols and act_cols count elements (H and I padded to 128).
 * Scale words: for row r and 128-column block b the word sits at index
 *   ((r / 128) * nblk + b) * 128 + 4 * (r % 32) + (r % 128) / 32
 * and holds the UE8M0 byte (e + 127) replicated in all four bytes; for
 * MOE_W_FP4_ACT_FP4 byte j holds the exponent byte (n + 127) of the 1x32
 * sub-block j of the 128 columns.
 */
typedef struct {
  size_t total_bytes;
  size_t status, counts, offsets, padded_offsets, perm, inv, row_slot, tiles;
  size_t xq, xsf, act, asf, y;
  int32_t row_capacity;  /* M */
  int32_t row_align;     /* group alignment A */
  int32_t xq_cols, act_cols;
  int32_t x_blocks, act_blocks; /* ceil(H/128), ceil(I/128) */
} moe_workspace_layout;

moe_status moe_query_workspace_layout(int fmt, int T, int H, int I, int E, int K, moe_workspace_layout* layout);

/*
 * Debug tap for tests: the forward of moe_experts_forward (same arguments,
 * same results) run as the multi-kernel sequence (routing, quantization,
 * GEMM1, GEMM2, combine as separate launches, also for the small FP4 decode
 * batches that moe_experts_forward runs as one launch), which also stores,
 * from GEMM1's epilogue, the
 * fp32 SwiGLU values it requantizes -- act = silu(gate) * up after the
 * optional clamp -- so that the requantized bytes (workspace regions act and
 * asf) can be checked bit for bit against the 1x128 rule (the 1x32 e2m1 rule
 * for MOE_W_FP4_ACT_FP4) applied to exactly these values. Row r of the padded grouped layout goes to
 * act_f32[r * act_cols + j], j < act_cols (moe_query_workspace_layout;
 * columns j >= I hold 0); padding rows are not written.
 *   act_f32  device fp32, >= row_capacity * act_cols * 4 bytes, 32-byte
 *            aligned (MOE_ERR_INVALID_ARG if null, MOE_ERR_ALIGNMENT,
 *            MOE_ERR_WORKSPACE_TOO_SMALL if short).
 * Other errors as moe_experts_forward. The extra stores make GEMM1 slower:
 * not for timing.
 */
moe_status moe_debug_forward_act_f32(const void* hidden, const int32_t* topk_idx, const float* topk_w, int T,
                                     int H, int I, int E, int K, int fmt, const void* w13_prep,
                                     const void* w2_prep, float swiglu_limit, void* workspace,
                                     size_t workspace_bytes, void* out, float* act_f32, size_t act_f32_bytes,
                                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSMOE_MOE_EXPERTS_H_ */

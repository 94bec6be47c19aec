// A forward that allocates nothing and takes no workspace argument.
//
// Some callers cannot allocate device memory at the point where they run the
// experts forward: a host runtime that owns all device allocations and hands
// out only the tensors of the model, a plugin called inside a region where
// allocation is forbidden, or a C caller without a device allocator of its
// own. For them the scratch memory of the forward lives in one file-scope
// device array of fixed size, kStaticWorkspaceBytes, which every GPU that
// loads this library holds until the process exits. Calls larger than that
// are refused with MOE_ERR_WORKSPACE_TOO_SMALL.
#include <mutex>

#include "moe_internal.cuh"

namespace bsmoe {

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
struct CachedAddr {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
};
CachedAddr g_workspace_addr[kMaxDevices];
std::mutex g_workspace_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id (for the life of the process) of the calling thread's current
// context, 0 when there is none or the driver cannot say.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the array on the current device. In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, with that device current. It is looked up once per
// device and context: if the context is destroyed and made again (for
// example after cudaDeviceReset) the module is loaded again and the array
// may move, so a changed context id triggers a new lookup.
moe_status static_workspace(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE_MISMATCH;
  std::lock_guard<std::mutex> lock(g_workspace_mu);
  CachedAddr& c = g_workspace_addr[dev];
  const unsigned long long id = current_ctx_id();
  if (c.ptr == nullptr || id == 0 || id != c.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    c.ptr = p;
    // the lookup has made the context current if it was not yet
    c.ctx_id = current_ctx_id();
  }
  *addr = c.ptr;
  return MOE_OK;
}

}  // namespace

}  // namespace bsmoe

extern "C" size_t moe_static_workspace_capacity(void) { return bsmoe::kStaticWorkspaceBytes; }

extern "C" moe_status moe_experts_forward_static(const void* hidden, const int32_t* topk_idx, const float* topk_w,
                                                 int T, int H, int I, int E, int K, int fmt,
                                                 const void* w13_prep, const void* w2_prep, float swiglu_limit,
                                                 void* out, void* stream) {
  using namespace bsmoe;
  // the same checks, in the same order, as moe_experts_forward
  if (T < 0 || K < 1 || K > kMaxTopK) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_bytes(fmt, T, H, I, E, K);
  if (need == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (need > kStaticWorkspaceBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (T == 0) return MOE_OK;
  void* ws = nullptr;
  const moe_status s = static_workspace(&ws);
  if (s != MOE_OK) return s;
  return forward_impl(hidden, topk_idx, topk_w, T, H, I, E, K, fmt, w13_prep, w2_prep, swiglu_limit, ws,
                      kStaticWorkspaceBytes, out, stream, nullptr);
}

extern "C" moe_status moe_static_get_device_status(void* stream, uint32_t* flags) {
  using namespace bsmoe;
  if (flags == nullptr) return MOE_ERR_INVALID_ARG;
  void* ws = nullptr;
  const moe_status s = static_workspace(&ws);
  if (s != MOE_OK) return s;
  return moe_get_device_status(ws, stream, flags);
}

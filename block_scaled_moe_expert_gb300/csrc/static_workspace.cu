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
void* g_workspace_addr[kMaxDevices] = {};
std::mutex g_workspace_mu;

// Device address of the array on the current device. In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
moe_status static_workspace(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE_MISMATCH;
  std::lock_guard<std::mutex> lock(g_workspace_mu);
  if (g_workspace_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_workspace_addr[dev] = p;
  }
  *addr = g_workspace_addr[dev];
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
  const size_t need = moe_workspace_bytes(fmt, T, H, I, E, K);
  if (need == 0) return (T < 0 || K < 1) ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  if (need > kStaticWorkspaceBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (T == 0) return MOE_OK;
  void* ws = nullptr;
  const moe_status s = static_workspace(&ws);
  if (s != MOE_OK) return s;
  return forward_impl(hidden, topk_idx, topk_w, T, H, I, E, K, fmt, w13_prep, w2_prep, swiglu_limit, ws,
                      kStaticWorkspaceBytes, out, stream, nullptr);
}

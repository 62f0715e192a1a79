// mla_noalloc.cu -- decode for callers that cannot allocate device memory.
//
// mla_decode needs a caller-provided workspace (split plan, per-split partial outputs,
// status word). Some callers cannot obtain one: an inference engine that has reserved
// nearly all device memory for its own pools before this library is loaded, or a
// latency-critical loop that must not call cudaMalloc/cudaFree because they can
// synchronise the whole device. For them this file keeps one fixed-size workspace in a
// file-scope __device__ array and runs the ordinary decode path on it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "mla_internal.cuh"

namespace {

// The library-owned workspace. Every GPU on which this module is loaded holds these
// MLA_STATIC_WS_BYTES of device memory until the process exits.
static __device__ __align__(256) unsigned char g_static_ws[MLA_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
// Per device: the context the address was looked up in, and the address. A device reset
// (or a primary context destroyed and created again) reloads the module, possibly at
// another address, so the address is looked up again whenever the context changes.
CUcontext g_ws_ctx[kMaxDevices] = {nullptr};
void* g_ws_ptr[kMaxDevices] = {nullptr};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no link-time dependency on the
// driver library).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

// Device address of g_static_ws on `device`, which must be current. In host code the name
// g_static_ws is only a host-side stand-in, so the real address is looked up with
// cudaGetSymbolAddress the first time a device (in its current context) is seen, and
// cached.
void* static_ws_address(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (ctx && g_ws_ptr[device] && g_ws_ctx[device] == ctx) return g_ws_ptr[device];
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  // the symbol query made the device's primary context current if nothing was yet
  if (get(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
  g_ws_ptr[device] = ptr;
  g_ws_ctx[device] = ctx;
  return ptr;
}

}  // namespace

extern "C" mla_status_t mla_decode_static_ws(const mla_kv_t* kv, const void* q, int B, int H,
                                             float sm_scale, void* out, float* lse,
                                             void* stream) {
  if (B < 0 || H < 1 || H > MLA_MAX_HEADS) return (B < 0) ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const size_t need = mla_workspace_size(MLA_OP_DECODE, B, H, 1, device);
  if (need == 0) return MLA_ERR_CUDA;
  if (need > MLA_STATIC_WS_BYTES) return MLA_ERR_WORKSPACE;  // batch too large for the fixed workspace
  void* ws = static_ws_address(device);
  if (!ws) return MLA_ERR_CUDA;
  return mla_decode(kv, q, B, H, sm_scale, out, lse, ws, MLA_STATIC_WS_BYTES, stream);
}

extern "C" mla_status_t mla_read_status_static(void* stream) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  void* ws = static_ws_address(device);
  if (!ws) return MLA_ERR_CUDA;
  return mla_read_status(ws, MLA_STATIC_WS_BYTES, stream);
}

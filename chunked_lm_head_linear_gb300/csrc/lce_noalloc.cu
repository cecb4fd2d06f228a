// lce_forward_noalloc: the forward (loss and lse) for callers that cannot
// allocate device memory. Its scratch lives in a fixed array in this
// library's device image instead of a caller-provided workspace.
//
// Who needs it: code whose device memory is entirely owned by another
// allocator (a framework's caching pool or an inference runtime's arena that
// has reserved the free memory), where a side cudaMalloc either fails or is
// not permitted, and code that must not call cudaMalloc / cudaFree because
// those calls can block or synchronise the device. Such a caller still owns
// the inputs and outputs; only the scratch moves into the library.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes. Every
// GPU that loads this library holds it until the process exits. Host code
// must not pass the array's name to a kernel: on the host that name is a
// stand-in, not a device address. The device address belongs to one CUDA
// context: the runtime loads this library's device image into each context
// separately (the device's primary context, a context the caller created
// with the driver API, the new primary context after cudaDeviceReset), each
// copy at its own address. So the address is looked up with
// cudaGetSymbolAddress once per context, with that context current, and
// cached under the context's unique id (never reused within a process), not
// under the device number.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "../../include/lce.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverCalls {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverCalls& driver_calls() {
  static DriverCalls calls;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      calls.get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      calls.get_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  return calls;
}

std::mutex g_mu;
std::unordered_map<unsigned long long, void*> g_scratch_by_ctx;  // context id -> device address

// Device address of the scratch array in the calling thread's current context
// (looked up on the first call in each context).
int scratch_address(void** out) {
  const DriverCalls& dc = driver_calls();
  if (dc.get_current == nullptr || dc.get_id == nullptr) return LCE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (dc.get_current(&ctx) != CUDA_SUCCESS) return LCE_ERR_CUDA;
  if (ctx == nullptr) {
    // No context yet on this thread: the runtime's first call makes the
    // current device's primary context current.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return LCE_ERR_CUDA;
    if (dc.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return LCE_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (dc.get_id(ctx, &id) != CUDA_SUCCESS) return LCE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_scratch_by_ctx.find(id);
  if (it == g_scratch_by_ctx.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LCE_ERR_CUDA;
    it = g_scratch_by_ctx.emplace(id, p).first;
  }
  *out = it->second;
  return LCE_OK;
}

}  // namespace

extern "C" int lce_forward_noalloc(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                                   float* loss, float* lse, const lce_opts* opts, void* stream) {
  const size_t need = lce_workspace_size(LCE_OP_FORWARD, N, d, V, opts);
  if (need == 0) return LCE_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return LCE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != LCE_OK) return rc;
  return lce_forward(H, W, y, N, d, V, loss, lse, opts, scratch, kNoAllocScratchBytes, stream);
}

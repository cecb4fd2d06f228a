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
// stand-in, not a device address. The device address is looked up once per
// device with cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/lce.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LCE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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

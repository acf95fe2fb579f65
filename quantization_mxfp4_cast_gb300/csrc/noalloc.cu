// gemm_fp4_bf16_fwd_noalloc: the bf16 forward MXFP4 GEMM for callers that
// cannot allocate device memory.
//
// Some callers have no way to get a workspace buffer: code that runs where
// CUDA allocation calls are not allowed (for example a host function enqueued
// on a stream, which must not make CUDA API calls that allocate), or a plugin
// whose device memory belongs to the host framework's allocator and which is
// handed only its inputs and outputs.  This entry point needs no workspace:
// the quantized copies of X and W live in one file-scope device array of
// MXFP4_NOALLOC_SCRATCH_BYTES, which every GPU that loads this library holds
// until the process exits.  The operation itself is exactly
// gemm_fp4_bf16_fwd; it has no counterpart on the pages.
//
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the first call on each device, with that
// device current, looks up the address with cudaGetSymbolAddress and caches
// it.  That first call should come before any stream capture.  Every call
// shares the one array and overwrites it completely (codes and every scale
// byte, padding included), so nothing has to start at zero; calls whose work
// overlaps on the GPU (different streams, or several host threads) race on it.
#include <mutex>

#include "../../include/mxfp4.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = MXFP4_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
mxfp4_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXFP4_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXFP4_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MXFP4_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MXFP4_OK;
}

}  // namespace

extern "C" mxfp4_status gemm_fp4_bf16_fwd_noalloc(const uint16_t* x, const uint16_t* w,
                                                   uint16_t* y, int64_t M, int64_t N, int64_t K,
                                                   void* stream) {
  if (M < 0 || N < 0 || K < 0) return MXFP4_ERR_INVALID_ARG;
  if (mxfp4_workspace_bytes(MXFP4_OP_FWD, M, N, K) > kScratchBytes) return MXFP4_ERR_WORKSPACE;
  if (y == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (M > 0 && N > 0) {  // scratch of the device that holds the output
    const cudaError_t e = mxfp4::bind_device_of(y);
    if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;
    if (e != cudaSuccess) return MXFP4_ERR_CUDA;
  }
  void* scratch = nullptr;
  const mxfp4_status st = scratch_address(&scratch);
  if (st != MXFP4_OK) return st;
  return gemm_fp4_bf16_fwd(x, w, y, M, N, K, scratch, kScratchBytes, stream);
}

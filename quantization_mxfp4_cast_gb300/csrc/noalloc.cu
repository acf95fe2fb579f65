// gemm_fp4_bf16_fwd_noalloc: the bf16 forward MXFP4 GEMM for callers that
// cannot allocate device memory.
//
// Some callers have no way to get a workspace buffer: a plugin or extension
// whose device memory all belongs to the host framework's caching allocator
// and which is handed only its inputs and outputs, or code that must not
// make allocating CUDA calls at the point where it runs.  This entry point
// needs no workspace: the quantized copies of X and W live in one file-scope
// device array of MXFP4_NOALLOC_SCRATCH_BYTES.  The operation itself is
// exactly gemm_fp4_bf16_fwd; it has no counterpart on the pages.
//
// The array is part of this file's device module.  CUDA loads modules
// lazily by default, so the first call on each device loads it: that load
// is where the array's 32 MiB of device memory is taken, and it fails (the
// call returns MXFP4_ERR_CUDA, cudaErrorMemoryAllocation in
// mxfp4_last_cuda_error) if the device is already full.  Make the first call
// on each device early -- before the framework reserves its memory pool, and
// before any stream capture.  Every later call allocates nothing.
//
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so that first call, with the device current,
// also looks up the address with cudaGetSymbolAddress and caches it.  Every
// call shares the one array and overwrites it completely (codes and every
// scale byte, padding included), so nothing has to start at zero; calls
// whose work overlaps on the GPU (different streams, or several host
// threads) race on it.
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
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<mxfp4_status>(mxfp4::status_from_cuda(e));
  if (dev < 0 || dev >= kMaxDevices) return MXFP4_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<mxfp4_status>(mxfp4::status_from_cuda(e));
    if (p == nullptr) return MXFP4_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MXFP4_OK;
}

}  // namespace

extern "C" mxfp4_status gemm_fp4_bf16_fwd_noalloc(const uint16_t* x, const uint16_t* w,
                                                   uint16_t* y, int64_t M, int64_t N, int64_t K,
                                                   void* stream) {
  // gemm_fp4_bf16_fwd's own argument checks and order, then the array's limit
  const mxfp4_status st = static_cast<mxfp4_status>(mxfp4::check_fwd_args(x, w, y, M, N, K));
  if (st != MXFP4_OK || M == 0 || N == 0) return st;
  if (mxfp4_workspace_bytes(MXFP4_OP_FWD, M, N, K) > kScratchBytes) return MXFP4_ERR_WORKSPACE;
  // the scratch array of the device that holds the output
  const cudaError_t e = mxfp4::bind_device_of(y);
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;  // not device memory
  if (e != cudaSuccess) return static_cast<mxfp4_status>(mxfp4::status_from_cuda(e));
  void* scratch = nullptr;
  const mxfp4_status sa = scratch_address(&scratch);
  if (sa != MXFP4_OK) return sa;
  return gemm_fp4_bf16_fwd(x, w, y, M, N, K, scratch, kScratchBytes, stream);
}

// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxfp4 {

constexpr uint32_t kFlagHadamardRow = 1u;
constexpr uint32_t kFlagHadamardCol = 2u;
constexpr uint32_t kFlagScaleLinear = 4u;
constexpr uint32_t kFlagFp8 = 1u << 16;  // internal: E4M3 elements (column output only)

struct CastArgs {
  const uint16_t* x;  // bf16 bits [rows, cols], pitch ldx
  int64_t rows, cols, ldx;
  uint8_t* q_row;   // [rows, cols/2] or null (no row-wise output)
  uint8_t* sf_row;  // scales of the row-wise output
  uint8_t* q_col;   // [cols, rows/2] or null (no column-wise output)
  uint8_t* sf_col;  // scales of the column-wise output
  uint32_t flags;
};

// One launch over 128 x 128 tiles of x; writes whichever outputs are non-null.
cudaError_t launch_cast(const CastArgs& args, cudaStream_t stream);
// Up to 4 casts of one kind (the same outputs and element format; each its
// own shape and Hadamard flags) in one launch, their tiles numbered one cast
// after another; cudaErrorInvalidValue for count outside 1..4 or mixed kinds.
cudaError_t launch_cast_grouped(const CastArgs* list, int count, cudaStream_t stream);

// Makes the device that holds `data` current in this library's CUDA runtime
// for the calling thread (binding its primary context); cudaErrorInvalidValue
// if `data` is not device memory.
cudaError_t bind_device_of(const void* data);

struct GemmArgs {
  const uint8_t* a;     // codes [M, K/2]
  const uint8_t* a_sf;  // tiled scales, M rows x K/32 blocks
  const uint8_t* b;     // codes [N, K/2]
  const uint8_t* b_sf;  // tiled scales, N rows x K/32 blocks
  uint16_t* c;          // bf16 [M, N], pitch ldc
  int64_t M, N, K, ldc;
};

cudaError_t launch_gemm(const GemmArgs& args, cudaStream_t stream);
// Up to 4 independent GEMMs in one persistent launch (their tiles numbered
// one after the other); cudaErrorInvalidValue for count outside 1..4.
cudaError_t launch_gemm_grouped(const GemmArgs* list, int count, cudaStream_t stream);

// The MXFP4 dual cast of the GEMM's own bf16 output, written by its epilogue.
struct CastOutArgs {
  uint8_t* q_row;   // codes [M, N/2] of C quantized along N, or null
  uint8_t* sf_row;  // its tile-layout scales (null iff q_row is)
  uint8_t* q_col;   // codes [N, M/2] of C^T quantized along M, or null
  uint8_t* sf_col;  // its tile-layout scales (null iff q_col is)
  uint32_t flags;   // kFlagHadamardRow, kFlagHadamardCol
};
// Requires M % 32 == 0 and N % 32 == 0.  args.c may be null (no bf16 C is
// written) when at least one cast output is given.
cudaError_t launch_gemm_cast_out(const GemmArgs& args, const CastOutArgs& out, cudaStream_t stream);
// Self-test of the bounded waits: the MXFP4 GEMM with the given wait limit and
// its first "stage ready" signal withheld, so that a wait runs out, the
// kernel records MXFP4_ERR_TIMEOUT in the status word and every role leaves
// (after its loads and MMAs in flight have completed).  C is not written.
cudaError_t launch_gemm_selftest_timeout(const GemmArgs& args, unsigned long long wait_limit_ns,
                                         cudaStream_t stream);
// The same GEMM on MXFP8 (E4M3) operands: codes [rows, K] bytes, same scale layout.
cudaError_t launch_gemm_mxfp8(const GemmArgs& args, cudaStream_t stream);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (so the library needs no link-time dependency on libcuda); null if missing.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Device address of the library's status word on the current device (looked
// up once per device); null on failure.  Kernels with bounded waits record
// MXFP4_ERR_TIMEOUT there.
int* device_status_word();

// Reads (and optionally clears) the device status word.  Synchronous.
cudaError_t read_device_status(int* value, bool reset);

// Records e as the calling thread's last CUDA error (mxfp4_last_cuda_error)
// and returns the matching status: MXFP4_OK or MXFP4_ERR_CUDA.
int status_from_cuda(cudaError_t e);

// The argument checks gemm_fp4_bf16_fwd runs before its workspace check, in
// the same order; MXFP4_OK also when M == 0 or N == 0 (nothing to launch).
int check_fwd_args(const uint16_t* x, const uint16_t* w, const uint16_t* y, int64_t M, int64_t N, int64_t K);

// Zero-fill of a bf16 matrix (used when K == 0).
cudaError_t launch_fill_zero_bf16(uint16_t* c, int64_t M, int64_t N, int64_t ldc,
                                  cudaStream_t stream);

}  // namespace mxfp4

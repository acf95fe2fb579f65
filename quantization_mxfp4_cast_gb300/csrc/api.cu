// C ABI of the MXFP4 library (declared in include/mxfp4.h): argument
// validation on the host, workspace carving, and launches on the caller's
// stream.  Nothing here allocates memory or synchronizes (except
// mxfp4_device_status, which reads the device status word).
//
// Operations: jax-aiter README, "Supported ops" table (MXFP4 Cast, FP4 GEMM
// low-level, FP4 GEMM training) and "MXFP4 training architecture" (forward =
// activation cast + weight cast + GEMM; backward = gradient cast + dA GEMM,
// plus the dB GEMM).
#include <algorithm>
#include <atomic>

#include "../../include/mxfp4.h"
#include "internal.h"
#include "ptx.cuh"

using mxfp4::CastArgs;
using mxfp4::GemmArgs;

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 31;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The CUDA error behind this thread's last MXFP4_ERR_CUDA.
thread_local int t_last_cuda_error = 0;

mxfp4_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MXFP4_OK;
  t_last_cuda_error = static_cast<int>(e);
  return MXFP4_ERR_CUDA;
}

}  // namespace

int mxfp4::status_from_cuda(cudaError_t e) { return from_cuda(e); }

// This library links its own CUDA runtime, whose per-thread current device is
// separate from the caller's (torch's) runtime: a thread that torch created
// (an autograd worker, say) may have no current context here at all, and
// the tensor-map encode is a driver call that needs one.  So every entry
// point makes the device that holds its data current in this runtime, which
// also binds that device's primary context to the calling thread.
cudaError_t mxfp4::bind_device_of(const void* data) {
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, data);
  if (e != cudaSuccess) return e;
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return cudaErrorInvalidValue;
  return cudaSetDevice(attr.device);
}

namespace {

// Binds the data's device (above), which must be compute capability 10.3.
// The answer per device is cached (it cannot change within a process):
// 0 unknown, 1 yes, 2 no.
mxfp4_status check_device(const void* data) {
  static std::atomic<int> known[64];
  cudaError_t e = mxfp4::bind_device_of(data);
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;  // not device memory
  if (e != cudaSuccess) return from_cuda(e);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  int k = (dev >= 0 && dev < 64) ? known[dev].load(std::memory_order_relaxed) : 0;
  if (k == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return from_cuda(e);
    k = (major == 10 && minor == 3) ? 1 : 2;
    if (dev >= 0 && dev < 64) known[dev].store(k, std::memory_order_relaxed);
  }
  return k == 1 ? MXFP4_OK : MXFP4_ERR_UNSUPPORTED_DEVICE;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t tile_scale_bytes(int64_t rows, int64_t cols) {
  return static_cast<size_t>(ceil_div(rows, 128) * ceil_div(cols / 32, 4) * 512);
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Common checks of a bf16 input tensor.
mxfp4_status check_bf16_in(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return MXFP4_ERR_INVALID_ARG;
  if (cols % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (ldx < cols) return MXFP4_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MXFP4_OK;
  if (x == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx % 8) != 0) return MXFP4_ERR_MISALIGNED;
  if (ceil_div(rows, 128) > 65535) return MXFP4_ERR_INVALID_ARG;  // grid.y limit
  return MXFP4_OK;
}

mxfp4_status check_out(const void* p) {
  if (p == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (!aligned16(p)) return MXFP4_ERR_MISALIGNED;
  return MXFP4_OK;
}

}  // namespace

// The argument checks of gemm_fp4_bf16_fwd before its workspace check, in its
// order; MXFP4_OK for M == 0 or N == 0 (nothing to do).
int mxfp4::check_fwd_args(const uint16_t* x, const uint16_t* w, const uint16_t* y, int64_t M, int64_t N,
                          int64_t K) {
  mxfp4_status st = check_bf16_in(x, M, K, K);
  if (st == MXFP4_OK) st = check_bf16_in(w, N, K, K);
  if (st != MXFP4_OK || M == 0 || N == 0) return st;
  st = check_out(y);
  if (st == MXFP4_OK && N % 8 != 0) st = MXFP4_ERR_MISALIGNED;
  return st;
}

namespace {

#define MXFP4_TRY(expr)                      \
  do {                                       \
    mxfp4_status _s = (expr);                \
    if (_s != MXFP4_OK) return _s;           \
  } while (0)

// Row-wise cast of an internal operand into the workspace.
struct QuantView {
  uint8_t* q;
  uint8_t* sf;
};

QuantView carve(uint8_t*& cursor, int64_t rows, int64_t cols) {
  QuantView v;
  v.q = cursor;
  cursor += align256(static_cast<size_t>(rows) * static_cast<size_t>(cols / 2));
  v.sf = cursor;
  cursor += align256(tile_scale_bytes(rows, cols));
  return v;
}

size_t carve_bytes(int64_t rows, int64_t cols) {
  return align256(static_cast<size_t>(rows) * static_cast<size_t>(cols / 2)) +
         align256(tile_scale_bytes(rows, cols));
}

// MXFP8 operand in the workspace: codes [rows, cols] bytes, tile scales.
QuantView carve_fp8(uint8_t*& cursor, int64_t rows, int64_t cols) {
  QuantView v;
  v.q = cursor;
  cursor += align256(static_cast<size_t>(rows) * static_cast<size_t>(cols));
  v.sf = cursor;
  cursor += align256(tile_scale_bytes(rows, cols));
  return v;
}

size_t carve_fp8_bytes(int64_t rows, int64_t cols) {
  return align256(static_cast<size_t>(rows) * static_cast<size_t>(cols)) +
         align256(tile_scale_bytes(rows, cols));
}

// The argument checks of gemm_fp4, in order; on MXFP4_OK the device of c is
// bound (nothing to check or bind when *empty: M == 0 or N == 0).
mxfp4_status check_gemm(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                        const uint16_t* c, int64_t M, int64_t N, int64_t K, int64_t ldc, bool* empty) {
  *empty = false;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MXFP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldc < N) return MXFP4_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    *empty = true;
    return MXFP4_OK;
  }
  MXFP4_TRY(check_out(c));
  if (ldc % 8 != 0) return MXFP4_ERR_MISALIGNED;
  if (K > 0) {
    MXFP4_TRY(check_out(a));
    MXFP4_TRY(check_out(a_sf));
    MXFP4_TRY(check_out(b));
    MXFP4_TRY(check_out(b_sf));
  }
  return check_device(c);
}

mxfp4_status gemm_checked(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                          const uint8_t* b_sf, uint16_t* c, int64_t M, int64_t N, int64_t K,
                          int64_t ldc, cudaStream_t s, bool fp8 = false) {
  GemmArgs g{a, a_sf, b, b_sf, c, M, N, K, ldc};
  cudaError_t e = fp8 ? mxfp4::launch_gemm_mxfp8(g, s) : mxfp4::launch_gemm(g, s);
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(e);
}

}  // namespace

extern "C" {

int mxfp4_abi_version(void) { return 1; }

int mxfp4_last_cuda_error(void) { return t_last_cuda_error; }

const char* mxfp4_cuda_error_string(int cuda_error) {
  return cudaGetErrorName(static_cast<cudaError_t>(cuda_error));
}

const char* mxfp4_status_string(int status) {
  switch (status) {
    case MXFP4_OK: return "MXFP4_OK";
    case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG";
    case MXFP4_ERR_MISALIGNED: return "MXFP4_ERR_MISALIGNED";
    case MXFP4_ERR_UNSUPPORTED_DEVICE: return "MXFP4_ERR_UNSUPPORTED_DEVICE";
    case MXFP4_ERR_WORKSPACE: return "MXFP4_ERR_WORKSPACE";
    case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA";
    case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT";
    case MXFP4_ERR_NOT_IMPLEMENTED: return "MXFP4_ERR_NOT_IMPLEMENTED";
    default: return "MXFP4_UNKNOWN_STATUS";
  }
}

size_t mxfp4_codes_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return static_cast<size_t>(rows) * static_cast<size_t>(cols / 2);
}

size_t mxfp4_scales_bytes(int64_t rows, int64_t cols, uint32_t flags) {
  if (rows < 0 || cols < 0) return 0;
  if (flags & MXFP4_SCALE_LINEAR) return static_cast<size_t>(rows) * static_cast<size_t>(cols / 32);
  return tile_scale_bytes(rows, cols);
}

mxfp4_status mxfp4_cast(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                        uint8_t* sf, uint32_t flags, void* stream) {
  if (flags & ~(MXFP4_HADAMARD_ROW | MXFP4_SCALE_LINEAR)) return MXFP4_ERR_INVALID_ARG;
  MXFP4_TRY(check_bf16_in(x, rows, cols, ldx));
  if (rows == 0 || cols == 0) return MXFP4_OK;
  MXFP4_TRY(check_out(q));
  MXFP4_TRY(check_out(sf));
  MXFP4_TRY(check_device(x));
  CastArgs a{x, rows, cols, ldx, q, sf, nullptr, nullptr, flags};
  return from_cuda(mxfp4::launch_cast(a, static_cast<cudaStream_t>(stream)));
}

// The checks of mxfp4_cast_dual, in its order; binds the device of x.
// `*empty` is set when there is nothing to cast.
static mxfp4_status check_cast_dual(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                                    const uint8_t* q_row, const uint8_t* sf_row, const uint8_t* q_col,
                                    const uint8_t* sf_col, uint32_t flags, bool* empty) {
  *empty = false;
  if (flags & ~(MXFP4_HADAMARD_ROW | MXFP4_HADAMARD_COL | MXFP4_SCALE_LINEAR))
    return MXFP4_ERR_INVALID_ARG;
  MXFP4_TRY(check_bf16_in(x, rows, cols, ldx));
  if (rows % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) {
    *empty = true;
    return MXFP4_OK;
  }
  MXFP4_TRY(check_out(q_row));
  MXFP4_TRY(check_out(sf_row));
  MXFP4_TRY(check_out(q_col));
  MXFP4_TRY(check_out(sf_col));
  return check_device(x);
}

mxfp4_status mxfp4_cast_dual(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                             uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                             uint32_t flags, void* stream) {
  bool empty = false;
  MXFP4_TRY(check_cast_dual(x, rows, cols, ldx, q_row, sf_row, q_col, sf_col, flags, &empty));
  if (empty) return MXFP4_OK;
  CastArgs a{x, rows, cols, ldx, q_row, sf_row, q_col, sf_col, flags};
  return from_cuda(mxfp4::launch_cast(a, static_cast<cudaStream_t>(stream)));
}

mxfp4_status mxfp4_cast_dual_grouped(const mxfp4_cast_desc* casts, int count, void* stream) {
  if (casts == nullptr || count < 1 || count > MXFP4_GROUP_MAX) return MXFP4_ERR_INVALID_ARG;
  CastArgs list[MXFP4_GROUP_MAX];
  int n = 0, dev = -1;
  for (int i = 0; i < count; ++i) {
    const mxfp4_cast_desc& d = casts[i];
    bool empty = false;
    MXFP4_TRY(check_cast_dual(d.x, d.rows, d.cols, d.ldx, d.q_row, d.sf_row, d.q_col, d.sf_col, d.flags,
                              &empty));
    if (empty) continue;
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);  // the device check_cast_dual bound
    if (e != cudaSuccess) return from_cuda(e);
    if (dev >= 0 && cur != dev) return MXFP4_ERR_INVALID_ARG;  // one launch, one device
    dev = cur;
    list[n++] = CastArgs{d.x, d.rows, d.cols, d.ldx, d.q_row, d.sf_row, d.q_col, d.sf_col, d.flags};
  }
  if (n == 0) return MXFP4_OK;
  cudaError_t e = mxfp4::launch_cast_grouped(list, n, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(e);
}

mxfp4_status gemm_fp4(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                      uint16_t* c, int64_t M, int64_t N, int64_t K, int64_t ldc, void* stream) {
  bool empty = false;
  MXFP4_TRY(check_gemm(a, a_sf, b, b_sf, c, M, N, K, ldc, &empty));
  if (empty) return MXFP4_OK;
  return gemm_checked(a, a_sf, b, b_sf, c, M, N, K, ldc, static_cast<cudaStream_t>(stream));
}

mxfp4_status gemm_fp4_grouped(const mxfp4_gemm_desc* gemms, int count, void* stream) {
  if (gemms == nullptr || count < 1 || count > MXFP4_GROUP_MAX) return MXFP4_ERR_INVALID_ARG;
  GemmArgs list[MXFP4_GROUP_MAX];
  int n = 0, dev = -1;
  for (int i = 0; i < count; ++i) {
    const mxfp4_gemm_desc& d = gemms[i];
    bool empty = false;
    MXFP4_TRY(check_gemm(d.a, d.a_sf, d.b, d.b_sf, d.c, d.M, d.N, d.K, d.ldc, &empty));
    if (empty) continue;
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);  // the device check_gemm bound
    if (e != cudaSuccess) return from_cuda(e);
    if (dev >= 0 && cur != dev) return MXFP4_ERR_INVALID_ARG;  // one launch, one device
    dev = cur;
    list[n++] = GemmArgs{d.a, d.a_sf, d.b, d.b_sf, d.c, d.M, d.N, d.K, d.ldc};
  }
  if (n == 0) return MXFP4_OK;
  cudaError_t e = mxfp4::launch_gemm_grouped(list, n, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(e);
}

mxfp4_status gemm_mxfp8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                        uint16_t* c, int64_t M, int64_t N, int64_t K, int64_t ldc, void* stream) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MXFP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldc < N) return MXFP4_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MXFP4_OK;
  MXFP4_TRY(check_out(c));
  if (ldc % 8 != 0) return MXFP4_ERR_MISALIGNED;
  if (K > 0) {
    MXFP4_TRY(check_out(a));
    MXFP4_TRY(check_out(a_sf));
    MXFP4_TRY(check_out(b));
    MXFP4_TRY(check_out(b_sf));
  }
  MXFP4_TRY(check_device(c));
  return gemm_checked(a, a_sf, b, b_sf, c, M, N, K, ldc, static_cast<cudaStream_t>(stream), true);
}

mxfp4_status gemm_fp4_cast_out(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                               const uint8_t* b_sf, uint16_t* c, int64_t M, int64_t N, int64_t K,
                               int64_t ldc, uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col,
                               uint8_t* sf_col, uint32_t flags, void* stream) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MXFP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || M % 32 != 0 || N % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (flags & ~(MXFP4_HADAMARD_ROW | MXFP4_HADAMARD_COL)) return MXFP4_ERR_INVALID_ARG;
  if ((q_row == nullptr) != (sf_row == nullptr) || (q_col == nullptr) != (sf_col == nullptr))
    return MXFP4_ERR_INVALID_ARG;
  if (c != nullptr && ldc < N) return MXFP4_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MXFP4_OK;
  if (c == nullptr && q_row == nullptr && q_col == nullptr) return MXFP4_ERR_INVALID_ARG;  // no output
  if (c != nullptr) {
    MXFP4_TRY(check_out(c));
    if (ldc % 8 != 0) return MXFP4_ERR_MISALIGNED;
  }
  if (q_row != nullptr) {
    MXFP4_TRY(check_out(q_row));
    MXFP4_TRY(check_out(sf_row));
  }
  if (q_col != nullptr) {
    MXFP4_TRY(check_out(q_col));
    MXFP4_TRY(check_out(sf_col));
  }
  if (K > 0) {
    MXFP4_TRY(check_out(a));
    MXFP4_TRY(check_out(a_sf));
    MXFP4_TRY(check_out(b));
    MXFP4_TRY(check_out(b_sf));
  }
  MXFP4_TRY(check_device(c != nullptr ? static_cast<const void*>(c)
                                       : (q_row != nullptr ? static_cast<const void*>(q_row) : q_col)));
  const GemmArgs g{a, a_sf, b, b_sf, c, M, N, K, ldc};
  const mxfp4::CastOutArgs out{q_row, sf_row, q_col, sf_col, flags};
  const cudaError_t e = mxfp4::launch_gemm_cast_out(g, out, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(e);
}

mxfp4_status mxfp8_cast_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                             uint8_t* q_col, uint8_t* sf_col, uint32_t flags, void* stream) {
  if (flags & ~(MXFP4_HADAMARD_COL | MXFP4_SCALE_LINEAR)) return MXFP4_ERR_INVALID_ARG;
  MXFP4_TRY(check_bf16_in(x, rows, cols, ldx));
  if (rows % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MXFP4_OK;
  MXFP4_TRY(check_out(q_col));
  MXFP4_TRY(check_out(sf_col));
  MXFP4_TRY(check_device(x));
  CastArgs a{x, rows, cols, ldx, nullptr, nullptr, q_col, sf_col, flags | mxfp4::kFlagFp8};
  return from_cuda(mxfp4::launch_cast(a, static_cast<cudaStream_t>(stream)));
}

mxfp4_status gemm_fp8_bf16_wgrad(const uint16_t* dy, const uint16_t* x, uint16_t* dw, int64_t M,
                                 int64_t N, int64_t K, uint32_t flags, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (flags & ~MXFP4_HADAMARD_COL) return MXFP4_ERR_INVALID_ARG;
  MXFP4_TRY(check_bf16_in(dy, M, N, N));
  MXFP4_TRY(check_bf16_in(x, M, K, K));
  if (M % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return MXFP4_OK;
  MXFP4_TRY(check_out(dw));
  if (ws == nullptr || ws_bytes < mxfp4_workspace_bytes(MXFP4_OP_WGRAD_FP8, M, N, K) || !aligned16(ws))
    return MXFP4_ERR_WORKSPACE;
  MXFP4_TRY(check_device(dw));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) return from_cuda(mxfp4::launch_fill_zero_bf16(dw, N, K, K, s));
  uint8_t* cur = static_cast<uint8_t*>(ws);
  QuantView qdyt = carve_fp8(cur, N, M), qxt = carve_fp8(cur, K, M);
  const uint32_t cf = ((flags & MXFP4_HADAMARD_COL) ? mxfp4::kFlagHadamardCol : 0u) | mxfp4::kFlagFp8;
  CastArgs cdy{dy, M, N, N, nullptr, nullptr, qdyt.q, qdyt.sf, cf};  // dY^T along M
  CastArgs cx{x, M, K, K, nullptr, nullptr, qxt.q, qxt.sf, cf};      // X^T along M
  const CastArgs casts[2] = {cdy, cx};  // one launch: the same kind of cast
  MXFP4_TRY(from_cuda(mxfp4::launch_cast_grouped(casts, 2, s)));
  return gemm_checked(qdyt.q, qdyt.sf, qxt.q, qxt.sf, dw, N, K, M, K, s, true);
}

size_t mxfp4_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  switch (op) {
    case MXFP4_OP_WGRAD_FP8: return carve_fp8_bytes(N, M) + carve_fp8_bytes(K, M);  // col(dY), col(X)
    case MXFP4_OP_FWD: return carve_bytes(M, K) + carve_bytes(N, K);    // row(X), row(W)
    case MXFP4_OP_DGRAD: return carve_bytes(M, N) + carve_bytes(K, N);  // row(dY), col(W)
    case MXFP4_OP_WGRAD: return carve_bytes(N, M) + carve_bytes(K, M);  // col(dY), col(X)
    default: return 0;
  }
}

mxfp4_status gemm_fp4_bf16_fwd(const uint16_t* x, const uint16_t* w, uint16_t* y, int64_t M,
                               int64_t N, int64_t K, void* ws, size_t ws_bytes, void* stream) {
  MXFP4_TRY(static_cast<mxfp4_status>(mxfp4::check_fwd_args(x, w, y, M, N, K)));
  if (M == 0 || N == 0) return MXFP4_OK;
  if (ws == nullptr || ws_bytes < mxfp4_workspace_bytes(MXFP4_OP_FWD, M, N, K) || !aligned16(ws))
    return MXFP4_ERR_WORKSPACE;
  MXFP4_TRY(check_device(y));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(mxfp4::launch_fill_zero_bf16(y, M, N, N, s));
  uint8_t* cur = static_cast<uint8_t*>(ws);
  QuantView qx = carve(cur, M, K), qw = carve(cur, N, K);
  CastArgs cx{x, M, K, K, qx.q, qx.sf, nullptr, nullptr, 0};
  CastArgs cw{w, N, K, K, qw.q, qw.sf, nullptr, nullptr, 0};
  const CastArgs casts[2] = {cx, cw};  // one launch: both row-wise
  MXFP4_TRY(from_cuda(mxfp4::launch_cast_grouped(casts, 2, s)));
  return gemm_checked(qx.q, qx.sf, qw.q, qw.sf, y, M, N, K, N, s);
}

mxfp4_status gemm_fp4_bf16_dgrad(const uint16_t* dy, const uint16_t* w, uint16_t* dx, int64_t M,
                                 int64_t N, int64_t K, void* ws, size_t ws_bytes, void* stream) {
  MXFP4_TRY(check_bf16_in(dy, M, N, N));
  MXFP4_TRY(check_bf16_in(w, N, K, K));
  if (N % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return MXFP4_OK;
  MXFP4_TRY(check_out(dx));
  if (ws == nullptr || ws_bytes < mxfp4_workspace_bytes(MXFP4_OP_DGRAD, M, N, K) || !aligned16(ws))
    return MXFP4_ERR_WORKSPACE;
  MXFP4_TRY(check_device(dx));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) return from_cuda(mxfp4::launch_fill_zero_bf16(dx, M, K, K, s));
  uint8_t* cur = static_cast<uint8_t*>(ws);
  QuantView qdy = carve(cur, M, N), qwt = carve(cur, K, N);
  CastArgs cdy{dy, M, N, N, qdy.q, qdy.sf, nullptr, nullptr, 0};
  CastArgs cw{w, N, K, K, nullptr, nullptr, qwt.q, qwt.sf, 0};  // W^T, quantized along N
  MXFP4_TRY(from_cuda(mxfp4::launch_cast(cdy, s)));
  MXFP4_TRY(from_cuda(mxfp4::launch_cast(cw, s)));
  return gemm_checked(qdy.q, qdy.sf, qwt.q, qwt.sf, dx, M, K, N, K, s);
}

mxfp4_status gemm_fp4_bf16_wgrad(const uint16_t* dy, const uint16_t* x, uint16_t* dw, int64_t M,
                                 int64_t N, int64_t K, uint32_t flags, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (flags & ~MXFP4_HADAMARD_COL) return MXFP4_ERR_INVALID_ARG;
  MXFP4_TRY(check_bf16_in(dy, M, N, N));
  MXFP4_TRY(check_bf16_in(x, M, K, K));
  if (M % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return MXFP4_OK;
  MXFP4_TRY(check_out(dw));
  if (ws == nullptr || ws_bytes < mxfp4_workspace_bytes(MXFP4_OP_WGRAD, M, N, K) || !aligned16(ws))
    return MXFP4_ERR_WORKSPACE;
  MXFP4_TRY(check_device(dw));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) return from_cuda(mxfp4::launch_fill_zero_bf16(dw, N, K, K, s));
  uint8_t* cur = static_cast<uint8_t*>(ws);
  QuantView qdyt = carve(cur, N, M), qxt = carve(cur, K, M);
  const uint32_t cf = (flags & MXFP4_HADAMARD_COL) ? mxfp4::kFlagHadamardCol : 0u;
  CastArgs cdy{dy, M, N, N, nullptr, nullptr, qdyt.q, qdyt.sf, cf};  // dY^T along M
  CastArgs cx{x, M, K, K, nullptr, nullptr, qxt.q, qxt.sf, cf};      // X^T along M
  const CastArgs casts[2] = {cdy, cx};  // one launch: the same kind of cast
  MXFP4_TRY(from_cuda(mxfp4::launch_cast_grouped(casts, 2, s)));
  return gemm_checked(qdyt.q, qdyt.sf, qxt.q, qxt.sf, dw, N, K, M, K, s);
}

mxfp4_status mxfp4_selftest_wait_timeout(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                         const uint8_t* b_sf, uint16_t* c, int64_t M, int64_t N, int64_t K,
                                         int64_t ldc, uint64_t wait_limit_ns, void* stream) {
  if (wait_limit_ns < 1000000ull || wait_limit_ns > 2000000000ull) return MXFP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return MXFP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldc < N) return MXFP4_ERR_INVALID_ARG;
  MXFP4_TRY(check_out(c));
  if (ldc % 8 != 0) return MXFP4_ERR_MISALIGNED;
  MXFP4_TRY(check_out(a));
  MXFP4_TRY(check_out(a_sf));
  MXFP4_TRY(check_out(b));
  MXFP4_TRY(check_out(b_sf));
  MXFP4_TRY(check_device(c));
  GemmArgs g{a, a_sf, b, b_sf, c, M, N, K, ldc};
  const cudaError_t e = mxfp4::launch_gemm_selftest_timeout(g, wait_limit_ns, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(e);
}

mxfp4_status mxfp4_device_status(int reset, int* out_status) {
  if (out_status == nullptr) return MXFP4_ERR_INVALID_ARG;
  int v = 0;
  if (mxfp4::read_device_status(&v, reset != 0) != cudaSuccess) return MXFP4_ERR_CUDA;
  *out_status = v;
  return MXFP4_OK;
}

}  // extern "C"

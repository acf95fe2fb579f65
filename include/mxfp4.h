/*
 * mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 training-GEMM library.
 *
 * What the operations are (page title, section):
 *   - jax-aiter README, "Supported ops" table, row "MXFP4 Cast"
 *     (CastMxfp4JA / CastMxfp4DualJA): BF16 -> MXFP4, i.e. E2M1 elements with
 *     E8M0 block scales, with a transposed copy and a GEMM-ready ("shuffled")
 *     scale layout.                                   -> mxfp4_cast, mxfp4_cast_dual
 *   - same table, row "FP4 GEMM (low-level)": gemm_fp4(a, b, a_scale,
 *     b_scale) on pre-quantized fp4x2 inputs with e8m0 scales.   -> gemm_fp4
 *   - same table, row "FP4 GEMM (training)", "Quick start" and "MXFP4
 *     training architecture": BF16 in/out, A[M,K] . B[N,K]^T, FP4 forward,
 *     FP4 dA, FP4 dB, grad_out cast with a Hadamard transform.
 *                      -> gemm_fp4_bf16_fwd, gemm_fp4_bf16_dgrad, gemm_fp4_bf16_wgrad
 *
 * Numerics (the pages fix none of them; these are the library's readings):
 *   block = 32 elements along the contraction dimension; scale byte
 *   s = clamp(floor(log2 amax) - 2, -127, 127) + 127 (amax = 0 -> 0x00;
 *   a NaN/Inf in the block -> 0xFF with all codes 0); element code =
 *   x * 2^(127 - s) rounded to nearest-even onto {0,.5,1,1.5,2,3,4,6},
 *   saturating at 6, sign kept; element 2j in the low nibble of byte j.
 *   Optional 32-point orthonormal Walsh-Hadamard transform (Sylvester order)
 *   of each block before quantization, in fp32.
 *   GEMM: fp32 accumulation of the exact block-scaled products, one
 *   round-to-nearest-even to bf16.
 *
 * Data layouts (all row-major, all buffers owned by the caller):
 *   bf16 tensors are passed as uint16_t bit patterns.
 *   codes  of a tensor T[R, C] quantized along C: [R, C/2] bytes, pitch C/2.
 *   scales, default ("tile") layout: tiles of 128 rows x 4 blocks (512 bytes),
 *     ceil(R/128) x ceil(C/128) tiles stored row-tile-major; inside a tile the
 *     scale of row r, block b sits at byte (r%32)*16 + ((r%128)/32)*4 + b%4.
 *     Size: mxfp4_scales_bytes().  The cast writes 0x00 into padding bytes;
 *     gemm_fp4 requires padding bytes to hold finite scales (not 0xFF).
 *   scales, MXFP4_SCALE_LINEAR: [R, C/32] bytes (for inspection; the GEMMs
 *     take the tile layout only).
 *   "col" outputs of mxfp4_cast_dual quantize T^T: codes [C, R/2], scales as
 *     a tensor of C rows with R/32 blocks per row.
 *
 * Execution: every call validates its arguments on the host (nothing is
 * launched on an error), then enqueues its kernels on `stream` (a
 * cudaStream_t; NULL means the legacy default stream) and returns without
 * synchronizing.  The library allocates nothing and keeps no per-call state.
 * Pointers must be device pointers on the current device, 16-byte aligned;
 * leading dimensions must make every row start 16-byte aligned.  The device
 * must have compute capability 10.3 (GB300).
 */
#ifndef MXFP4_H_
#define MXFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXFP4_OK = 0,
  MXFP4_ERR_INVALID_ARG = 1,        /* null pointer, bad shape, bad flags */
  MXFP4_ERR_MISALIGNED = 2,         /* pointer or leading dimension not 16-byte aligned */
  MXFP4_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  MXFP4_ERR_WORKSPACE = 4,          /* workspace missing or smaller than mxfp4_workspace_bytes() */
  MXFP4_ERR_CUDA = 5,               /* a CUDA runtime call failed (launch error, ...) */
  MXFP4_ERR_TIMEOUT = 6,            /* a GEMM pipeline wait ran out (see mxfp4_device_status) */
  MXFP4_ERR_NOT_IMPLEMENTED = 7
} mxfp4_status;

/* Cast flags. */
#define MXFP4_HADAMARD_ROW 1u /* transform each 32-block of the row-wise output first */
#define MXFP4_HADAMARD_COL 2u /* transform each 32-block of the column-wise output first */
#define MXFP4_SCALE_LINEAR 4u /* write scales as [R, C/32] instead of the tile layout */

/* Workspace queries for the bf16 entry points. */
#define MXFP4_OP_FWD 0
#define MXFP4_OP_DGRAD 1
#define MXFP4_OP_WGRAD 2
#define MXFP4_OP_WGRAD_FP8 3 /* gemm_fp8_bf16_wgrad */

/* Version of this ABI (bumped on any signature change). */
int mxfp4_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* mxfp4_status_string(int status);

/* The CUDA runtime error code behind the calling thread's most recent
 * MXFP4_ERR_CUDA (0 if there was none), and the CUDA runtime's name for a
 * code (static string).  No counterpart in the pages: a diagnostic for the
 * one status that wraps another library's error. */
int mxfp4_last_cuda_error(void);
const char* mxfp4_cuda_error_string(int cuda_error);

/* Bytes of codes for a [rows, cols] tensor quantized along cols: rows*cols/2. */
size_t mxfp4_codes_bytes(int64_t rows, int64_t cols);

/* Bytes of scales for a [rows, cols] tensor quantized along cols, in the
 * layout `flags` selects (MXFP4_SCALE_LINEAR or the tile layout). */
size_t mxfp4_scales_bytes(int64_t rows, int64_t cols, uint32_t flags);

/*
 * mxfp4_cast -- row-wise BF16 -> MXFP4 cast (CastMxfp4JA).
 *   x     : bf16 [rows, cols], row pitch ldx elements (ldx >= cols, ldx % 8 == 0)
 *   q     : out, codes [rows, cols/2]
 *   sf    : out, scales (tile layout, or linear with MXFP4_SCALE_LINEAR)
 *   flags : MXFP4_HADAMARD_ROW | MXFP4_SCALE_LINEAR
 * Requires rows >= 0, cols % 32 == 0.  rows == 0 or cols == 0 is a no-op.
 */
mxfp4_status mxfp4_cast(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                        uint8_t* sf, uint32_t flags, void* stream);

/*
 * mxfp4_cast_dual -- row-wise and column-wise (transposed) cast in one pass
 * over x (CastMxfp4DualJA).
 *   q_row/sf_row : row-wise output as in mxfp4_cast
 *   q_col/sf_col : column-wise output: codes [cols, rows/2]; scales of a
 *                  [cols, rows] tensor (tile layout: ceil(cols/128) x
 *                  ceil(rows/128) tiles)
 *   flags        : MXFP4_HADAMARD_ROW, MXFP4_HADAMARD_COL (each applies to
 *                  its own output only), MXFP4_SCALE_LINEAR (both outputs)
 * Requires rows % 32 == 0 and cols % 32 == 0.
 */
mxfp4_status mxfp4_cast_dual(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                             uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                             uint32_t flags, void* stream);

/*
 * mxfp4_cast_dual_grouped -- up to MXFP4_GROUP_MAX independent mxfp4_cast_dual
 * calls in one launch.  A training step casts X, W and dY before its GEMMs
 * (the "FP4 GEMM (training)" row: every operand goes through the cast); one
 * persistent launch over all their tiles (numbered cast after cast) fills
 * and drains the pipeline once instead of once per cast.  The pages describe
 * no grouped call: this is a scheduling form of mxfp4_cast_dual with the same
 * results, every byte equal to the mxfp4_cast_dual call with the same
 * arguments.
 *   casts : host array of `count` descriptors, read during the call only;
 *           each field means what the mxfp4_cast_dual argument of the same
 *           name means (each its own shape and flags)
 *   count : 1 .. MXFP4_GROUP_MAX
 * Each descriptor is checked as mxfp4_cast_dual checks its arguments, in
 * that order.  The first failing descriptor's status is returned and nothing
 * is launched.  Descriptors with rows == 0 or cols == 0 are skipped.  Every
 * cast's memory must be on one device (MXFP4_ERR_INVALID_ARG otherwise).
 * The casts run concurrently: no output may overlap another descriptor's
 * input or outputs.
 */
typedef struct mxfp4_cast_desc {
  const uint16_t* x;
  int64_t rows, cols, ldx;
  uint8_t* q_row;
  uint8_t* sf_row;
  uint8_t* q_col;
  uint8_t* sf_col;
  uint32_t flags;
} mxfp4_cast_desc;
mxfp4_status mxfp4_cast_dual_grouped(const mxfp4_cast_desc* casts, int count, void* stream);

/*
 * gemm_fp4 -- C[M,N] = A[M,K] . B[N,K]^T on MXFP4 operands, bf16 output
 * (gemm_fp4 of the "FP4 GEMM (low-level)" row).
 *   a, a_sf : codes [M, K/2], scales (tile layout, M rows, K/32 blocks)
 *   b, b_sf : codes [N, K/2], scales (tile layout, N rows, K/32 blocks)
 *   c       : out, bf16 [M, N], row pitch ldc elements (ldc >= N, ldc % 8 == 0)
 * Requires M, N >= 0, K >= 0, K % 32 == 0; M*N == 0 is a no-op; K == 0
 * writes zeros.
 */
mxfp4_status gemm_fp4(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                      uint16_t* c, int64_t M, int64_t N, int64_t K, int64_t ldc, void* stream);

/*
 * gemm_fp4_grouped -- up to MXFP4_GROUP_MAX independent gemm_fp4 calls in one
 * launch.  The "FP4 GEMM (training)" row runs the forward GEMM, dA and dB
 * through gemm_fp4. In a training step their operands are ready together,
 * and one persistent launch over all their tiles (numbered GEMM after GEMM)
 * leaves a single partial last wave of tiles where separate launches leave
 * one each.  The pages describe no grouped call: this is a scheduling form of
 * gemm_fp4 with the same results, each C bit-identical to the gemm_fp4 call
 * with the same arguments.
 *   gemms : host array of `count` descriptors, read during the call only; each
 *           field means what the gemm_fp4 argument of the same name means
 *   count : 1 .. MXFP4_GROUP_MAX
 * Each descriptor is checked as gemm_fp4 checks its arguments, in that
 * order. The first failing descriptor's status is returned and nothing is
 * launched. Descriptors with M == 0 or N == 0 are skipped; K == 0 writes
 * zeros. Every GEMM's memory must be on one device (MXFP4_ERR_INVALID_ARG
 * otherwise). The GEMMs run concurrently: no C may overlap another
 * descriptor's C or operands.
 */
#define MXFP4_GROUP_MAX 4
typedef struct mxfp4_gemm_desc {
  const uint8_t* a;
  const uint8_t* a_sf;
  const uint8_t* b;
  const uint8_t* b_sf;
  uint16_t* c;
  int64_t M, N, K, ldc;
} mxfp4_gemm_desc;
mxfp4_status gemm_fp4_grouped(const mxfp4_gemm_desc* gemms, int count, void* stream);

/*
 * gemm_fp4_cast_out -- gemm_fp4 whose epilogue also casts its own output to
 * MXFP4, so the next GEMM's operand comes without a separate cast of C (the
 * gradient one GEMM produces is the next one's grad_out: jax-aiter README,
 * "MXFP4 training architecture"; the pages run the casts as separate calls).
 *   a .. ldc     : as gemm_fp4; c may be NULL (then no bf16 C is written and
 *                  ldc is ignored) when at least one cast output is given
 *   q_row/sf_row : C quantized along N: codes [M, N/2], tile scales (M rows,
 *                  N/32 blocks) -- what mxfp4_cast_dual writes as its row
 *                  output for x = C; both NULL to skip
 *   q_col/sf_col : C^T quantized along M: codes [N, M/2], tile scales (N rows,
 *                  M/32 blocks) -- mxfp4_cast_dual's column output; both NULL
 *                  to skip
 *   flags        : MXFP4_HADAMARD_ROW, MXFP4_HADAMARD_COL (tile layout only)
 * The cast outputs are bit-identical to mxfp4_cast_dual(C, flags) on the bf16
 * C (whether or not it is stored), scale padding (0x00) included.  Requires
 * M % 32 == 0, N % 32 == 0, K % 32 == 0; M*N == 0 is a no-op; K == 0 writes
 * zeros and the casts of a zero matrix (all bytes 0x00).
 */
mxfp4_status gemm_fp4_cast_out(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                               const uint8_t* b_sf, uint16_t* c, int64_t M, int64_t N, int64_t K,
                               int64_t ldc, uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col,
                               uint8_t* sf_col, uint32_t flags, void* stream);

/*
 * MXFP8: the FP8 alternative for the wgrad operands (jax-aiter README,
 * "MXFP4 training architecture": an FP8 dB path next to the FP4 one).
 * E4M3 elements (one byte each, round to nearest even, saturating at 448)
 * with the same E8M0 scales per 32 elements, scale byte
 * floor(log2 amax) - 8 + 127 (clamped), the same NaN/Inf, zero-block and
 * tile-layout conventions as MXFP4.
 *
 * mxfp8_cast_cols -- column-wise (transposed) MXFP8 cast of bf16 x[rows, cols]
 * (row pitch ldx elements): q_col [cols, rows] bytes, sf_col scales of the
 * [cols, rows/32] blocks (tile layout, or linear with MXFP4_SCALE_LINEAR).
 * flags: MXFP4_HADAMARD_COL, MXFP4_SCALE_LINEAR.  rows, cols % 32 == 0.
 */
mxfp4_status mxfp8_cast_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                             uint8_t* q_col, uint8_t* sf_col, uint32_t flags, void* stream);

/*
 * gemm_mxfp8 -- C[M,N] = A[M,K] . B[N,K]^T on MXFP8 operands, bf16 output:
 *   a, a_sf : codes [M, K] bytes, scales (tile layout, M rows, K/32 blocks)
 *   b, b_sf : codes [N, K] bytes, scales (tile layout, N rows, K/32 blocks)
 *   c       : out, bf16 [M, N], row pitch ldc (ldc >= N, ldc % 8 == 0)
 * Requires K % 32 == 0; M*N == 0 is a no-op; K == 0 writes zeros.
 */
mxfp4_status gemm_mxfp8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                        uint16_t* c, int64_t M, int64_t N, int64_t K, int64_t ldc, void* stream);

/*
 * gemm_fp8_bf16_wgrad -- dW[N,K] = dY[M,N]^T . X[M,K] like gemm_fp4_bf16_wgrad,
 * with both operands cast to MXFP8 along M (column-wise) into `ws`
 * (mxfp4_workspace_bytes(MXFP4_OP_WGRAD_FP8, M, N, K) bytes).
 * flags: MXFP4_HADAMARD_COL (both operands).  M % 32 == 0.
 */
mxfp4_status gemm_fp8_bf16_wgrad(const uint16_t* dy, const uint16_t* x, uint16_t* dw, int64_t M,
                                 int64_t N, int64_t K, uint32_t flags, void* ws, size_t ws_bytes,
                                 void* stream);

/* Workspace bytes that gemm_fp4_bf16_{fwd,dgrad,wgrad} (op = MXFP4_OP_*)
 * need for the quantized copies of their operands; 0 for a bad op. */
size_t mxfp4_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/*
 * gemm_fp4_bf16_fwd -- Y[M,N] = X[M,K] . W[N,K]^T: casts X and W row-wise
 * into `ws`, then gemm_fp4.  x, w, y dense row-major.  K % 32 == 0.
 */
mxfp4_status gemm_fp4_bf16_fwd(const uint16_t* x, const uint16_t* w, uint16_t* y, int64_t M,
                               int64_t N, int64_t K, void* ws, size_t ws_bytes, void* stream);

/*
 * gemm_fp4_bf16_dgrad -- dX[M,K] = dY[M,N] . W[N,K]: A = dY quantized along N
 * (row-wise), B = W quantized along N (column-wise), contraction over N.
 * N % 32 == 0, K % 32 == 0.
 */
mxfp4_status gemm_fp4_bf16_dgrad(const uint16_t* dy, const uint16_t* w, uint16_t* dx, int64_t M,
                                 int64_t N, int64_t K, void* ws, size_t ws_bytes, void* stream);

/*
 * gemm_fp4_bf16_wgrad -- dW[N,K] = dY[M,N]^T . X[M,K]: both operands
 * quantized along the token dimension M (column-wise), contraction over M.
 * flags: MXFP4_HADAMARD_COL transforms BOTH operands along M, so that the
 * orthonormal transform cancels in the product.  M % 32 == 0.
 */
mxfp4_status gemm_fp4_bf16_wgrad(const uint16_t* dy, const uint16_t* x, uint16_t* dw, int64_t M,
                                 int64_t N, int64_t K, uint32_t flags, void* ws, size_t ws_bytes,
                                 void* stream);

/*
 * mxfp4_device_status -- reads (and with reset != 0 clears) the library's
 * device-side status word on the current device: MXFP4_OK, or
 * MXFP4_ERR_TIMEOUT if a GEMM pipeline wait gave up (the kernel then stopped
 * early and its output is incomplete).  Synchronizes the device.
 */
mxfp4_status mxfp4_device_status(int reset, int* out_status);

/*
 * mxfp4_selftest_wait_timeout -- a self-test of the GEMM's bounded waits, for
 * tests and diagnostics (not part of any computation; the pages have no
 * counterpart).  Launches gemm_fp4's kernel on the given operands with every
 * pipeline wait limited to wait_limit_ns (1 ms .. 2 s; the product launches
 * use 2 s) and the first "stage ready" signal of the first tile withheld, so
 * that the tensor-core warp's wait runs out: the kernel records
 * MXFP4_ERR_TIMEOUT in the device status word (mxfp4_device_status), lets its
 * loads and tensor-core operations in flight complete, and ends; C is left
 * unwritten or partly written.  No fault, trap or hang is involved and the
 * context stays usable.  Arguments as gemm_fp4 (M, N, K > 0).
 */
mxfp4_status mxfp4_selftest_wait_timeout(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b,
                                         const uint8_t* b_sf, uint16_t* c, int64_t M, int64_t N, int64_t K,
                                         int64_t ldc, uint64_t wait_limit_ns, void* stream);

/* Size of the library-owned device scratch array used by
 * gemm_fp4_bf16_fwd_noalloc (32 MiB; taken on a device by the first call
 * there, held until the process exits). */
#define MXFP4_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * gemm_fp4_bf16_fwd_noalloc -- the same operation as gemm_fp4_bf16_fwd
 * (Y[M,N] = X[M,K] . W[N,K]^T through MXFP4, bf16 in/out) for callers that
 * cannot allocate device memory: a plugin whose device memory all belongs to
 * the host framework's allocator and which is handed only its inputs and
 * outputs, or code that must not make allocating CUDA calls where it runs.
 * It takes no workspace; the quantized X and W go to a file-scope device
 * array of MXFP4_NOALLOC_SCRATCH_BYTES inside the library.  The pages have no
 * counterpart to this entry point: it exists for those callers only.
 *   Arguments: checked as gemm_fp4_bf16_fwd checks them, in the same order
 *   and with the same errors; M == 0 or N == 0 is a no-op.  Then
 *   mxfp4_workspace_bytes(MXFP4_OP_FWD, M, N, K) must not exceed
 *   MXFP4_NOALLOC_SCRATCH_BYTES, else MXFP4_ERR_WORKSPACE and nothing is
 *   launched.
 *   First call on a device: CUDA loads the library's device code lazily, so
 *   the first call on each device loads the array -- the one moment its
 *   32 MiB of device memory is taken.  That call fails with MXFP4_ERR_CUDA
 *   (cudaErrorMemoryAllocation in mxfp4_last_cuda_error) if the device is
 *   full: make it before the host framework reserves its memory pool, and
 *   before any stream capture.  It also looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it.  Later
 *   calls allocate nothing: no cudaMalloc, cudaFree or allocating library
 *   call.
 *   All calls share the one array: calls whose work overlaps on the GPU
 *   (other streams, other host threads) race on it.
 */
mxfp4_status gemm_fp4_bf16_fwd_noalloc(const uint16_t* x, const uint16_t* w, uint16_t* y,
                                       int64_t M, int64_t N, int64_t K, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_H_ */

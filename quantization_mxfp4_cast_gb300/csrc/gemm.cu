// Block-scaled MXFP4 GEMM, C[M,N] (bf16) = A[M,K] . B[N,K]^T, on the
// fifth-generation tensor cores of sm_103a.
//
// Method: jax-aiter README, "Supported ops" table, rows "FP4 GEMM (low-level)"
// (pre-quantized fp4x2 inputs with e8m0 block scales) and "FP4 GEMM
// (training)" (A[M,K] . B[N,K]^T with BF16 output; forward, dA and dB all
// run through it).  The pages' kernels are AMD assembly for MI355X; this is an
// independent design for GB300:
//   * persistent CTAs (one per SM), tile 128 x 256 of C, K step 256;
//   * warp 0 lane 0: TMA producer -- codes by cp.async.bulk.tensor with the
//     128-byte swizzle (one 256-element K slab is exactly one 128-byte
//     swizzle row), scales by plain bulk copies of whole 512-byte scale tiles
//     (the cast writes scales in the tensor-memory copy layout, so no
//     reshuffle is needed), into a 4-stage shared-memory ring;
//   * warp 1 lane 0: tensor-core issuer -- tcgen05.cp moves each stage's
//     scales into tensor memory, then four tcgen05.mma.kind::mxf4 (K = 64
//     each, two UE8M0 scales per row per MMA) accumulate into a 128 x 256
//     fp32 tensor-memory accumulator; tcgen05.commit releases the stage;
//   * warps 2-5: epilogue -- tcgen05.ld of the accumulator (each warp its
//     32-lane sub-partition), fp32 -> bf16 round-to-nearest-even, stores.
// M and N tails come from the TMA out-of-bounds zero fill plus masked stores;
// a K tail (K % 64 == 32) reads zero codes past K.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

// Device-side status word: MXFP4_OK (0), or MXFP4_ERR_TIMEOUT once a pipeline
// wait of the GEMM gave up.
__device__ int g_device_status = 0;

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 256;              // elements per stage
constexpr int kBKBytes = kBK / 2;     // 128 bytes = one swizzle row
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBKBytes;          // 16 KiB
constexpr int kBStage = kBN * kBKBytes;          // 32 KiB
constexpr int kSfaStage = (kBM / 128) * 2 * 512;  // 1 row tile x 2 K tiles
constexpr int kSfbStage = (kBN / 128) * 2 * 512;  // 2 row tiles x 2 K tiles
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;
constexpr uint32_t kSfCol0 = kBN;
// per stage: SFA 2 K tiles x 4 columns, SFB 2 K tiles x 2 row tiles x 4 columns
constexpr uint32_t kSfaCols = 8;
constexpr uint32_t kSfStageCols = kSfaCols + 16;
static_assert(kSfCol0 + kStages * kSfStageCols <= kTmemCols, "tensor memory budget");

constexpr int kRingBytes = kStages * (kAStage + kBStage + kSfaStage + kSfbStage);
constexpr int kSmemBytes = kRingBytes + 256 + 1024;  // + barriers, + alignment slack

// Instruction descriptor, kind::mxf4: A and B E2M1 (format 1) K-major, D fp32,
// N >> 3 at bit 17, UE8M0 scales (bit 23), M >> 4 at bit 24.  The scale
// factor ids (bits 4-5 for B, 29-30 for A) select which byte pair of the
// 32-bit tensor-memory scale column an MMA reads.
constexpr uint32_t kIdescBase = (1u << 7) | (1u << 10) | (uint32_t(kBN >> 3) << 17) | (1u << 23) |
                                (uint32_t(kBM >> 4) << 24);

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(__uint_as_float(hi_f32)),
      "f"(__uint_as_float(lo_f32)));
  return out;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs args, int num_mt, int num_nt, int num_kt, int ktiles128,
                     int b_rowtiles) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled operand tiles.
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStages * kAStage;
  uint8_t* sSfa = sB + kStages * kBStage;
  uint8_t* sSfb = sSfa + kStages * kSfaStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSfb + kStages * kSfbStage);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4 * 32);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = num_mt * num_nt;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        const int mt = t % num_mt, nt = t / num_mt;
        const int nbt = min(2, b_rowtiles - nt * 2);
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_device_status)) {
            ok = false;
            break;
          }
          const int kg0 = kt * 2;
          const uint32_t sf_bytes = uint32_t(min(2, ktiles128 - kg0)) * 512u;
          mbar_arrive_expect_tx(&full[stage], kAStage + kBStage + sf_bytes * (1 + nbt));
          tma_load_2d(sA + stage * kAStage, &tmA, &full[stage], kt * kBKBytes, mt * kBM);
          tma_load_2d(sB + stage * kBStage, &tmB, &full[stage], kt * kBKBytes, nt * kBN);
          bulk_load(sSfa + stage * kSfaStage,
                    args.a_sf + (static_cast<int64_t>(mt) * ktiles128 + kg0) * 512, sf_bytes,
                    &full[stage]);
          for (int j = 0; j < nbt; ++j)
            bulk_load(sSfb + stage * kSfbStage + j * 1024,
                      args.b_sf + (static_cast<int64_t>(nt * 2 + j) * ktiles128 + kg0) * 512,
                      sf_bytes, &full[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, &g_device_status)) break;
        tc_fence_after();
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&full[stage], phase, abort_flag, &g_device_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nkg = min(2, ktiles128 - kt * 2);
          const uint32_t sf_col = tmem_base + kSfCol0 + stage * kSfStageCols;
          const uint32_t sfa_addr = smem_u32(sSfa + stage * kSfaStage);
          const uint32_t sfb_addr = smem_u32(sSfb + stage * kSfbStage);
          for (int g = 0; g < nkg; ++g) {
            tc_cp_32x128b_warpx4(sf_col + g * 4, make_smem_desc(sfa_addr + g * 512, 0, 128, 0));
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tc_cp_32x128b_warpx4(sf_col + kSfaCols + g * 8 + j * 4,
                                   make_smem_desc(sfb_addr + j * 1024 + g * 512, 0, 128, 0));
          }
          const uint32_t a_addr = smem_u32(sA + stage * kAStage);
          const uint32_t b_addr = smem_u32(sB + stage * kBStage);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            if (static_cast<int64_t>(kt) * kBK + ks * 64 >= args.K) break;
            const uint32_t g = ks >> 1, sf_id = (ks & 1) * 2;
            const uint64_t adesc = make_smem_desc(a_addr + ks * 32, 16, 1024, 2);
            const uint64_t bdesc = make_smem_desc(b_addr + ks * 32, 16, 1024, 2);
            const uint32_t idesc = kIdescBase | (sf_id << 4) | (sf_id << 29);
            tc_mma_mxf4(tmem_base + kAccCol, adesc, bdesc, idesc, sf_col + g * 4,
                        sf_col + kSfaCols + g * 8, (kt | ks) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // the tensor-memory lane quarter this warp may read
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const int mt = t % num_mt, nt = t / num_mt;
      if (!mbar_wait(acc_full, acc_phase, abort_flag, &g_device_status)) break;
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + ch * 32, r);
        tmem_ld_wait();
        const int64_t col = static_cast<int64_t>(nt) * kBN + ch * 32;
        if (row < args.M && col < args.N) {
          uint32_t p[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) p[j] = pack_bf16x2(r[2 * j], r[2 * j + 1]);
          uint16_t* dst = args.c + row * args.ldc + col;
          if (col + 32 <= args.N) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
          } else {
            const int n_left = static_cast<int>(args.N - col);
            for (int e = 0; e < n_left; ++e)
              dst[e] = static_cast<uint16_t>((e & 1) ? (p[e >> 1] >> 16) : (p[e >> 1] & 0xFFFFu));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty);
      acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

__global__ void fill_zero_bf16_kernel(uint16_t* c, int64_t M, int64_t N, int64_t ldc) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c[(i / N) * ldc + (i % N)] = 0;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D map over a [rows, K/2] byte matrix, boxes of box_rows x 128 bytes,
// 128-byte swizzle, zero fill out of bounds.
bool make_codes_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t k_bytes,
                    uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(k_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), box_rows};
  cuuint32_t estrides[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides,
                  box, estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t read_device_status(int* value, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_status, sizeof(int));
  if (e != cudaSuccess || !reset) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
}

cudaError_t launch_fill_zero_bf16(uint16_t* c, int64_t M, int64_t N, int64_t ldc,
                                  cudaStream_t stream) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int64_t total = M * N;
  const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 152 * 8));
  fill_zero_bf16_kernel<<<blocks, 256, 0, stream>>>(c, M, N, ldc);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs& args, cudaStream_t stream) {
  if (args.M == 0 || args.N == 0) return cudaSuccess;
  if (args.K == 0) return launch_fill_zero_bf16(args.c, args.M, args.N, args.ldc, stream);
  CUtensorMap tmA, tmB;
  if (!make_codes_map(&tmA, args.a, args.M, args.K / 2, kBM) ||
      !make_codes_map(&tmB, args.b, args.N, args.K / 2, kBN))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_mxf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int num_mt = static_cast<int>((args.M + kBM - 1) / kBM);
  const int num_nt = static_cast<int>((args.N + kBN - 1) / kBN);
  const int num_kt = static_cast<int>((args.K + kBK - 1) / kBK);
  const int ktiles128 = static_cast<int>((args.K + 127) / 128);
  const int b_rowtiles = static_cast<int>((args.N + 127) / 128);
  const int64_t tiles = static_cast<int64_t>(num_mt) * num_nt;
  const int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
  gemm_mxf4_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, args, num_mt, num_nt, num_kt,
                                                           ktiles128, b_rowtiles);
  return cudaGetLastError();
}

}  // namespace mxfp4

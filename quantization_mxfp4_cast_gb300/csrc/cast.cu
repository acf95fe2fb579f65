// BF16 -> MXFP4 cast kernels (row-wise, column-wise transposed, or both in
// one pass), with the optional 32-point Walsh-Hadamard transform per block.
//
// Method: jax-aiter README, "Supported ops" table, row "MXFP4 Cast"
// (CastMxfp4JA / CastMxfp4DualJA: BF16 to E2M1 elements + E8M0 block scales,
// with a transposed copy and a GEMM-ready scale layout), and "Quick start"
// (grad_out is cast with a Hadamard transform).  Numeric readings: block of
// 32, scale 2^(floor(log2 amax) - 2) clamped to [2^-127, 2^127], round to
// nearest even onto the E2M1 grid with saturation at 6, sign kept, NaN/Inf
// block -> scale 0xFF and codes 0.
//
// Design (HBM-bound: 2 bytes read, ~0.53 bytes written per element per
// direction; the arithmetic is kept to a few instructions per element so the
// ALU pipes stay below the memory rate):
//   * persistent CTAs (as many as fit on the GPU), 256 threads each, walking
//     128 x 128 tiles of x; each tile arrives in shared memory by two TMA
//     loads (64-column halves, 128-byte swizzle, zero fill past the edges)
//     into a double buffer, so the next tile's load overlaps this tile's
//     arithmetic and stores;
//   * row pass: from the shared-memory tile, one lane per 32-element block
//     (four 16-byte reads, conflict-free because of the swizzle); block amax
//     as a tree of packed, NaN-propagating bf16 magnitude maxima; the
//     power-of-two scaling as an exact bf16x2 multiply; packing by
//     cvt.rn.satfinite.e2m1x2.f32 (which keeps the sign of values that round
//     to zero); the row-wise Hadamard in registers;
//   * column pass: from the same shared-memory tile (untransformed); each
//     thread takes a column pair x 32 rows (conflict-free 4-byte reads) and
//     treats the two columns as the two halves of packed words -- one packed
//     max per row gives both amaxes, one bf16x2 multiply scales both, and the column
//     Hadamard runs both columns through one f32x2 butterfly network; 16
//     bytes of codes are stored per column;
//   * a 128 x 128 tile owns exactly one 512-byte scale tile of each output
//     (128 rows x 4 blocks), assembled in shared memory (double-buffered, so
//     one barrier per tile suffices) and written with one coalesced store,
//     padding included.
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mxfp4 {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;

// E4M3 codes of 4 values, element 0 in the low byte.  The conversion rounds
// to nearest even and saturates at +-448 (cvt puts its first source in the
// upper byte, hence the swapped operands).
__device__ __forceinline__ uint32_t cvt4_e4m3(float v0, float v1, float v2, float v3) {
  uint32_t out;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return out;
}

// Code words of one 32-element block from an accessor v(i) of its scaled fp32
// values: 4 words of E2M1 pairs (MXFP4) or 8 words of E4M3 bytes (MXFP8).
template <bool kFp8, typename V>
__device__ __forceinline__ void block_codes(V v, uint32_t* out) {
  if constexpr (kFp8) {
#pragma unroll
    for (int g = 0; g < 8; ++g) out[g] = cvt4_e4m3(v(4 * g), v(4 * g + 1), v(4 * g + 2), v(4 * g + 3));
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g)
      out[g] = cvt8_e2m1(v(8 * g), v(8 * g + 1), v(8 * g + 2), v(8 * g + 3), v(8 * g + 4), v(8 * g + 5),
                         v(8 * g + 6), v(8 * g + 7));
  }
}

__device__ __forceinline__ int sf_in_tile(int r, int b) { return (r & 31) * 16 + (r >> 5) * 4 + b; }

// A 128 x 128 bf16 tile in shared memory is two 128-row halves of 64 columns
// (128 bytes per row), each written by one TMA load with the 128-byte
// swizzle: the 16-byte chunk k of row r sits at chunk position k ^ (r % 8).
// Both passes below read it without bank conflicts: eight lanes reading the
// same chunk of eight consecutive rows, or 32 lanes reading 4-byte words of
// one row, always land on distinct banks.
constexpr int kHalfBytes = kTile * 128;
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr int kSfTileBytes = 512;
constexpr int kCastSmemBytes = 2 * kTileBytes + 4 * kSfTileBytes + 64 + 1024;

template <bool kRow, bool kCol, bool kFp8>
__global__ void __launch_bounds__(kThreads, 3)
    cast_kernel(const __grid_constant__ CUtensorMap tmX, const CastArgs args, int col_tiles,
                int num_tiles, int* status) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: the swizzle pattern follows address bits 7..9.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* bufs = smem;                               // two tiles
  uint8_t* sf_row_tiles = smem + 2 * kTileBytes;      // two 512-byte scale tiles (row output)
  uint8_t* sf_col_tiles = sf_row_tiles + 2 * kSfTileBytes;  // two (column output)
  uint64_t* full = reinterpret_cast<uint64_t*>(sf_col_tiles + 2 * kSfTileBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t rows = args.rows, cols = args.cols;
  const bool linear = (args.flags & kFlagScaleLinear) != 0;

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Tile t covers rows 128 * (t / col_tiles), columns 128 * (t % col_tiles).
  // The TMA zero-fills whatever lies past the tensor's edge (including a
  // half that starts beyond the last column).
  auto issue = [&](int t, int b) {
    const int x = (t % col_tiles) * kTile, y = (t / col_tiles) * kTile;
    uint8_t* dst = bufs + b * kTileBytes;
    mbar_arrive_expect_tx(&full[b], kTileBytes);
    tma_load_2d(dst, &tmX, &full[b], x, y);
    tma_load_2d(dst + kHalfBytes, &tmX, &full[b], x + kTile / 2, y);
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmX);
    for (int b = 0; b < 2; ++b) {
      const int t = static_cast<int>(blockIdx.x) + b * static_cast<int>(gridDim.x);
      if (t < num_tiles) issue(t, b);
    }
  }

  // Tile coordinates advance by the grid size each step.
  int tile_x = static_cast<int>(blockIdx.x) % col_tiles;
  int tile_y = static_cast<int>(blockIdx.x) / col_tiles;
  const int step_x = static_cast<int>(gridDim.x) % col_tiles;
  const int step_y = static_cast<int>(gridDim.x) / col_tiles;

  int it = 0;
  for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
  const int b = it & 1;
  if (!mbar_wait(&full[b], (it >> 1) & 1, abort_flag, status)) break;
  const uint8_t* tile = bufs + b * kTileBytes;
  const int64_t c0 = static_cast<int64_t>(tile_x) * kTile;
  const int64_t r0 = static_cast<int64_t>(tile_y) * kTile;
  uint8_t* sf_row_tile = sf_row_tiles + b * kSfTileBytes;
  uint8_t* sf_col_tile = sf_col_tiles + b * kSfTileBytes;

  static_assert(!(kFp8 && kRow), "MXFP8 is produced column-wise only");
  // ---------------------------------------------------------------- row pass
  // One lane per 32-element block: warp w, lane l take tile row
  // 8 w + (l % 8) (+ 64 in the second iteration), block l / 8 of that row.
  if constexpr (kRow) {
    const bool had = (args.flags & kFlagHadamardRow) != 0;
    const int kb = lane >> 3;
    const int xk = ((kb & 1) * 4) ^ (lane & 7);  // chunk 4 (kb % 2) + j sits at xk ^ j
    const bool col_ok = c0 + kb * 32 < cols;      // cols is a multiple of 32
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const int row = warp * 8 + (lane & 7) + ri * 64;
      const uint8_t* rowp = tile + (kb >> 1) * kHalfBytes + row * 128;
      uint32_t v[16];  // elements 2i (low half), 2i + 1 of the block
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 q = *reinterpret_cast<const uint4*>(rowp + ((xk ^ j) << 4));
        v[4 * j] = q.x;
        v[4 * j + 1] = q.y;
        v[4 * j + 2] = q.z;
        v[4 * j + 3] = q.w;
      }
      uint4 codes;
      BlockScale s;
      if (!had) {
        uint32_t m = tree_absmax_bf16x2<16>(v);
        m = absmax_bf16x2(m, __byte_perm(m, 0, 0x1032));  // both halves hold the block max
        s = block_scale((m & 0x7FFFu) << 16);
        const uint16_t mb = static_cast<uint16_t>(s.mult_bf16);
        codes.x = quantize8_bf16(v[0], v[1], v[2], v[3], mb);
        codes.y = quantize8_bf16(v[4], v[5], v[6], v[7], mb);
        codes.z = quantize8_bf16(v[8], v[9], v[10], v[11], mb);
        codes.w = quantize8_bf16(v[12], v[13], v[14], v[15], mb);
        if (s.nonfinite) codes = make_uint4(0u, 0u, 0u, 0u);
      } else {
        float y[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          y[2 * i] = bf16_times<false>(v[i], kBf16One);
          y[2 * i + 1] = bf16_times<true>(v[i], kBf16One);
        }
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j & h) continue;
            const float a = y[j], c = y[j + h];
            y[j] = __fadd_rn(a, c);
            y[j + h] = __fsub_rn(a, c);
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __fmul_rn(y[j], kInvSqrt32);
        s = block_scale(__float_as_uint(amax32([&](int i) { return y[i]; })));
        codes.x = quantize8(y, s);
        codes.y = quantize8(y + 8, s);
        codes.z = quantize8(y + 16, s);
        codes.w = quantize8(y + 24, s);
      }
      const int64_t grow = r0 + row;
      if (col_ok && grow < rows)
        *reinterpret_cast<uint4*>(args.q_row + grow * (cols / 2) + (c0 + kb * 32) / 2) = codes;
      if (linear) {
        if (col_ok && grow < rows) args.sf_row[grow * (cols / 32) + (c0 / 32) + kb] = (uint8_t)s.byte;
      } else {
        sf_row_tile[sf_in_tile(row, kb)] = (uint8_t)s.byte;
      }
    }
  }

  // ---------------------------------------------------------------- column pass
  if constexpr (kCol) {
    const bool had = (args.flags & kFlagHadamardCol) != 0;
    const int p = tid & 63;   // column pair: tile columns 2p (low halves), 2p+1 (high halves)
    const int rb = tid >> 6;  // 32-row block of the tile
    const uint8_t* colp = tile + (p >> 5) * kHalfBytes + rb * 32 * 128 + (p & 3) * 4;
    const int ch = (p & 31) >> 2;  // 16-byte chunk of the pair within its row half
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
      w[i] = *reinterpret_cast<const uint32_t*>(colp + i * 128 + ((ch ^ (i & 7)) << 4));
    const bool rows_ok = r0 + rb * 32 < rows;  // rows is a multiple of 32
    // MXFP4: 16 code bytes per column block; MXFP8 (E4M3, column output only): 32
    constexpr int kWords = kFp8 ? 8 : 4;
    constexpr int kEmax = kFp8 ? 8 : 2;
    BlockScale sa, sb;
    uint32_t ca[kWords], cb[kWords];  // codes of column 2p and 2p+1
    if (!had) {
      const uint32_t m = tree_absmax_bf16x2<32>(w) & 0x7FFF7FFFu;
      sa = block_scale<kEmax>(m << 16);
      sb = block_scale<kEmax>(m & 0xFFFF0000u);
      const uint16_t ma = static_cast<uint16_t>(sa.mult_bf16), mb = static_cast<uint16_t>(sb.mult_bf16);
      block_codes<kFp8>([&](int i) { return bf16_times<false>(w[i], ma); }, ca);
      block_codes<kFp8>([&](int i) { return bf16_times<true>(w[i], mb); }, cb);
    } else {
      // both columns through one 32-point butterfly network on fp32 pairs
      uint64_t y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = pk2(bf16_times<false>(w[i], kBf16One), bf16_times<true>(w[i], kBf16One));
#pragma unroll
      for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j & h) continue;
          const uint64_t a = y[j], c = y[j + h];
          y[j] = add2(a, c);
          y[j + h] = sub2(a, c);
        }
      }
      // amax of the transformed block: rounding is monotonic, so the largest
      // |RN(h * c)| is RN(max |h| * c); the NaN-propagating max keeps NaN/Inf.
      const float ha = amax32([&](int i) { return lo2(y[i]); });
      const float hb = amax32([&](int i) { return hi2(y[i]); });
      sa = block_scale<kEmax>(__float_as_uint(__fmul_rn(ha, kInvSqrt32)));
      sb = block_scale<kEmax>(__float_as_uint(__fmul_rn(hb, kInvSqrt32)));
      // v = RN(h * c) * 2^-e.  RN(h * (c * 2^-e)) is the same number when
      // c * 2^-e stays normal (scale byte <= 250) and every transformed value
      // RN(h * c) that is subnormal in fp32 (< 2^-126, so |v| < 2^(1 - byte))
      // lands below the format's zero threshold either way: byte >= 3 for
      // E2M1 (|v| < 1/4), byte >= 11 for E4M3 (|v| <= 2^-10).  Outside that
      // range the two roundings are kept apart.
      constexpr uint32_t kFusedMin = kFp8 ? 11u : 3u;
      if ((sa.byte - kFusedMin) <= 250u - kFusedMin && (sb.byte - kFusedMin) <= 250u - kFusedMin) {
        const uint64_t m2 = pk2(__fmul_rn(kInvSqrt32, sa.mult), __fmul_rn(kInvSqrt32, sb.mult));
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = mul2(y[i], m2);
      } else {
        const uint64_t c2 = pk2(kInvSqrt32, kInvSqrt32);
        const uint64_t m2 = pk2(sa.mult, sb.mult);
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = mul2(mul2(y[i], c2), m2);
      }
      block_codes<kFp8>([&](int i) { return lo2(y[i]); }, ca);
      block_codes<kFp8>([&](int i) { return hi2(y[i]); }, cb);
    }
    if (sa.nonfinite) {
#pragma unroll
      for (int g = 0; g < kWords; ++g) ca[g] = 0u;
    }
    if (sb.nonfinite) {
#pragma unroll
      for (int g = 0; g < kWords; ++g) cb[g] = 0u;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = 2 * p + half;
      const BlockScale& s = half ? sb : sa;
      const uint32_t* cw = half ? cb : ca;
      const int64_t gcol = c0 + c;
      if (gcol < cols && rows_ok) {
        // codes of T^T: [cols, rows] bytes (MXFP8) or [cols, rows / 2] (MXFP4)
        uint4* dst = reinterpret_cast<uint4*>(args.q_col + (gcol * rows + r0 + rb * 32) / (kFp8 ? 1 : 2));
        dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        if constexpr (kFp8) dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      }
      if (linear) {
        if (gcol < cols && rows_ok) args.sf_col[gcol * (rows / 32) + (r0 / 32) + rb] = (uint8_t)s.byte;
      } else {
        sf_col_tile[sf_in_tile(c, rb)] = (uint8_t)s.byte;
      }
    }
  }

  // ---------------------------------------------------------------- scale tiles
  // One barrier per tile: the tile buffer is consumed and both scale tiles
  // are complete.  The scale tiles are double-buffered, so the next tile's
  // passes write the other pair while warps 0 and 1 copy these out; the
  // pair is reused only after the next tile's barrier, which those warps
  // reach after their copies.
  __syncthreads();
  if (tid == 0) {
    const int tn = t + 2 * static_cast<int>(gridDim.x);
    if (tn < num_tiles) {
      fence_proxy_async_shared();  // order this tile's generic reads before the async refill
      issue(tn, b);
    }
  }
  if (!linear) {
    if constexpr (kRow) {
      if (warp == 0) {
        const int64_t ktiles = (cols + kTile - 1) / kTile;
        const int64_t tile_idx = static_cast<int64_t>(tile_y) * ktiles + tile_x;
        reinterpret_cast<uint4*>(args.sf_row + tile_idx * 512)[lane] =
            reinterpret_cast<const uint4*>(sf_row_tile)[lane];
      }
    }
    if constexpr (kCol) {
      if (warp == 1) {
        const int64_t ktiles = (rows + kTile - 1) / kTile;
        const int64_t tile_idx = static_cast<int64_t>(tile_x) * ktiles + tile_y;
        reinterpret_cast<uint4*>(args.sf_col + tile_idx * 512)[lane] =
            reinterpret_cast<const uint4*>(sf_col_tile)[lane];
      }
    }
  }
  tile_x += step_x;
  tile_y += step_y;
  if (tile_x >= col_tiles) {
    tile_x -= col_tiles;
    ++tile_y;
  }
  }
}

}  // namespace

namespace {

template <bool kRow, bool kCol, bool kFp8 = false>
cudaError_t launch_cast_t(const CUtensorMap& tm, const CastArgs& args, int col_tiles, int num_tiles,
                          int dev, cudaStream_t stream) {
  static std::atomic<int> ctas_per_sm[64];
  int per_sm = (dev >= 0 && dev < 64) ? ctas_per_sm[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(cast_kernel<kRow, kCol, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kCastSmemBytes);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, cast_kernel<kRow, kCol, kFp8>, kThreads,
                                                      kCastSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    per_sm = std::max(1, occ) * sms;  // resident CTAs on the whole GPU
    if (dev >= 0 && dev < 64) ctas_per_sm[dev].store(per_sm, std::memory_order_relaxed);
  }
  int* status = device_status_word();
  if (status == nullptr) return cudaErrorUnknown;
  // cudaLaunchKernelEx reports this launch's own error; the thread's last
  // error may hold a stale, unrelated one (e.g. a not-ready query result).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(num_tiles, per_sm)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kCastSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, cast_kernel<kRow, kCol, kFp8>, tm, args, col_tiles, num_tiles, status);
}

}  // namespace

cudaError_t launch_cast(const CastArgs& args, cudaStream_t stream) {
  if (args.rows == 0 || args.cols == 0) return cudaSuccess;
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap tm;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(args.cols), static_cast<cuuint64_t>(args.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(args.ldx) * 2};
  cuuint32_t box[2] = {kTile / 2, kTile};  // 64 columns (128 bytes) x 128 rows
  cuuint32_t estrides[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(args.x), dims, strides, box,
         estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int64_t col_tiles = (args.cols + kTile - 1) / kTile;
  const int64_t row_tiles = (args.rows + kTile - 1) / kTile;
  if (col_tiles * row_tiles > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  const int num_tiles = static_cast<int>(col_tiles * row_tiles);
  const bool row = args.q_row != nullptr, col = args.q_col != nullptr;
  if (args.flags & kFlagFp8) {
    if (row || !col) return cudaErrorInvalidValue;  // MXFP8: column output only
    return launch_cast_t<false, true, true>(tm, args, int(col_tiles), num_tiles, dev, stream);
  }
  if (row && col) return launch_cast_t<true, true>(tm, args, int(col_tiles), num_tiles, dev, stream);
  if (row) return launch_cast_t<true, false>(tm, args, int(col_tiles), num_tiles, dev, stream);
  if (col) return launch_cast_t<false, true>(tm, args, int(col_tiles), num_tiles, dev, stream);
  return cudaSuccess;
}

}  // namespace mxfp4

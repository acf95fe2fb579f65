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
// Design (HBM-bound: 2 bytes read, ~1.06 bytes written per element per
// direction):
//   * one CTA = one 128 x 128 tile of x, 256 threads;
//   * row pass: 16-byte coalesced loads, 4 lanes per 32-element block (8
//     elements each), block amax by two xor-shuffles on the integer
//     magnitude bits (NaN/Inf sort above every finite value), the row-wise
//     Hadamard as three in-register butterfly stages plus two shuffle stages,
//     packing by cvt.rn.satfinite.e2m1x2.f32;
//   * column pass: the untransformed tile is staged in shared memory; each
//     thread takes a column pair x 32 rows (conflict-free 4-byte reads), runs
//     the column Hadamard in registers, and stores 16 bytes of codes per
//     column;
//   * a 128 x 128 tile owns exactly one 512-byte scale tile of each output
//     (128 rows x 4 blocks), assembled in shared memory and written with one
//     coalesced store, padding included.
#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr uint32_t kFullMask = 0xFFFFFFFFu;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// E2M1 codes of 8 values, element 0 in the low nibble of byte 0.  The
// conversion rounds to nearest even and saturates at +-6.
__device__ __forceinline__ uint32_t cvt8_e2m1(float v0, float v1, float v2, float v3, float v4,
                                              float v5, float v6, float v7) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return out;
}

// Sign bit of each of the 8 inputs moved to bit 3 of its nibble, so that a
// negative value that rounds to zero (and -0) keeps its sign.
__device__ __forceinline__ uint32_t sign_nibbles(const float* y) {
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s |= (__float_as_uint(y[i]) >> 31) << (4 * i + 3);
  return s;
}

__device__ __forceinline__ uint32_t abs_bits(float f) { return __float_as_uint(f) & 0x7FFFFFFFu; }

// From the largest magnitude's bit pattern: scale byte and the exact
// power-of-two multiplier 2^-e.  For a finite amax with biased exponent E,
// floor(log2 amax) - 2 + 127 = E - 129 + 127 = E - 2, clamped at 0 (E = 0
// covers zero and subnormals).
struct BlockScale {
  uint32_t byte;
  float mult;
  bool nonfinite;
};

__device__ __forceinline__ BlockScale block_scale(uint32_t amax_bits) {
  BlockScale s;
  s.nonfinite = amax_bits >= 0x7F800000u;
  const int e_biased = static_cast<int>(amax_bits >> 23);
  const int byte = e_biased > 2 ? e_biased - 2 : 0;
  s.mult = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);
  s.byte = s.nonfinite ? 0xFFu : static_cast<uint32_t>(byte);
  return s;
}

// Codes of 8 elements under the block's scale.
__device__ __forceinline__ uint32_t quantize8(const float* y, const BlockScale& s) {
  if (s.nonfinite) return 0u;
  const float m = s.mult;
  uint32_t c = cvt8_e2m1(__fmul_rn(y[0], m), __fmul_rn(y[1], m), __fmul_rn(y[2], m),
                         __fmul_rn(y[3], m), __fmul_rn(y[4], m), __fmul_rn(y[5], m),
                         __fmul_rn(y[6], m), __fmul_rn(y[7], m));
  return c | sign_nibbles(y);
}

// fp32 value nearest to 1/sqrt(32).
constexpr float kInvSqrt32 = 0x1.6a09e6p-3f;  // bit pattern 0x3E3504F3

// Butterfly stages h = 1, 2, 4 of the 32-point transform on this thread's 8
// consecutive elements: pair (j, j+h), j & h == 0, becomes (a + b, a - b).
__device__ __forceinline__ void fwht_local8(float* y) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j & h) continue;
      const float a = y[j], b = y[j + h];
      y[j] = __fadd_rn(a, b);
      y[j + h] = __fsub_rn(a, b);
    }
  }
}

// Stage across lanes: this lane's element j pairs with element j of lane
// (lane ^ lane_mask).  The lane holding the lower index keeps a + b, the
// other keeps a - b with a the lower lane's value.
__device__ __forceinline__ void fwht_cross(float* y, int lane_mask, bool upper) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float p = __shfl_xor_sync(kFullMask, y[j], lane_mask);
    y[j] = upper ? __fsub_rn(p, y[j]) : __fadd_rn(y[j], p);
  }
}

__device__ __forceinline__ void fwht32_inreg(float* y) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j & h) continue;
      const float a = y[j], b = y[j + h];
      y[j] = __fadd_rn(a, b);
      y[j + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) y[j] = __fmul_rn(y[j], kInvSqrt32);
}

__device__ __forceinline__ int sf_in_tile(int r, int b) { return (r & 31) * 16 + (r >> 5) * 4 + b; }

template <bool kRow, bool kCol>
__global__ void __launch_bounds__(kThreads) cast_kernel(const CastArgs args) {
  __shared__ __align__(16) uint16_t xs[kCol ? kTile : 1][kCol ? kTile : 8];
  __shared__ __align__(16) uint8_t sf_row_tile[kRow ? 512 : 16];
  __shared__ __align__(16) uint8_t sf_col_tile[kCol ? 512 : 16];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t rows = args.rows, cols = args.cols;
  const bool linear = (args.flags & kFlagScaleLinear) != 0;

  // ---------------------------------------------------------------- load
  // Iteration i covers tile rows 16i .. 16i+15: warp w takes rows 16i+2w and
  // 16i+2w+1, 16 lanes x 8 elements per row.
  const int c8 = (lane & 15) * 8;
  const bool col_ok = c0 + c8 < cols;  // cols is a multiple of 32
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = i * 16 + warp * 2 + (lane >> 4);
    if (col_ok && r0 + row < rows)
      v[i] = ld_stream_16(args.x + (r0 + row) * args.ldx + c0 + c8);
    else
      v[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  if constexpr (kCol) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = i * 16 + warp * 2 + (lane >> 4);
      *reinterpret_cast<uint4*>(&xs[row][c8]) = v[i];
    }
  }

  // ---------------------------------------------------------------- row pass
  if constexpr (kRow) {
    const bool had = (args.flags & kFlagHadamardRow) != 0;
    const int q = lane & 3;  // which 8 of the block's 32 elements
    const int kb = (lane & 15) >> 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = i * 16 + warp * 2 + (lane >> 4);
      float y[8] = {bf16lo(v[i].x), bf16hi(v[i].x), bf16lo(v[i].y), bf16hi(v[i].y),
                    bf16lo(v[i].z), bf16hi(v[i].z), bf16lo(v[i].w), bf16hi(v[i].w)};
      if (had) {
        fwht_local8(y);
        fwht_cross(y, 1, (q & 1) != 0);
        fwht_cross(y, 2, (q & 2) != 0);
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(y[j], kInvSqrt32);
      }
      uint32_t amax = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = max(amax, abs_bits(y[j]));
      amax = max(amax, __shfl_xor_sync(kFullMask, amax, 1));
      amax = max(amax, __shfl_xor_sync(kFullMask, amax, 2));
      const BlockScale s = block_scale(amax);
      const uint32_t codes = quantize8(y, s);
      const int64_t grow = r0 + row;
      if (col_ok && grow < rows)
        *reinterpret_cast<uint32_t*>(args.q_row + grow * (cols / 2) + (c0 + c8) / 2) = codes;
      if (q == 0) {
        if (linear) {
          if (col_ok && grow < rows) args.sf_row[grow * (cols / 32) + (c0 + c8) / 32] = (uint8_t)s.byte;
        } else {
          sf_row_tile[sf_in_tile(row, kb)] = (uint8_t)s.byte;
        }
      }
    }
  }

  // ---------------------------------------------------------------- column pass
  if constexpr (kCol) {
    __syncthreads();
    const bool had = (args.flags & kFlagHadamardCol) != 0;
    const int p = tid & 63;   // column pair: tile columns 2p, 2p+1
    const int rb = tid >> 6;  // 32-row block of the tile
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(&xs[rb * 32 + i][2 * p]);
    const bool rows_ok = r0 + rb * 32 < rows;  // rows is a multiple of 32
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = 2 * p + half;
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = half ? bf16hi(w[i]) : bf16lo(w[i]);
      if (had) fwht32_inreg(y);
      uint32_t amax = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = max(amax, abs_bits(y[i]));
      const BlockScale s = block_scale(amax);
      uint4 codes;
      codes.x = quantize8(y + 0, s);
      codes.y = quantize8(y + 8, s);
      codes.z = quantize8(y + 16, s);
      codes.w = quantize8(y + 24, s);
      const int64_t gcol = c0 + c;
      if (gcol < cols && rows_ok)
        *reinterpret_cast<uint4*>(args.q_col + gcol * (rows / 2) + (r0 + rb * 32) / 2) = codes;
      if (linear) {
        if (gcol < cols && rows_ok) args.sf_col[gcol * (rows / 32) + (r0 / 32) + rb] = (uint8_t)s.byte;
      } else {
        sf_col_tile[sf_in_tile(c, rb)] = (uint8_t)s.byte;
      }
    }
  }

  // ---------------------------------------------------------------- scale tiles
  if (!linear) {
    __syncthreads();
    if constexpr (kRow) {
      if (tid < 32) {
        const int64_t ktiles = (cols + kTile - 1) / kTile;
        const int64_t tile = static_cast<int64_t>(blockIdx.y) * ktiles + blockIdx.x;
        reinterpret_cast<uint4*>(args.sf_row + tile * 512)[tid] =
            reinterpret_cast<const uint4*>(sf_row_tile)[tid];
      }
    }
    if constexpr (kCol) {
      if (tid >= 32 && tid < 64) {
        const int64_t ktiles = (rows + kTile - 1) / kTile;
        const int64_t tile = static_cast<int64_t>(blockIdx.x) * ktiles + blockIdx.y;
        reinterpret_cast<uint4*>(args.sf_col + tile * 512)[tid - 32] =
            reinterpret_cast<const uint4*>(sf_col_tile)[tid - 32];
      }
    }
  }
}

}  // namespace

cudaError_t launch_cast(const CastArgs& args, cudaStream_t stream) {
  if (args.rows == 0 || args.cols == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((args.cols + kTile - 1) / kTile),
            static_cast<unsigned>((args.rows + kTile - 1) / kTile));
  const bool row = args.q_row != nullptr, col = args.q_col != nullptr;
  if (row && col)
    cast_kernel<true, true><<<grid, kThreads, 0, stream>>>(args);
  else if (row)
    cast_kernel<true, false><<<grid, kThreads, 0, stream>>>(args);
  else if (col)
    cast_kernel<false, true><<<grid, kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace mxfp4

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
//     128 x 128 tiles of x; each tile arrives in shared memory by one TMA
//     load (zero fill past the edges) into a double buffer, so the next
//     tile's load overlaps this tile's arithmetic and stores;
//   * row pass: from the shared-memory tile, 2 lanes per 32-element block
//     (16 elements each); block amax as a packed, NaN-propagating bf16
//     magnitude max plus one xor-shuffle; the power-of-two scaling as an
//     exact bf16x2 multiply; packing by cvt.rn.satfinite.e2m1x2.f32 (which
//     keeps the sign of values that round to zero); the row-wise Hadamard as
//     four in-register butterfly stages plus one shuffle stage;
//   * column pass: from the same shared-memory tile (untransformed); each
//     thread takes a column pair x 32 rows (conflict-free 4-byte reads) and
//     treats the two columns as the two halves of packed words -- one packed
//     max per row gives both amaxes, one bf16x2 multiply scales both, and the column
//     Hadamard runs both columns through one f32x2 butterfly network; 16
//     bytes of codes are stored per column;
//   * a 128 x 128 tile owns exactly one 512-byte scale tile of each output
//     (128 rows x 4 blocks), assembled in shared memory and written with one
//     coalesced store, padding included.
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr uint32_t kFullMask = 0xFFFFFFFFu;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

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

__device__ __forceinline__ uint32_t abs_bits(float f) { return __float_as_uint(f) & 0x7FFFFFFFu; }

// max(m, |x|) with NaN propagation (an Inf or NaN anywhere makes the block
// non-finite).
__device__ __forceinline__ float max_nan_abs(float m, float x) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(x)));
  return r;
}

// Elementwise max(|a|, |b|) of bf16 pairs, NaN-propagating (sign bits of
// the result are the XOR of the inputs' and must be masked off).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic, IEEE round-to-nearest per lane).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// From the largest magnitude's bit pattern: scale byte and the exact
// power-of-two multiplier 2^-e (as fp32, and as a bf16 bit pattern).  For a
// finite amax with biased exponent E, floor(log2 amax) - 2 + 127 = E - 2,
// clamped at 0 (E = 0 covers zero and subnormals).
struct BlockScale {
  uint32_t byte;
  float mult;
  uint32_t mult_bf16;
  bool nonfinite;
};

__device__ __forceinline__ BlockScale block_scale(uint32_t amax_bits) {
  BlockScale s;
  s.nonfinite = amax_bits >= 0x7F800000u;
  const int e_biased = static_cast<int>(amax_bits >> 23);
  const int byte = e_biased > 2 ? e_biased - 2 : 0;
  s.mult = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);
  s.mult_bf16 = static_cast<uint32_t>(254 - byte) << 7;
  s.byte = s.nonfinite ? 0xFFu : static_cast<uint32_t>(byte);
  return s;
}

// Codes of 8 fp32 elements under the block's scale (the conversion keeps the
// sign of values that round to zero, so no fix-up is needed).
__device__ __forceinline__ uint32_t quantize8(const float* y, const BlockScale& s) {
  if (s.nonfinite) return 0u;
  const float m = s.mult;
  return cvt8_e2m1(__fmul_rn(y[0], m), __fmul_rn(y[1], m), __fmul_rn(y[2], m),
                   __fmul_rn(y[3], m), __fmul_rn(y[4], m), __fmul_rn(y[5], m),
                   __fmul_rn(y[6], m), __fmul_rn(y[7], m));
}

// Codes of the 8 bf16 elements in 4 packed words (element 2i in the low half
// of word i), scaled in bf16: the product of a bf16 and a power of two is
// exact down to 2^-126, and anything smaller rounds to a signed zero code
// either way.
__device__ __forceinline__ uint32_t quantize8_bf16(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                                   uint32_t mult2) {
  const uint32_t p0 = mul_bf16x2(w0, mult2), p1 = mul_bf16x2(w1, mult2);
  const uint32_t p2 = mul_bf16x2(w2, mult2), p3 = mul_bf16x2(w3, mult2);
  return cvt8_e2m1(bf16lo(p0), bf16hi(p0), bf16lo(p1), bf16hi(p1), bf16lo(p2), bf16hi(p2),
                   bf16lo(p3), bf16hi(p3));
}

// fp32 value nearest to 1/sqrt(32).
constexpr float kInvSqrt32 = 0x1.6a09e6p-3f;  // bit pattern 0x3E3504F3

__device__ __forceinline__ int sf_in_tile(int r, int b) { return (r & 31) * 16 + (r >> 5) * 4 + b; }

constexpr int kTileBytes = kTile * kTile * 2;  // one 128 x 128 bf16 tile
constexpr int kCastSmemBytes = 2 * kTileBytes + 2 * 512 + 64 + 128;

template <bool kRow, bool kCol>
__global__ void __launch_bounds__(kThreads, 3)
    cast_kernel(const __grid_constant__ CUtensorMap tmX, const CastArgs args, int col_tiles,
                int num_tiles, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  uint16_t* bufs = reinterpret_cast<uint16_t*>(smem);  // two [128][128] bf16 tiles
  uint8_t* sf_row_tile = smem + 2 * kTileBytes;
  uint8_t* sf_col_tile = sf_row_tile + 512;
  uint64_t* full = reinterpret_cast<uint64_t*>(sf_col_tile + 512);
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
  // The TMA zero-fills whatever lies past the tensor's edge.
  auto issue = [&](int t, int b) {
    mbar_arrive_expect_tx(&full[b], kTileBytes);
    tma_load_2d(bufs + b * kTile * kTile, &tmX, &full[b], (t % col_tiles) * kTile,
                (t / col_tiles) * kTile);
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmX);
    for (int b = 0; b < 2; ++b) {
      const int t = static_cast<int>(blockIdx.x) + b * static_cast<int>(gridDim.x);
      if (t < num_tiles) issue(t, b);
    }
  }

  int it = 0;
  for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
  const int b = it & 1;
  if (!mbar_wait(&full[b], (it >> 1) & 1, abort_flag, status)) break;
  const uint16_t* xs = bufs + b * kTile * kTile;  // xs[row * kTile + col]
  const int64_t c0 = static_cast<int64_t>(t % col_tiles) * kTile;
  const int64_t r0 = static_cast<int64_t>(t / col_tiles) * kTile;
  const int tile_x = t % col_tiles, tile_y = t / col_tiles;

  // ---------------------------------------------------------------- row pass
  // Iteration it covers tile rows 32 it .. 32 it + 31: warp w takes rows
  // 32 it + 4 w .. + 3; two lanes per 32-element block, 16 elements each.
  if constexpr (kRow) {
    const bool had = (args.flags & kFlagHadamardRow) != 0;
    const int kb = (lane >> 1) & 3;  // block of the row (tile-local)
    const int hf = lane & 1;         // which 16 of the block's 32 elements
    const int e0 = kb * 32 + hf * 16;
    const bool col_ok = c0 + kb * 32 < cols;  // cols is a multiple of 32
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int row = it * 32 + warp * 4 + (lane >> 3);
      const uint4 va = *reinterpret_cast<const uint4*>(xs + row * kTile + e0);
      const uint4 vb = *reinterpret_cast<const uint4*>(xs + row * kTile + e0 + 8);
      uint2 codes;
      BlockScale s;
      if (!had) {
        uint32_t m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(va.x, va.y), absmax_bf16x2(va.z, va.w)),
                                   absmax_bf16x2(absmax_bf16x2(vb.x, vb.y), absmax_bf16x2(vb.z, vb.w)));
        m = absmax_bf16x2(m, __shfl_xor_sync(kFullMask, m, 1));
        m = absmax_bf16x2(m, __byte_perm(m, 0, 0x1032));  // both halves hold the block max
        s = block_scale((m & 0x7FFFu) << 16);
        const uint32_t mult2 = s.mult_bf16 * 0x00010001u;
        codes.x = quantize8_bf16(va.x, va.y, va.z, va.w, mult2);
        codes.y = quantize8_bf16(vb.x, vb.y, vb.z, vb.w, mult2);
        if (s.nonfinite) codes = make_uint2(0u, 0u);
      } else {
        // 32-point transform: stages h = 1, 2, 4, 8 inside the lane's 16
        // elements, h = 16 across the lane pair.
        float y[16] = {bf16lo(va.x), bf16hi(va.x), bf16lo(va.y), bf16hi(va.y),
                       bf16lo(va.z), bf16hi(va.z), bf16lo(va.w), bf16hi(va.w),
                       bf16lo(vb.x), bf16hi(vb.x), bf16lo(vb.y), bf16hi(vb.y),
                       bf16lo(vb.z), bf16hi(vb.z), bf16lo(vb.w), bf16hi(vb.w)};
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j & h) continue;
            const float a = y[j], b = y[j + h];
            y[j] = __fadd_rn(a, b);
            y[j + h] = __fsub_rn(a, b);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float q = __shfl_xor_sync(kFullMask, y[j], 1);
          y[j] = hf ? __fsub_rn(q, y[j]) : __fadd_rn(y[j], q);
        }
        uint32_t amax = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          y[j] = __fmul_rn(y[j], kInvSqrt32);
          amax = max(amax, abs_bits(y[j]));
        }
        amax = max(amax, __shfl_xor_sync(kFullMask, amax, 1));
        s = block_scale(amax);
        codes.x = quantize8(y, s);
        codes.y = quantize8(y + 8, s);
      }
      const int64_t grow = r0 + row;
      if (col_ok && grow < rows)
        *reinterpret_cast<uint2*>(args.q_row + grow * (cols / 2) + (c0 + e0) / 2) = codes;
      if (hf == 0) {
        if (linear) {
          if (col_ok && grow < rows) args.sf_row[grow * (cols / 32) + (c0 / 32) + kb] = (uint8_t)s.byte;
        } else {
          sf_row_tile[sf_in_tile(row, kb)] = (uint8_t)s.byte;
        }
      }
    }
  }

  // ---------------------------------------------------------------- column pass
  if constexpr (kCol) {
    const bool had = (args.flags & kFlagHadamardCol) != 0;
    const int p = tid & 63;   // column pair: tile columns 2p (low halves), 2p+1 (high halves)
    const int rb = tid >> 6;  // 32-row block of the tile
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(xs + (rb * 32 + i) * kTile + 2 * p);
    const bool rows_ok = r0 + rb * 32 < rows;  // rows is a multiple of 32
    BlockScale sa, sb;
    uint4 ca, cb;  // codes of column 2p and 2p+1
    if (!had) {
      uint32_t m = w[0];
#pragma unroll
      for (int i = 1; i < 32; ++i) m = absmax_bf16x2(m, w[i]);
      m &= 0x7FFF7FFFu;
      sa = block_scale(m << 16);
      sb = block_scale(m & 0xFFFF0000u);
      const uint32_t mult2 = sa.mult_bf16 | (sb.mult_bf16 << 16);
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = mul_bf16x2(w[i], mult2);
      uint32_t* pa = &ca.x;
      uint32_t* pb = &cb.x;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t* u = w + 8 * g;
        pa[g] = cvt8_e2m1(bf16lo(u[0]), bf16lo(u[1]), bf16lo(u[2]), bf16lo(u[3]), bf16lo(u[4]),
                          bf16lo(u[5]), bf16lo(u[6]), bf16lo(u[7]));
        pb[g] = cvt8_e2m1(bf16hi(u[0]), bf16hi(u[1]), bf16hi(u[2]), bf16hi(u[3]), bf16hi(u[4]),
                          bf16hi(u[5]), bf16hi(u[6]), bf16hi(u[7]));
      }
      if (sa.nonfinite) ca = make_uint4(0u, 0u, 0u, 0u);
      if (sb.nonfinite) cb = make_uint4(0u, 0u, 0u, 0u);
    } else {
      // both columns through one 32-point butterfly network on fp32 pairs
      uint64_t y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = pk2(bf16lo(w[i]), bf16hi(w[i]));
#pragma unroll
      for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j & h) continue;
          const uint64_t a = y[j], b = y[j + h];
          y[j] = add2(a, b);
          y[j + h] = sub2(a, b);
        }
      }
      // amax of the transformed block: rounding is monotonic, so the largest
      // |RN(h * c)| is RN(max |h| * c); the NaN-propagating max keeps NaN/Inf.
      float ha = 0.f, hb = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        ha = max_nan_abs(ha, lo2(y[i]));
        hb = max_nan_abs(hb, hi2(y[i]));
      }
      sa = block_scale(__float_as_uint(__fmul_rn(ha, kInvSqrt32)));
      sb = block_scale(__float_as_uint(__fmul_rn(hb, kInvSqrt32)));
      // v = RN(h * c) * 2^-e.  For scale bytes 3..250 this equals
      // RN(h * (c * 2^-e)) exactly: c * 2^-e stays normal, and a transformed
      // value RN(h * c) small enough to be subnormal gives |v| < 1/4, code 0
      // either way.  Outside that range the two roundings are kept apart.
      if ((sa.byte - 3u) <= 247u && (sb.byte - 3u) <= 247u) {
        const uint64_t m2 = pk2(__fmul_rn(kInvSqrt32, sa.mult), __fmul_rn(kInvSqrt32, sb.mult));
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = mul2(y[i], m2);
      } else {
        const uint64_t c2 = pk2(kInvSqrt32, kInvSqrt32);
        const uint64_t m2 = pk2(sa.mult, sb.mult);
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = mul2(mul2(y[i], c2), m2);
      }
      uint32_t* pa = &ca.x;
      uint32_t* pb = &cb.x;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint64_t* u = y + 8 * g;
        pa[g] = cvt8_e2m1(lo2(u[0]), lo2(u[1]), lo2(u[2]), lo2(u[3]), lo2(u[4]), lo2(u[5]),
                          lo2(u[6]), lo2(u[7]));
        pb[g] = cvt8_e2m1(hi2(u[0]), hi2(u[1]), hi2(u[2]), hi2(u[3]), hi2(u[4]), hi2(u[5]),
                          hi2(u[6]), hi2(u[7]));
      }
      if (sa.nonfinite) ca = make_uint4(0u, 0u, 0u, 0u);
      if (sb.nonfinite) cb = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = 2 * p + half;
      const BlockScale& s = half ? sb : sa;
      const int64_t gcol = c0 + c;
      if (gcol < cols && rows_ok)
        *reinterpret_cast<uint4*>(args.q_col + gcol * (rows / 2) + (r0 + rb * 32) / 2) = half ? cb : ca;
      if (linear) {
        if (gcol < cols && rows_ok) args.sf_col[gcol * (rows / 32) + (r0 / 32) + rb] = (uint8_t)s.byte;
      } else {
        sf_col_tile[sf_in_tile(c, rb)] = (uint8_t)s.byte;
      }
    }
  }

  // ---------------------------------------------------------------- scale tiles
  __syncthreads();  // the tile buffer is consumed and both scale tiles are complete
  if (tid == 0) {
    const int tn = t + 2 * static_cast<int>(gridDim.x);
    if (tn < num_tiles) {
      fence_proxy_async_shared();  // order this tile's generic reads before the async refill
      issue(tn, b);
    }
  }
  if (!linear) {
    if constexpr (kRow) {
      if (tid < 32) {
        const int64_t ktiles = (cols + kTile - 1) / kTile;
        const int64_t tile = static_cast<int64_t>(tile_y) * ktiles + tile_x;
        reinterpret_cast<uint4*>(args.sf_row + tile * 512)[tid] =
            reinterpret_cast<const uint4*>(sf_row_tile)[tid];
      }
    }
    if constexpr (kCol) {
      if (tid >= 32 && tid < 64) {
        const int64_t ktiles = (rows + kTile - 1) / kTile;
        const int64_t tile = static_cast<int64_t>(tile_x) * ktiles + tile_y;
        reinterpret_cast<uint4*>(args.sf_col + tile * 512)[tid - 32] =
            reinterpret_cast<const uint4*>(sf_col_tile)[tid - 32];
      }
    }
  }
  __syncthreads();  // scale tiles written out before the next tile refills them
  }
}

}  // namespace

namespace {

template <bool kRow, bool kCol>
cudaError_t launch_cast_t(const CUtensorMap& tm, const CastArgs& args, int col_tiles, int num_tiles,
                          int dev, cudaStream_t stream) {
  static std::atomic<int> ctas_per_sm[64];
  int per_sm = (dev >= 0 && dev < 64) ? ctas_per_sm[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(cast_kernel<kRow, kCol>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kCastSmemBytes);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, cast_kernel<kRow, kCol>, kThreads,
                                                      kCastSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    per_sm = std::max(1, occ) * sms;  // resident CTAs on the whole GPU
    if (dev >= 0 && dev < 64) ctas_per_sm[dev].store(per_sm, std::memory_order_relaxed);
  }
  int* status = device_status_word();
  if (status == nullptr) return cudaErrorUnknown;
  const int grid = std::min(num_tiles, per_sm);
  cast_kernel<kRow, kCol><<<grid, kThreads, kCastSmemBytes, stream>>>(tm, args, col_tiles, num_tiles,
                                                                     status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cast(const CastArgs& args, cudaStream_t stream) {
  if (args.rows == 0 || args.cols == 0) return cudaSuccess;
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap tm;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(args.cols), static_cast<cuuint64_t>(args.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(args.ldx) * 2};
  cuuint32_t box[2] = {kTile, kTile};
  cuuint32_t estrides[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(args.x), dims, strides, box,
         estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
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
  if (row && col) return launch_cast_t<true, true>(tm, args, int(col_tiles), num_tiles, dev, stream);
  if (row) return launch_cast_t<true, false>(tm, args, int(col_tiles), num_tiles, dev, stream);
  if (col) return launch_cast_t<false, true>(tm, args, int(col_tiles), num_tiles, dev, stream);
  return cudaSuccess;
}

}  // namespace mxfp4

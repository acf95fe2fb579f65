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
// issue slots stay below the memory rate):
//   * the work unit is a slab of 32 rows x 128 columns (8 KB of bf16) that ONE
//     warp quantizes completely -- its 128 row blocks and its 128 column
//     blocks -- so no warp waits for another one to finish a tile;
//   * one persistent CTA per SM owns the 128 x 128 tiles blockIdx.x + k *
//     gridDim.x.  A producer thread streams their slabs with TMA (two 32 x 64
//     boxes, 128-byte swizzle, zero fill past the edges) into a ring of 20
//     slots (measured: 24 slots leave no room for the column-code buffers
//     below, 16 are 4-8% slower); 15 consumer warps take the slabs in order
//     from a shared counter as they become free, so the four slabs of a tile
//     are quantized side by
//     side (balanced to within one slab per SM, with loads in flight beyond the
//     slabs being quantized).  A slot's sequence word tells a consumer when
//     the producer has claimed the slot for its slab (and publishes the
//     slab's coordinates), so no consumer waits on a barrier phase that
//     belongs to an earlier use of the slot;
//   * one launch may cast up to four tensors (mxfp4_cast_dual_grouped): their
//     tiles are numbered one cast after another and every slab carries its
//     cast's index, so the pipeline fills and drains once for all of them.
//     Hadamard flags that differ between the casts are read per slab at run
//     time; otherwise they are template parameters;
//   * a tile's column codes (128 columns x 64 bytes: four 16-byte pieces per
//     column, one from each slab's warp) and its two 512-byte scale tiles are
//     assembled in shared memory; the warp that finishes the tile's last slab
//     writes the codes with one TMA store (64-byte swizzle, clipped at the
//     tensor's edges) and the scale tiles whole.  Each warp storing its 16-byte
//     pieces straight to memory, 32 columns apart per instruction, made the
//     dual cast's column output the bottleneck (measured: with no arithmetic
//     at all the old kernel ran as fast as the real one; staging the pieces
//     took X[8192, 14336] from 5.1 to 6.4 TB/s, 0.94 of the copy rate).  A
//     partial last round of tiles, dealt out slab by slab over the CTAs, and
//     the linear scale layout keep the direct stores;
//   * row blocks: lane l takes row 8i + l % 8 (i = 0..3), block l / 8, read as
//     four 16-byte chunks (conflict-free under the swizzle); a store
//     instruction writes 8 rows x 64 contiguous bytes;
//   * column blocks: each lane takes two column pairs x 32 rows as the halves
//     of packed 4-byte words (conflict-free reads), so one packed max gives
//     both amaxes and one f32x2 butterfly network transforms both columns;
//   * block amax as a tree of packed, NaN-propagating bf16 magnitude maxima;
//     scaling by the exact power of two with the mixed-precision fma (or the
//     fused 1/sqrt(32) * 2^-e multiply after the transform, where that is
//     exact); packing by cvt.rn.satfinite.e2m1x2.f32, which keeps the sign of
//     values that round to zero;
//   * row blocks are padded to whole 128-row tiles (slabs past the last row
//     are zero fill), so every byte of every scale tile, padding included, is
//     written (0x00 for padding);
//   * launched with programmatic stream serialization: the barrier set-up
//     overlaps the end of the previous kernel in the stream, and every read of
//     x and write of an output waits for that kernel to complete.
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mxfp4 {
namespace {

constexpr int kSlabRows = 32;
constexpr int kSlabCols = 128;
constexpr int kHalfBytes = kSlabRows * 128;  // one 64-column half: 32 rows x 128 bytes
constexpr int kSlabBytes = 2 * kHalfBytes;   // 8 KB
constexpr int kStages = 20;                  // ring slots
constexpr int kConsumerWarps = 15;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + the producer warp
constexpr int kSfBufs = 8;                   // scale-tile staging buffers (tiles in progress)
constexpr int kCqBufs = 6;                   // column-code staging buffers (tiles in progress)
constexpr int kCqBytes = 128 * 64;           // a tile's column codes: 128 columns x 64 bytes
constexpr int kSfStageBytes = 2 * 512;       // one tile's row and column scale tiles
constexpr int kBarrierBytes = 2 * kStages * 8 + 3 * kStages * 4 + 2 * kSfBufs * 4 + kCqBufs * 4 + 16;
constexpr int kCastSmemBytes =
    kStages * kSlabBytes + kSfBufs * kSfStageBytes + kCqBufs * kCqBytes + kBarrierBytes + 1024;
static_assert(kCastSmemBytes <= 232448, "shared memory");
static_assert(kStages % 4 == 0, "a tile's four slabs take four consecutive ring slots");
constexpr uint32_t kNoSlab = 0xFFFFFFFFu;

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

// Up to kMaxCastGroup casts in one launch: their tiles are numbered one cast
// after another, and every slab carries its cast's index.
constexpr int kMaxCastGroup = 4;
struct CastMaps {
  CUtensorMap x[kMaxCastGroup];   // bf16 input, 32 x 64 boxes
  CUtensorMap qc[kMaxCastGroup];  // MXFP4 column codes, 128 x 64-byte boxes
};
struct CastGroup {
  CastArgs args;
  int col_tiles, row_tiles128;
  int tile_end;  // tiles of this cast and the ones before it
};
struct CastGroups {
  CastGroup g[kMaxCastGroup];
  int count, num_tiles;
};

// The cast of tile t (0 <= t < num_tiles) and t's index within that cast.
__device__ __forceinline__ int cast_of_tile(const CastGroups& p, int t, int& lt) {
  int g = 0;
  while (g + 1 < p.count && t >= p.g[g].tile_end) ++g;
  lt = g == 0 ? t : t - p.g[g - 1].tile_end;
  return g;
}

// Byte of (row r, block b) inside a 512-byte scale tile of 128 rows x 4 blocks.
__device__ __forceinline__ int sf_in_tile(int r, int b) { return (r & 31) * 16 + ((r >> 5) & 3) * 4 + b; }

// Bounded wait until a shared word holds `want` (acquire).  The polls back
// off with a short sleep, so that waiting warps leave the issue slots to the
// producer and to the warps that have data.
__device__ __forceinline__ bool wait_word(const uint32_t* p, uint32_t want, volatile int* abort_flag,
                                          int* status_word) {
  if (ld_acquire_shared(p) == want) return true;
  const unsigned long long t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    __nanosleep(64);
    if (ld_acquire_shared(p) == want) return true;
    if ((++spins & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicExch(status_word, 6 /* MXFP4_ERR_TIMEOUT */);
        return false;
      }
    }
  }
}

// Tile t of x covers rows 128 * (t / col_tiles) and columns 128 * (t %
// col_tiles).  With G = gridDim.x, the first floor(num_tiles / G) * G tiles
// are dealt out whole: the CTA owns tiles t = blockIdx.x + k * G, and its local
// slab i = 4k + j is tile k's 32-row block j, so the four slabs of a tile are
// handed out one after the other and quantized side by side by four warps --
// the column codes of a tile's column (four 16-byte pieces) are written
// together, and its two 512-byte scale tiles are assembled in shared memory
// and written whole by the warp that finishes the tile's last slab.  The
// slabs of the last, partial round of tiles are dealt out one by one over all
// CTAs (tail slab u goes to CTA u mod G), so that every CTA's work is within
// one slab of every other's; a tail slab writes its scale bytes directly.
template <bool kRow, bool kCol, bool kFp8, int kHadRowMode, int kHadColMode>
__global__ void __launch_bounds__(kThreads, 1)
    cast_kernel(const __grid_constant__ CastMaps maps, const __grid_constant__ CastGroups p, int* status) {
  static_assert(!(kFp8 && kRow), "MXFP8 is produced column-wise only");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: the swizzle pattern follows address bits 7..9.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint8_t* sf_stage = smem + kStages * kSlabBytes;  // [kSfBufs][row tile, column tile]
  uint8_t* cq_stage = sf_stage + kSfBufs * kSfStageBytes;  // [kCqBufs][128 columns x 64 B], 64-byte swizzle
  uint64_t* full = reinterpret_cast<uint64_t*>(cq_stage + kCqBufs * kCqBytes);
  uint64_t* empty = full + kStages;
  uint32_t* seq = reinterpret_cast<uint32_t*>(empty + kStages);  // local slab that owns each slot
  uint32_t* slot_rb = seq + kStages;                                // its 32-row block
  uint32_t* slot_ct = slot_rb + kStages;                            // its 128-column tile
  uint32_t* sf_free = slot_ct + kStages;   // staging buffer b is free for local tile sf_free[b]
  int* tile_done = reinterpret_cast<int*>(sf_free + kSfBufs);      // slabs of the tile in b finished
  // column-code buffer b is free for local tile cq_free[b]
  uint32_t* cq_free = reinterpret_cast<uint32_t*>(tile_done + kSfBufs);
  int* counter = reinterpret_cast<int*>(cq_free + kCqBufs);          // next local slab to hand out
  volatile int* abort_flag = counter + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.num_tiles;
  // local slabs of this CTA: four per whole tile, then its tail slabs
  const int grid = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const int full_rounds = num_tiles / grid;
  const int tail_slabs = 4 * (num_tiles - full_rounds * grid);
  const int n_whole = 4 * full_rounds;
  const int n_local = n_whole + (cta < tail_slabs ? (tail_slabs - cta + grid - 1) / grid : 0);

  {  // set-up spread over the threads (one thread took ~1 us for it)
    const int t = threadIdx.x;
    if (t < kStages) {
      mbar_init(&full[t], 1);
      mbar_init(&empty[t], 1);
      seq[t] = kNoSlab;
      fence_barrier_init();
    } else if (t < kStages + kSfBufs) {
      sf_free[t - kStages] = static_cast<uint32_t>(t - kStages);
      tile_done[t - kStages] = 0;
    } else if (t < kStages + kSfBufs + kCqBufs) {
      cq_free[t - kStages - kSfBufs] = static_cast<uint32_t>(t - kStages - kSfBufs);
    } else if (t == kStages + kSfBufs + kCqBufs) {
      *counter = 0;
      *abort_flag = 0;
    }
  }
  if (threadIdx.x == 32 * kConsumerWarps)
    for (int g = 0; g < p.count; ++g) tma_prefetch_desc(&maps.x[g]);
  __syncthreads();
  // x may be the output of the previous kernel in the stream, and the outputs
  // may still be read by it: nothing below touches global memory before it ends.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      int slot = 0;
      uint32_t empty_parity = 1;  // from the second pass on: parity of the slot's previous release
      bool ok = true;
      int g = 0, tx = 0, ty = 0;  // the current whole tile: its cast and coordinates
      for (int i = 0; ok && i < n_local; ++i) {
        const int j = i & 3;
        int rb, ct;
        uint32_t tail_bit = 0;
        if (i < n_whole) {
          if (j == 0) {  // a new whole tile (32-bit divisions, once per four slabs)
            int lt;
            g = cast_of_tile(p, cta + (i >> 2) * grid, lt);
            ty = lt / p.g[g].col_tiles;
            tx = lt - ty * p.g[g].col_tiles;
          }
          rb = 4 * ty + j;
          ct = tx;
        } else {  // tail slab u of the partial round (a handful per CTA)
          const int u = cta + (i - n_whole) * grid;
          int lt;
          g = cast_of_tile(p, full_rounds * grid + u / 4, lt);
          rb = 4 * (lt / p.g[g].col_tiles) + (u & 3);
          ct = lt % p.g[g].col_tiles;
          tail_bit = 0x80000000u;
        }
        // the slot's previous slab (i - kStages) has been quantized
        if (i >= kStages && !mbar_wait(&empty[slot], empty_parity, abort_flag, status)) {
          ok = false;
          break;
        }
        slot_rb[slot] = static_cast<uint32_t>(rb) | tail_bit;
        slot_ct[slot] = static_cast<uint32_t>(ct) | (static_cast<uint32_t>(g) << 28);
        st_release_shared(&seq[slot], static_cast<uint32_t>(i));  // publishes the coordinates too
        uint8_t* dst = ring + slot * kSlabBytes;
        mbar_arrive_expect_tx(&full[slot], kSlabBytes);
        tma_load_2d(dst, &maps.x[g], &full[slot], ct * kSlabCols, rb * kSlabRows);
        tma_load_2d(dst + kHalfBytes, &maps.x[g], &full[slot], ct * kSlabCols + kSlabCols / 2, rb * kSlabRows);
        issued = i + 1;
        if (++slot == kStages) {
          slot = 0;
          empty_parity ^= 1u;
        }
      }
      // Every load issued has landed before the CTA may end (a consumer that
      // gave up may have left one unconsumed).  The last load into a slot
      // completes the phase its slab index gives; nothing follows it.
      volatile int keep_waiting = 0;  // not the CTA's abort flag: this wait must run its course
      for (int sl = 0; sl < kStages && sl < issued; ++sl) {
        const int last = sl + ((issued - 1 - sl) / kStages) * kStages;
        mbar_wait(&full[sl], (last / kStages) & 1, &keep_waiting, status);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  for (;;) {
    int i = 0;
    if (lane == 0) i = atomicAdd(counter, 1);
    i = __shfl_sync(0xFFFFFFFFu, i, 0);
    if (i >= n_local) break;
    const int slot = i % kStages;
    if (!wait_word(&seq[slot], static_cast<uint32_t>(i), abort_flag, status)) break;
    const uint32_t rbw = slot_rb[slot];  // 32-row block (published with seq), bit 31: tail slab
    const int rb = static_cast<int>(rbw & 0x7FFFFFFFu);
    const uint32_t ctw = slot_ct[slot];  // 128-column tile, bits 28-29: the cast
    const int ct = static_cast<int>(ctw & 0x0FFFFFFFu);
    const int g = static_cast<int>(ctw >> 28);
    const CastArgs& args = p.g[g].args;
    const int col_tiles = p.g[g].col_tiles, row_tiles128 = p.g[g].row_tiles128;
    const int64_t rows = args.rows, cols = args.cols;
    const bool linear = (args.flags & kFlagScaleLinear) != 0;
    const bool had_row = kHadRowMode == 2 ? (args.flags & kFlagHadamardRow) != 0 : kHadRowMode == 1;
    const bool had_col = kHadColMode == 2 ? (args.flags & kFlagHadamardCol) != 0 : kHadColMode == 1;
    // scale bytes: staged per whole tile, or straight to the tile layout (tail slab)
    const bool staged = !linear && (rbw >> 31) == 0;
    const int sfb = (i >> 2) % kSfBufs;  // the whole tile's staging buffer
    uint8_t* sf_row_stage = staged ? sf_stage + sfb * kSfStageBytes
                                   : args.sf_row + (static_cast<size_t>(rb >> 2) * col_tiles + ct) * 512;
    uint8_t* sf_col_stage = staged ? sf_row_stage + 512
                                   : args.sf_col + (static_cast<size_t>(ct) * row_tiles128 + (rb >> 2)) * 512;
    if (staged && !wait_word(&sf_free[sfb], static_cast<uint32_t>(i >> 2), abort_flag, status)) break;
    // column codes: assembled per whole tile in shared memory (64 contiguous
    // bytes per column) and written by one TMA store
    const bool cq_staged = staged && kCol && !kFp8;
    const int cqb = (i >> 2) % kCqBufs;
    if (cq_staged && !wait_word(&cq_free[cqb], static_cast<uint32_t>(i >> 2), abort_flag, status)) break;
    if (!mbar_wait(&full[slot], (i / kStages) & 1, abort_flag, status)) break;
    const uint8_t* tile = ring + slot * kSlabBytes;
    const int64_t c0 = static_cast<int64_t>(ct) * kSlabCols;
    const int64_t r0 = static_cast<int64_t>(rb) * kSlabRows;

    // ---------------------------------------------------------- row blocks
    if constexpr (kRow) {
      const int kb = lane >> 3;
      const int xk = ((kb & 1) * 4) ^ (lane & 7);  // chunk 4 (kb % 2) + j sits at xk ^ j
      const bool col_ok = c0 + kb * 32 < cols;      // cols is a multiple of 32
      const uint8_t* half = tile + (kb >> 1) * kHalfBytes;
#pragma unroll 1
      for (int it = 0; it < 4; ++it) {
        const int row = it * 8 + (lane & 7);
        const uint8_t* rowp = half + row * 128;
        uint32_t v[16];  // elements 2i (low half), 2i + 1 of the block
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 q = *reinterpret_cast<const uint4*>(rowp + ((xk ^ j) << 4));
          v[4 * j] = q.x;
          v[4 * j + 1] = q.y;
          v[4 * j + 2] = q.z;
          v[4 * j + 3] = q.w;
        }
        uint32_t c[4];
        BlockScale sc;
        if (!had_row) {
          sc = quantize_bf16_block(v, c);
        } else {
          float y[32];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            y[2 * k] = __uint_as_float(v[k] << 16);
            y[2 * k + 1] = __uint_as_float(v[k] & 0xFFFF0000u);
          }
          sc = quantize_hadamard_block(y, c);
        }
        const int64_t grow = r0 + row;
        if (col_ok && grow < rows)
          *reinterpret_cast<uint4*>(args.q_row + grow * (cols / 2) + (c0 + kb * 32) / 2) =
              make_uint4(c[0], c[1], c[2], c[3]);
        if (linear) {
          if (col_ok && grow < rows) args.sf_row[grow * (cols / 32) + (c0 / 32) + kb] = (uint8_t)sc.byte;
        } else {
          sf_row_stage[sf_in_tile(rb * 32 + row, kb)] = (uint8_t)sc.byte;
        }
      }
    }

    // ---------------------------------------------------------- column blocks
    if constexpr (kCol) {
      const bool rows_ok = r0 < rows;  // rows is a multiple of 32
      const int ch = lane >> 2;        // 16-byte chunk of the pair within its row half
      // MXFP4: 16 code bytes per column block; MXFP8 (E4M3, column output only): 32
      constexpr int kWords = kFp8 ? 8 : 4;
      constexpr int kEmax = kFp8 ? 8 : 2;
#pragma unroll 1
      for (int hp = 0; hp < 2; ++hp) {
        const uint8_t* colp = tile + hp * kHalfBytes + (lane & 3) * 4;
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
          w[k] = *reinterpret_cast<const uint32_t*>(colp + k * 128 + ((ch ^ (k & 7)) << 4));
        BlockScale sa, sb;
        uint32_t ca[kWords], cb[kWords];  // codes of columns 2p and 2p + 1
        if (!had_col) {
          const uint32_t m = tree_absmax_bf16x2<32>(w) & 0x7FFF7FFFu;
          sa = block_scale<kEmax>(m << 16);
          sb = block_scale<kEmax>(m & 0xFFFF0000u);
          const uint16_t ma = static_cast<uint16_t>(sa.mult_bf16), mb = static_cast<uint16_t>(sb.mult_bf16);
          block_codes<kFp8>([&](int k) { return bf16_times<false>(w[k], ma); }, ca);
          block_codes<kFp8>([&](int k) { return bf16_times<true>(w[k], mb); }, cb);
        } else {
          // both columns through one 32-point butterfly network on fp32 pairs
          uint64_t y[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) y[k] = pk2(bf16_times<false>(w[k], kBf16One), bf16_times<true>(w[k], kBf16One));
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
          const float ha = amax32([&](int k) { return lo2(y[k]); });
          const float hb = amax32([&](int k) { return hi2(y[k]); });
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
            for (int k = 0; k < 32; ++k) y[k] = mul2(y[k], m2);
          } else {
            const uint64_t c2 = pk2(kInvSqrt32, kInvSqrt32);
            const uint64_t m2 = pk2(sa.mult, sb.mult);
#pragma unroll
            for (int k = 0; k < 32; ++k) y[k] = mul2(mul2(y[k], c2), m2);
          }
          block_codes<kFp8>([&](int k) { return lo2(y[k]); }, ca);
          block_codes<kFp8>([&](int k) { return hi2(y[k]); }, cb);
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
          const int c = 64 * hp + 2 * lane + half;  // column within the slab
          const BlockScale& sc = half ? sb : sa;
          const uint32_t* cw = half ? cb : ca;
          const int64_t gcol = c0 + c;
          if (cq_staged) {
            // column c's 16 bytes of this slab (slab j = rb % 4 of the tile), chunk j of
            // the column's 64-byte row under the 64-byte swizzle the TMA store undoes
            const uint32_t dst =
                smem_u32(cq_stage + cqb * kCqBytes) + c * 64 + (((rb & 3) ^ ((c >> 1) & 3)) << 4);
            sts128(dst, cw[0], cw[1], cw[2], cw[3]);
          } else if (gcol < cols && rows_ok) {
            // codes of T^T: [cols, rows] bytes (MXFP8) or [cols, rows / 2] (MXFP4)
            uint4* dst = reinterpret_cast<uint4*>(args.q_col + (gcol * rows + r0) / (kFp8 ? 1 : 2));
            dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            if constexpr (kFp8) dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
          }
          if (linear) {
            if (gcol < cols && rows_ok) args.sf_col[gcol * (rows / 32) + rb] = (uint8_t)sc.byte;
          } else {
            sf_col_stage[sf_in_tile(c, rb & 3)] = (uint8_t)sc.byte;
          }
        }
      }
    }
    if (cq_staged) fence_proxy_async_shared();  // this lane's column codes, before the TMA store reads them
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // the slot may be refilled
    if (staged) {
      // the warp that finishes the tile's last slab writes its scale tiles
      int done = 0;
      if (lane == 0) {
        __threadfence_block();  // this warp's staging bytes before the count
        done = atomicAdd(&tile_done[sfb], 1);
      }
      if (__shfl_sync(0xFFFFFFFFu, done, 0) == 3) {
        __threadfence_block();  // the other three warps' staging bytes
        const size_t tile_y = static_cast<size_t>(rb >> 2), tile_x = static_cast<size_t>(ct);
        if constexpr (kRow)
          reinterpret_cast<uint4*>(args.sf_row + (tile_y * col_tiles + tile_x) * 512)[lane] =
              reinterpret_cast<const uint4*>(sf_row_stage)[lane];
        if constexpr (kCol)
          reinterpret_cast<uint4*>(args.sf_col + (tile_x * row_tiles128 + tile_y) * 512)[lane] =
              reinterpret_cast<const uint4*>(sf_col_stage)[lane];
        if (cq_staged && lane == 0) {
          // the tile's column codes: 128 columns x 64 bytes (rows past the end
          // and columns past cols are clipped by the store)
          tma_store_2d(&maps.qc[g], cq_stage + cqb * kCqBytes, static_cast<int32_t>(tile_y * 64),
                       static_cast<int32_t>(tile_x * 128));
          bulk_commit_group();
          bulk_wait_group_read0();  // the buffer has been read
          st_release_shared(&cq_free[cqb], static_cast<uint32_t>((i >> 2) + kCqBufs));
        }
        __syncwarp();
        if (lane == 0) {
          tile_done[sfb] = 0;
          st_release_shared(&sf_free[sfb], static_cast<uint32_t>((i >> 2) + kSfBufs));
        }
      }
    }
  }
  if (lane == 0) bulk_wait_group0();  // this warp's column-code stores are complete
}

template <bool kRow, bool kCol, bool kFp8, int kHadRowMode, int kHadColMode>
cudaError_t launch_cast_t(const CastMaps& maps, const CastGroups& groups, int dev, cudaStream_t stream) {
  auto kernel = cast_kernel<kRow, kCol, kFp8, kHadRowMode, kHadColMode>;
  static std::atomic<int> ctas[64];  // resident CTAs on the whole GPU, per device
  int grid = (dev >= 0 && dev < 64) ? ctas[dev].load(std::memory_order_relaxed) : 0;
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCastSmemBytes);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, kCastSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    grid = std::max(1, occ) * sms;
    if (dev >= 0 && dev < 64) ctas[dev].store(grid, std::memory_order_relaxed);
  }
  int* status = device_status_word();
  if (status == nullptr) return cudaErrorUnknown;
  // cudaLaunchKernelEx reports this launch's own error; the thread's last
  // error may hold a stale, unrelated one (e.g. a not-ready query result).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(4 * static_cast<int64_t>(groups.num_tiles), grid)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kCastSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, maps, groups, status);
}

// Hadamard flags of a launch: off (0) or on (1) for every cast in it, or per
// cast at run time (2) where they differ.
template <bool kRow, bool kCol, bool kFp8>
cudaError_t launch_had(const CastMaps& maps, const CastGroups& groups, int dev, cudaStream_t stream) {
  auto mode = [&](uint32_t flag, bool applies) {
    if (!applies) return 0;
    int on = 0;
    for (int g = 0; g < groups.count; ++g) on += (groups.g[g].args.flags & flag) != 0;
    return on == 0 ? 0 : (on == groups.count ? 1 : 2);
  };
  const int hr = mode(kFlagHadamardRow, kRow), hc = mode(kFlagHadamardCol, kCol);
  if constexpr (kRow && kCol) {
    if (hr == 2 || hc == 2) return launch_cast_t<true, true, kFp8, 2, 2>(maps, groups, dev, stream);
    if (hr && hc) return launch_cast_t<true, true, kFp8, 1, 1>(maps, groups, dev, stream);
    if (hr) return launch_cast_t<true, true, kFp8, 1, 0>(maps, groups, dev, stream);
    if (hc) return launch_cast_t<true, true, kFp8, 0, 1>(maps, groups, dev, stream);
    return launch_cast_t<true, true, kFp8, 0, 0>(maps, groups, dev, stream);
  } else if constexpr (kRow) {
    if (hr == 2) return launch_cast_t<true, false, kFp8, 2, 0>(maps, groups, dev, stream);
    if (hr) return launch_cast_t<true, false, kFp8, 1, 0>(maps, groups, dev, stream);
    return launch_cast_t<true, false, kFp8, 0, 0>(maps, groups, dev, stream);
  } else {
    if (hc == 2) return launch_cast_t<false, true, kFp8, 0, 2>(maps, groups, dev, stream);
    if (hc) return launch_cast_t<false, true, kFp8, 0, 1>(maps, groups, dev, stream);
    return launch_cast_t<false, true, kFp8, 0, 0>(maps, groups, dev, stream);
  }
}

// Tensor maps and tile counts of one cast; false if a map cannot be encoded
// or the tile counts leave the 32-bit range.
bool prepare_cast(const CastArgs& args, EncodeTiledFn fn, CUtensorMap* tm, CUtensorMap* tm_qc, CastGroup* grp) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(args.cols), static_cast<cuuint64_t>(args.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(args.ldx) * 2};
  cuuint32_t box[2] = {kSlabCols / 2, kSlabRows};  // 64 columns (128 bytes) x 32 rows
  cuuint32_t estrides[2] = {1, 1};
  if (fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(args.x), dims, strides, box,
         estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // column codes [cols, rows / 2] (MXFP4), stored a tile (128 columns x 64
  // bytes) at a time from a 64-byte-swizzled staging buffer
  *tm_qc = *tm;
  if (args.q_col != nullptr && (args.flags & kFlagFp8) == 0) {
    cuuint64_t qdims[2] = {static_cast<cuuint64_t>(args.rows / 2), static_cast<cuuint64_t>(args.cols)};
    cuuint64_t qstrides[1] = {static_cast<cuuint64_t>(args.rows / 2)};
    cuuint32_t qbox[2] = {64, 128};
    if (fn(tm_qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, args.q_col, qdims, qstrides, qbox, estrides,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const int64_t col_tiles = (args.cols + kSlabCols - 1) / kSlabCols;
  const int64_t row_tiles128 = (args.rows + 127) / 128;
  // whole 128 x 128 tiles: the slabs past the last row only write the zero
  // scales of the tile padding
  const int64_t num_tiles = row_tiles128 * col_tiles;
  if (4 * num_tiles > (int64_t(1) << 31) - 1 || row_tiles128 * 128 > (int64_t(1) << 31) - 1 ||
      col_tiles >= (int64_t(1) << 28))
    return false;
  grp->args = args;
  grp->col_tiles = static_cast<int>(col_tiles);
  grp->row_tiles128 = static_cast<int>(row_tiles128);
  grp->tile_end = static_cast<int>(num_tiles);  // made cumulative by the caller
  return true;
}

}  // namespace

cudaError_t launch_cast_grouped(const CastArgs* list, int count, cudaStream_t stream) {
  if (count < 1 || count > kMaxCastGroup) return cudaErrorInvalidValue;
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  CastMaps maps = {};
  CastGroups groups = {};
  int64_t tiles = 0;
  bool row = false, col = false, fp8 = false, first = true;
  for (int i = 0; i < count; ++i) {
    const CastArgs& args = list[i];
    if (args.rows == 0 || args.cols == 0) continue;
    const bool r = args.q_row != nullptr, c = args.q_col != nullptr, f = (args.flags & kFlagFp8) != 0;
    if (!r && !c) continue;
    // one kind of cast per launch: the same outputs and element format
    if (!first && (r != row || c != col || f != fp8)) return cudaErrorInvalidValue;
    row = r, col = c, fp8 = f, first = false;
    CastGroup& grp = groups.g[groups.count];
    if (!prepare_cast(args, fn, &maps.x[groups.count], &maps.qc[groups.count], &grp))
      return cudaErrorInvalidValue;
    tiles += grp.tile_end;
    if (4 * tiles > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
    grp.tile_end = static_cast<int>(tiles);
    ++groups.count;
  }
  if (groups.count == 0) return cudaSuccess;
  groups.num_tiles = static_cast<int>(tiles);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (fp8) {
    if (row || !col) return cudaErrorInvalidValue;  // MXFP8: column output only
    return launch_had<false, true, true>(maps, groups, dev, stream);
  }
  if (row && col) return launch_had<true, true, false>(maps, groups, dev, stream);
  if (row) return launch_had<true, false, false>(maps, groups, dev, stream);
  return launch_had<false, true, false>(maps, groups, dev, stream);
}

cudaError_t launch_cast(const CastArgs& args, cudaStream_t stream) {
  return launch_cast_grouped(&args, 1, stream);
}

}  // namespace mxfp4

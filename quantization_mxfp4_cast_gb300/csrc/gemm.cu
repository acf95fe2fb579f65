// Block-scaled MXFP4 GEMM, C[M,N] (bf16) = A[M,K] . B[N,K]^T, on the
// fifth-generation tensor cores of sm_103a.
//
// Method: jax-aiter README, "Supported ops" table, rows "FP4 GEMM (low-level)"
// (pre-quantized fp4x2 inputs with e8m0 block scales) and "FP4 GEMM
// (training)" (A[M,K] . B[N,K]^T with BF16 output; forward, dA and dB all
// run through it).  The pages' kernels are AMD assembly for MI355X; this is an
// independent design for GB300:
//   * CTA pairs (clusters of 2 on neighbouring SMs) run tcgen05.mma with
//     cta_group::2: one 256 x 256 output tile per pair, each SM holding 128
//     rows of A and 128 of the 256 rows of B, so every SM streams 8 KiB of
//     operands per 64-deep MMA step instead of 12 KiB;
//   * persistent: one pair per two SMs walks the tiles in groups of row
//     tiles, column tiles outer (L2 reuse of A and B across the concurrently
//     running tiles); a group holds as many row tiles as keep its A panel
//     within 24 MiB (measured at the Llama-3.1-8B down-projection shapes: 8
//     row tiles for K = 14336, 32 for K = 4096, 16 for K = 8192, each 1-3%
//     faster than the other two sizes);
//   * grouped: one launch may carry up to four independent GEMMs (their
//     tensor maps and tile counts in the kernel parameters), whose tiles are
//     numbered one GEMM after another; every role decodes a tile index the
//     same way, and the ring's stages run on across GEMMs of different K.
//     A training step's fwd, dgrad and wgrad then leave one partial last wave
//     instead of three (gemm_fp4_grouped; a gemm_fp4 call is the one-GEMM case);
//   * warps 0 and 14: TMA producers in each CTA -- warp 0 the FP4 codes with
//     the 128-byte swizzle (a 256-element K slab is one 128-byte swizzle row),
//     warp 14 the 512-byte scale tiles, which the cast already writes in the
//     tensor-memory copy layout (B's two 128-row tiles in one 3-D box), into
//     a 6-stage shared-memory ring (measured: 4 stages are 11% slower; the
//     5-stage ring of the output-cast instance is 4-6% slower with no cast
//     work).  The ring, not the tensor pipe, sets the pace: a stage's release
//     (the commit of its MMAs) comes ~1,000-2,000 cycles after they are
//     issued, so every link from release to refill counts;
//   * warps 2-5, in each CTA: scale stagers -- each takes one 32-lane quarter
//     of tensor memory and writes the stage's A and B scales there with
//     tcgen05.st (the layout the block-scaled MMA reads: lane i of every
//     quarter, column j = scales of row 32j + i), so the scale traffic never
//     sits on the MMA issue path (measured: staging by tcgen05.cp in front of
//     each stage's MMAs halved the MMA rate, tcgen05.st by four warps costs
//     ~50 cycles per stage off the tensor pipe).  The scale tiles land on a
//     barrier of their own, so the stagers copy them while the stage's codes
//     are still landing and then wait for the codes before they report
//     (measured: the output-cast instance 1.6-1.9% faster, the plain GEMM
//     unchanged);
//   * warp 1 of the first CTA: tensor-core issuer -- four
//     tcgen05.mma.kind::mxf4 per stage (K = 64, two UE8M0 scales per row each)
//     update a 256 x 256 fp32 accumulator (128 lanes x 256 columns in each
//     SM); tcgen05.commit multicasts the stage release to both CTAs.  One
//     elected lane runs the whole loop, stepping the operand descriptors
//     from stage to stage (~160 cycles from "scales ready" to the commit).
//     The stagers of both CTAs report "stage ready" straight to the first
//     CTA's barrier (their own data has landed by then), so no relay hop;
//   * warps 6-13: epilogue -- each warp reads 32 lanes x 128 columns of the
//     accumulator into registers as bf16 pairs, frees tensor memory at once,
//     then stages four 32 x 32 blocks in 64-byte-swizzled shared memory; the
//     four warps of a 128-column half stage side by side and one of them
//     writes each 128 x 32 block with a TMA store, so the global writes are
//     whole-line and asynchronous while the next tile's MMAs run.
// M and N tails come from the TMA out-of-bounds zero fill on loads and the
// TMA clipping of stores; a K tail (K % 64 == 32) reads zero codes past K.
//
// Output cast (the kCastOut instance): the epilogue also writes C as MXFP4,
// row-wise (C quantized along N) and column-wise (C^T quantized along M),
// each optional, with the optional Hadamard per output -- the same bytes a
// separate dual cast of the bf16 C would write, without reading C back
// (jax-aiter README, "MXFP4 training architecture": the gradient that one
// GEMM produces is cast for the next).  Each epilogue lane holds one row of
// its 128 columns, so the row blocks are quantized from registers; the column
// blocks are read back, one column per lane, from the 32 x 32 bf16 blocks the
// epilogue already stages in shared memory for the C store.  Row codes leave
// through one more TMA store per warp and tile; the four warps of a 128-column
// half stage their column codes side by side (64 bytes per column) for one
// store per half and tile, instead of one 16-byte piece per column and warp
// (measured: dgrad 161-162 -> 159 us).  Scales are direct stores.
// Rows past M and columns past N hold exact zeros (zero-filled operands), so
// the scale padding comes out 0x00 as the cast writes it.  The two code
// staging buffers take the room of one ring stage (5 stages instead of 6).
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mxfp4 {

// Device-side status word: MXFP4_OK (0), or MXFP4_ERR_TIMEOUT once a pipeline
// wait of the GEMM gave up.
__device__ int g_device_status = 0;

namespace {

constexpr int kMaxGroup = 4;            // GEMMs per grouped launch
constexpr int kBM = 256;                // rows of C per CTA pair
constexpr int kRowsPerCta = 128;        // rows of A (and of B) held by each CTA
constexpr int kBN = 256;                // columns of C per tile
constexpr int kBKBytes = 128;           // code bytes per row per stage = one swizzle row
constexpr int kAStage = kRowsPerCta * kBKBytes;  // 16 KiB
constexpr int kBStage = kRowsPerCta * kBKBytes;  // 16 KiB
constexpr int64_t kRasterPanelBytes = int64_t(24) << 20;  // A panel of one raster group
constexpr int kScaleWarps = 4;   // warps 2-5
constexpr int kEpiWarps = 8;     // warps 6-13
constexpr int kFirstEpiWarp = 2 + kScaleWarps;
constexpr int kSfLoadWarp = kFirstEpiWarp + kEpiWarps;  // warp 14: the scale-tile loads
constexpr int kThreads = 32 * (kSfLoadWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;
constexpr uint32_t kSfCol0 = kBN;
constexpr int kOutStageBytes = 32 * 32 * 2;  // per epilogue warp: 32 rows x 32 bf16 columns
// The dynamic shared-memory window starts 1024-byte aligned in practice; the
// spare bytes below cover a smaller alignment and the kernel checks it.
constexpr int kSmemBytes = 232448;

// Operand element format.  MXFP4 (E2M1, two per byte): a 128-byte swizzle row
// holds 256 K, consumed by four K = 64 kind::mxf4 MMAs, each reading a pair of
// scale bytes (scale_vec::2X).  MXFP8 (E4M3, one per byte): 128 K per stage,
// four K = 32 kind::mxf8f6f4 MMAs with one scale byte each (scale_vec::1X).
// Scales come in 512-byte tiles of 128 rows x 4 K-blocks (128 K).
template <bool kFp8, bool kCastOut = false>
struct Fmt {
  static_assert(!(kFp8 && kCastOut), "the output cast is MXFP4 only");
  static constexpr int kStages = kCastOut ? 5 : 6;
  static constexpr int kBK = kFp8 ? 128 : 256;     // K elements per stage
  static constexpr int kKTiles = kBK / 128;         // scale K-tiles per stage
  static constexpr int kMmaK = kBK / 4;             // K per MMA
  static constexpr int kMmasPerKTile = 4 / kKTiles;
  static constexpr int kSfaStage = kKTiles * 512;        // own 128-row tile
  static constexpr int kSfbStage = 2 * kKTiles * 512;    // both 128-row tiles of B
  static constexpr uint32_t kStageBytes = kAStage + kBStage + kSfaStage + kSfbStage;
  static constexpr uint32_t kSfaCols = kKTiles * 4;      // 4 tensor-memory columns per tile
  static constexpr uint32_t kSfStageCols = kSfaCols + 2 * kKTiles * 4;
  static constexpr int kRingBytes = kStages * static_cast<int>(kStageBytes);
  // epilogue staging per warp: the bf16 C block, plus row and column codes
  static constexpr int kEpiBytes = kEpiWarps * kOutStageBytes * (kCastOut ? 3 : 1);
  static constexpr int kBarrierBytes = (4 * kStages + 3) * 8 + 16;
  static constexpr uint32_t kSmemSlack = kSmemBytes - (kRingBytes + kEpiBytes + kBarrierBytes);
  // Instruction descriptor: A and B types (kind::mxf4: E2M1 = 1;
  // kind::mxf8f6f4: E4M3 = 0) at bits 7 and 10, both K-major, fp32
  // accumulator, N >> 3 at bit 17, UE8M0 scales (bit 23), M >> 4 at bit 24
  // (M = 256: the pair).  The scale-factor ids (bits 4-5 for B, 29-30 for A)
  // pick the byte(s) of the 32-bit tensor-memory scale column an MMA reads.
  static constexpr uint32_t kIdescBase = (kFp8 ? 0u : ((1u << 7) | (1u << 10))) |
                                         (uint32_t(kBN >> 3) << 17) | (1u << 23) |
                                         (uint32_t(kBM >> 4) << 24);
  static_assert(kSfCol0 + kStages * kSfStageCols <= kTmemCols, "tensor memory budget");
  static_assert(kRingBytes + kEpiBytes + kBarrierBytes <= kSmemBytes, "shared memory");
};

// Named barriers 1 and 2: the four epilogue warps of one 128-column half of
// the tile (128 threads).  named_bar_and also returns the AND of `ok` over
// them, so that the four warps leave the tile loop together or not at all.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ bool named_bar_and(int id, int count, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
      : "=r"(out)
      : "f"(__uint_as_float(hi_f32)), "f"(__uint_as_float(lo_f32)));
  return out;
}

// Tile t -> (pair row tile, column tile): groups of group_m row tiles, column
// tiles outer within a group, so concurrently running tiles share A and B.
__device__ __forceinline__ void tile_coords(int t, int num_mt, int num_nt, int group_m, int& mt,
                                            int& nt) {
  const int per_group = group_m * num_nt;
  const int g = t / per_group;
  const int first = g * group_m;
  const int gm = min(group_m, num_mt - first);
  const int r = t - g * per_group;
  mt = first + r % gm;
  nt = r / gm;
}

// Tile counts of one GEMM of the launch.  A launch runs up to kMaxGroup
// independent GEMMs (gemm_fp4_grouped): their tiles are numbered one after
// the other, GEMM g owning [tile_end[g-1], tile_end[g]).
struct GroupTiles {
  int num_mt, num_nt, num_kt, ktiles128;
  int group_m;   // raster group, in pair row tiles
  int last_nks;  // 64-deep k-steps of the last stage (K % 64 == 32 rounds up: zero codes)
  int tile_end;  // one past the GEMM's last tile in the launch's numbering
  int has_c;     // 0: no bf16 C (the cast-only form of the output-cast instance)
};

// Tensor maps of a launch: operands, scales and C of each GEMM, and the
// output-cast code maps (kCastOut instance, one GEMM).
struct GemmMaps {
  CUtensorMap a[kMaxGroup], b[kMaxGroup], sfa[kMaxGroup], sfb[kMaxGroup], c[kMaxGroup], c128[kMaxGroup];
  CUtensorMap qr, qc;
};

struct PairGemmParams {
  GroupTiles g[kMaxGroup];
  int groups;     // GEMMs in the launch, 1..kMaxGroup
  int num_tiles;  // tiles of all of them
  // output cast (kCastOut instance): tile-layout scales of C along N and of
  // C^T along M (each null when that output is not wanted), Hadamard flags,
  // and the scale tile counts ceil(M / 128), ceil(N / 128)
  uint8_t* sf_row;
  uint8_t* sf_col;
  uint32_t cast_flags;
  int m_tiles128, n_tiles128;
  // time without progress after which a pipeline wait gives up (2 s), and the
  // self-test knob: when set, the scale stagers withhold their "stage ready"
  // signal for the first stage of the first tile, so the MMA warp's wait runs
  // out (mxfp4_selftest_wait_timeout); 0 on every product launch
  unsigned long long wait_limit_ns;
  int withhold_first_scale_signal;
};

// The GEMM that owns launch tile t, and t's index within that GEMM.
__device__ __forceinline__ int tile_group(const PairGemmParams& p, int t, int& lt) {
  int g = 0, begin = 0;
  while (g + 1 < p.groups && t >= p.g[g].tile_end) {
    begin = p.g[g].tile_end;
    ++g;
  }
  lt = t - begin;
  return g;
}

template <bool kFp8, bool kCastOut>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_pair_kernel(const __grid_constant__ GemmMaps maps, const PairGemmParams p) {
  using F = Fmt<kFp8, kCastOut>;
  constexpr int kStages = F::kStages;
  constexpr int kSfaStage = F::kSfaStage, kSfbStage = F::kSfbStage;
  constexpr uint32_t kSfaCols = F::kSfaCols, kSfStageCols = F::kSfStageCols;
  constexpr uint32_t kSmemSlack = F::kSmemSlack;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled operand tiles (same offset
  // in both CTAs: identical kernels, identical static layout).
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  if (pad > kSmemSlack) {  // cannot place the ring: report and leave (uniform over the grid)
    if (threadIdx.x == 0) atomicExch(&g_device_status, 5 /* MXFP4_ERR_CUDA */);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStages * kAStage;
  uint8_t* sSfa = sB + kStages * kBStage;
  uint8_t* sSfb = sSfa + kStages * kSfaStage;
  uint8_t* sOut = sSfb + kStages * kSfbStage;  // epilogue staging, 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + F::kEpiBytes);
  uint64_t* empty = full + kStages;
  uint64_t* sf_ready = empty + kStages;
  uint64_t* sf_full = sf_ready + kStages;  // the stage's scale tiles have landed
  uint64_t* acc_full = sf_full + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* mma_drain = acc_empty + 1;  // leader: every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();  // 0 = the CTA that issues the MMAs
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
      // leader only: the four stager warps of each CTA arrive here
      mbar_init(&sf_ready[s], 2 * kScaleWarps);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * kEpiWarps);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.groups; ++g) {
      tma_prefetch_desc(&maps.a[g]);
      tma_prefetch_desc(&maps.b[g]);
      tma_prefetch_desc(&maps.sfa[g]);
      tma_prefetch_desc(&maps.sfb[g]);
      if (p.g[g].has_c) tma_prefetch_desc(&maps.c[g]);
    }
    if constexpr (kCastOut) {
      if (p.sf_row != nullptr) tma_prefetch_desc(&maps.qr);
      if (p.sf_col != nullptr) tma_prefetch_desc(&maps.qc);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialized before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = p.num_tiles;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);

  if (warp == 0 || warp == kSfLoadWarp) {
    // ------------------------------------------------------------ producers (both CTAs)
    // Warp 0 arms each stage's code barrier and loads the A and B codes;
    // warp 14 arms the stage's scale barrier and loads the two scale boxes
    // once the stage is free.  Two threads issuing
    // the four loads side by side, instead of one issuing them in turn,
    // shorten the path from a stage's release to its refill (measured: 4-9%
    // faster GEMMs at the Llama shapes).
    const bool code_loads = warp == 0;
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int issued = 0;  // stage loads issued so far
      for (int t = pair; ok && t < num_tiles; t += num_pairs) {
        int lt, mt, nt;
        const int g = tile_group(p, t, lt);
        const GroupTiles& G = p.g[g];
        tile_coords(lt, G.num_mt, G.num_nt, G.group_m, mt, nt);
        const int a_row = mt * kBM + static_cast<int>(rank) * kRowsPerCta;
        const int b_row = nt * kBN + static_cast<int>(rank) * kRowsPerCta;
        const int a_rt = a_row / 128;  // this CTA's scale row tile of A
        for (int kt = 0; kt < G.num_kt; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_device_status, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          if (code_loads) {
            mbar_arrive_expect_tx(&full[stage], kAStage + kBStage);
            tma_load_2d(sA + stage * kAStage, &maps.a[g], &full[stage], kt * kBKBytes, a_row);
            tma_load_2d(sB + stage * kBStage, &maps.b[g], &full[stage], kt * kBKBytes, b_row);
          } else {
            const int kg0 = kt * F::kKTiles;
            mbar_arrive_expect_tx(&sf_full[stage], kSfaStage + kSfbStage);
            tma_load_2d(sSfa + stage * kSfaStage, &maps.sfa[g], &sf_full[stage], 0,
                        (a_rt * G.ktiles128 + kg0) * 4);
            // both 128-row scale tiles of B in one box (measured: 4-7% faster
            // than two 2-D loads)
            tma_load_3d(sSfb + stage * kSfbStage, &maps.sfb[g], &sf_full[stage], 0, kg0 * 4, nt * 2);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load issued has landed before the CTA may end: the stagers wait
      // for all of them unless a wait gave up.  The last load into a stage
      // completes the phase its index gives; nothing follows it.  Each
      // producer waits on the barrier it armed, for the stages it loaded into.
      volatile int keep_waiting = 0;  // not the CTA's abort flag: this wait must run its course
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / kStages) * kStages;
        uint64_t* landed = code_loads ? &full[s] : &sf_full[s];
        if (!mbar_wait(landed, (last / kStages) & 1, &keep_waiting, &g_device_status, p.wait_limit_ns)) break;
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ------------------------------------------------------------ MMA issuer
      // One elected lane runs the whole loop: the waits, four MMAs and the
      // commit per stage, with the descriptors stepped from stage to stage.
      // Measured: ~160 cycles from a stage's scales being ready to its
      // commit, against ~300 with the whole warp running the loop and
      // electing a lane per stage (a vote, an elect and a re-convergence
      // each time); the GEMMs at the Llama shapes ran 1-3% faster.
      if (elect_one_sync()) {
        uint32_t stage = 0, phase = 0, acc_phase = 0;
        bool ok = true;
        // Descriptor start addresses are in 16-byte units: a stage is
        // kAStage / 16 further, a 64-deep k-step 32 bytes (2 units).
        const uint64_t adesc0 = make_smem_desc(smem_u32(sA), 16, 1024, 2);
        const uint64_t bdesc0 = make_smem_desc(smem_u32(sB), 16, 1024, 2);
        uint64_t a_d = adesc0, b_d = bdesc0;
        uint32_t sf_col = tmem_base + kSfCol0;
        for (int t = pair; ok && t < num_tiles; t += num_pairs) {
          int lt;
          const GroupTiles& G = p.g[tile_group(p, t, lt)];
          ok = mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, &g_device_status, p.wait_limit_ns);
          if (!ok) break;
          tc_fence_after();
          for (int kt = 0; kt < G.num_kt; ++kt) {
            ok = mbar_wait(&sf_ready[stage], phase, abort_flag, &g_device_status, p.wait_limit_ns);
            if (!ok) break;
            tc_fence_after();
            const int nks = kt + 1 < G.num_kt ? 4 : G.last_nks;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (ks < nks) {
                // K-tile g of the stage; byte (FP8) or byte pair (FP4) sf_id of its columns
                const uint32_t g = ks / F::kMmasPerKTile;
                const uint32_t sf_id = (ks % F::kMmasPerKTile) * (4 / F::kMmasPerKTile);
                const uint32_t idesc = F::kIdescBase | (sf_id << 4) | (sf_id << 29);
                if constexpr (kFp8)
                  tc_mma_pair_mxf8f6f4(tmem_base + kAccCol, a_d + 2 * ks, b_d + 2 * ks, idesc,
                                       sf_col + g * 4, sf_col + kSfaCols + g * 8, (kt | ks) != 0);
                else
                  tc_mma_pair_mxf4(tmem_base + kAccCol, a_d + 2 * ks, b_d + 2 * ks, idesc,
                                   sf_col + g * 4, sf_col + kSfaCols + g * 8, (kt | ks) != 0);
              }
            }
            tc_commit_pair(&empty[stage], 0x3);
            a_d += kAStage >> 4;
            b_d += kBStage >> 4;
            sf_col += kSfStageCols;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
              a_d = adesc0;
              b_d = bdesc0;
              sf_col = tmem_base + kSfCol0;
            }
          }
          if (!ok) break;
          tc_commit_pair(acc_full, 0x3);
          acc_phase ^= 1u;
        }
        // Every MMA issued (they read both CTAs' shared memory and write their
        // tensor memory) has completed before the teardown: already so on the
        // normal path, not when a wait gave up mid-tile.
        tc_commit_pair(mma_drain, 0x1);
        volatile int keep_waiting = 0;
        mbar_wait(mma_drain, 0, &keep_waiting, &g_device_status, p.wait_limit_ns);
        tc_fence_after();
      }
      __syncwarp();
    }
  } else if (warp < kFirstEpiWarp) {
    // ------------------------------------------------------------ scale stagers (both CTAs)
    // Quarter q of tensor memory (lanes 32q .. 32q+31); thread i writes lane
    // 32q + i.  Shared-memory scale tiles hold row r's 4 block scales at byte
    // (r % 32) * 16 + (r / 32) * 4, so lane i's 16 bytes of a tile are exactly
    // the 4 columns (rows i, i+32, i+64, i+96) the MMA reads for that tile.
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t leader_ready0 = map_to_cta(&sf_ready[0], 0);
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int t = pair; ok && t < num_tiles; t += num_pairs) {
      int lt;
      const int num_kt = p.g[tile_group(p, t, lt)].num_kt;
      for (int kt = 0; kt < num_kt; ++kt) {
        if (!mbar_wait(&sf_full[stage], phase, abort_flag, &g_device_status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint8_t* sfa = sSfa + stage * kSfaStage + lane * 16;
        const uint8_t* sfb = sSfb + stage * kSfbStage + lane * 16;  // [row tile][K tile][512]
        const uint32_t taddr = tmem_base + lane_base + kSfCol0 + stage * kSfStageCols;
        if constexpr (kFp8) {
          // columns 0-3: A; 4-11: B (row tiles 0, 1), one K tile
          const uint4 a0 = lds128(sfa), b0 = lds128(sfb), b1 = lds128(sfb + 512);
          tmem_st_32x32b_x4(taddr + 0, a0.x, a0.y, a0.z, a0.w);
          tmem_st_32x32b_x8(taddr + 4, b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w);
        } else {
          // columns 0-7: A, K tiles 0 and 1; 8-15: B K tile 0 (row tiles 0, 1); 16-23: B K tile 1
          const uint4 a0 = lds128(sfa), a1 = lds128(sfa + 512);
          const uint4 b00 = lds128(sfb), b10 = lds128(sfb + 1024);
          const uint4 b01 = lds128(sfb + 512), b11 = lds128(sfb + 1536);
          tmem_st_32x32b_x8(taddr + 0, a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w);
          tmem_st_32x32b_x8(taddr + 8, b00.x, b00.y, b00.z, b00.w, b10.x, b10.y, b10.z, b10.w);
          tmem_st_32x32b_x8(taddr + 16, b01.x, b01.y, b01.z, b01.w, b11.x, b11.y, b11.z, b11.w);
        }
        tmem_st_wait();
        tc_fence_before();
        // both CTAs' codes must have landed before the issuing CTA hears "ready"
        if (!mbar_wait(&full[stage], phase, abort_flag, &g_device_status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        __syncwarp();
        const bool withhold = p.withhold_first_scale_signal && t == pair && kt == 0;
        if (lane == 0 && !withhold) mbar_arrive_cluster(leader_ready0 + stage * 8u);  // the issuing CTA's barrier
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                         // tensor-memory lane quarter this warp may read
    const int h = (warp - kFirstEpiWarp) >> 2;      // which 128-column half of the tile
    const uint32_t acc_empty_leader = map_to_cta(acc_empty, 0);
    const int ew = warp - kFirstEpiWarp;
    // C staging: the plain kernel keeps the four lane quarters of a half in
    // consecutive buffers (rows 0-127 of the half, in order) for one
    // 128-row store per block; the output-cast instance, one buffer per warp
    const int stage_idx = kCastOut ? ew : h * 4 + q;
    const uint32_t out_buf = smem_u32(sOut + stage_idx * kOutStageBytes);
    // output cast: row-code block (32 rows x 64 bytes, 64-byte swizzle like
    // the C block) and column codes (128 column rows x 16 bytes)
    const uint32_t rq_buf = smem_u32(sOut + (kEpiWarps + ew) * kOutStageBytes);
    // column codes of the half's 128 rows: 128 columns x 64 bytes, warp q's
    // 16 bytes at chunk q under the 64-byte swizzle, one TMA store per tile
    const uint32_t cq_half = smem_u32(sOut + (2 * kEpiWarps + 4 * h) * kOutStageBytes);
    const bool do_row = kCastOut && p.sf_row != nullptr;
    const bool do_col = kCastOut && p.sf_col != nullptr;
    const bool had_row = (p.cast_flags & kFlagHadamardRow) != 0;
    const bool had_col = (p.cast_flags & kFlagHadamardCol) != 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < num_tiles; t += num_pairs) {
      int lt, mt, nt;
      const int g = tile_group(p, t, lt);
      const GroupTiles& G = p.g[g];
      tile_coords(lt, G.num_mt, G.num_nt, G.group_m, mt, nt);
      {
        bool okw = mbar_wait(acc_full, acc_phase, abort_flag, &g_device_status, p.wait_limit_ns);
        // the half's four warps meet at named barriers below: one that gave up
        // takes the other three out of the loop with it.  In the output-cast
        // instance the half's column-code block is free once this meeting is
        // passed: its store of the previous tile has read it.
        if constexpr (kCastOut) {
          if (do_col && q == 0 && lane == 0) bulk_wait_group_read0();
        }
        okw = named_bar_and(1 + h, 128, okw);
        if (!okw) break;
      }
      tc_fence_after();
      // Read all 128 columns (4 x 32) as bf16 pairs, then release the accumulator.
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + h * 128;
      const int32_t row0 = mt * kBM + static_cast<int32_t>(rank) * kRowsPerCta + q * 32;
      const int32_t col0 = nt * kBN + h * 128;
      // output cast: this warp's 32 rows and 128 columns sit in one 128-row
      // scale tile of each output (row tile mt * 2 + rank, column tile
      // nt * 2 + h); tiles past the padded extent are not written
      const int rt128 = mt * 2 + static_cast<int>(rank), ct128 = nt * 2 + h;
      const bool sf_tiles_ok = kCastOut && rt128 < p.m_tiles128 && ct128 < p.n_tiles128;
      const size_t row_sf_tile = (static_cast<size_t>(rt128) * p.n_tiles128 + ct128) * 512;
      const size_t col_sf_tile = (static_cast<size_t>(ct128) * p.m_tiles128 + rt128) * 512;
      uint32_t row_sf = 0;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[c * 16 + j] = pack_bf16x2(r[2 * j], r[2 * j + 1]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);  // accumulator free for the next tile
      // Four 32 x 32 blocks: row `lane` is 64 bytes = four 16-byte chunks, chunk j
      // stored at j ^ ((row / 2) % 4) (the 64-byte swizzle), conflict-free.
      if constexpr (!kCastOut) {
        // The half's four warps stage block c side by side (128 rows x 32
        // columns) and one thread stores it with a single TMA store: a quarter
        // of the store operations of one store per warp (measured: dgrad and
        // the other K = 4096-8192 shapes 2-3% faster, results unchanged).
        const int32_t row_half = mt * kBM + static_cast<int32_t>(rank) * kRowsPerCta;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            sts128(out_buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16), pk[c * 16 + 4 * j],
                   pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2], pk[c * 16 + 4 * j + 3]);
          fence_proxy_async_shared();
          named_bar_sync(1 + h, 128);  // the half's 128 rows are staged
          if (q == 0 && lane == 0) {
            if (G.has_c) tma_store_2d(&maps.c128[g], sOut + h * 4 * kOutStageBytes, col0 + c * 32, row_half);
            bulk_commit_group();
            bulk_wait_group_read0();  // the store has read the staging buffer
          }
          named_bar_sync(1 + h, 128);  // buffer free for the next block
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (lane == 0) bulk_wait_group_read0();  // the previous block has left the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            sts128(out_buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16), pk[c * 16 + 4 * j],
                   pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2], pk[c * 16 + 4 * j + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            if (G.has_c)  // the cast-only form writes no bf16 C
              tma_store_2d(&maps.c[g], sOut + ew * kOutStageBytes, col0 + c * 32, row0);
            bulk_commit_group();
          }
          if constexpr (kCastOut) {
            if (do_row) {  // block c of this lane's row, read back from the staged block
              // (from shared memory rather than the packed registers: the cast then
              // cannot be scheduled ahead of the accumulator release, and pk dies
              // with the block stores -- measured 7-14% faster, no spills)
              uint32_t w[16], q4[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 v = lds128(sOut + ew * kOutStageBytes + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4));
                w[4 * j] = v.x;
                w[4 * j + 1] = v.y;
                w[4 * j + 2] = v.z;
                w[4 * j + 3] = v.w;
              }
              BlockScale s;
              if (!had_row) {
                s = quantize_bf16_block(w, q4);
              } else {
                float y[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  y[2 * i] = __uint_as_float(w[i] << 16);
                  y[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                }
                s = quantize_hadamard_block(y, q4);
              }
              row_sf |= s.byte << (8 * c);
              sts128(rq_buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), q4[0], q4[1], q4[2], q4[3]);
            }
            if (do_col) {  // column c * 32 + lane of the staged block: 32 rows
              uint32_t q4[4];
              const uint32_t cb = out_buf + (lane & 7) * 2;
              auto elem = [&](int r) { return lds_u16(cb + r * 64 + (((lane >> 3) ^ ((r >> 1) & 3)) << 4)); };
              BlockScale s;
              if (!had_col) {
                uint32_t w[16];  // rows 2i, 2i + 1 as one bf16 pair
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = __byte_perm(elem(2 * i), elem(2 * i + 1), 0x5410);
                s = quantize_bf16_block(w, q4);
              } else {
                float y[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) y[r] = __uint_as_float(elem(r) << 16);
                s = quantize_hadamard_block(y, q4);
              }
              const int colx = c * 32 + lane;
              sts128(cq_half + colx * 64 + ((q ^ ((colx >> 1) & 3)) << 4), q4[0], q4[1], q4[2], q4[3]);
              if (sf_tiles_ok) p.sf_col[col_sf_tile + lane * 16 + c * 4 + q] = static_cast<uint8_t>(s.byte);
            }
          }
        }
      }
      if constexpr (kCastOut) {
        fence_proxy_async_shared();
        if (do_col) named_bar_sync(1 + h, 128);  // the half's column codes are staged
        else __syncwarp();
        if (lane == 0 && (do_row || (do_col && q == 0))) {
          if (do_row) tma_store_2d(&maps.qr, sOut + (kEpiWarps + ew) * kOutStageBytes, col0 / 2, row0);
          if (do_col && q == 0)
            tma_store_2d(&maps.qc, sOut + (2 * kEpiWarps + 4 * h) * kOutStageBytes,
                         (mt * kBM + static_cast<int32_t>(rank) * kRowsPerCta) / 2, col0);
          bulk_commit_group();
        }
        // scales of this lane's row: blocks 0-3 of the 128-column tile, one word
        if (do_row && sf_tiles_ok)
          *reinterpret_cast<uint32_t*>(p.sf_row + row_sf_tile + lane * 16 + q * 4) = row_sf;
      }
      acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  cluster_sync();  // neither CTA leaves while its peer may still touch its barriers or memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

__global__ void fill_zero_bf16_kernel(uint16_t* c, int64_t M, int64_t N, int64_t ldc) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c[(i / N) * ldc + (i % N)] = 0;
}

// 2-D byte matrix [rows, row_bytes] (pitch row_bytes), boxes of box_rows x
// box_bytes, zero fill out of bounds.
bool make_byte_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t row_bytes,
                   uint32_t box_bytes, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estrides[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides,
                  box, estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scale tiles of an operand as a 3-D byte tensor [row tiles][K tiles x 4][128]
// (each 512-byte tile is four 128-byte rows); boxes of 2 row tiles x
// box_rows rows (box_rows / 4 K tiles) x 128 bytes, zero fill past the edges.
bool make_scale_pair_map(CUtensorMap* map, const uint8_t* base, int64_t row_tiles, int64_t ktiles128,
                         uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(ktiles128 * 4), static_cast<cuuint64_t>(row_tiles)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(ktiles128 * 512)};
  cuuint32_t box[3] = {128, box_rows, 2};
  cuuint32_t estrides[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box,
                  estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map: bf16 [M, N] with row pitch ldc elements, boxes of box_rows rows
// x 32 columns (64 bytes, 64-byte swizzle); stores clip at M and N.
bool make_bf16_out_map(CUtensorMap* map, uint16_t* base, int64_t M, int64_t N, int64_t ldc, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * 2};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estrides[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estrides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Shared-memory opt-in of the kernel, once per device.
template <bool kFp8, bool kCastOut>
cudaError_t prepare_kernel(int dev) {
  static std::atomic<bool> done[64];
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_mxf4_pair_kernel<kFp8, kCastOut>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}

// Largest number of co-resident CTA pairs, per device (cached).
template <bool kFp8, bool kCastOut>
int max_pairs(int dev) {
  static std::atomic<int> cache[64];
  if (dev >= 0 && dev < 64 && cache[dev].load(std::memory_order_relaxed) > 0)
    return cache[dev].load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_mxf4_pair_kernel<kFp8, kCastOut>, &cfg) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = std::max(1, sms / 2);
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

int* device_status_word() {
  static std::atomic<int*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int* p = cache[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return nullptr;
    p = static_cast<int*>(addr);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, fill_zero_bf16_kernel, c, M, N, ldc);
}

namespace {

// One launch over the tiles of `count` independent GEMMs (1..kMaxGroup; the
// output-cast instance takes one).  GEMMs with M or N == 0 are skipped; those
// with K == 0 get C = 0 (and zero casts) from separate fills, enqueued first.
template <bool kFp8, bool kCastOut = false>
cudaError_t launch_gemm_fmt(const GemmArgs* list, int count, cudaStream_t stream,
                            const CastOutArgs* out = nullptr,
                            unsigned long long wait_limit_ns = kWaitLimitNs, bool withhold = false) {
  using F = Fmt<kFp8, kCastOut>;
  if (count < 1 || count > kMaxGroup || (kCastOut && count != 1)) return cudaErrorInvalidValue;
  GemmMaps maps = {};
  PairGemmParams p = {};
  int64_t tiles = 0;
  int groups = 0;
  for (int i = 0; i < count; ++i) {
    const GemmArgs& args = list[i];
    if (args.M == 0 || args.N == 0) continue;
    if (args.K == 0) {  // C = 0, and its casts are those of a zero matrix: all bytes 0x00
      cudaError_t e = args.c != nullptr ? launch_fill_zero_bf16(args.c, args.M, args.N, args.ldc, stream)
                                        : cudaSuccess;
      if (e != cudaSuccess) return e;
      if (kCastOut) {
        const size_t code_bytes = static_cast<size_t>(args.M) * static_cast<size_t>(args.N / 2);
        const size_t sf_bytes = static_cast<size_t>((args.M + 127) / 128) * ((args.N + 127) / 128) * 512;
        if (out->q_row != nullptr && e == cudaSuccess) e = cudaMemsetAsync(out->q_row, 0, code_bytes, stream);
        if (out->sf_row != nullptr && e == cudaSuccess) e = cudaMemsetAsync(out->sf_row, 0, sf_bytes, stream);
        if (out->q_col != nullptr && e == cudaSuccess) e = cudaMemsetAsync(out->q_col, 0, code_bytes, stream);
        if (out->sf_col != nullptr && e == cudaSuccess) e = cudaMemsetAsync(out->sf_col, 0, sf_bytes, stream);
        if (e != cudaSuccess) return e;
      }
      continue;
    }
    const int64_t ktiles128 = (args.K + 127) / 128;
    const int64_t a_sf_rows = (args.M + 127) / 128 * ktiles128 * 4;  // 128-byte rows of the scale buffer
    const int64_t row_bytes = kFp8 ? args.K : args.K / 2;             // code bytes per row
    const int g = groups;
    if (!make_byte_map(&maps.a[g], args.a, args.M, row_bytes, kBKBytes, kRowsPerCta,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_byte_map(&maps.b[g], args.b, args.N, row_bytes, kBKBytes, kRowsPerCta,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_byte_map(&maps.sfa[g], args.a_sf, a_sf_rows, 128, 128, 4 * F::kKTiles,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_scale_pair_map(&maps.sfb[g], args.b_sf, (args.N + 127) / 128, ktiles128, 4 * F::kKTiles))
      return cudaErrorInvalidValue;
    if (args.c != nullptr && (!make_bf16_out_map(&maps.c[g], args.c, args.M, args.N, args.ldc, 32) ||
                              !make_bf16_out_map(&maps.c128[g], args.c, args.M, args.N, args.ldc, 128)))
      return cudaErrorInvalidValue;
    GroupTiles& G = p.g[g];
    G.num_mt = static_cast<int>((args.M + kBM - 1) / kBM);
    G.num_nt = static_cast<int>((args.N + kBN - 1) / kBN);
    G.num_kt = static_cast<int>((args.K + F::kBK - 1) / F::kBK);
    G.ktiles128 = static_cast<int>(ktiles128);
    G.last_nks = static_cast<int>((args.K - static_cast<int64_t>(G.num_kt - 1) * F::kBK + F::kMmaK - 1) /
                                  F::kMmaK);
    // Raster group: powers of two up to 64 row tiles while the group's A panel,
    // counted in FP4 bytes (K / 2 per row), stays within the budget.  An MXFP8
    // panel of the same K is twice the bytes and still fits the L2; sizing it
    // by its own bytes halved the group and streamed B twice (measured on the
    // wgrad of the 8B down projection: 1.8x the operand bytes read from DRAM).
    G.group_m = 1;
    while (G.group_m < 64 && 2 * G.group_m * kBM * (args.K / 2) <= kRasterPanelBytes) G.group_m *= 2;
    G.has_c = args.c != nullptr ? 1 : 0;
    tiles += static_cast<int64_t>(G.num_mt) * G.num_nt;
    if (tiles > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    G.tile_end = static_cast<int>(tiles);
    ++groups;
  }
  if (groups == 0) return cudaSuccess;
  p.groups = groups;
  p.num_tiles = static_cast<int>(tiles);
  if constexpr (kCastOut) {
    // output cast: row codes [M, N/2] in 32-row x 64-byte boxes, column codes
    // [N, M/2] in 128-row x 64-byte boxes (64-byte swizzle both)
    const GemmArgs& args = list[0];
    if (out->q_row != nullptr &&
        !make_byte_map(&maps.qr, out->q_row, args.M, args.N / 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    if (out->q_col != nullptr &&
        !make_byte_map(&maps.qc, out->q_col, args.N, args.M / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    p.sf_row = out->sf_row;
    p.sf_col = out->sf_col;
    p.cast_flags = out->flags;
    p.m_tiles128 = static_cast<int>((args.M + 127) / 128);
    p.n_tiles128 = static_cast<int>((args.N + 127) / 128);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = prepare_kernel<kFp8, kCastOut>(dev);
  if (e != cudaSuccess) return e;
  p.wait_limit_ns = wait_limit_ns;
  p.withhold_first_scale_signal = withhold ? 1 : 0;
  const int pairs = static_cast<int>(std::min<int64_t>(tiles, max_pairs<kFp8, kCastOut>(dev)));

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the launch's own result (the thread's last error may be stale and unrelated)
  return cudaLaunchKernelEx(&cfg, gemm_mxf4_pair_kernel<kFp8, kCastOut>, maps, p);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& args, cudaStream_t stream) {
  return launch_gemm_fmt<false>(&args, 1, stream);
}

cudaError_t launch_gemm_grouped(const GemmArgs* list, int count, cudaStream_t stream) {
  return launch_gemm_fmt<false>(list, count, stream);
}

cudaError_t launch_gemm_mxfp8(const GemmArgs& args, cudaStream_t stream) {
  return launch_gemm_fmt<true>(&args, 1, stream);
}

cudaError_t launch_gemm_cast_out(const GemmArgs& args, const CastOutArgs& out, cudaStream_t stream) {
  return launch_gemm_fmt<false, true>(&args, 1, stream, &out);
}

cudaError_t launch_gemm_selftest_timeout(const GemmArgs& args, unsigned long long wait_limit_ns,
                                         cudaStream_t stream) {
  return launch_gemm_fmt<false>(&args, 1, stream, nullptr, wait_limit_ns, true);
}

}  // namespace mxfp4

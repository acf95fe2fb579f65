// MMA-only rate of the fifth-generation tensor cores on this GPU: back-to-back
// tcgen05.mma issued by one elected lane, operands in zeroed shared memory,
// no loads, cycles per instruction (clock64 around the issue loop and the
// final commit).  This is the ceiling the block-scaled FP4 GEMM is measured
// against: a 256 x 256 x 64 pair MMA of kind::mxf4 per N cycles.
//
// Test infrastructure (built and run by tests/test_gpu_mma_ceiling.py); it
// uses the library's inline-PTX wrappers and shares no arithmetic with it.
// Prints one "RESULT <name> <cycles per MMA> <FLOP/clk/SM> <err>" line per case.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../quantization_mxfp4_cast_gb300/csrc/ptx.cuh"

using namespace mxfp4;

__device__ unsigned long long g_cycles[512];
__device__ int g_err;

enum Kind { MXF4 = 0, NVF4_4X = 1, MXF8 = 2, BF16 = 3 };

template <int KIND>
__device__ __forceinline__ void pair_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb) {
  const uint32_t acc = 1;
#define PAIR_MMA_SCALED(KIND_STR)                                                              \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2." KIND_STR \
               " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),                             \
               "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)                        \
               : "memory")
  if constexpr (KIND == MXF4) PAIR_MMA_SCALED("kind::mxf4.block_scale.scale_vec::2X");
  if constexpr (KIND == NVF4_4X) PAIR_MMA_SCALED("kind::mxf4nvf4.block_scale.scale_vec::4X");
  if constexpr (KIND == MXF8) PAIR_MMA_SCALED("kind::mxf8f6f4.block_scale.scale_vec::1X");
  if constexpr (KIND == BF16)
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
#undef PAIR_MMA_SCALED
}

// Instruction descriptor: M = 256 (pair), N, K-major operands; element and
// scale types per kind (block-scaled kinds: UE8M0 at bit 23 unless UE4M3).
template <int KIND, int N>
__host__ __device__ constexpr uint32_t idesc_of() {
  constexpr uint32_t nm = (uint32_t(N >> 3) << 17) | (uint32_t(256 >> 4) << 24);
  if (KIND == MXF4) return nm | (1u << 7) | (1u << 10) | (1u << 23);
  if (KIND == NVF4_4X) return nm | (1u << 7) | (1u << 10);
  if (KIND == MXF8) return nm | (1u << 23);
  return nm | (1u << 4) | (1u << 7) | (1u << 10);  // bf16 x bf16 -> f32
}

template <int KIND>
__host__ __device__ constexpr int k_of() { return KIND == BF16 ? 16 : (KIND == MXF8 ? 32 : 64); }

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) {
      atomicExch(&g_err, 1);
      return false;
    }
  }
}

// More than half of an SM's shared memory: one CTA per SM, so two CTAs never
// compete for the same SM's tensor memory.
constexpr int kSmem = 120 * 1024;

template <int KIND, int N>
__global__ void __launch_bounds__(128, 1) mma_rate(int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;          // 128 rows x 128 bytes
  uint8_t* sB = smem + 16384;  // up to 128 rows x 128 bytes
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 32768);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  fence_proxy_async_shared();
  __syncthreads();
  if (warp == 0) {
    tmem_alloc_pair(slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t base = *slot;
  {  // scale columns 256..287 of every lane: 1.0 in the kind's scale type
    const uint32_t v = KIND == NVF4_4X ? 0x38383838u : 0x7F7F7F7Fu;
    const uint32_t t = base + (static_cast<uint32_t>(warp * 32) << 16) + 256;
    for (int c = 0; c < 32; c += 8) tmem_st_32x32b_x8(t + c, v, v, v, v, v, v, v, v);
    tmem_st_wait();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const bool leader = cluster_cta_rank() == 0;
  if (warp == 0) {
    constexpr uint32_t idesc = idesc_of<KIND, N>();
    const uint64_t ad = make_smem_desc(smem_u32(sA), 16, 1024, 2);
    const uint64_t bd = make_smem_desc(smem_u32(sB), 16, 1024, 2);
    const unsigned long long c0 = clock64();
    if (leader) {
      for (int s = 0; s < stages; ++s) {
        if (elect_one_sync()) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) pair_mma<KIND>(base, ad + 2 * ks, bd + 2 * ks, idesc, base + 256, base + 264);
          tc_commit_pair(&bar[0], 0x3);  // a commit per 4 MMAs, as a GEMM stage does
        }
        __syncwarp();
      }
      if (elect_one_sync()) tc_commit_pair(&bar[1], 0x3);
      __syncwarp();
    }
    bounded_wait(&bar[1], 0);  // both CTAs: every MMA has completed
    tc_fence_after();
    const unsigned long long c1 = clock64();
    if (leader && lane == 0) g_cycles[blockIdx.x >> 1] = c1 - c0;
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(base, 512);
  }
}

#define CK(x)                                                                            \
  do {                                                                                   \
    cudaError_t e_ = (x);                                                                \
    if (e_ != cudaSuccess) {                                                             \
      printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__);            \
      exit(1);                                                                           \
    }                                                                                    \
  } while (0)

template <int KIND, int N>
void run(const char* name, int pairs, int stages) {
  auto kern = mma_rate<KIND, N>;
  CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  CK(cudaLaunchKernelEx(&cfg, kern, 16));  // warm-up
  CK(cudaDeviceSynchronize());
  CK(cudaLaunchKernelEx(&cfg, kern, stages));
  CK(cudaDeviceSynchronize());
  int err = 0;
  CK(cudaMemcpyFromSymbol(&err, g_err, sizeof(int)));
  std::vector<unsigned long long> cyc(pairs);
  CK(cudaMemcpyFromSymbol(cyc.data(), g_cycles, pairs * sizeof(unsigned long long)));
  double mean = 0;
  for (int i = 0; i < pairs; ++i) mean += static_cast<double>(cyc[i]) / pairs;
  const double per_mma = mean / (4.0 * stages);
  const double flop_per_clk_sm = 2.0 * 128 * N * k_of<KIND>() / per_mma;  // 128 rows of D per SM
  printf("RESULT %s_%dpairs %.2f %.0f %d\n", name, pairs, per_mma, flop_per_clk_sm, err);
}

int main() {
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  const int stages = 4000;
  for (int pairs : {1, sms / 2}) {
    run<MXF4, 256>("mxf4_n256", pairs, stages);
    run<NVF4_4X, 256>("mxf4nvf4_4x_n256", pairs, stages);
    run<MXF8, 256>("mxf8f6f4_n256", pairs, stages);
    run<BF16, 256>("bf16_n256", pairs, stages);
    run<MXF4, 224>("mxf4_n224", pairs, stages);
    run<MXF4, 192>("mxf4_n192", pairs, stages);
    run<MXF4, 128>("mxf4_n128", pairs, stages);
    run<MXF4, 16>("mxf4_n16", pairs, stages);
  }
  return 0;
}

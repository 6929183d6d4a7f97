// fp4_peak_probe.cu -- measures the dense NVFP4 tensor-core rate of this GPU.
//
// The roofline of the compute-bound (prefill) grouped GEMM needs the dense
// e2m1 x e2m1 MMA rate of the GPU it runs on.  This kernel issues the same
// instruction the grouped GEMM uses (tcgen05.mma kind::mxf4nvf4, ue4m3 scales
// per 16 K-elements, M = 128, K = 64) back to back from shared-memory operands
// into a tensor-memory accumulator, on one CTA per SM, with no global-memory
// traffic; the caller times the launch.  Operands hold a fixed pseudo-random
// pattern (all-zero operands would under-report power and over-report rate).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kProbeN = 256;                       // MMA N (the largest for M = 128)
constexpr int kProbeABytes = 128 * 128;            // 128 rows x 256 K-elements
constexpr int kProbeBBytes = kProbeN * 128;        // 256 rows x 256 K-elements
constexpr int kProbeMaxIters = 1000000;
constexpr int kProbeSmem = kProbeABytes + kProbeBBytes + 2 * 2048 + 1024 + 64;

__global__ void __launch_bounds__(128, 1) fp4_peak_kernel(int iters, int32_t* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a = smem;
  uint8_t* b = a + kProbeABytes;
  uint8_t* sfa = b + kProbeBBytes;
  uint8_t* sfb = sfa + 2048;
  uint64_t* done = reinterpret_cast<uint64_t*>(sfb + 2048);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5;

  // pseudo-random codes; scales 1.0 (e4m3 0x38) so every product is finite
  for (int i = threadIdx.x; i < (kProbeABytes + kProbeBBytes) / 4; i += blockDim.x) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u ^ (blockIdx.x * 40503u);
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    reinterpret_cast<uint32_t*>(a)[i] = h;
  }
  for (int i = threadIdx.x; i < 4096 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sfa)[i] = 0x38383838u;
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_barrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  if (threadIdx.x == 0) {
    // TMEM columns: accumulator [0, 256); per K step g the A scales at 256 + 4g (one atom, 128 rows)
    // and the B scales at 272 + 8g (two atoms: rows 0-127 then 128-255).
    const uint32_t sf_col = tmem + 256;
    for (int g = 0; g < 4; ++g) {
      tmem_cp_32x128b_x4(sf_col + 4 * g, smem_desc(smem_u32(sfa) + 512 * g, 0, 128, 0));
      tmem_cp_32x128b_x4(sf_col + 16 + 8 * g, smem_desc(smem_u32(sfb) + 512 * g, 0, 128, 0));
      tmem_cp_32x128b_x4(sf_col + 16 + 8 * g + 4, smem_desc(smem_u32(sfb) + 512 * g, 0, 128, 0));
    }
    const uint32_t idesc = idesc_mxf4nvf4(kProbeN);
    for (int it = 0; it < iters; ++it) {
      const int g = it & 3;
      mma_mxf4nvf4(tmem, smem_desc(smem_u32(a) + 32 * g, 16, 1024, 2), smem_desc(smem_u32(b) + 32 * g, 16, 1024, 2),
                   idesc, sf_col + 4 * g, sf_col + 16 + 8 * g, it != 0);
    }
    mma_commit(done);
    volatile int no_abort = 0;
    if (!mbar_wait_bounded(done, 0, timeout_ns, &no_abort)) record_error(err, MOE_ERR_TIMEOUT, 20);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_fp4_mma_probe(int iters, int blocks, double* flops_per_launch, void* stream) {
  if (iters < 1 || blocks < 0 || !flops_per_launch) return MOE_ERR_INVALID_ARG;
  // The launch ends with a bounded wait for its MMAs, after which tensor memory is
  // freed: keep the MMA chain far inside that bound (one MMA takes well under
  // 200 ns even at a low clock), so the memory is never freed under a running MMA.
  if (iters > kProbeMaxIters || static_cast<uint64_t>(iters) * 200u > wait_timeout_ns()) return MOE_ERR_INVALID_ARG;
  const int grid = blocks > 0 ? blocks : num_sms();
  if (grid < 1) return MOE_ERR_CUDA;
  int32_t* err = device_error_word();
  if (!err) return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(fp4_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) != cudaSuccess)
    return MOE_ERR_RESOURCE;
  fp4_peak_kernel<<<grid, 128, kProbeSmem, static_cast<cudaStream_t>(stream)>>>(iters, err, wait_timeout_ns());
  *flops_per_launch = 2.0 * 128.0 * kProbeN * 64.0 * static_cast<double>(iters) * grid;
  return check_launch();
}

// ---------------------------------------------------------------------------
// The same measurement for the CTA-pair form (tcgen05 cta_group::2): one thread
// of each even CTA issues M = 256, N = 256, K = 64 MMAs whose A and B halves sit
// in the two CTAs' shared memory; each SM computes 128 x 256 of every MMA.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kPairHalfBytes = 128 * 128;          // 128 rows x 256 K-elements per CTA, for A and for B
constexpr int kPairSmem = 2 * kPairHalfBytes + 1024 + 64;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    fp4_peak_pair_kernel(int iters, int32_t* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a = smem;
  uint8_t* b = a + kPairHalfBytes;
  uint64_t* done = reinterpret_cast<uint64_t*>(b + kPairHalfBytes);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();

  for (int i = threadIdx.x; i < 2 * kPairHalfBytes / 4; i += blockDim.x) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u ^ (blockIdx.x * 40503u);
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    reinterpret_cast<uint32_t*>(a)[i] = h;
  }
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_barrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {  // one warp of each CTA: the pair's allocation is made by both together
    tmem_alloc_pair(s_tmem, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // scale 1.0 (e4m3 0x38) in every scale column [256, 512) of every lane: each warp its lane quadrant
  {
    uint32_t ones[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) ones[i] = 0x38383838u;
    for (int c = 256; c < 512; c += 32) tmem_st_32cols(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c, ones);
    tmem_st_wait();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs: operands written, barrier initialised, tensor memory allocated
  tc_fence_after();
  if (rank == 0 && threadIdx.x == 0) {
    const uint32_t idesc = idesc_mxf4nvf4(256, 256);
    for (int it = 0; it < iters; ++it) {
      const int g = it & 3;
      // A scales of K step g at column 256 + 4g, B scales (256 rows) at 272 + 8g
      mma_mxf4nvf4_pair(tmem, smem_desc(smem_u32(a) + 32 * g, 16, 1024, 2),
                        smem_desc(smem_u32(b) + 32 * g, 16, 1024, 2), idesc, tmem + 256 + 4 * g,
                        tmem + 272 + 8 * g, it != 0);
    }
    mma_commit_pair(done, 0x3);  // both CTAs learn that the MMAs writing their tensor memory are done
  }
  if (threadIdx.x == 0) {
    volatile int no_abort = 0;
    if (!mbar_wait_bounded(done, 0, timeout_ns, &no_abort)) record_error(err, MOE_ERR_TIMEOUT, 21);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA frees its half while the other may still use the pair
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_fp4_mma_probe_pair(int iters, int pairs, double* flops_per_launch, void* stream) {
  if (iters < 1 || pairs < 0 || !flops_per_launch) return MOE_ERR_INVALID_ARG;
  if (iters > kProbeMaxIters || static_cast<uint64_t>(iters) * 200u > wait_timeout_ns()) return MOE_ERR_INVALID_ARG;
  int32_t* err = device_error_word();
  if (!err) return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(fp4_peak_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem) !=
      cudaSuccess)
    return MOE_ERR_RESOURCE;
  int n = pairs;
  if (n == 0) {  // as many pairs as can be resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = kPairSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fp4_peak_pair_kernel, &cfg) != cudaSuccess || n < 1) return MOE_ERR_CUDA;
  }
  fp4_peak_pair_kernel<<<2 * n, 128, kPairSmem, static_cast<cudaStream_t>(stream)>>>(iters, err, wait_timeout_ns());
  *flops_per_launch = 2.0 * 256.0 * 256.0 * 64.0 * static_cast<double>(iters) * n;
  return check_launch();
}

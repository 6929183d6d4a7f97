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

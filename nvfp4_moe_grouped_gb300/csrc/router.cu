// router.cu -- the router in front of the routing step: the logits GEMM
//   logits[t][e] = sum_h x[t][h] * w_gate[e][h]      (bf16 inputs, FP32 sums)
// on the 5th-generation tensor cores, then the top-k routing and stable
// permutation of route_permute.cu on those logits.
//
// "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on Blackwell
// SM120", section "The Broader Context": every token is scored against the 256
// experts and the 8 best are kept.  The pages give no gate formula; the plain
// reading is a bias-free linear gate over the hidden state, logits in FP32.
//
// The contraction is small (T x E x H = 1024 x 256 x 6144 at decode) and its
// inputs are read once, so the launch is spread over the GPU by splitting K:
// CTA (tile, split) multiplies 128 tokens by all E (<= 256) experts over its
// share of H with tcgen05.mma kind::f16 (M = 128 tokens, N = E rounded up to 16,
// K = 16, FP32 accumulator in tensor memory) and stores its FP32 partial tile.
// The routing kernel adds the partials in split order (deterministic) as it
// reads each token's logits, so the logits never make a round trip of their
// own.  Roles in the GEMM CTA: lane 0 of warp 0 issues the TMA loads (128-byte
// swizzle, rows past T or E read as zeros), lane 0 of warp 1 the MMAs, warps 2
// and 3 (when asked) take max |x| over the x tiles for the activation
// quantiser, half of each stage each, two |bf16| patterns per 32-bit word
// (one warp taking them one by one held the mainloop to its pace); all four
// warps then drain the accumulator.  Every wait is bounded.
#include "common.cuh"

namespace moe {
moe_status route_permute_enqueue(const float* logits, const float* part, int splits, int NE, float* logits_out,
                                 const uint32_t* x_amax_bits, float* x_scale, int T, int E, int k, int32_t* topk_id,
                                 float* topk_w, int32_t* expert_offsets, int32_t* perm_to_expanded,
                                 int32_t* expanded_to_perm, int32_t* expanded_to_row, void* ws, cudaStream_t st);
namespace {

constexpr int kRThreads = 128;
constexpr int kRStages = 4;
constexpr int kRBK = 64;                     // bf16 elements per K block (128 bytes of a row)
constexpr int kRAStage = 128 * 128;          // 128 tokens x 128 bytes
constexpr int kRBStage = 256 * 128;          // up to 256 experts x 128 bytes
constexpr int kRSmem = kRStages * (kRAStage + kRBStage) + 128 + 1024;  // stages, barriers, alignment slack
constexpr uint32_t kRTmemCols = 256;

struct RouterParams {
  int T, E, NE, KB, splits;
  float* part;           // [tiles][splits][128][NE]
  uint32_t* amax_bits;   // optional: max |x| (bit pattern), for the activation quantiser
  int32_t* err;
  uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kRThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = smem;
  uint8_t* s_b = smem + kRStages * kRAStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_b + kRStages * kRBStage);
  uint64_t* empty = full + kRStages;
  uint64_t* acc_full = empty + kRStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * p.KB / p.splits);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.KB / p.splits);
  const int nk = kb1 - kb0;  // >= 1: splits <= KB
  const uint32_t b_bytes = static_cast<uint32_t>(p.NE) * 128;

  const bool amax_on = p.amax_bits != nullptr;
  if (threadIdx.x == 0) {
    // a stage is free once the MMAs and (when x's amax is wanted) warps 2 and 3 are done with it
    for (int s = 0; s < kRStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], amax_on ? 3 : 1); }
    mbar_init(acc_full, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kRTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0 && lane == 0) {
    // ---- producer ----
    const uint64_t pol = l2_policy_evict_first();
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kRStages;
      const uint32_t ph = static_cast<uint32_t>(i / kRStages) & 1u;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.timeout_ns, s_abort)) {
        if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 30);
        *s_abort = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[s], kRAStage + b_bytes);
      tma_load_2d(s_a + s * kRAStage, &tm_x, &full[s], (kb0 + i) * kRBK, tile * 128, pol);
      tma_load_2d(s_b + s * kRBStage, &tm_w, &full[s], (kb0 + i) * kRBK, 0, pol);
      issued = i + 1;
    }
    // let the copies this CTA started land before it can exit (the last kRStages fills)
    int zero = 0;
    for (int i = issued - kRStages > 0 ? issued - kRStages : 0; i < issued; ++i)
      mbar_wait_bounded(&full[i % kRStages], static_cast<uint32_t>(i / kRStages) & 1u, p.timeout_ns,
                        reinterpret_cast<volatile int*>(&zero));
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = idesc_bf16_f32(p.NE);
    for (int i = 0; i < nk; ++i) {
      const int s = i % kRStages;
      const uint32_t ph = static_cast<uint32_t>(i / kRStages) & 1u;
      if (!mbar_wait_bounded(&full[s], ph, p.timeout_ns, s_abort)) {
        if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 31);
        *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint64_t adesc = smem_desc(smem_u32(s_a + s * kRAStage), 16, 1024, 2);
      const uint64_t bdesc = smem_desc(smem_u32(s_b + s * kRBStage), 16, 1024, 2);
#pragma unroll
      for (int g = 0; g < 4; ++g)  // K = 16 per MMA: 32 bytes along the swizzled row
        mma_bf16(tmem, adesc + 2 * g, bdesc + 2 * g, idesc, (i | g) != 0);
      mma_commit(&empty[s]);
    }
    mma_commit(acc_full);  // arrives once every MMA issued above has completed
  } else if ((warp == 2 || warp == 3) && amax_on) {
    // ---- max |x| over this CTA's x tiles (each x element is in exactly one CTA's tiles; rows past T
    // are zero-filled), for the NVFP4 decode multiplier of the activation quantiser: warp 2 the first
    // half of every stage, warp 3 the second; |bf16| bit patterns order like the values ----
    const int hw = warp - 2;
    uint32_t m2 = 0;  // maxima of the two halfwords
    for (int i = 0; i < nk; ++i) {
      const int s = i % kRStages;
      const uint32_t ph = static_cast<uint32_t>(i / kRStages) & 1u;
      const bool got = mbar_wait_bounded(&full[s], ph, p.timeout_ns, s_abort);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 33);
          *s_abort = 1;
        }
        break;
      }
      const uint4* a4 = reinterpret_cast<const uint4*>(s_a + s * kRAStage + hw * (kRAStage / 2));
#pragma unroll 8
      for (int j = lane; j < kRAStage / 32; j += 32) {
        const uint4 u = a4[j];
        m2 = __vmaxu2(m2, u.x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, u.y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, u.z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, u.w & 0x7FFF7FFFu);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && m > 0) atomicMax(p.amax_bits, m << 16);  // the bf16 pattern as an f32 pattern
  }
  __syncwarp();

  // ---- epilogue: all four warps; thread = token row of the tile (its TMEM lane) ----
  const bool got = mbar_wait_bounded(acc_full, 0, p.timeout_ns, s_abort);
  const int bad = __syncthreads_or(!got || *s_abort);
  tc_fence_after();
  if (!bad) {
    const int r = warp * 32 + lane;
    float* dst = p.part + (static_cast<int64_t>(tile * p.splits + split) * 128 + r) * p.NE;
    for (int c0 = 0; c0 < p.NE; c0 += 32) {
      uint32_t v[32];
      tmem_ld_32cols(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
      tmem_ld_wait();
      const int cn = min(32, p.NE - c0);  // NE is a multiple of 16
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        if (j < cn)
          *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                 __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
    }
  } else if (threadIdx.x == 0 && !got) {
    record_error(p.err, MOE_ERR_TIMEOUT, 32);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kRTmemCols);
  }
}

struct RouterShape {
  int tiles, splits, NE, KB;
  size_t part_bytes;
};

RouterShape router_shape(int T, int E, int H) {
  RouterShape s;
  s.tiles = (T + 127) / 128;
  s.NE = (E + 15) / 16 * 16;
  s.KB = H / kRBK;
  const int sms = num_sms() > 0 ? num_sms() : 148;
  // up to one CTA per SM, but at most 8 splits: each split adds T x E floats of partial sums that the
  // routing kernel reads back per token
  int splits = (sms + s.tiles - 1) / s.tiles;
  if (splits > s.KB) splits = s.KB;
  if (splits > 8) splits = 8;
  if (splits < 1) splits = 1;
  s.splits = splits;
  s.part_bytes = (static_cast<size_t>(s.tiles) * splits * 128 * s.NE * sizeof(float) + 255) / 256 * 256;
  return s;
}

// 2D bf16 map over [rows][cols], boxes of 64 columns (128 bytes) x box_rows, 128-byte swizzle.
bool make_bf16_map(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kRBK), box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_router_workspace_size(int T, int E, int H, int k) {
  if (T < 1 || E < 1 || H < kRBK || k < 1) return 0;
  const RouterShape s = router_shape(T, E, H);
  return s.part_bytes + 256 + moe_route_permute_workspace_size(T, E, k);  // 256: the amax word
}

extern "C" moe_status moe_router(const uint16_t* x, const uint16_t* w_gate, int T, int E, int H, int k,
                                 float* logits, float* x_scale, int32_t* topk_id, float* topk_w,
                                 int32_t* expert_offsets, int32_t* perm_to_expanded, int32_t* expanded_to_perm,
                                 int32_t* expanded_to_row, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !w_gate || !topk_id || !topk_w || !expert_offsets || !perm_to_expanded || !expanded_to_perm ||
      !expanded_to_row)
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || H < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 256 || k > 32 || H % kRBK) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * k > 0x7FFFFFFF || static_cast<int64_t>(T) * E > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(ws) || (logits && !aligned16(logits))) return MOE_ERR_MISALIGNED;
  if (!ws || ws_bytes < moe_router_workspace_size(T, E, H, k)) return MOE_ERR_WORKSPACE;
  const RouterShape s = router_shape(T, E, H);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float* part = reinterpret_cast<float*>(w8);
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(w8 + s.part_bytes);
  void* route_ws = w8 + s.part_bytes + 256;

  RouterParams p{};
  p.T = T;
  p.E = E;
  p.NE = s.NE;
  p.KB = s.KB;
  p.splits = s.splits;
  p.part = part;
  p.amax_bits = x_scale ? amax_bits : nullptr;
  p.err = device_error_word();
  p.timeout_ns = wait_timeout_ns();
  if (!p.err) return MOE_ERR_CUDA;
  CUtensorMap tm_x, tm_w;
  if (!make_bf16_map(&tm_x, x, static_cast<uint64_t>(T), static_cast<uint64_t>(H), 128)) return MOE_ERR_CUDA;
  if (!make_bf16_map(&tm_w, w_gate, static_cast<uint64_t>(E), static_cast<uint64_t>(H), static_cast<uint32_t>(s.NE)))
    return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem) != cudaSuccess)
    return MOE_ERR_RESOURCE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (x_scale && cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  router_gemm_kernel<<<dim3(s.tiles, s.splits), kRThreads, kRSmem, st>>>(tm_x, tm_w, p);
  moe_status rs = check_launch();
  if (rs != MOE_OK) return rs;
  // the routing kernel adds the partial sums (in split order) as it reads each token's logits
  return route_permute_enqueue(nullptr, part, s.splits, s.NE, logits, x_scale ? amax_bits : nullptr, x_scale, T, E,
                               k, topk_id, topk_w, expert_offsets, perm_to_expanded, expanded_to_perm,
                               expanded_to_row, route_ws, st);
}

// router.cu -- the router in front of the routing step: the logits GEMM
//   logits[t][e] = sum_h x[t][h] * w_gate[e][h]      (bf16 inputs, FP32 sums)
// on the 5th-generation tensor cores, with the top-k and softmax of every
// token in the same kernel; then the stable permutation's scan and scatter.
//
// "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on Blackwell
// SM120", section "The Broader Context": every token is scored against the 256
// experts and the 8 best are kept.  The pages give no gate formula; the plain
// reading is a bias-free linear gate over the hidden state, logits in FP32.
//
// The contraction is small (T x E x H = 1024 x 256 x 6144 at decode) and its
// inputs are read once, so the launch is spread over the GPU by splitting K:
// the S (<= 16) CTAs of a cluster share one tile of 128 tokens, CTA (tile,
// split) multiplying the tile by all E (<= 256) experts over its share of H
// with tcgen05.mma kind::f16 (M = 128 tokens, N = E rounded up to 16, K = 16,
// FP32 accumulator in tensor memory).  The partial sums then never leave the
// cluster: each CTA drains its accumulator and stores every token row into the
// shared memory of the CTA that owns the token (128 / S tokens per CTA); each
// owner adds its rows' S partial rows in split order (deterministic), and one
// warp per token runs the top-k and softmax (k rounds of a warp max and a warp
// min reduction), writing the routing and the counts of its chunk of (token,
// slot) items; the scan and the stable scatter of route_permute.cu follow.
// Roles: lane 0 of warp 0 issues the TMA loads (128-byte swizzle, rows past T
// or E read as zeros), lane 0 of warp 1 the MMAs, warps 2 and 3 (when asked)
// take max |x| over the x tiles for the activation quantiser (the scan kernel
// combines the CTAs' words into x's decode multiplier); all sixteen warps
// drain and route (the phases after the MMAs are latency-bound, so more warps
// shorten them).  Every mbarrier wait is bounded; every CTA reaches both
// cluster barriers on every path, and a CTA whose waits gave up marks the tile
// void in its peers.
#include <algorithm>

#include "common.cuh"

namespace moe {
int& gemm_debug_flags();
moe_status route_scan_scatter_enqueue(int T, int E, int k, int chunk_tokens, const int32_t* topk_id,
                                      int32_t* chunk_counts, int32_t* pad_offsets, int32_t* expert_totals,
                                      const uint32_t* amax_part, int n_parts, float* x_scale,
                                      int32_t* expert_offsets, int32_t* perm_to_expanded, int32_t* expanded_to_perm,
                                      int32_t* expanded_to_row, cudaStream_t st);
namespace {

constexpr int kRThreads = 512;
constexpr int kRStages = 4;
constexpr int kRBK = 64;                     // bf16 elements per K block (128 bytes of a row)
constexpr int kRAStage = 128 * 128;          // 128 tokens x 128 bytes
constexpr int kRBStage = 256 * 128;          // up to 256 experts x 128 bytes
constexpr int kRStageArea = kRStages * (kRAStage + kRBStage);
constexpr int kRMaxSplits = 16;              // 16 only where the device places clusters that large
constexpr int kRAmaxWarps = 2;               // warps 2 and 3 take max |x|, half of each x stage each
// after the MMAs the stage area holds the partial rows this CTA owns ([S][128 / S][NE] floats, 128 KB at
// NE = 256), its chunk counts (at most 16 chunks x E ints: a chunk holds at least 8 tokens) and one void
// flag per peer (at most 16)
constexpr int kRRecvBytes = 128 * 256 * 4;
constexpr int kRHistOff = kRRecvBytes;
constexpr int kRHistBytes = 16 * 256 * 4;
constexpr int kRFlagOff = kRHistOff + kRHistBytes;
static_assert(kRFlagOff + 64 <= kRStageArea, "exchange area fits the stage area");
constexpr int kRSmem = kRStageArea + 128 + 1024;  // stages, barriers, alignment slack
constexpr uint32_t kRTmemCols = 256;
constexpr int kRDrainStep = 32 * (kRThreads / 128);  // columns between a drain warp's two 32-column blocks
static_assert(2 * kRDrainStep >= static_cast<int>(kRTmemCols), "two blocks per drain warp cover the accumulator");

struct RouterParams {
  int T, E, NE, KB, k, group, chunk_tokens, n_chunks;
  uint32_t* amax_part;   // optional: max |x| (bit pattern) of each amax warp's x tiles, [tiles * splits * 2]
  float* logits;         // optional [T][E]
  int32_t* topk_id;
  float* topk_w;
  int32_t* chunk_counts;  // [n_chunks][E]: items of each expert in each chunk of chunk_tokens tokens
  int32_t* err;
  uint64_t timeout_ns;
  int debug_flags;  // bit 0: CTA (0, 0) never fills its first stage (bounded-wait test hook)
};

MOE_DEVINL void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
MOE_DEVINL void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// The partial logits a CTA owns sit column-major: [split][float4 chunk c of
// the experts][token slot g], so a warp storing one chunk of 32 consecutive
// token rows, and a thread reading its token's chunks in order, both touch
// consecutive 16-byte words.
MOE_DEVINL int recv_off(int split, int c, int g, int G, int nc4) { return ((split * nc4 + c) * G + g) * 4; }

template <int NV>  // logits per lane: 32 NV >= E
__global__ void __launch_bounds__(kRThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = smem;
  uint8_t* s_b = smem + kRStages * kRAStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRStageArea);
  uint64_t* empty = full + kRStages;
  uint64_t* acc_full = empty + kRStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  float* s_recv = reinterpret_cast<float*>(smem);
  int* s_hist = reinterpret_cast<int*>(smem + kRHistOff);
  volatile int* s_void = reinterpret_cast<volatile int*>(smem + kRFlagOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y, S = gridDim.y;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * p.KB / S);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.KB / S);
  const int nk = kb1 - kb0;  // >= 1: splits <= KB
  const uint32_t b_bytes = static_cast<uint32_t>(p.NE) * 128;

  const bool amax_on = p.amax_part != nullptr;
  if (threadIdx.x == 0) {
    // a stage is free once the MMAs and (when x's amax is wanted) both amax warps are done with it
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], amax_on ? 1 + kRAmaxWarps : 1);
    }
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
    const bool skip_first = (p.debug_flags & 1) != 0 && tile == 0 && split == 0;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kRStages;
      const uint32_t ph = static_cast<uint32_t>(i / kRStages) & 1u;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.timeout_ns, s_abort)) {
        if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 30);
        *s_abort = 1;
        break;
      }
      if (i == 0 && skip_first) continue;  // stage 0 never fills: the MMA thread's wait gives up
      mbar_arrive_expect_tx(&full[s], kRAStage + b_bytes);
      tma_load_2d(s_a + s * kRAStage, &tm_x, &full[s], (kb0 + i) * kRBK, tile * 128, pol);
      tma_load_2d(s_b + s * kRBStage, &tm_w, &full[s], (kb0 + i) * kRBK, 0, pol);
      issued = i + 1;
    }
    // let the copies this CTA started land before the stage area is reused (the last kRStages fills)
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
    // ---- max |x| over this CTA's x tiles (each x element is in exactly one CTA's tiles; rows past T are
    // zero-filled), for the NVFP4 decode multiplier of the activation quantiser: warp 2 the first half
    // of every stage, warp 3 the second; |bf16| patterns order like the values, two per 32-bit word ----
    const int hw = warp - 2;
    uint32_t m2 = 0;  // per-halfword maxima
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
    if (lane == 0) p.amax_part[(tile * S + split) * kRAmaxWarps + hw] = m << 16;  // as an f32 pattern
  }
  __syncwarp();

  // ---- epilogue: all eight warps ----
  const bool got = mbar_wait_bounded(acc_full, 0, p.timeout_ns, s_abort);
  const int bad = __syncthreads_or(!got || *s_abort);
  if (threadIdx.x == 0 && !got && !*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 32);
  tc_fence_after();
  // the stage area was last written by the tensor-memory copies (async proxy); order those writes before
  // the generic stores made into it from here on (the void flags below, the peers' rows after the barrier)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x < kRMaxSplits) s_void[threadIdx.x] = 0;  // peers write here only after the barrier
  cluster_sync_all();  // every CTA of the tile is done with its stage area
  const int G = p.group;
  if (!bad) {
    // this CTA's partial row of token r (its TMEM lane) goes to owner r / G, slot [split][r % G]; warp w
    // drains lane quadrant w % 4, the 32-column blocks 32 * (w / 4) and 32 * (w / 4) + 128, both loads in
    // flight before one wait
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int nc4 = p.NE / 4;
    const uint32_t base = map_shared_rank(smem_u32(s_recv), static_cast<uint32_t>(r / G));
    const uint32_t lane_cols = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const int c0 = 32 * (warp >> 2);
    uint32_t v[2][32];
    if (c0 < p.NE) tmem_ld_32cols(lane_cols + c0, v[0]);
    if (c0 + kRDrainStep < p.NE) tmem_ld_32cols(lane_cols + c0 + kRDrainStep, v[1]);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cb = c0 + h * kRDrainStep;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = (cb >> 2) + i;
        if (cb < p.NE && c < nc4)  // NE is a multiple of 16
          st_cluster_v4(base + 4 * recv_off(split, c, r % G, G, nc4), v[h][4 * i], v[h][4 * i + 1],
                        v[h][4 * i + 2], v[h][4 * i + 3]);
      }
    }
  } else if (threadIdx.x < S) {
    // this tile's routing cannot be computed: say so to every CTA of the tile
    st_cluster_u32(map_shared_rank(smem_u32(const_cast<int*>(s_void) + split), threadIdx.x), 1u);
  }
  cluster_sync_all();  // every partial row (or void flag) has landed
  int void_any = 0;
  for (int q = 0; q < S; ++q) void_any |= s_void[q];
  // ---- the owner of tokens [tok0, tok0 + G): their S partial rows summed in split order into slot 0
  // (and written out as logits when asked), then one warp per token: top-k, softmax, chunk counts.
  // A void tile (its error already recorded) routes every token to experts 0..k-1 with weight 0, so that
  // the scan and scatter after it stay within their buffers.
  const int tok0 = tile * 128 + split * G;
  const int CT = p.chunk_tokens;
  const int n_cl = G / CT;  // chunks of this CTA's tokens
  for (int i = threadIdx.x; i < n_cl * p.E; i += kRThreads) s_hist[i] = 0;
  if (!void_any && (S > 1 || p.logits)) {  // one split and no logits wanted: slot 0 holds the sums already
    const int nc4 = p.NE / 4;  // float4 chunks of a row
    for (int i = threadIdx.x; i < G * nc4; i += kRThreads) {
      const int c = i / G, g = i - c * G, e0 = 4 * c;
      float4* dst = reinterpret_cast<float4*>(s_recv + recv_off(0, c, g, G, nc4));
      float4 v = *dst;
      for (int q = 1; q < S; ++q) {
        const float4 u = *reinterpret_cast<const float4*>(s_recv + recv_off(q, c, g, G, nc4));
        v.x = __fadd_rn(v.x, u.x);
        v.y = __fadd_rn(v.y, u.y);
        v.z = __fadd_rn(v.z, u.z);
        v.w = __fadd_rn(v.w, u.w);
      }
      if (S > 1) *dst = v;
      const int t = tok0 + g;
      if (p.logits && t < p.T && e0 < p.E) {
        float* lrow = p.logits + static_cast<int64_t>(t) * p.E + e0;
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j < p.E) lrow[j] = vv[j];
      }
    }
  }
  __syncthreads();
  const int nc4 = p.NE / 4;
  // one warp per token: its summed row from shared memory, the warp top-k and softmax, the routing out
  // and its items counted in their chunk
  for (int g = warp; g < G; g += kRThreads / 32) {
    const int t = tok0 + g;
    if (t >= p.T) break;  // the same for the whole warp
    float v[NV];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = 0.0f;
      if (e >= p.E) taken |= 1u << i;
      else if (!void_any) v[i] = s_recv[recv_off(0, e >> 2, g, G, nc4) + (e & 3)];
    }
    int id = lane;
    float w = 0.0f;
    if (!void_any) warp_topk_softmax<NV>(v, taken, p.k, &id, &w);
    if (lane < p.k) {
      p.topk_id[static_cast<int64_t>(t) * p.k + lane] = id;
      p.topk_w[static_cast<int64_t>(t) * p.k + lane] = w;
      atomicAdd(&s_hist[(g / CT) * p.E + id], 1);
    }
  }
  __syncthreads();
  const int c_first = tok0 / CT;
  for (int i = threadIdx.x; i < n_cl * p.E; i += kRThreads) {
    const int c = c_first + i / p.E;
    if (c < p.n_chunks) p.chunk_counts[static_cast<int64_t>(c) * p.E + i % p.E] = s_hist[i];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kRTmemCols);
  }
}

struct RouterShape {
  int tiles, splits, NE, KB, group, chunk_tokens, n_chunks;
};

int pow2_floor(int v) {
  int r = 1;
  while (2 * r <= v) r *= 2;
  return r;
}

// Chunk of tokens whose items the scan counts together: a power of two that
// divides the tokens a CTA routes (128 / splits) and keeps a chunk's items
// within one scatter block (256).
int router_chunk_tokens(int splits, int k) { return pow2_floor(std::min(128 / splits, std::max(1, 256 / k))); }

// Clusters of 16 CTAs of one router kernel variant that the current device
// holds at once (0 where it refuses the non-portable size).
template <int NV>
int router_clusters16_of() {
  auto kern = router_topk_kernel<NV>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, 16, 1);
    cfg.blockDim = dim3(kRThreads, 1, 1);
    cfg.dynamicSmemBytes = kRSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 16;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refusal above is an answer, not an error of a later launch
  return n;
}

int router_nv_index(int NE) {
  const int nv = (NE + 31) / 32;
  return nv <= 1 ? 0 : nv <= 2 ? 1 : nv <= 4 ? 2 : 3;
}

// Looked up once per device and variant, never while `st` is being captured
// into a graph (a call made then takes 8-CTA clusters and looks up later).
int router_clusters16(int NE, cudaStream_t st) {
  static int cached[64][4] = {};  // clusters + 1; 0 = not looked up
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int i = router_nv_index(NE);
  if (cached[dev][i] == 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return 0;
    }
    const int n = i == 0 ? router_clusters16_of<1>()
                  : i == 1 ? router_clusters16_of<2>()
                  : i == 2 ? router_clusters16_of<4>()
                           : router_clusters16_of<8>();
    cached[dev][i] = n + 1;
  }
  return cached[dev][i] - 1;
}

// Splits: a power of two, so that the tiles x splits CTAs fill the SMs, each
// with at least one K block; 16 (a non-portable cluster) only where the device
// holds every tile's cluster at once, else at most 8.
RouterShape router_shape(int T, int E, int H, int k, cudaStream_t st) {
  RouterShape s;
  s.tiles = (T + 127) / 128;
  s.NE = (E + 15) / 16 * 16;
  s.KB = H / kRBK;
  const int sms = num_sms() > 0 ? num_sms() : 148;
  int splits = pow2_floor(std::max(1, sms / s.tiles));
  splits = std::min(splits, std::min(kRMaxSplits, pow2_floor(s.KB)));
  if (splits > 8 && router_clusters16(s.NE, st) < s.tiles) splits = 8;
  s.splits = splits;
  s.group = 128 / splits;
  s.chunk_tokens = router_chunk_tokens(splits, k);
  s.n_chunks = (T + s.chunk_tokens - 1) / s.chunk_tokens;
  return s;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace: per-CTA amax words, then the chunk counts, the padded offsets and
// each expert's total; sized for the most CTAs and the most chunks any split
// count gives.
struct RouterWs {
  size_t amax_off, counts_off, pads_off, totals_off, total;
};
RouterWs router_ws(int T, int E, int k) {
  RouterWs w;
  const int tiles = (T + 127) / 128;
  const int ct_min = router_chunk_tokens(kRMaxSplits, k);
  const int64_t chunks_max = (T + ct_min - 1) / ct_min;
  w.amax_off = 0;
  w.counts_off = align256(static_cast<size_t>(tiles) * kRMaxSplits * kRAmaxWarps * sizeof(uint32_t));
  w.pads_off = w.counts_off + align256(static_cast<size_t>(chunks_max) * E * sizeof(int32_t));
  w.totals_off = w.pads_off + align256(static_cast<size_t>(E + 1) * sizeof(int32_t));
  w.total = w.totals_off + align256(static_cast<size_t>(E) * sizeof(int32_t));
  return w;
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

template <int NV>
moe_status launch_router(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterParams& p, int tiles,
                         int splits, cudaStream_t st) {
  auto kern = router_topk_kernel<NV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem) != cudaSuccess)
    return MOE_ERR_RESOURCE;
  if (splits > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return MOE_ERR_RESOURCE;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(tiles, splits, 1);
  cfg.blockDim = dim3(kRThreads, 1, 1);
  cfg.dynamicSmemBytes = kRSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of one tile form a cluster
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, p) != cudaSuccess) return MOE_ERR_CUDA;
  return check_launch();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_router_workspace_size(int T, int E, int H, int k) {
  if (T < 1 || E < 1 || H < kRBK || k < 1) return 0;
  return router_ws(T, E, k).total;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const RouterShape s = router_shape(T, E, H, k, st);
  const RouterWs L = router_ws(T, E, k);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint32_t* amax_part = reinterpret_cast<uint32_t*>(w8 + L.amax_off);
  int32_t* counts = reinterpret_cast<int32_t*>(w8 + L.counts_off);
  int32_t* pads = reinterpret_cast<int32_t*>(w8 + L.pads_off);
  int32_t* totals = reinterpret_cast<int32_t*>(w8 + L.totals_off);

  RouterParams p{};
  p.T = T;
  p.E = E;
  p.NE = s.NE;
  p.KB = s.KB;
  p.k = k;
  p.group = s.group;
  p.chunk_tokens = s.chunk_tokens;
  p.n_chunks = s.n_chunks;
  p.amax_part = x_scale ? amax_part : nullptr;
  p.logits = logits;
  p.topk_id = topk_id;
  p.topk_w = topk_w;
  p.chunk_counts = counts;
  p.err = device_error_word();
  p.timeout_ns = wait_timeout_ns();
  p.debug_flags = gemm_debug_flags();
  if (!p.err) return MOE_ERR_CUDA;
  CUtensorMap tm_x, tm_w;
  if (!make_bf16_map(&tm_x, x, static_cast<uint64_t>(T), static_cast<uint64_t>(H), 128)) return MOE_ERR_CUDA;
  if (!make_bf16_map(&tm_w, w_gate, static_cast<uint64_t>(E), static_cast<uint64_t>(H), static_cast<uint32_t>(s.NE)))
    return MOE_ERR_CUDA;
  const int nv = (s.NE + 31) / 32;
  moe_status rs = nv <= 1   ? launch_router<1>(tm_x, tm_w, p, s.tiles, s.splits, st)
                  : nv <= 2 ? launch_router<2>(tm_x, tm_w, p, s.tiles, s.splits, st)
                  : nv <= 4 ? launch_router<4>(tm_x, tm_w, p, s.tiles, s.splits, st)
                            : launch_router<8>(tm_x, tm_w, p, s.tiles, s.splits, st);
  if (rs != MOE_OK) return rs;
  // expert offsets, padded offsets and the stable scatter from the routing kernel's chunk counts; x's
  // decode multiplier from the CTAs' amax words
  return route_scan_scatter_enqueue(T, E, k, s.chunk_tokens, topk_id, counts, pads, totals,
                                    x_scale ? amax_part : nullptr, s.tiles * s.splits * kRAmaxWarps, x_scale,
                                    expert_offsets, perm_to_expanded, expanded_to_perm, expanded_to_row, st);
}

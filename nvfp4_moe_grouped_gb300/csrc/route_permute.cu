// route_permute.cu -- top-k routing of tokens to experts and the stable
// counting-sort permutation that groups the routed rows by expert.
//
// "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on Blackwell
// SM120", section "The Broader Context": 256 experts, 8 active per token;
// section "Input Knowledge Required": one GEMM per expert over that expert's
// rows.  Selection rule (largest logits, ties to the lower index) and weights
// (softmax over the k selected logits) as stated in nvfp4_moe.h.
//
// Three launches, all deterministic:
//   1. route_kernel: one warp per token does a warp-shuffle top-k over the E
//      logits held in registers, the softmax of the selected k, and each block
//      counts the expert histogram of its chunk of (token, slot) items.
//   2. scan_kernel: one block turns the per-chunk histograms into expert
//      offsets, padded (128-row) offsets and per-chunk base positions.
//   3. scatter_kernel: each block ranks its chunk's items stably within each
//      expert (warp match + warps in order) and writes the permutation.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;      // scatter: one thread per (token, slot) item of a chunk
constexpr int kTopkThreads = 1024;      // top-k (a single-chunk layer): one warp per token

struct RouteDims {
  int T, E, k, chunk_tokens, n_chunks;
};

inline RouteDims route_dims(int T, int E, int k) {
  RouteDims d;
  d.T = T; d.E = E; d.k = k;
  d.chunk_tokens = kRouteThreads / k;
  if (d.chunk_tokens < 1) d.chunk_tokens = 1;
  d.n_chunks = (T + d.chunk_tokens - 1) / d.chunk_tokens;
  return d;
}

// Top-k and softmax of tokens [t0, t1), one warp per token (warps of the whole
// block in turn); counts each selected expert in the shared histogram `hist`.
// For E <= 256 a warp loads its next token's row while it ranks the current
// one.
template <int NV>  // logits per lane, NV * 32 >= E
MOE_DEVINL void route_tokens(const float* __restrict__ logits, const RouteDims& d, int t0, int t1,
                             int32_t* __restrict__ topk_id, float* __restrict__ topk_w, int* hist) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x / 32;
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (lane + 32 * i >= d.E) taken |= 1u << i;
  constexpr bool kAhead = NV <= 8;
  float nxt[NV];  // the row of the warp's next token
  if (kAhead) {
    const float* row = logits + static_cast<int64_t>(t0 + warp < t1 ? t0 + warp : t0) * d.E;
#pragma unroll
    for (int i = 0; i < NV; ++i) nxt[i] = (t0 + warp < t1 && !(taken >> i & 1u)) ? __ldg(row + lane + 32 * i) : 0.0f;
  }
  for (int t = t0 + warp; t < t1; t += nw) {
    float v[NV];
    if (kAhead) {
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = nxt[i];
      if (t + nw < t1) {
        const float* row = logits + static_cast<int64_t>(t + nw) * d.E;
#pragma unroll
        for (int i = 0; i < NV; ++i) nxt[i] = (taken >> i & 1u) ? 0.0f : __ldg(row + lane + 32 * i);
      }
    } else {
      const float* row = logits + static_cast<int64_t>(t) * d.E;
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = (taken >> i & 1u) ? 0.0f : __ldg(row + lane + 32 * i);
    }
    int my_i;
    float my_w;
    warp_topk_softmax<NV>(v, taken, d.k, &my_i, &my_w);
    if (lane < d.k) {
      int64_t o = static_cast<int64_t>(t) * d.k + lane;
      topk_id[o] = my_i;
      topk_w[o] = my_w;
      atomicAdd(&hist[my_i], 1);
    }
  }
}

template <int NV>
__global__ void __launch_bounds__(kRouteThreads, NV > 8 ? 1 : 4) route_kernel(const float* __restrict__ logits,
                                                                             RouteDims d,
                                                                             int32_t* __restrict__ topk_id,
                                                                             float* __restrict__ topk_w,
                                                                             int32_t* __restrict__ chunk_counts) {
  extern __shared__ int hist[];  // [E]
  const int t0 = blockIdx.x * d.chunk_tokens;
  const int t1 = min(d.T, t0 + d.chunk_tokens);
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  route_tokens<NV>(logits, d, t0, t1, topk_id, topk_w, hist);
  __syncthreads();
  int32_t* out = chunk_counts + static_cast<int64_t>(blockIdx.x) * d.E;
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) out[e] = hist[e];
}

// Exclusive scan of one value per thread over a block of up to 1024 threads.
MOE_DEVINL int block_exclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int nw = (blockDim.x + 31) >> 5;
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) warp_tot[lane] = t;  // inclusive warp prefix
  }
  __syncthreads();
  int before = warp ? warp_tot[warp - 1] : 0;
  int r = before + x - v;
  __syncthreads();
  return r;
}

// Each expert's items before every chunk: chunk_counts[b][e] (items of expert e
// in chunk b) becomes the exclusive prefix over chunks b' < b, and
// expert_total[e] the sum over all chunks.  Block x covers the 32 experts
// 32 x .. 32 x + 31 (one per lane, so a warp reads 128 contiguous bytes of a
// chunk's row) and splits the chunks into 32 groups, one per warp; the group
// sums are scanned per expert in shared memory, then every thread rewrites its
// chunks from its group's base.  The expert offsets themselves (a scan over
// experts) are left to the scatter.  With `amax_part` (n_parts max |x| words,
// f32 bit patterns, from the router's CTAs), block 0's first warp also writes
// x's NVFP4 decode multiplier s = amax / (6 * 448) (1 when amax = 0).
__global__ void __launch_bounds__(1024) chunk_scan_kernel(RouteDims d, int32_t* __restrict__ chunk_counts,
                                                          int32_t* __restrict__ expert_total,
                                                          const uint32_t* __restrict__ amax_part, int n_parts,
                                                          float* __restrict__ x_scale) {
  __shared__ int part[32][33];  // [group][expert of the block], then each group's base
  constexpr int kB = 8;         // loads issued together
  const int g = threadIdx.x >> 5, c = threadIdx.x & 31;
  if (amax_part && blockIdx.x == 0 && g == 0) {
    uint32_t m = 0;
    for (int i = c; i < n_parts; i += 32) m = max(m, amax_part[i]);  // non-negative patterns order as values
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (c == 0) {
      const float a = __uint_as_float(m);
      *x_scale = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
    }
  }
  const int e = blockIdx.x * 32 + c;
  const bool act = e < d.E;
  const int b0 = static_cast<int>(static_cast<int64_t>(g) * d.n_chunks / 32);
  const int b1 = static_cast<int>(static_cast<int64_t>(g + 1) * d.n_chunks / 32);
  int sub = 0;
  if (act) {
    for (int b = b0; b < b1; b += kB) {
      int v[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) v[u] = b + u < b1 ? chunk_counts[static_cast<int64_t>(b + u) * d.E + e] : 0;
#pragma unroll
      for (int u = 0; u < kB; ++u) sub += v[u];
    }
  }
  part[g][c] = sub;
  __syncthreads();
  {  // warp g scans expert 32 x + g over the groups: lane c holds group c
    const int v = part[c][g];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (c >= o) x += y;
    }
    part[c][g] = x - v;
    const int eg = blockIdx.x * 32 + g;
    if (c == 31 && eg < d.E) expert_total[eg] = x;
  }
  __syncthreads();
  if (act) {
    int run = part[g][c];
    for (int b = b0; b < b1; b += kB) {
      int v[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) v[u] = b + u < b1 ? chunk_counts[static_cast<int64_t>(b + u) * d.E + e] : 0;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if (b + u < b1) chunk_counts[static_cast<int64_t>(b + u) * d.E + e] = run;
        run += v[u];
      }
    }
  }
}

// Expert offsets and 128-row padded offsets from the per-expert totals, into
// shared `off` and `poff` (every block of the scatter computes them; block 0
// also writes them out, with the grand totals at index E).  256 threads, each
// over up to four consecutive experts (E <= 1024).
MOE_DEVINL void expert_offsets_from_totals(const RouteDims& d, const int32_t* __restrict__ expert_total, int* off,
                                           int* poff, int* warp_tot, int32_t* __restrict__ expert_offsets,
                                           int32_t* __restrict__ pad_offsets) {
  const int per = (d.E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = threadIdx.x * per;
  int tot[4], s = 0, ps = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    tot[u] = (u < per && e0 + u < d.E) ? expert_total[e0 + u] : 0;
    s += tot[u];
    ps += (tot[u] + 127) / 128 * 128;
  }
  int o = block_exclusive_scan(s, warp_tot);
  int po = block_exclusive_scan(ps, warp_tot);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (u < per && e0 + u < d.E) {
      off[e0 + u] = o;
      poff[e0 + u] = po;
      if (blockIdx.x == 0) {
        expert_offsets[e0 + u] = o;
        pad_offsets[e0 + u] = po;
      }
      o += tot[u];
      po += (tot[u] + 127) / 128 * 128;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == kRouteThreads - 1) {  // past the last expert: the grand totals
    expert_offsets[d.E] = o;
    pad_offsets[d.E] = po;
  }
}

// Stable scatter of one chunk of items: item i = t * k + j of expert e goes to
// position off[e] + (items of e in earlier chunks) + (items of e before it in
// this chunk), warps in order and peers by lane.
__global__ void __launch_bounds__(kRouteThreads) scatter_kernel(RouteDims d, const int32_t* __restrict__ topk_id,
                                                                const int32_t* __restrict__ chunk_base,
                                                                const int32_t* __restrict__ expert_total,
                                                                int32_t* __restrict__ expert_offsets,
                                                                int32_t* __restrict__ pad_offsets,
                                                                int32_t* __restrict__ perm_to_expanded,
                                                                int32_t* __restrict__ expanded_to_perm,
                                                                int32_t* __restrict__ expanded_to_row) {
  extern __shared__ int sm[];
  int* cnt = sm;             // [E] items of each expert seen so far in this chunk
  int* off = sm + d.E;       // [E] expert offsets
  int* poff = sm + 2 * d.E;  // [E] padded expert offsets
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * d.chunk_tokens * d.k;
  const int64_t i1 = min(static_cast<int64_t>(d.T) * d.k, i0 + static_cast<int64_t>(d.chunk_tokens) * d.k);
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) cnt[e] = 0;
  expert_offsets_from_totals(d, expert_total, off, poff, warp_tot, expert_offsets, pad_offsets);
  const int64_t i = i0 + threadIdx.x;
  const int e_in = i < i1 ? topk_id[i] : -1;
  const bool valid = e_in >= 0 && e_in < d.E;  // an expert id out of range is never placed
  const int e = valid ? e_in : -1;
  const unsigned active = __ballot_sync(0xffffffffu, valid);
  unsigned peers = 0;
  if (valid) peers = __match_any_sync(active, e);
  const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
  for (int w = 0; w < kRouteThreads / 32; ++w) {
    __syncthreads();
    if (warp == w && valid) {
      int base = cnt[e];
      __syncwarp(active);
      int leader = __ffs(peers) - 1;
      if (lane == leader) cnt[e] = base + __popc(peers);
      const int within = chunk_base[static_cast<int64_t>(blockIdx.x) * d.E + e] + base + rank_in_warp;
      const int p = off[e] + within;
      perm_to_expanded[p] = static_cast<int32_t>(i);
      expanded_to_perm[i] = p;
      expanded_to_row[i] = poff[e] + within;
    }
  }
}

// The whole routing step in one block when every (token, slot) item fits one
// chunk (T * k <= 256): top-k, expert offsets and the stable scatter, without
// the scan and scatter launches (small decode batches are launch-bound).
// 1024 threads, E <= 1024; dynamic shared memory 2 * E ints.
template <int NV>
__global__ void __launch_bounds__(kTopkThreads) route_one_chunk_kernel(
    const float* __restrict__ logits, RouteDims d, int32_t* __restrict__ topk_id, float* __restrict__ topk_w,
    int32_t* __restrict__ expert_offsets, int32_t* __restrict__ pad_offsets, int32_t* __restrict__ perm_to_expanded,
    int32_t* __restrict__ expanded_to_perm, int32_t* __restrict__ expanded_to_row) {
  extern __shared__ int sm[];
  int* hist = sm;        // [E] items per expert, then each expert's first position
  int* cnt = sm + d.E;   // [E] items of each expert placed so far
  __shared__ int warp_tot[32];
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) { hist[e] = 0; cnt[e] = 0; }
  __syncthreads();
  route_tokens<NV>(logits, d, 0, d.T, topk_id, topk_w, hist);
  __syncthreads();
  // expert offsets and padded (128-row) offsets: thread e holds expert e
  const int e = threadIdx.x;
  const int total = e < d.E ? hist[e] : 0;
  const int off = block_exclusive_scan(total, warp_tot);
  const int padded = e < d.E ? ((total + 127) / 128) * 128 : 0;
  const int poff = block_exclusive_scan(padded, warp_tot);
  if (e < d.E) {
    expert_offsets[e] = off;
    pad_offsets[e] = poff;
    if (e == d.E - 1) {
      expert_offsets[d.E] = off + total;
      pad_offsets[d.E] = poff + padded;
    }
    hist[e] = off;
  }
  __syncthreads();
  // stable scatter: item i = t * k + j, ranked within its expert by i (warps in order, peers by lane)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = d.T * d.k;
  const int i = threadIdx.x;
  const bool valid = i < n;
  const int ex = valid ? topk_id[i] : -1;
  const unsigned active = __ballot_sync(0xffffffffu, valid);
  unsigned peers = 0;
  if (valid) peers = __match_any_sync(active, ex);
  const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
  for (int w = 0; w < kRouteThreads / 32; ++w) {
    __syncthreads();
    if (warp == w && valid) {
      const int base = cnt[ex];
      __syncwarp(active);
      const int leader = __ffs(peers) - 1;
      if (lane == leader) cnt[ex] = base + __popc(peers);
      const int pos = hist[ex] + base + rank_in_warp;
      perm_to_expanded[pos] = i;
      expanded_to_perm[i] = pos;
      expanded_to_row[i] = pad_offsets[ex] + (pos - expert_offsets[ex]);
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_permute_workspace_size(int T, int E, int k) {
  if (T < 1 || E < 1 || k < 1) return 0;
  RouteDims d = route_dims(T, E, k);
  size_t counts = static_cast<size_t>(d.n_chunks) * E * sizeof(int32_t);
  size_t pads = static_cast<size_t>(E + 1) * sizeof(int32_t);  // padded offsets, then each expert's total
  return ((counts + 255) / 256) * 256 + 2 * (((pads + 255) / 256) * 256);
}

namespace moe {
// True when routing T tokens takes one launch (every item fits one chunk).
bool route_one_chunk(int T, int E, int k) { return route_dims(T, E, k).n_chunks == 1; }

// Padded offsets live right after the chunk counts in the routing workspace,
// each expert's total (E ints, 256-byte aligned) right after them.
int32_t* route_pad_offsets(void* ws, int T, int E, int k) {
  RouteDims d = route_dims(T, E, k);
  size_t counts = static_cast<size_t>(d.n_chunks) * E * sizeof(int32_t);
  return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + ((counts + 255) / 256) * 256);
}
}  // namespace moe

namespace moe {
// Routing and permutation from full logits.  Arguments are validated by the
// callers.
moe_status route_permute_enqueue(const float* logits, int T, int E, int k, int32_t* topk_id, float* topk_w,
                                 int32_t* expert_offsets, int32_t* perm_to_expanded, int32_t* expanded_to_perm,
                                 int32_t* expanded_to_row, void* ws, cudaStream_t st) {
  RouteDims d = route_dims(T, E, k);
  int32_t* counts = static_cast<int32_t*>(ws);
  int32_t* pads = route_pad_offsets(ws, T, E, k);
  int32_t* totals = pads + ((static_cast<size_t>(E + 1) * sizeof(int32_t) + 255) / 256) * 256 / sizeof(int32_t);
  const size_t hist_bytes = sizeof(int) * E;
  const int nv = (E + 31) / 32;
  if (d.n_chunks == 1) {
    const size_t one_bytes = 2 * sizeof(int) * E;
#define MOE_ROUTE1(NV)                                                                                           \
  route_one_chunk_kernel<NV><<<1, kTopkThreads, one_bytes, st>>>(logits, d, topk_id, topk_w, expert_offsets, pads, \
                                                                 perm_to_expanded, expanded_to_perm, expanded_to_row)
    if (nv <= 1) MOE_ROUTE1(1);
    else if (nv <= 2) MOE_ROUTE1(2);
    else if (nv <= 4) MOE_ROUTE1(4);
    else if (nv <= 8) MOE_ROUTE1(8);
    else if (nv <= 16) MOE_ROUTE1(16);
    else MOE_ROUTE1(32);
#undef MOE_ROUTE1
    return check_launch();
  }
#define MOE_ROUTE(NV) route_kernel<NV><<<d.n_chunks, kRouteThreads, hist_bytes, st>>>(logits, d, topk_id, topk_w, counts)
  if (nv <= 1) MOE_ROUTE(1);
  else if (nv <= 2) MOE_ROUTE(2);
  else if (nv <= 4) MOE_ROUTE(4);
  else if (nv <= 8) MOE_ROUTE(8);
  else if (nv <= 16) MOE_ROUTE(16);
  else MOE_ROUTE(32);
#undef MOE_ROUTE
  chunk_scan_kernel<<<(E + 31) / 32, 1024, 0, st>>>(d, counts, totals, nullptr, 0, nullptr);
  scatter_kernel<<<d.n_chunks, kRouteThreads, 3 * hist_bytes, st>>>(d, topk_id, counts, totals, expert_offsets, pads,
                                                                    perm_to_expanded, expanded_to_perm,
                                                                    expanded_to_row);
  return check_launch();
}
}  // namespace moe

namespace moe {
// Scan and stable scatter of routing already in topk_id, whose per-chunk expert
// counts (chunks of chunk_tokens tokens, chunk_tokens * k <= 256) are in
// chunk_counts; the router's per-CTA amax words (optional) become x's decode
// multiplier.  pad_offsets and expert_totals: E + 1 and E ints of scratch.
moe_status route_scan_scatter_enqueue(int T, int E, int k, int chunk_tokens, const int32_t* topk_id,
                                      int32_t* chunk_counts, int32_t* pad_offsets, int32_t* expert_totals,
                                      const uint32_t* amax_part, int n_parts, float* x_scale,
                                      int32_t* expert_offsets, int32_t* perm_to_expanded, int32_t* expanded_to_perm,
                                      int32_t* expanded_to_row, cudaStream_t st) {
  if (chunk_tokens < 1 || static_cast<int64_t>(chunk_tokens) * k > kRouteThreads) return MOE_ERR_INVALID_ARG;
  RouteDims d;
  d.T = T;
  d.E = E;
  d.k = k;
  d.chunk_tokens = chunk_tokens;
  d.n_chunks = (T + chunk_tokens - 1) / chunk_tokens;
  chunk_scan_kernel<<<(E + 31) / 32, 1024, 0, st>>>(d, chunk_counts, expert_totals, amax_part, n_parts, x_scale);
  scatter_kernel<<<d.n_chunks, kRouteThreads, 3 * sizeof(int) * E, st>>>(
      d, topk_id, chunk_counts, expert_totals, expert_offsets, pad_offsets, perm_to_expanded, expanded_to_perm,
      expanded_to_row);
  return check_launch();
}
}  // namespace moe

extern "C" moe_status moe_route_permute(const float* logits, int T, int E, int k, int32_t* topk_id, float* topk_w,
                                        int32_t* expert_offsets, int32_t* perm_to_expanded,
                                        int32_t* expanded_to_perm, int32_t* expanded_to_row, void* ws,
                                        size_t ws_bytes, void* stream) {
  if (!logits || !topk_id || !topk_w || !expert_offsets || !perm_to_expanded || !expanded_to_perm ||
      !expanded_to_row)
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * k > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < moe_route_permute_workspace_size(T, E, k)) return MOE_ERR_WORKSPACE;
  return route_permute_enqueue(logits, T, E, k, topk_id, topk_w,
                               expert_offsets, perm_to_expanded, expanded_to_perm, expanded_to_row, ws,
                               static_cast<cudaStream_t>(stream));
}

// small_layer.cu -- the whole MoE layer in ONE launch, for layers so small that
// launch latency, not bandwidth or tensor-core throughput, sets their time
// (a few dozen routed rows: 16 tokens, 8 experts, top-2, H = 256, I = 128).
//
// "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on Blackwell
// SM120", section "Conclusion": persistent kernel designs as the way past
// per-kernel overheads.  The layer computes exactly what moe_forward's staged
// kernels compute (routing and permutation bit for bit, the same NVFP4
// quantisation of x and of the intermediate h, FINALIZE in FP32 rounded once to
// bf16); only the order of the FP32 sums inside the two contractions differs.
//
// Design: ONE thread-block cluster of G CTAs (16, or 8 where a 16-CTA cluster
// cannot be placed); the cluster barrier is the only wait between CTAs.
//   1. Every CTA routes all T tokens itself (T*k <= 64 items: a warp per token,
//      the shared warp top-k; counts and stable ranks by warp match) and takes
//      x's amax itself; CTA 0 publishes the routing, the permutation and the
//      activation multiplier.
//   2. Phase 1: the units (expert e, 32 columns of h) are dealt to the CTAs in
//      contiguous ranges, so a CTA's units are mostly of one expert.  For each
//      expert in its range the CTA quantises the expert's x rows once per pass
//      of eight routed rows (published by the CTA holding the expert's first
//      unit), runs gate_up for up to eight of its units at once (64 weight rows
//      each: 32 gate, 32 up; 8, 4, 2 or 1 lanes per row, each a strided share of
//      K; FP32 sums of exact e2m1 x e4m3 products), then SiLU-mul (a thread per
//      h element) and the NVFP4 requantisation of the units' h columns into the
//      routed-row h buffers.
//   3. Cluster barrier (release / acquire at cluster scope).
//   4. Phase 2: CTA c takes output columns [c H/G, (c+1) H/G) of every token:
//      one thread per (item, column) runs down over the item's quantised h row
//      (codes and block scales, all of a row's loads issued together), scales it
//      by the router weight, and the token's k slots are summed in slot order and
//      rounded to bf16 -- FINALIZE without atomics or a second pass.
// The contractions run on the CUDA cores: at a few dozen rows they are a few
// million multiply-adds, less than the set-up of a tensor-memory pipeline.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kSmallThreads = 512;
constexpr int kSmallMaxItems = 64;  // T * k
constexpr int kSmallMaxE = 64;
constexpr int kSmallMaxH = 1024;
constexpr int kSmallMaxI = 512;
constexpr int kSmallMaxEI = 4096;   // E * I: at most 128 phase-1 units
constexpr int kSmallRows = 8;       // routed rows per gate_up pass
constexpr int kSmallUnitCols = 32;  // h columns per phase-1 unit (64 weight rows)
constexpr int kSmallBatch = 8;      // units at most in one gate_up batch (512 weight rows)
// Decoded x rows in shared memory keep each 32-element chunk 36 floats apart, so
// the lanes of a weight row, reading different chunks at once, hit different banks.
constexpr int kChunkStride = 36;

struct SmallParams {
  const uint16_t* x;
  const float* logits;
  const uint8_t* w13;
  const float* w13_scale;
  const uint8_t* w2;
  const float* w2_scale;
  int T, E, k, H, I;
  float h_scale;
  uint16_t* out;
  int32_t *topk_id, *expert_offsets, *perm_to_expanded, *expanded_to_perm, *expanded_to_row;
  float *topk_w, *x_scale, *h_scale_out;
  uint8_t *x_codes, *x_sf, *h_codes, *h_sf;
};

// Value of an e2m1 code (bit 3 the sign): magnitudes 0, .5, 1, 1.5 for codes
// 0-3 and 2, 3, 4, 6 for codes 4-7.
MOE_DEVINL float e2m1_value(uint32_t c) {
  const uint32_t a = c & 7u;
  const float mag = a < 4u ? 0.5f * static_cast<float>(a) : static_cast<float>((a == 7u) ? 6u : a - 2u);
  return (c & 8u) ? -mag : mag;
}

// The two e2m1 values of a code byte as FP32 (the hardware conversion to
// f16x2, exact; the low nibble holds the even element).
MOE_DEVINL float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 q;\n\tcvt.u8.u32 q, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, q;\n\t}" : "=r"(h2) : "r"(byte));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}

// acc[r] += s_blk * sum_i code_i * v[r][i] for one 16-element block: `lo`, `hi`
// the block's eight code bytes, v the block's first element of row 0 (rows
// `ld` floats apart).  The products of e2m1 values with the decoded activation
// values are exact; the block sum is rounded once per element, then scaled.
MOE_DEVINL void block16_fma(uint32_t lo, uint32_t hi, float s_blk, const float* v, int ld, int R, float (&acc)[8]) {
  float w[16];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 a = e2m1x2_to_f32x2((lo >> (8 * b)) & 0xFFu);
    const float2 c = e2m1x2_to_f32x2((hi >> (8 * b)) & 0xFFu);
    w[2 * b] = a.x;
    w[2 * b + 1] = a.y;
    w[8 + 2 * b] = c.x;
    w[8 + 2 * b + 1] = c.y;
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (r < R) {
      const float4* vr = reinterpret_cast<const float4*>(v + r * ld);
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 xv = vr[i];
        part = __fmaf_rn(w[4 * i], xv.x, part);
        part = __fmaf_rn(w[4 * i + 1], xv.y, part);
        part = __fmaf_rn(w[4 * i + 2], xv.z, part);
        part = __fmaf_rn(w[4 * i + 3], xv.w, part);
      }
      acc[r] = __fmaf_rn(s_blk, part, acc[r]);
    }
  }
}

// Chunk q (K elements 32 q .. 32 q + 31) of row rr of one 128-row block of a
// blocked weight matrix (K tiles of 256 elements, kBlockedTileBytes apart):
// its 16 code bytes (tile q / 8, logical chunk q % 8 stored at (q % 8) ^ (rr % 8))
// and the scale word of its 64-element K-step, whose bytes 2 (q % 2) and
// 2 (q % 2) + 1 are the chunk's two block scales.
struct Chunk {
  uint4 c;
  uint32_t sw;
};

MOE_DEVINL const uint8_t* chunk_tile(const uint8_t* blk, int q) {
  return blk + static_cast<int64_t>(q >> 3) * kBlockedTileBytes;
}

MOE_DEVINL void load_chunk(const uint8_t* blk, int rr, int q, Chunk& t) {
  const uint8_t* tile = chunk_tile(blk, q);
  const int cq = q & 7;
  t.c = __ldg(reinterpret_cast<const uint4*>(tile + rr * 128) + (cq ^ (rr & 7)));
  t.sw = __ldg(reinterpret_cast<const uint32_t*>(tile + 16384 + (cq >> 1) * 512 + (rr & 31) * 16 + (rr >> 5) * 4));
}

MOE_DEVINL void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }

MOE_DEVINL float chunk_scale(const Chunk& t, int q, int b) {
  return e4m3_decode((t.sw >> (16 * (q & 1) + 8 * b)) & 0xFFu);
}

// Block q of decoded rows: acc[r] += s * sum_i code_i * v[r][i] for the two
// 16-element blocks of chunk t (rows `ld` floats apart, the chunk's first
// element at v).
MOE_DEVINL void chunk_fma(const Chunk& t, int q, const float* v, int ld, int R, float (&acc)[kSmallRows]) {
  block16_fma(t.c.x, t.c.y, chunk_scale(t, q, 0), v, ld, R, acc);
  block16_fma(t.c.z, t.c.w, chunk_scale(t, q, 1), v + 16, ld, R, acc);
}

// Eight e2m1 codes (a 32-bit word, element j in bits 4j..4j+3) as four f16x2
// pairs (the hardware conversion, exact; the even element in the low half).
MOE_DEVINL void e2m1x8_to_h2x4(uint32_t w, __half2 (&h)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t h2;
    asm("{\n\t.reg .b8 q;\n\tcvt.u8.u32 q, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, q;\n\t}" : "=r"(h2) : "r"((w >> (8 * j)) & 0xFFu));
    h[j] = *reinterpret_cast<const __half2*>(&h2);
  }
}

// acc + the dot product of chunk t of a weight row with the 32 h elements of
// the same K range: hc their e2m1 codes (element j in bits 4j.. of the byte
// string), hsf the four h block scales of the chunk's 64-element K-step.  Per
// 16-element block: (sum of the e2m1 x e2m1 products) x h scale x weight
// scale.  The products (at most 36 in magnitude, multiples of 1/4) and their
// sums over eight elements (at most 288) are exact in f16, so the block sum is
// taken with packed f16x2 multiply-adds, each half over eight products, and the
// two halves are added in FP32: the exact sum, as an FP32 chain would give it.
MOE_DEVINL float chunk_dot_codes(const Chunk& t, int q, const uint4& hc, uint32_t hsf, float acc) {
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    __half2 w[4], h[4];
    __half2 s2 = __float2half2_rn(0.0f);
#pragma unroll
    for (int half8 = 0; half8 < 2; ++half8) {
      const uint32_t ww = b ? (half8 ? t.c.w : t.c.z) : (half8 ? t.c.y : t.c.x);
      const uint32_t hw = b ? (half8 ? hc.w : hc.z) : (half8 ? hc.y : hc.x);
      e2m1x8_to_h2x4(ww, w);
      e2m1x8_to_h2x4(hw, h);
#pragma unroll
      for (int j = 0; j < 4; ++j) s2 = __hfma2(w[j], h[j], s2);
    }
    const float part = __fadd_rn(__low2float(s2), __high2float(s2));
    const float hs = e4m3_decode((hsf >> (16 * (q & 1) + 8 * b)) & 0xFFu);
    acc = __fmaf_rn(__fmul_rn(hs, chunk_scale(t, q, b)), part, acc);
  }
  return acc;
}

// Blocked weight row of h column i's gate row in a gate_up matrix (gate and up
// rows interleaved per 64 inside each 128-row block); the up row is 64 further.
MOE_DEVINL int gate_row(int i) { return (i >> 6) * 128 + (i & 63); }

MOE_DEVINL uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

MOE_DEVINL uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Lanes per weight row in a gate_up batch of nb units: the largest power of two
// with 64 nb rows x lanes <= the block.
MOE_DEVINL int batch_lanes(int nb) { return nb <= 1 ? 8 : nb == 2 ? 4 : nb <= 4 ? 2 : 1; }

__global__ void __launch_bounds__(kSmallThreads, 1) small_layer_kernel(const SmallParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, E = p.E, k = p.k, H = p.H, I = p.I;
  const int n_items = T * k;
  const int c = static_cast<int>(cluster_ctarank()), G = static_cast<int>(cluster_nctarank());
  const int Hc = H / G;                       // phase-2 output columns of this CTA
  const int units_e = I / kSmallUnitCols;     // phase-1 units per expert
  const int n_units = E * units_e;
  const int ua = c * n_units / G, ub = (c + 1) * n_units / G;  // this CTA's phase-1 units
  const int mt13 = 2 * I / 128, mt2 = H / 128;  // 128-row blocks per expert
  const int kt13 = (H + 255) / 256, kt2 = (I + 255) / 256;
  const int Hs = H / 32 * kChunkStride;       // floats per decoded x row
  // shared memory: x as loaded (bf16 [T][H]; phase 2 reuses the bytes for its results [T*k][Hc]),
  // decoded x rows [8][Hs], gate_up sums [8][512], h values [8][256], then small tables
  const size_t region_a = max(static_cast<size_t>(T) * H * 2, static_cast<size_t>(n_items) * Hc * 4);
  uint16_t* s_xin = reinterpret_cast<uint16_t*>(smem);
  float* s_y = reinterpret_cast<float*>(smem);
  float* s_x = reinterpret_cast<float*>(smem + (region_a + 15) / 16 * 16);
  float* s_pre = s_x + kSmallRows * Hs;
  float* s_hv = s_pre + kSmallRows * 2 * kSmallUnitCols * kSmallBatch;
  int* s_id = reinterpret_cast<int*>(s_hv + kSmallRows * kSmallUnitCols * kSmallBatch);  // [64] expert of each item
  float* s_w = reinterpret_cast<float*>(s_id + kSmallMaxItems);  // [64] router weight of each item
  int* s_perm = reinterpret_cast<int*>(s_w + kSmallMaxItems);    // [64] items in permuted order
  int* s_row = s_perm + kSmallMaxItems;                           // [64] routed row of each item
  int* s_cnt = s_row + kSmallMaxItems;                            // [64] items per expert
  int* s_cnt0 = s_cnt + kSmallMaxE;                               // [64] ... among items 0-31
  int* s_off = s_cnt0 + kSmallMaxE;                               // [65] expert offsets
  int* s_pad = s_off + kSmallMaxE + 1;                            // [65] padded offsets
  float* s_red = reinterpret_cast<float*>(s_pad + kSmallMaxE + 1);  // [16] warp maxima

  // weight row `wr` (0..64 nb - 1) of a batch starting at unit u0: gate rows 0-31, up rows 32-63 of
  // each unit
  auto batch_row = [&](int u0, int wr, int& rr, const uint8_t*& blk) {
    const int u = u0 + (wr >> 6), e = u / units_e;
    const int i = (u - e * units_e) * kSmallUnitCols + (wr & 31);
    const int jr = gate_row(i) + ((wr & 63) >= 32 ? 64 : 0);
    rr = jr & 127;
    blk = p.w13 + (static_cast<int64_t>(e) * mt13 + (jr >> 7)) * kt13 * kBlockedTileBytes;
  };
  // the first batch of this CTA: units [ua, end of ua's expert or ub), at most kSmallBatch of them
  const int nb0 = min(kSmallBatch, min(ub, (ua / units_e + 1) * units_e) - ua);
  const int L0 = batch_lanes(nb0);

  // ---- 0. inputs requested at once: x into shared memory; this thread's first two gate_up chunks of
  // its first batch into registers (the units' experts are known before routing); the lines of the rest
  // of this CTA's gate_up rows, and of its down rows of every expert, into L2
  {
    const int n16 = T * H / 8;  // 16-byte pieces of x
    for (int i = tid; i < n16; i += kSmallThreads)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(s_xin + 8 * i)), "l"(p.x + 8 * i)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  Chunk first[2] = {};
  if (nb0 > 0 && tid / L0 < 64 * nb0) {
    int rr;
    const uint8_t* blk;
    batch_row(ua, tid / L0, rr, blk);
#pragma unroll
    for (int f = 0; f < 2; ++f)
      if (tid % L0 + f * L0 < H / 32) load_chunk(blk, rr, tid % L0 + f * L0, first[f]);
  }
  for (int q = tid; q < (ub - ua) * 64 * kt13; q += kSmallThreads) {  // (weight row, K tile): its 128-byte row
    const int wr = q / kt13, kt = q - wr * kt13;
    int rr;
    const uint8_t* blk;
    batch_row(ua, wr, rr, blk);
    prefetch_l2(blk + static_cast<int64_t>(kt) * kBlockedTileBytes + rr * 128);
    if ((rr & 7) == 0)  // the scale words of eight rows share a line per K-step
      for (int st = 0; st < 4; ++st)
        prefetch_l2(blk + static_cast<int64_t>(kt) * kBlockedTileBytes + 16384 + st * 512 + (rr & 31) * 16);
  }
  for (int q = tid; q < E * Hc * kt2; q += kSmallThreads) {
    const int row = q / kt2, kt = q - row * kt2;
    const int e = row / Hc, n = c * Hc + (row - e * Hc);
    const uint8_t* tile = p.w2 + ((static_cast<int64_t>(e) * mt2 + (n >> 7)) * kt2 + kt) * kBlockedTileBytes;
    prefetch_l2(tile + (n & 127) * 128);
    if ((n & 7) == 0)
      for (int st = 0; st < 4; ++st) prefetch_l2(tile + 16384 + st * 512 + (n & 31) * 16);
  }

  // ---- 1. routing of every token (a warp per token), the same selection rule as moe_route_permute
  if (tid < kSmallMaxE) {
    s_cnt[tid] = 0;
    s_cnt0[tid] = 0;
  }
  for (int t = warp; t < T; t += kSmallThreads / 32) {
    float v[2];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int ex = lane + 32 * i;
      v[i] = ex < E ? __ldg(p.logits + static_cast<int64_t>(t) * E + ex) : 0.0f;
      if (ex >= E) taken |= 1u << i;
    }
    int id;
    float w;
    warp_topk_softmax<2>(v, taken, k, &id, &w);
    if (lane < k) {
      s_id[t * k + lane] = id;
      s_w[t * k + lane] = w;
      if (c == 0) {
        p.topk_id[t * k + lane] = id;
        p.topk_w[t * k + lane] = w;
      }
    }
  }
  __syncthreads();
  // items per expert and each item's rank among the earlier items of its expert (warps 0 and 1 hold
  // items 0-31 and 32-63; the leader of each group of equal experts adds the group)
  int my_ex = -1, my_rank = 0;
  if (warp < 2) {
    const bool valid = tid < n_items;
    my_ex = valid ? s_id[tid] : -1;
    const unsigned active = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const unsigned peers = __match_any_sync(active, my_ex);
      my_rank = __popc(peers & lanemask_lt());
      if ((peers & lanemask_lt()) == 0) {
        atomicAdd(&s_cnt[my_ex], __popc(peers));
        if (warp == 0) s_cnt0[my_ex] = __popc(peers);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // expert offsets and padded offsets: an exclusive scan over at most 64 experts, two per lane
    const int c0 = 2 * lane < E ? s_cnt[2 * lane] : 0, c1 = 2 * lane + 1 < E ? s_cnt[2 * lane + 1] : 0;
    const int p0 = (c0 + 127) / 128 * 128, p1 = (c1 + 127) / 128 * 128;
    int a = c0 + c1, b = p0 + p1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) { a += ya; b += yb; }
    }
    const int ea = a - c0 - c1, eb = b - p0 - p1;  // exclusive prefixes
    if (2 * lane < E) { s_off[2 * lane] = ea; s_pad[2 * lane] = eb; }
    if (2 * lane + 1 < E) { s_off[2 * lane + 1] = ea + c0; s_pad[2 * lane + 1] = eb + p0; }
    if (lane == 31) { s_off[E] = a; s_pad[E] = b; }  // the totals (the last lane's inclusive prefixes)
  }
  __syncthreads();
  if (tid < n_items) {
    const int rank = my_rank + (warp == 1 ? s_cnt0[my_ex] : 0);
    const int pos = s_off[my_ex] + rank;
    s_perm[pos] = tid;
    s_row[tid] = s_pad[my_ex] + rank;
    if (c == 0) {
      p.perm_to_expanded[pos] = tid;
      p.expanded_to_perm[tid] = pos;
      p.expanded_to_row[tid] = s_pad[my_ex] + rank;
    }
  }
  if (c == 0 && tid <= E) p.expert_offsets[tid] = s_off[tid];

  // ---- 2. x's decode multiplier: s = amax / (6 * 448), 1 when x is all zero
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  float amax = 0.0f;
  for (int i = tid; i < T * H / 8; i += kSmallThreads) {
    const uint4 q = reinterpret_cast<const uint4*>(s_xin)[i];
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_float(static_cast<uint16_t>(wv[j] & 0xFFFFu))));
      amax = fmaxf(amax, fabsf(bf16_bits_to_float(static_cast<uint16_t>(wv[j] >> 16))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_red[warp] = amax;
  __syncthreads();
  amax = 0.0f;
  for (int w = 0; w < kSmallThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
  const float xs = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  if (c == 0 && tid == 0) {
    *p.x_scale = xs;
    *p.h_scale_out = p.h_scale;
  }

  // ---- 3. phase 1: this CTA's units expert by expert, eight routed rows at a time
  for (int e = ua / units_e; ua < ub && e <= (ub - 1) / units_e; ++e) {
    const int sa = max(ua, e * units_e), sb = min(ub, (e + 1) * units_e);  // the expert's units here
    const int m_e = s_cnt[e];
    if (m_e == 0) continue;  // the same for the whole CTA
    const float alpha1 = __fmul_rn(xs, __ldg(p.w13_scale + e));
    for (int r0 = 0; r0 < m_e; r0 += kSmallRows) {
      const int R = min(kSmallRows, m_e - r0);
      __syncthreads();  // the previous pass is done with the shared rows
      // 3a. quantise x rows into decoded values (and, from the CTA holding the expert's first unit,
      // into the routed-row buffers, as the quantiser would)
      for (int q = tid; q < R * (H / 16); q += kSmallThreads) {
        const int r = q / (H / 16), cb = q - r * (H / 16);
        const int item = s_perm[s_off[e] + r0 + r];
        const int t = item / k;
        const int64_t dst = s_pad[e] + r0 + r;
        float v[16];
        const uint4* src = reinterpret_cast<const uint4*>(s_xin + static_cast<int64_t>(t) * H + 16 * cb);
        const uint4 q0 = src[0], q1 = src[1];
        const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        float bm = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[2 * j] = bf16_bits_to_float(static_cast<uint16_t>(wv[j] & 0xFFFFu));
          v[2 * j + 1] = bf16_bits_to_float(static_cast<uint16_t>(wv[j] >> 16));
          bm = fmaxf(bm, fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
        }
        float recip;
        const uint32_t sfb = nvfp4_block_scale(bm, xs, &recip);
        const uint32_t lo = nvfp4_codes8(v, recip), hi = nvfp4_codes8(v + 8, recip);
        if (sa == e * units_e) {
          *reinterpret_cast<uint2*>(p.x_codes + dst * (H / 2) + 8 * cb) = make_uint2(lo, hi);
          p.x_sf[tiled_sf_offset(dst, cb, H)] = static_cast<uint8_t>(sfb);
        }
        const float sd = e4m3_decode(sfb);
        float* xr = s_x + r * Hs + (cb >> 1) * kChunkStride + 16 * (cb & 1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          xr[j] = __fmul_rn(e2m1_value((lo >> (4 * j)) & 15u), sd);
          xr[8 + j] = __fmul_rn(e2m1_value((hi >> (4 * j)) & 15u), sd);
        }
      }
      for (int s0 = sa; s0 < sb; s0 += kSmallBatch) {
        const int nb = min(kSmallBatch, sb - s0), L = batch_lanes(nb);
        const int wr = tid / L, kp = tid % L;
        __syncthreads();  // decoded rows written; the previous batch is done with the sums
        // 3b. gate_up: weight row wr of the batch by the L lanes L (tid / L) .. + L - 1, lane kp taking
        // chunks kp, kp + L, ...
        float acc[kSmallRows];
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) acc[r] = 0.0f;
        if (wr < 64 * nb) {
          int rr;
          const uint8_t* blk;
          batch_row(s0, wr, rr, blk);
          for (int q = kp; q < H / 32; q += L) {
            Chunk t;
            if (s0 == ua && r0 == 0 && q == kp) t = first[0];
            else if (s0 == ua && r0 == 0 && q == kp + L) t = first[1];
            else load_chunk(blk, rr, q, t);
            chunk_fma(t, q, s_x + q * kChunkStride, Hs, R, acc);
          }
        }
        for (int o = 1; o < L; o <<= 1) {
#pragma unroll
          for (int r = 0; r < kSmallRows; ++r) acc[r] = __fadd_rn(acc[r], __shfl_xor_sync(0xffffffffu, acc[r], o));
        }
        if (wr < 64 * nb && kp == 0) {
#pragma unroll
          for (int r = 0; r < kSmallRows; ++r)
            if (r < R) s_pre[r * 512 + wr] = acc[r];
        }
        __syncthreads();
        // 3c. h = SiLU(gate) * up, a thread per element of the batch's 32 nb columns of each row
        const int nh = 32 * nb;
        for (int q = tid; q < R * nh; q += kSmallThreads) {
          const int r = q / nh, j = q - r * nh;  // column j of the batch: unit j / 32, column j % 32
          const float* pre = s_pre + r * 512 + 64 * (j >> 5) + (j & 31);
          s_hv[r * 256 + j] = silu_mul(__fmul_rn(alpha1, pre[0]), __fmul_rn(alpha1, pre[32]));
        }
        __syncthreads();
        // ... requantised with the static multiplier, a thread per 16-column block
        for (int q = tid; q < R * 2 * nb; q += kSmallThreads) {
          const int r = q / (2 * nb), b = q - r * (2 * nb);
          const int64_t dst = s_pad[e] + r0 + r;
          const float* h = s_hv + r * 256 + 16 * b;
          float bm = 0.0f;
#pragma unroll
          for (int t = 0; t < 16; ++t) bm = fmaxf(bm, fabsf(h[t]));
          float recip;
          const uint32_t sfb = nvfp4_block_scale(bm, p.h_scale, &recip);
          const uint32_t lo = nvfp4_codes8(h, recip), hi = nvfp4_codes8(h + 8, recip);
          const int ib = (s0 - e * units_e) * kSmallUnitCols + 16 * b;  // h column of the block
          *reinterpret_cast<uint2*>(p.h_codes + dst * (I / 2) + ib / 2) = make_uint2(lo, hi);
          p.h_sf[tiled_sf_offset(dst, ib / 16, I)] = static_cast<uint8_t>(sfb);
        }
      }
    }
  }

  // ---- 4. every item's quantised h is written: the cluster barrier publishes it to every CTA.  Between
  // its arrive and its wait each thread requests the first four K chunks of its first down row (they do
  // not depend on phase 1), so only the h loads follow the barrier.
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  Chunk w2first[4];
  float w2s_first = 0.0f;
  if (tid < n_items * Hc) {
    const int item = tid / Hc, n = c * Hc + (tid - (tid / Hc) * Hc);
    const uint8_t* blk =
        p.w2 + (static_cast<int64_t>(s_id[item]) * mt2 + (n >> 7)) * kt2 * kBlockedTileBytes;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < I / 32) load_chunk(blk, n & 127, j, w2first[j]);
    w2s_first = __ldg(p.w2_scale + s_id[item]);
  }
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");

  // ---- 5. phase 2: down + FINALIZE for output columns [c Hc, c Hc + Hc): one thread per (item, column),
  // four K chunks of the weight row and of the item's h row requested together
  for (int q = tid; q < n_items * Hc; q += kSmallThreads) {
    const int item = q / Hc, col = q - item * Hc;
    const int n = c * Hc + col;
    const int e = s_id[item];
    const uint8_t* blk = p.w2 + (static_cast<int64_t>(e) * mt2 + (n >> 7)) * kt2 * kBlockedTileBytes;
    const int64_t hrow = s_row[item];
    const uint4* hcodes = reinterpret_cast<const uint4*>(p.h_codes + hrow * (I / 2));
    float acc = 0.0f;
    for (int q0 = 0; q0 < I / 32; q0 += 4) {
      Chunk t[4];
      uint4 hc[4];
      uint32_t hsf[2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (q0 + j < I / 32) {
          if (q == tid && q0 == 0) t[j] = w2first[j];
          else load_chunk(blk, n & 127, q0 + j, t[j]);
          hc[j] = __ldcg(hcodes + q0 + j);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)  // the K-steps of the four chunks: four h scales each
        if (q0 + 2 * j < I / 32)
          hsf[j] = __ldcg(reinterpret_cast<const unsigned int*>(p.h_sf + tiled_sf_offset(hrow, 2 * (q0 + 2 * j), I)));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (q0 + j < I / 32) acc = chunk_dot_codes(t[j], q0 + j, hc[j], hsf[j >> 1], acc);
    }
    const float alpha2 = __fmul_rn(p.h_scale, q == tid ? w2s_first : __ldg(p.w2_scale + e));
    s_y[q] = __fmul_rn(__fmul_rn(s_w[item], alpha2), acc);
  }
  __syncthreads();
  // each token's k weighted rows summed in slot order, rounded once to bf16
  for (int q = tid; q < T * Hc; q += kSmallThreads) {
    const int t = q / Hc, col = q - t * Hc;
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, s_y[(t * k + j) * Hc + col]);
    p.out[static_cast<int64_t>(t) * H + c * Hc + col] = float_to_bf16_bits(sum);
  }
}

size_t small_smem_bytes(int T, int k, int H, int G) {
  const size_t region_a = std::max(static_cast<size_t>(T) * H * 2, static_cast<size_t>(T) * k * (H / G) * 4);
  return (region_a + 15) / 16 * 16 +
         (static_cast<size_t>(kSmallRows) * (H / 32 * kChunkStride) +
          static_cast<size_t>(kSmallRows) * kSmallBatch * 3 * kSmallUnitCols) *
             sizeof(float) +
         (4 * kSmallMaxItems + 2 * kSmallMaxE + 2 * (kSmallMaxE + 1)) * sizeof(int) +
         (kSmallThreads / 32) * sizeof(float) + 16;
}

// Cluster size for this device and layer: 16 CTAs where such a cluster can be
// placed, else 8 (portable); 0 if neither can.
int small_cluster_size(int T, int k, int H) {
  static int cached[64][2] = {};  // per device: [placeable 16, placeable 8] as 1/2 (0 = not looked up)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  for (int i = 0; i < 2; ++i) {
    const int G = i == 0 ? 16 : 8;
    const size_t smem = small_smem_bytes(T, k, H, G);
    if (cached[dev][i] == 0) {
      int n = 0;
      if (i == 0 && cudaFuncSetAttribute(small_layer_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                        cudaSuccess)
        n = 0;
      else if (cudaFuncSetAttribute(small_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem)) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(G, 1, 1);
        cfg.blockDim = dim3(kSmallThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = G;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, small_layer_kernel, &cfg) != cudaSuccess) n = 0;
      }
      cudaGetLastError();  // a refused query leaves no sticky error
      // the largest layer's shared memory decides, so the answer holds for every eligible shape
      cached[dev][i] = n > 0 ? 1 : 2;
    }
    if (cached[dev][i] == 1) return G;
  }
  return 0;
}

}  // namespace

// Shapes the single-launch layer takes.
bool small_layer_eligible(int T, int E, int k, int H, int I) {
  return static_cast<int64_t>(T) * k <= kSmallMaxItems && E <= kSmallMaxE && H <= kSmallMaxH && I <= kSmallMaxI &&
         E * I <= kSmallMaxEI && H % 128 == 0 && I % 64 == 0 && k <= 32;
}

// Scratch of the single-launch layer inside the moe_forward workspace: 256
// bytes reserved (every intermediate lives in the layout's own buffers).
size_t small_layer_scratch_bytes(int T, int k, int I) {
  (void)T;
  (void)k;
  (void)I;
  return 256;
}

moe_status small_layer_enqueue(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k,
                               int H, int I, float h_scale, uint16_t* out, int32_t* topk_id, float* topk_w,
                               int32_t* offs, int32_t* p2e, int32_t* e2p, int32_t* e2r, float* x_scale,
                               uint8_t* x_codes, uint8_t* x_sf, float* hs, uint8_t* h_codes, uint8_t* h_sf,
                               void* scratch, cudaStream_t st) {
  SmallParams p{};
  p.x = x;
  p.logits = logits;
  p.w13 = w->w13;
  p.w13_scale = w->w13_scale;
  p.w2 = w->w2;
  p.w2_scale = w->w2_scale;
  p.T = T;
  p.E = E;
  p.k = k;
  p.H = H;
  p.I = I;
  p.h_scale = h_scale;
  p.out = out;
  p.topk_id = topk_id;
  p.topk_w = topk_w;
  p.expert_offsets = offs;
  p.perm_to_expanded = p2e;
  p.expanded_to_perm = e2p;
  p.expanded_to_row = e2r;
  p.x_scale = x_scale;
  p.h_scale_out = hs;
  p.x_codes = x_codes;
  p.x_sf = x_sf;
  p.h_codes = h_codes;
  p.h_sf = h_sf;
  (void)scratch;
  const int G = small_cluster_size(kSmallMaxItems, 1, kSmallMaxH);
  if (G == 0) return MOE_ERR_RESOURCE;
  const size_t smem = small_smem_bytes(T, k, H, G);
  if (cudaFuncSetAttribute(small_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_RESOURCE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(kSmallThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = G;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, small_layer_kernel, p) != cudaSuccess) return MOE_ERR_CUDA;
  return check_launch();
}

}  // namespace moe

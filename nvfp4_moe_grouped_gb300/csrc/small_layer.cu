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
// Design: one CTA per expert, no CTA ever waits on another.
//   1. Every CTA routes all T tokens itself (T*k <= 64 items: a warp per token,
//      the shared warp top-k) and derives the expert offsets and the stable
//      permutation from the item list in shared memory; CTA 0 publishes them.
//   2. Every CTA takes x's amax itself (T*H elements) and so knows the
//      activation multiplier; CTA 0 publishes it.
//   3. CTA e quantises the rows routed to expert e (into the routed-row
//      buffers, as the quantiser would), keeps their decoded values in shared
//      memory, and runs gate_up (a thread per blocked weight row, FP32 sums of
//      exact e2m1 x e4m3 products), SiLU-mul + requantisation of h, and down (a
//      thread per output column), eight routed rows at a time.  Each routed
//      row's output times its router weight goes to a per-item FP32 scratch row.
//   4. The last CTA to finish (a ticket taken after a memory fence) sums each
//      token's k scratch rows in slot order, rounds to bf16, and resets the
//      ticket for the next launch.
// The contractions run on the CUDA cores: at a few dozen rows they are a few
// million multiply-adds, less than the set-up of a tensor-memory pipeline.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kSmallThreads = 512;
constexpr int kSmallMaxItems = 64;  // T * k
constexpr int kSmallMaxE = 64;
constexpr int kSmallMaxH = 1024;
constexpr int kSmallMaxI = 512;
constexpr int kSmallRows = 8;       // routed rows per pass

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
  float* yw;              // [T * k][H] router-weighted expert rows, expanded order
  unsigned int* ticket;   // 0 between launches
};

// Value of an e2m1 code (bit 3 the sign): magnitudes 0, .5, 1, 1.5 for codes
// 0-3 and 2, 3, 4, 6 for codes 4-7.
MOE_DEVINL float e2m1_value(uint32_t c) {
  const uint32_t a = c & 7u;
  const float mag = a < 4u ? 0.5f * static_cast<float>(a) : static_cast<float>((a == 7u) ? 6u : a - 2u);
  return (c & 8u) ? -mag : mag;
}

// Half of row `rr` of one blocked weight tile: logical 32-element chunks
// [4 * half, 4 * half + 4) of its eight (stored swizzled: logical chunk c at
// chunk c ^ (rr % 8)) and the two scale words (K-steps 2 * half, 2 * half + 1),
// requested together so the half row costs one memory latency.
struct HalfRow {
  uint4 q[4];
  uint32_t sf[2];
};

MOE_DEVINL void load_half_row(const uint8_t* tile, int rr, int half, HalfRow& t) {
  const uint4* row = reinterpret_cast<const uint4*>(tile + rr * 128);
#pragma unroll
  for (int c = 0; c < 4; ++c) t.q[c] = __ldg(row + ((4 * half + c) ^ (rr & 7)));
#pragma unroll
  for (int g = 0; g < 2; ++g)
    t.sf[g] = __ldg(
        reinterpret_cast<const uint32_t*>(tile + 16384 + (2 * half + g) * 512 + (rr & 31) * 16 + (rr >> 5) * 4));
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

// acc[r] += (half row) . v[r] over the elements the half row holds below K
// (kk0: the tile's first K-element).
MOE_DEVINL void half_row_fma(const HalfRow& t, int half, int kk0, int K, const float* v, int ld, int R,
                             float (&acc)[8]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int k0 = kk0 + 32 * (4 * half + c);
    if (k0 >= K) break;
    const uint4 q = t.q[c];
    const uint32_t sfw = t.sf[c >> 1];  // the K-step (64 elements) of this chunk: four scale bytes
    const float s0 = e4m3_decode((sfw >> (16 * (c & 1))) & 0xFFu);
    const float s1 = e4m3_decode((sfw >> (16 * (c & 1) + 8)) & 0xFFu);
    block16_fma(q.x, q.y, s0, v + k0, ld, R, acc);
    block16_fma(q.z, q.w, s1, v + k0 + 16, ld, R, acc);
  }
}

// One weight row's half (`half` of every 256-element tile) against R rows of
// v: the first tile's half row may already be loaded.  The two halves of a row
// are lanes l and l ^ 16 of one warp; the caller adds them.
MOE_DEVINL void dot_half(const uint8_t* w, int64_t blk, int kt_count, int rr, int half, int K, const float* v, int ld,
                         int R, const HalfRow& first, float (&acc)[8]) {
  half_row_fma(first, half, 0, K, v, ld, R, acc);
  for (int kt = 1; kt < kt_count; ++kt) {
    HalfRow t;
    load_half_row(w + (blk * kt_count + kt) * kBlockedTileBytes, rr, half, t);
    half_row_fma(t, half, kt * 256, K, v, ld, R, acc);
  }
}

__global__ void __launch_bounds__(kSmallThreads, 1) small_layer_kernel(const SmallParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, E = p.E, k = p.k, H = p.H, I = p.I;
  const int n_items = T * k;
  const int e = blockIdx.x;
  // shared memory: x as loaded (bf16 [T][H]), decoded x rows [8][H], gate_up sums [8][2I], decoded h
  // [8][I], then small tables
  uint16_t* s_xin = reinterpret_cast<uint16_t*>(smem);
  float* s_x = reinterpret_cast<float*>(smem + static_cast<size_t>(T) * H * 2);
  float* s_pre = s_x + kSmallRows * H;
  float* s_h = s_pre + kSmallRows * 2 * I;
  int* s_id = reinterpret_cast<int*>(s_h + kSmallRows * I);  // [64] expert of each item
  float* s_w = reinterpret_cast<float*>(s_id + kSmallMaxItems);  // [64] router weight of each item
  int* s_items = reinterpret_cast<int*>(s_w + kSmallMaxItems);   // [64] this expert's items in order
  int* s_cnt = s_items + kSmallMaxItems;                          // [64] items per expert
  int* s_off = s_cnt + kSmallMaxE;                                // [65] expert offsets
  int* s_pad = s_off + kSmallMaxE + 1;                            // [65] padded offsets
  float* s_red = reinterpret_cast<float*>(s_pad + kSmallMaxE + 1);  // [16] warp maxima
  int* s_last = reinterpret_cast<int*>(s_red + kSmallThreads / 32);

  // ---- 0. every input this CTA reads from memory, requested at once: x into shared memory, the
  // first half rows of this thread's gate_up and down weight rows into registers, this warp's first
  // token's logits; one memory latency instead of one per phase
  const int mt13 = 2 * I / 128, mt2 = H / 128;  // 128-row blocks per expert
  const int kt13 = (H + 255) / 256, kt2 = (I + 255) / 256;
  const int half = (lane >> 4) & 1;                          // the K half of this thread's weight row
  const int rsub = warp * 16 + (lane & 15);                  // this thread's row within a pass of 256 rows
  {
    const int n16 = T * H / 8;  // 16-byte pieces of x
    for (int i = tid; i < n16; i += kSmallThreads)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(s_xin + 8 * i)), "l"(p.x + 8 * i)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  HalfRow w13_first, w2_first;
  if (rsub < 2 * I)
    load_half_row(p.w13 + (static_cast<int64_t>(e) * mt13 + (rsub >> 7)) * kt13 * kBlockedTileBytes, rsub & 127,
                  half, w13_first);
  if (rsub < H)
    load_half_row(p.w2 + (static_cast<int64_t>(e) * mt2 + (rsub >> 7)) * kt2 * kBlockedTileBytes, rsub & 127, half,
                  w2_first);

  // ---- 1. routing of every token (a warp per token), the same selection rule as moe_route_permute
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
      if (e == 0) {
        p.topk_id[t * k + lane] = id;
        p.topk_w[t * k + lane] = w;
      }
    }
  }
  __syncthreads();
  if (tid < E) {
    int c = 0;
    for (int i = 0; i < n_items; ++i) c += s_id[i] == tid;
    s_cnt[tid] = c;
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
  // stable rank of every item within its expert (items in expanded order)
  if (tid < n_items) {
    const int ex = s_id[tid];
    int rank = 0;
    for (int i = 0; i < tid; ++i) rank += s_id[i] == ex;
    if (ex == e) s_items[rank] = tid;
    if (e == 0) {
      const int pos = s_off[ex] + rank;
      p.perm_to_expanded[pos] = tid;
      p.expanded_to_perm[tid] = pos;
      p.expanded_to_row[tid] = s_pad[ex] + rank;
    }
  }
  if (e == 0 && tid <= E) p.expert_offsets[tid] = s_off[tid];

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
  if (e == 0 && tid == 0) {
    *p.x_scale = xs;
    *p.h_scale_out = p.h_scale;
  }

  // ---- 3. this expert's rows, eight at a time
  const int m_e = s_cnt[e];
  const float alpha1 = __fmul_rn(xs, __ldg(p.w13_scale + e));
  const float alpha2 = __fmul_rn(p.h_scale, __ldg(p.w2_scale + e));
  for (int r0 = 0; r0 < m_e; r0 += kSmallRows) {
    const int R = min(kSmallRows, m_e - r0);
    __syncthreads();  // the previous pass is done with the shared rows
    // 3a. quantise x rows into the routed-row buffers and keep their decoded values
    for (int q = tid; q < R * (H / 16); q += kSmallThreads) {
      const int r = q / (H / 16), c = q - r * (H / 16);
      const int item = s_items[r0 + r];
      const int t = item / k;
      const int64_t dst = s_pad[e] + r0 + r;
      float v[16];
      const uint4* src = reinterpret_cast<const uint4*>(s_xin + static_cast<int64_t>(t) * H + 16 * c);
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
      *reinterpret_cast<uint2*>(p.x_codes + dst * (H / 2) + 8 * c) = make_uint2(lo, hi);
      p.x_sf[tiled_sf_offset(dst, c, H)] = static_cast<uint8_t>(sfb);
      const float sd = e4m3_decode(sfb);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s_x[r * H + 16 * c + j] = __fmul_rn(e2m1_value((lo >> (4 * j)) & 15u), sd);
        s_x[r * H + 16 * c + 8 + j] = __fmul_rn(e2m1_value((hi >> (4 * j)) & 15u), sd);
      }
    }
    __syncthreads();
    // 3b. gate_up: each blocked weight row (of 2I, gate/up interleaved per 64) by two lanes, one K half each
    for (int j = rsub; j - rsub < 2 * I; j += 16 * (kSmallThreads / 32)) {
      float acc[kSmallRows];
#pragma unroll
      for (int r = 0; r < kSmallRows; ++r) acc[r] = 0.0f;
      if (j < 2 * I) {
        HalfRow t0;
        if (j == rsub) t0 = w13_first;
        else load_half_row(p.w13 + (static_cast<int64_t>(e) * mt13 + (j >> 7)) * kt13 * kBlockedTileBytes, j & 127,
                           half, t0);
        dot_half(p.w13, static_cast<int64_t>(e) * mt13 + (j >> 7), kt13, j & 127, half, H, s_x, H, R, t0, acc);
      }
#pragma unroll
      for (int r = 0; r < kSmallRows; ++r) acc[r] = __fadd_rn(acc[r], __shfl_xor_sync(0xffffffffu, acc[r], 16));
      if (j < 2 * I && half == 0) {
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r)
          if (r < R) s_pre[r * 2 * I + j] = acc[r];
      }
    }
    __syncthreads();
    // 3c. h = SiLU(gate) * up, requantised with the static multiplier; decoded h kept for down
    for (int q = tid; q < R * (I / 16); q += kSmallThreads) {
      const int r = q / (I / 16), b = q - r * (I / 16);
      const int64_t dst = s_pad[e] + r0 + r;
      float h[16];
      float bm = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int i = 16 * b + t;
        const int jg = (i >> 6) * 128 + (i & 63);  // gate row; the matching up row is 64 further
        const float g = __fmul_rn(alpha1, s_pre[r * 2 * I + jg]);
        const float u = __fmul_rn(alpha1, s_pre[r * 2 * I + jg + 64]);
        h[t] = silu_mul(g, u);
        bm = fmaxf(bm, fabsf(h[t]));
      }
      float recip;
      const uint32_t sfb = nvfp4_block_scale(bm, p.h_scale, &recip);
      const uint32_t lo = nvfp4_codes8(h, recip), hi = nvfp4_codes8(h + 8, recip);
      *reinterpret_cast<uint2*>(p.h_codes + dst * (I / 2) + 8 * b) = make_uint2(lo, hi);
      p.h_sf[tiled_sf_offset(dst, b, I)] = static_cast<uint8_t>(sfb);
      const float sd = e4m3_decode(sfb);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s_h[r * I + 16 * b + j] = __fmul_rn(e2m1_value((lo >> (4 * j)) & 15u), sd);
        s_h[r * I + 16 * b + 8 + j] = __fmul_rn(e2m1_value((hi >> (4 * j)) & 15u), sd);
      }
    }
    __syncthreads();
    // 3d. down: each output column by two lanes (one K half each); each routed row's result times its
    // router weight
    for (int n = rsub; n - rsub < H; n += 16 * (kSmallThreads / 32)) {
      float acc[kSmallRows];
#pragma unroll
      for (int r = 0; r < kSmallRows; ++r) acc[r] = 0.0f;
      if (n < H) {
        HalfRow t0;
        if (n == rsub) t0 = w2_first;
        else load_half_row(p.w2 + (static_cast<int64_t>(e) * mt2 + (n >> 7)) * kt2 * kBlockedTileBytes, n & 127,
                           half, t0);
        dot_half(p.w2, static_cast<int64_t>(e) * mt2 + (n >> 7), kt2, n & 127, half, I, s_h, I, R, t0, acc);
      }
#pragma unroll
      for (int r = 0; r < kSmallRows; ++r) acc[r] = __fadd_rn(acc[r], __shfl_xor_sync(0xffffffffu, acc[r], 16));
      if (n < H && half == 0) {
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) {
          if (r < R) {
            const int item = s_items[r0 + r];
            p.yw[static_cast<int64_t>(item) * H + n] = __fmul_rn(__fmul_rn(s_w[item], alpha2), acc[r]);
          }
        }
      }
    }
  }

  // ---- 4. the last CTA to finish sums every token's k rows in slot order
  __syncthreads();
  if (tid == 0) {
    __threadfence();  // this CTA's scratch rows are visible before its ticket
    const unsigned int v = atomicAdd(p.ticket, 1u);
    *s_last = v == static_cast<unsigned int>(E - 1);
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  // four consecutive outputs per thread and step (H % 128 == 0), slot loads issued together
  const int n4 = H / 4;
#pragma unroll 4
  for (int q = tid; q < T * n4; q += kSmallThreads) {
    const int t = q / n4, n = 4 * (q - t * n4);
    const float4* src = reinterpret_cast<const float4*>(p.yw + static_cast<int64_t>(t) * k * H + n);
    float4 v[4];
    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j0 = 0; j0 < k; j0 += 4) {
      const int nj = min(4, k - j0);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < nj) v[j] = __ldcg(src + static_cast<int64_t>(j0 + j) * n4);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < nj) {
          sum.x = __fadd_rn(sum.x, v[j].x);
          sum.y = __fadd_rn(sum.y, v[j].y);
          sum.z = __fadd_rn(sum.z, v[j].z);
          sum.w = __fadd_rn(sum.w, v[j].w);
        }
      }
    }
    uint2 o;
    o.x = static_cast<uint32_t>(float_to_bf16_bits(sum.x)) | (static_cast<uint32_t>(float_to_bf16_bits(sum.y)) << 16);
    o.y = static_cast<uint32_t>(float_to_bf16_bits(sum.z)) | (static_cast<uint32_t>(float_to_bf16_bits(sum.w)) << 16);
    *reinterpret_cast<uint2*>(p.out + static_cast<int64_t>(t) * H + n) = o;
  }
  if (tid == 0) *p.ticket = 0u;  // ready for the next launch
}

size_t small_smem_bytes(int T, int H, int I) {
  return static_cast<size_t>(T) * H * 2 + static_cast<size_t>(kSmallRows) * (H + 2 * I + I) * sizeof(float) +
         (3 * kSmallMaxItems + kSmallMaxE + 2 * (kSmallMaxE + 1)) * sizeof(int) +
         (kSmallThreads / 32) * sizeof(float) + 16;
}

}  // namespace

// Shapes the single-launch layer takes.
bool small_layer_eligible(int T, int E, int k, int H, int I) {
  return static_cast<int64_t>(T) * k <= kSmallMaxItems && E <= kSmallMaxE && H <= kSmallMaxH && I <= kSmallMaxI &&
         H % 128 == 0 && I % 64 == 0 && k <= 32;
}

// Scratch of the single-launch layer inside the moe_forward workspace: the
// per-item rows, then the ticket word.
size_t small_layer_scratch_bytes(int T, int k, int H) {
  return (static_cast<size_t>(T) * k * H * sizeof(float) + 255) / 256 * 256 + 256;
}

moe_status small_layer_enqueue(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k,
                               int H, int I, float h_scale, uint16_t* out, int32_t* topk_id, float* topk_w,
                               int32_t* offs, int32_t* p2e, int32_t* e2p, int32_t* e2r, float* x_scale,
                               uint8_t* x_codes, uint8_t* x_sf, float* hs, uint8_t* h_codes, uint8_t* h_sf,
                               void* scratch, bool clear_ticket, cudaStream_t st) {
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
  p.yw = static_cast<float*>(scratch);
  p.ticket = reinterpret_cast<unsigned int*>(static_cast<char*>(scratch) + small_layer_scratch_bytes(T, k, H) - 256);
  const size_t smem = small_smem_bytes(T, H, I);
  if (cudaFuncSetAttribute(small_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_RESOURCE;
  // the ticket is left at 0 by every launch; a stream-ordered clear before eager calls makes that
  // hold from the first launch on (a captured graph relies on the eager pass before its capture)
  if (clear_ticket && cudaMemsetAsync(p.ticket, 0, sizeof(unsigned int), st) != cudaSuccess) return MOE_ERR_CUDA;
  small_layer_kernel<<<E, kSmallThreads, smem, st>>>(p);
  return check_launch();
}

}  // namespace moe

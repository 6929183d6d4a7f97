// quantize.cu -- NVFP4 quantisation (e2m1 codes, e4m3 scale per 16 elements,
// FP32 decode multiplier per tensor or per group of rows).
//
// Format: "Cracking the SM120 Shared Memory Ceiling: A Deep Dive into CUTLASS
// Tile Configuration Debugging", section "The Shared Memory Calculation" (FP4
// packed at 4 bits per element, one FP8 scale per 16 elements along K).
// Scale rule: s = amax/(6*448) per tensor; sf = e4m3(amax_16/(6 s));
// q = e2m1(x / (e4m3(sf) s)) -- the reading stated in nvfp4_moe.h.
//
// HBM-bound: one read of x, one write of codes (K/2 bytes per row) and scales
// (K/16 bytes per row) per destination.  One warp per source row and slice of
// 32 x 64 elements; each lane owns 64 consecutive elements (four 16-element
// blocks), so a warp reads 4 KB of bf16 contiguously, quantises them once and
// writes them to every routed row that reads the source row.  The e2m1 codes
// come from the hardware conversion (e2m1x8 in common.cuh).  The dynamic
// per-tensor scale needs the amax of all of x first: a separate pass
// (amax_kernel).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kQuantWarps = 8;

// Eight bf16 values (one 16-byte word, element 2i in the low half of 32-bit
// word i) as FP32, exactly.
MOE_DEVINL void bf16x8_to_f32(const uint4& u, float* v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

template <int IN_F32>
MOE_DEVINL void load_block16(const void* x, int64_t row, int K, int blk, float (&v)[16]) {
  if (IN_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + row * K + blk * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 f = __ldg(p + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + row * K + blk * 16);
#pragma unroll
    for (int i = 0; i < 2; ++i) bf16x8_to_f32(__ldg(p + i), v + 8 * i);
  }
}

// max |element| of one 16-byte vector of bf16 (8) or FP32 (4) values
template <int IN_F32>
MOE_DEVINL float abs_max_vec(const uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (IN_F32) {
      m = fmaxf(m, fabsf(__uint_as_float(w[j])));
    } else {
      m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
  return m;
}

// Per-group absolute maximum over the group's rows (contiguous, a multiple of 16
// bytes long): 16-byte loads in a grid-stride loop, a block-wide reduction, then
// one atomicMax per block on the bit pattern, which orders non-negative floats
// like their values.
constexpr int kAmaxThreads = 256;
template <int IN_F32>
__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const void* __restrict__ x, int64_t rows_per_group,
                                                            int K, uint32_t* __restrict__ amax_bits) {
  __shared__ float warp_max[kAmaxThreads / 32];
  const int g = blockIdx.y;
  constexpr int kPerVec = IN_F32 ? 4 : 8;  // elements per 16-byte vector
  const int64_t n_vec = rows_per_group * K / kPerVec;
  const uint4* v = reinterpret_cast<const uint4*>(x) + static_cast<int64_t>(g) * n_vec;
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kAmaxThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x;
  for (; i + 3 * stride < n_vec; i += 4 * stride) {  // four loads in flight per thread
    uint4 u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) u[j] = __ldg(v + i + j * stride);
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, abs_max_vec<IN_F32>(u[j]));
  }
  for (; i < n_vec; i += stride) m = fmaxf(m, abs_max_vec<IN_F32>(__ldg(v + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 1; w < kAmaxThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    if (m > 0.0f) atomicMax(amax_bits + g, __float_as_uint(m));
  }
}

// Decode multiplier of every group from its amax (used when the quantise kernel
// does not visit every group's first row).
__global__ void scale_from_amax_kernel(const uint32_t* __restrict__ amax_bits, int groups, float* __restrict__ scale) {
  int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  float a = __uint_as_float(amax_bits[g]);
  scale[g] = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
}

// Destination of one 16-element block (8 code bytes + 1 scale byte) of row `dst`, column block `c`.
//   LAYOUT 0: linear codes and scales; 1: linear codes, tiled scales; 2: blocked weights (one
//   18432-byte block per 128 rows x 256 K-elements: the 128-byte-swizzled code tile, then its
//   four 512-byte scale atoms).
template <int LAYOUT>
MOE_DEVINL void block_dst(uint8_t* codes, uint8_t* sf, int64_t dst, int c, int K, uint8_t** code_at,
                          uint8_t** sf_at) {
  if (LAYOUT == 2) {
    const int kt_count = (K + 255) / 256;
    const int rr = static_cast<int>(dst & 127);
    const int cc = c & 15;
    uint8_t* base = codes + ((dst >> 7) * kt_count + (c >> 4)) * static_cast<int64_t>(kBlockedTileBytes);
    *code_at = base + rr * 128 + (((cc >> 1) ^ (rr & 7)) << 4) + (cc & 1) * 8;
    *sf_at = base + 16384 + (cc >> 2) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (cc & 3);
  } else {
    *code_at = codes + dst * (K / 2) + 8 * c;
    *sf_at = (LAYOUT == 1) ? sf + tiled_sf_offset(dst, c, K) : sf + dst * (K / 16) + c;
  }
}

// Quantises one 16-element block: codes of elements 0-7 in *lo, 8-15 in *hi
// (element 2i in the low nibble of byte i), returns the e4m3 scale byte.
MOE_DEVINL uint32_t quantize_values16(const float (&v)[16], float s, uint32_t* lo, uint32_t* hi) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  float recip;
  const uint32_t sfb = nvfp4_block_scale(amax, s, &recip);
  *lo = nvfp4_codes8(v, recip);
  *hi = nvfp4_codes8(v + 8, recip);
  return sfb;
}

template <int IN_F32>
MOE_DEVINL uint32_t quantize_block16(const void* x, int64_t row, int K, int blk, float s, uint32_t* lo,
                                     uint32_t* hi) {
  float v[16];
  load_block16<IN_F32>(x, row, K, blk, v);
  return quantize_values16(v, s, lo, hi);
}

// One warp per source row.  The row is quantised once and written to every
// item that reads it: items [src * fan, src * fan + fan) when fan > 1 (all
// items of a source row are consecutive when items map to rows i / src_div),
// or the single item `src` when fan == 1.  When K % 64 == 0 each lane owns 4
// consecutive blocks (64 elements), so every destination gets 32 bytes of
// codes and 4 contiguous scale bytes (one aligned word in every layout).
template <int IN_F32, int LAYOUT>
__global__ void __launch_bounds__(kQuantWarps * 32) quantize_kernel(
    const void* __restrict__ x, int64_t rows_per_group, int K, const uint32_t* __restrict__ amax_bits,
    float* __restrict__ scale, int64_t n_src, int n_slices, int fan, const int32_t* __restrict__ dst_row,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  const int64_t src = w / n_slices;
  const int slice = static_cast<int>(w - src * n_slices);
  if (src >= n_src) return;
  const int64_t g = src / rows_per_group;
  float s;
  if (amax_bits) {
    // dynamic scale: s = amax / (6 * 448) of the row's group (1 when the group is all zero); the
    // first warp of the group publishes it
    const float a = __uint_as_float(__ldg(amax_bits + g));
    s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
    if (src == g * rows_per_group && slice == 0 && lane == 0) scale[g] = s;
  } else {
    s = __ldg(scale + g);
  }
  if (K % 64 == 0) {
    // The row's destinations, one per lane (fan <= 32), loaded up front alongside x
    // and broadcast in the loop below instead of one dependent load per store.
    int64_t my_dst = 0;
    if (lane < fan) {
      const int64_t item = src * fan + lane;
      my_dst = dst_row ? static_cast<int64_t>(__ldg(dst_row + item)) : item;
    }
    // this warp's slice: quads [32 * slice, 32 * slice + 32), one per lane
    const int q = 32 * slice + lane;
    const bool act = q < K / 64;
    uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t sf4 = 0;
    if (act) {
      if (IN_F32) {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          sf4 |= quantize_block16<IN_F32>(x, src, K, 4 * q + b, s, &c[2 * b], &c[2 * b + 1]) << (8 * b);
      } else {
        // the lane's 128 bytes of bf16 x requested together before any arithmetic: one memory round trip
        // per warp instead of one per block
        const uint4* p4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + src * K + 64 * q);
        uint4 raw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) raw[i] = __ldg(p4 + i);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float v[16];
          bf16x8_to_f32(raw[2 * b], v);
          bf16x8_to_f32(raw[2 * b + 1], v + 8);
          sf4 |= quantize_values16(v, s, &c[2 * b], &c[2 * b + 1]) << (8 * b);
        }
      }
    }
    if (LAYOUT != 2) {
      // Linear codes: the slice's codes form one contiguous span of 32 B per quad.  Lane l
      // holds 16-byte chunks 2l and 2l+1; after this transpose it holds chunks l and 32 + l,
      // so each destination takes two fully coalesced 512-byte stores.
      const int nq = min(32, K / 64 - 32 * slice);  // quads in this slice
      const int src_a = lane >> 1, src_b = 16 + (lane >> 1);
      const bool odd = (lane & 1) != 0;
      uint32_t ca[4], cb[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t a_lo = __shfl_sync(0xffffffffu, c[t], src_a), a_hi = __shfl_sync(0xffffffffu, c[4 + t], src_a);
        const uint32_t b_lo = __shfl_sync(0xffffffffu, c[t], src_b), b_hi = __shfl_sync(0xffffffffu, c[4 + t], src_b);
        ca[t] = odd ? a_hi : a_lo;
        cb[t] = odd ? b_hi : b_lo;
      }
      const bool st_a = lane < 2 * nq, st_b = 32 + lane < 2 * nq;
      for (int j = 0; j < fan; ++j) {
        const int64_t dst = __shfl_sync(0xffffffffu, my_dst, j);
        uint8_t* span = codes + dst * (K / 2) + 32 * (32 * slice);
        if (st_a) *reinterpret_cast<uint4*>(span + 16 * lane) = make_uint4(ca[0], ca[1], ca[2], ca[3]);
        if (st_b) *reinterpret_cast<uint4*>(span + 512 + 16 * lane) = make_uint4(cb[0], cb[1], cb[2], cb[3]);
        if (act) {
          uint8_t* sf_at = (LAYOUT == 1) ? sf + tiled_sf_offset(dst, 4 * q, K) : sf + dst * (K / 16) + 4 * q;
          *reinterpret_cast<uint32_t*>(sf_at) = sf4;
        }
      }
    } else {
      for (int j = 0; j < fan; ++j) {
        const int64_t dst = __shfl_sync(0xffffffffu, my_dst, j);
        if (!act) continue;
        uint8_t *c0, *c1, *sf_at;
        if (LAYOUT == 2) {
          const int kt_count = (K + 255) / 256;
          const int rr = static_cast<int>(dst & 127);
          uint8_t* base = codes + ((dst >> 7) * kt_count + (q >> 2)) * static_cast<int64_t>(kBlockedTileBytes);
          const int chunk = 2 * (q & 3);
          c0 = base + rr * 128 + ((chunk ^ (rr & 7)) << 4);
          c1 = base + rr * 128 + (((chunk + 1) ^ (rr & 7)) << 4);
          sf_at = base + 16384 + (q & 3) * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
        } else {
          c0 = codes + dst * (K / 2) + 32 * q;
          c1 = c0 + 16;
          sf_at = (LAYOUT == 1) ? sf + tiled_sf_offset(dst, 4 * q, K) : sf + dst * (K / 16) + 4 * q;
        }
        *reinterpret_cast<uint4*>(c0) = make_uint4(c[0], c[1], c[2], c[3]);
        *reinterpret_cast<uint4*>(c1) = make_uint4(c[4], c[5], c[6], c[7]);
        *reinterpret_cast<uint32_t*>(sf_at) = sf4;
      }
    }
  } else {
    for (int blk = lane; blk < K / 16; blk += 32) {
      uint32_t lo, hi;
      const uint32_t sfb = quantize_block16<IN_F32>(x, src, K, blk, s, &lo, &hi);
      for (int j = 0; j < fan; ++j) {
        const int64_t item = src * fan + j;
        const int64_t dst = dst_row ? static_cast<int64_t>(__ldg(dst_row + item)) : item;
        uint8_t *code_at, *sf_at;
        block_dst<LAYOUT>(codes, sf, dst, blk, K, &code_at, &sf_at);
        *reinterpret_cast<uint2*>(code_at) = make_uint2(lo, hi);
        *sf_at = static_cast<uint8_t>(sfb);
      }
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_blocked_weight_bytes(int64_t rows, int K) {
  if (rows < 1 || K < 64 || rows % 128 || K % 64) return 0;
  return static_cast<size_t>(rows / 128) * ((K + 255) / 256) * kBlockedTileBytes;
}

extern "C" size_t nvfp4_quantize_workspace_size(int groups) {
  if (groups < 1) return 0;
  return static_cast<size_t>((groups * 4 + 255) / 256) * 256;
}

namespace moe {

moe_status quantize_amax_enqueue(const void* x, int in_dtype, int64_t rows_per_group, int K, int groups,
                                 uint32_t* amax, cudaStream_t st) {
  if (cudaMemsetAsync(amax, 0, sizeof(uint32_t) * groups, st) != cudaSuccess) return MOE_ERR_CUDA;
  // four 16-byte vectors per thread per pass; about four blocks per SM over all groups
  const int64_t n_vec = rows_per_group * K / (in_dtype == MOE_IN_F32 ? 4 : 8);
  int64_t bx64 = (n_vec + 4 * kAmaxThreads - 1) / (4 * kAmaxThreads);
  const int cap = (num_sms() * 4 + groups - 1) / groups;
  if (bx64 > cap) bx64 = cap < 1 ? 1 : cap;
  const int bx = static_cast<int>(bx64);
  dim3 grid(bx, groups);
  if (in_dtype == MOE_IN_F32)
    amax_kernel<1><<<grid, kAmaxThreads, 0, st>>>(x, rows_per_group, K, amax);
  else
    amax_kernel<0><<<grid, kAmaxThreads, 0, st>>>(x, rows_per_group, K, amax);
  return check_launch();
}

moe_status quantize_enqueue(const void* x, int in_dtype, int64_t src_rows, int K, int groups, float* tensor_scale,
                            int amax_mode, int64_t n_items, int src_div, const int32_t* dst_row, uint8_t* codes,
                            uint8_t* sf, int sf_layout, int64_t dst_rows_alloc, void* ws, size_t ws_bytes,
                            cudaStream_t st) {
  const int dynamic_scale = amax_mode != 0;
  if (!x || !tensor_scale || !codes || (!sf && sf_layout != MOE_SF_BLOCKED)) return MOE_ERR_INVALID_ARG;
  if (src_rows < 1 || K < 16 || groups < 1 || n_items < 0 || src_div < 1 || dst_rows_alloc < 1)
    return MOE_ERR_INVALID_ARG;
  if (in_dtype != MOE_IN_BF16 && in_dtype != MOE_IN_F32) return MOE_ERR_INVALID_ARG;
  if (sf_layout != MOE_SF_LINEAR && sf_layout != MOE_SF_TILED && sf_layout != MOE_SF_BLOCKED)
    return MOE_ERR_INVALID_ARG;
  if (K % 16) return MOE_ERR_UNSUPPORTED;
  if (sf_layout != MOE_SF_LINEAR && (K % 64 || dst_rows_alloc % 128)) return MOE_ERR_UNSUPPORTED;
  if (src_rows % groups) return MOE_ERR_INVALID_ARG;
  if ((n_items - 1) / src_div >= src_rows && n_items > 0) return MOE_ERR_INVALID_ARG;
  if (!dst_row && n_items > dst_rows_alloc) return MOE_ERR_INVALID_ARG;
  // A source row read by several items is quantised once and fanned out to all of them.
  if (src_div > 1 && (src_div > 32 || n_items != src_rows * src_div)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(codes) || (sf && !aligned16(sf))) return MOE_ERR_MISALIGNED;
  if (dynamic_scale && (!ws || ws_bytes < nvfp4_quantize_workspace_size(groups))) return MOE_ERR_WORKSPACE;
  // Launch geometry first, so a shape the grid cannot express is rejected before anything is enqueued.
  const bool fan_out = src_div > 1;
  const int fan = fan_out ? src_div : 1;
  const int64_t n_src = fan_out ? src_rows : n_items;
  // rows split into slices of 32 x 64 elements so short batches still fill the GPU
  const int n_slices = (K % 64 == 0) ? (K / 64 + 31) / 32 : 1;
  const int64_t blocks = (n_src * n_slices + kQuantWarps - 1) / kQuantWarps;
  if (blocks > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  const int64_t rows_per_group = src_rows / groups;
  if (amax_mode == 1) {
    const moe_status s = quantize_amax_enqueue(x, in_dtype, rows_per_group, K, groups, static_cast<uint32_t*>(ws), st);
    if (s != MOE_OK) return s;
  }
  const bool covers_all_rows = (src_div > 1) || (n_items == src_rows);
  if (dynamic_scale && (n_items == 0 || !covers_all_rows))
    scale_from_amax_kernel<<<(groups + 255) / 256, 256, 0, st>>>(static_cast<const uint32_t*>(ws), groups,
                                                                 tensor_scale);
  if (n_items > 0) {
    // Fan out when every source row is read by src_div consecutive items (the
    // routed-row gather); otherwise one item per warp.
    const bool f32 = in_dtype == MOE_IN_F32;
#define MOE_QLAUNCH(F, T)                                                                                     \
  quantize_kernel<F, T><<<static_cast<unsigned>(blocks), kQuantWarps * 32, 0, st>>>(                          \
      x, rows_per_group, K, (dynamic_scale && covers_all_rows) ? static_cast<const uint32_t*>(ws) : nullptr,      \
      tensor_scale, n_src, n_slices,                                                                           \
      fan, dst_row, codes, sf)
    if (f32) {
      if (sf_layout == MOE_SF_BLOCKED) MOE_QLAUNCH(1, 2);
      else if (sf_layout == MOE_SF_TILED) MOE_QLAUNCH(1, 1);
      else MOE_QLAUNCH(1, 0);
    } else {
      if (sf_layout == MOE_SF_BLOCKED) MOE_QLAUNCH(0, 2);
      else if (sf_layout == MOE_SF_TILED) MOE_QLAUNCH(0, 1);
      else MOE_QLAUNCH(0, 0);
    }
#undef MOE_QLAUNCH
  }
  return check_launch();
}

}  // namespace moe

extern "C" moe_status nvfp4_quantize(const void* x, int in_dtype, int64_t src_rows, int K, int groups,
                                     float* tensor_scale, int dynamic_scale, int64_t n_items, int src_div,
                                     const int32_t* dst_row, uint8_t* codes, uint8_t* sf, int sf_layout,
                                     int64_t dst_rows_alloc, void* ws, size_t ws_bytes, void* stream) {
  return quantize_enqueue(x, in_dtype, src_rows, K, groups, tensor_scale, dynamic_scale ? 1 : 0, n_items, src_div,
                          dst_row, codes, sf, sf_layout, dst_rows_alloc, ws, ws_bytes,
                          static_cast<cudaStream_t>(stream));
}

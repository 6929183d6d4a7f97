// finalize.cu -- FINALIZE: the router-weighted sum of each token's k expert
// rows back into one BF16 token row, and the FP32 -> BF16 store that closes
// the in-GEMM FINALIZE epilogue.
//
// "The Epilogue That Broke the Kernel: Tracing a CUTLASS Tile Configuration
// Failure on Blackwell GPUs", section "The Insight: FINALIZE vs NONE"
// (FINALIZE does work beyond the NONE store); "Cracking the SM120 Shared
// Memory Ceiling: A Deep Dive into CUTLASS Tile Configuration Debugging",
// section "The Shared Memory Calculation" (FP32 accumulator, BF16 output).
//
// HBM-bound gathers: each thread owns 8 consecutive output columns of one
// token (16-byte loads and stores) and sums the k expert rows in slot order.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) finalize_kernel(const uint16_t* __restrict__ y,
                                                       const float* __restrict__ topk_w,
                                                       const int32_t* __restrict__ row_of_item, int T, int k,
                                                       int N, int64_t y_rows, uint16_t* __restrict__ out,
                                                       int32_t* err) {
  const int vec_per_row = N / 8;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<int64_t>(T) * vec_per_row) return;
  const int t = static_cast<int>(gid / vec_per_row);
  const int c = static_cast<int>(gid % vec_per_row) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int64_t item = static_cast<int64_t>(t) * k + j;
    const float w = __ldg(topk_w + item);
    const int64_t r = __ldg(row_of_item + item);
    if (r < 0 || r >= y_rows) {  // a row map outside y: report it and leave the term out
      record_error(err, MOE_ERR_INVALID_ARG, 8);
      continue;
    }
    uint4 u = __ldg(reinterpret_cast<const uint4*>(y + r * N + c));
    uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = __fmaf_rn(w, __uint_as_float(p[i] << 16), acc[2 * i]);
      acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(p[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = static_cast<uint32_t>(float_to_bf16_bits(acc[2 * i])) |
           (static_cast<uint32_t>(float_to_bf16_bits(acc[2 * i + 1])) << 16);
  *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * N + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out,
                                                          int64_t n4) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 f = __ldg(in + i);
    uint32_t a = static_cast<uint32_t>(float_to_bf16_bits(f.x)) | (static_cast<uint32_t>(float_to_bf16_bits(f.y)) << 16);
    uint32_t b = static_cast<uint32_t>(float_to_bf16_bits(f.z)) | (static_cast<uint32_t>(float_to_bf16_bits(f.w)) << 16);
    out[i] = make_uint2(a, b);
  }
}

// out[t][n] = bf16( sum_{j<k} rows[t*k + j][n] ), summed in slot order in FP32.
__global__ void __launch_bounds__(256) finalize_sum_kernel(const float* __restrict__ rows, int T, int k, int N,
                                                           uint16_t* __restrict__ out) {
  const int vec_per_row = N / 4;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<int64_t>(T) * vec_per_row) return;
  const int64_t t = gid / vec_per_row;
  const int c = static_cast<int>(gid % vec_per_row) * 4;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int j = 0; j < k; ++j) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(rows + (t * k + j) * N + c));
    acc.x = __fadd_rn(acc.x, v.x);
    acc.y = __fadd_rn(acc.y, v.y);
    acc.z = __fadd_rn(acc.z, v.z);
    acc.w = __fadd_rn(acc.w, v.w);
  }
  const uint32_t a = static_cast<uint32_t>(float_to_bf16_bits(acc.x)) | (static_cast<uint32_t>(float_to_bf16_bits(acc.y)) << 16);
  const uint32_t b = static_cast<uint32_t>(float_to_bf16_bits(acc.z)) | (static_cast<uint32_t>(float_to_bf16_bits(acc.w)) << 16);
  *reinterpret_cast<uint2*>(out + t * N + c) = make_uint2(a, b);
}

}  // namespace

moe_status launch_finalize_sum(const float* rows, int T, int k, int N, uint16_t* out, cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(T) * (N / 4);
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  finalize_sum_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(rows, T, k, N, out);
  return check_launch();
}

// Converts n (a multiple of 4) FP32 values to BF16 (round to nearest even).
moe_status launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t st) {
  int64_t n4 = n / 4;
  int64_t blocks = (n4 + 255) / 256;
  int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  f32_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(reinterpret_cast<const float4*>(in),
                                                                     reinterpret_cast<uint2*>(out), n4);
  return check_launch();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_finalize(const uint16_t* y, int64_t y_rows, const float* topk_w, const int32_t* row_of_item,
                                   int T, int k, int N, uint16_t* out, void* stream) {
  if (!y || !topk_w || !row_of_item || !out) return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || N < 8 || y_rows < 1) return MOE_ERR_INVALID_ARG;
  if (N % 8) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(y) || !aligned16(out)) return MOE_ERR_MISALIGNED;
  int64_t threads = static_cast<int64_t>(T) * (N / 8);
  int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  int32_t* err = device_error_word();
  if (!err) return MOE_ERR_CUDA;
  finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      y, topk_w, row_of_item, T, k, N, y_rows, out, err);
  return check_launch();
}

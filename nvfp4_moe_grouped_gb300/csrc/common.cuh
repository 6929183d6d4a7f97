// common.cuh -- shared device helpers of the GB300 NVFP4 MoE kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA, tcgen05 (tensor memory, block-scaled
// MMA) and the small scalar pieces the kernels share: the NVFP4 encoders, the
// routing exp, bf16 rounding.  Nothing here allocates memory.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4_moe.h"

#define MOE_DEVINL __device__ __forceinline__

namespace moe {

// ----------------------------------------------------------------------------
// Host-side plumbing shared by the translation units (defined in capi.cu).
// ----------------------------------------------------------------------------
int32_t* device_error_word();          // device address of {code, where}
uint64_t wait_timeout_ns();            // bound of every device-side wait
int num_sms();                          // SM count of the current device
moe_status check_launch();              // maps cudaGetLastError to a status
// Pieces of the public calls that the layer's graph schedules on their own:
// the activation quantiser's amax pass (into `amax_ws`, nvfp4_quantize's
// workspace), the quantiser itself with amax_mode 0 = static scale, 1 = compute
// the amax here, 2 = the amax is already in the workspace, and the grouped GEMM
// with or without clearing its FINALIZE accumulator (the bytes to clear, 0 when
// FINALIZE gathers rows instead, come from finalize_accumulator_bytes).
moe_status quantize_amax_enqueue(const void* x, int in_dtype, int64_t rows_per_group, int K, int groups,
                                 uint32_t* amax_ws, cudaStream_t st);
moe_status quantize_enqueue(const void* x, int in_dtype, int64_t src_rows, int K, int groups, float* tensor_scale,
                            int amax_mode, int64_t n_items, int src_div, const int32_t* dst_row, uint8_t* codes,
                            uint8_t* sf, int sf_layout, int64_t dst_rows_alloc, void* ws, size_t ws_bytes,
                            cudaStream_t st);
moe_status grouped_gemm_enqueue(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                const uint8_t* b_blocked, const float* b_scale, const int32_t* expert_offsets, int E,
                                int64_t a_rows_alloc, int N, int K, int epilogue, const moe_epilogue_args* ep,
                                void* out, void* ws, size_t ws_bytes, bool clear_accumulator, cudaStream_t st);
size_t finalize_accumulator_bytes(int T, int N);
// cuTensorMapEncodeTiled from the driver, or nullptr when the driver lacks it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Blocked weight layout: one block per 128 rows x 256 K-elements, holding the
// 128-byte-swizzled code tile (16 KB, the shared-memory image the MMA reads)
// followed by its four 512-byte scale atoms.
constexpr int kBlockedTileBytes = 16384 + 2048;

// ----------------------------------------------------------------------------
// Scalars
// ----------------------------------------------------------------------------
MOE_DEVINL uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first error of a launch; later ones are dropped.
MOE_DEVINL void record_error(int32_t* err, int32_t code, int32_t where) {
  if (atomicCAS(err, 0, code) == 0) atomicExch(err + 1, where);
}

// exp for the router weights: Cody-Waite reduction x = n ln2 + r with ln 2
// split into an FP32 head and tail, then the degree-7 Taylor polynomial of
// e^r in Horner form with fused multiply-adds, then an exact scaling by 2^n.
// Results below e^-86 flush to 0 (all inputs here are <= 0).  Every operation
// is correctly rounded, so the host restatement gives identical bits.
MOE_DEVINL float route_exp(float x) {
  const float kLog2e = 0x1.715476p+0f;
  const float kLn2Hi = 0x1.62e43p-1f;
  const float kLn2Lo = -0x1.05c61p-29f;
  if (!(x >= -86.0f)) return 0.0f;
  if (x > 88.0f) return __int_as_float(0x7f800000);
  float n = rintf(__fmul_rn(x, kLog2e));
  float r = __fmaf_rn(-n, kLn2Hi, x);
  r = __fmaf_rn(-n, kLn2Lo, r);
  float p = 0x1.a01a02p-13f;                 // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);      // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);       // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);       // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);       // 1/3!
  p = __fmaf_rn(p, r, 0x1p-1f);              // 1/2!
  p = __fmaf_rn(p, r, 1.0f);                 // 1/1!
  p = __fmaf_rn(p, r, 1.0f);                 // 1/0!
  float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
  return __fmul_rn(p, two_n);
}

// Routing order of a logit as an unsigned integer: larger logits give larger
// codes, -0 and +0 the same one, and every non-NaN logit a code above 0, so 0
// can stand for "not a candidate".
MOE_DEVINL uint32_t route_order_bits(float x) {
  const uint32_t b = x == 0.0f ? 0u : __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The logit a routing code stands for (+0 for either zero).
MOE_DEVINL float route_order_value(uint32_t ob) {
  return __uint_as_float((ob & 0x80000000u) ? (ob & 0x7FFFFFFFu) : ~ob);
}

// Top-k and softmax of one token whose E logits a warp holds: lane l owns
// experts l + 32 i in v[i], and bit i of `taken` is set where that expert does
// not exist (>= E).  Slot j (descending logit, ties to the lower index) ends in
// lane j: *id its expert, *w its weight, the softmax of the k selected logits
// (exponentials of the differences to the largest, summed in slot order, one
// correctly rounded division).  Lanes >= k get *w = 0 and an unspecified *id.
// Each of the k rounds takes the largest remaining code with one warp max
// reduction and, among the experts holding it, the lowest index with one warp
// min reduction; the winner's code is then cleared.  NaN logits are not
// supported (their order is unspecified).
template <int NV>
MOE_DEVINL void warp_topk_softmax(const float (&v)[NV], uint32_t taken, int k, int* id, float* w) {
  const int lane = threadIdx.x & 31;
  uint32_t ob[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) ob[i] = (taken >> i & 1u) ? 0u : route_order_bits(v[i]);
  uint32_t my_ob = 0u;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t lm = ob[0];
#pragma unroll
    for (int i = 1; i < NV; ++i) lm = max(lm, ob[i]);
    const uint32_t m = __reduce_max_sync(0xffffffffu, lm);
    int ci = NV;  // this lane's lowest slot holding the maximum
#pragma unroll
    for (int i = NV - 1; i >= 0; --i) ci = ob[i] == m ? i : ci;
    const int bi = __reduce_min_sync(0xffffffffu, ci < NV ? lane + 32 * ci : 0x7fffffff);
    const int bd = bi - lane;  // 32 i in the winner's lane, not a multiple of 32 in the others
#pragma unroll
    for (int i = 0; i < NV; ++i) ob[i] = bd == 32 * i ? 0u : ob[i];
    if (lane == j) { my_ob = m; my_i = bi; }
  }
  const float my_v = route_order_value(my_ob);
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? route_exp(__fsub_rn(my_v, m)) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ex, j));
  *id = my_i;
  *w = (lane < k) ? __fdiv_rn(ex, sum) : 0.0f;
}

// e2m1 codes of eight values, v[i] in bits 4i..4i+3: the nearest of
// {0, .5, 1, 1.5, 2, 3, 4, 6} with the sign, ties to the even code, saturating
// above 6 (the hardware conversion, two values per instruction, the first
// operand to the high nibble); then the sign bit is cleared wherever the
// magnitude code is 0, so a value that rounds to zero is +0.
MOE_DEVINL uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t w;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  // bit 3 of every nibble whose magnitude (bits 0-2) is non-zero: m + 7 carries into it
  const uint32_t nonzero = ((w & 0x77777777u) + 0x77777777u) & 0x88888888u;
  return w & (0x77777777u | nonzero);
}

// e4m3 (fn) scale byte of a non-negative value: round to nearest even,
// saturating to 448.
MOE_DEVINL uint32_t e4m3_encode_satfinite(float v) {
  __nv_fp8_storage_t s = __nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(s) & 0xFFu;
}

MOE_DEVINL float e4m3_decode(uint32_t byte) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
  return __half2float(__half(h));
}

// The NVFP4 scale of one 16-element block with decode multiplier s.
// Returns the e4m3 byte and the reciprocal multiplier (0 when the block's
// decoded scale is 0, which zeroes every code of the block).
MOE_DEVINL uint32_t nvfp4_block_scale(float amax, float s, float* recip) {
  float sf_f = __fdiv_rn(amax, __fmul_rn(6.0f, s));
  uint32_t sf = e4m3_encode_satfinite(sf_f);
  float d = __fmul_rn(e4m3_decode(sf), s);
  *recip = (d == 0.0f) ? 0.0f : __frcp_rn(d);
  return sf;
}

// Codes of x[0..7] under the block's reciprocal multiplier (0 when the block's
// decoded scale is 0: every product is then a zero and every code 0).
MOE_DEVINL uint32_t nvfp4_codes8(const float* x, float recip) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(x[i], recip);
  return e2m1x8(v);
}

// h = silu(g) * u = g / (1 + e^-g) * u in FP32 with the fast hardware forms:
// __expf (the SFU's 2^x, error growing with |g|) and __fdividef (about 2 ulp),
// then a correctly rounded product.  Against the FP64 reference on the
// full-size layers, these flip 16 of 524,288 sampled requantised h codes (one
// grid step each, at rounding boundaries) in one of nine configurations and none
// in the other eight; correctly rounded division and expf flip none there, but
// cost the prefill gate_up launch about a quarter of its time (its epilogue
// shares the SM with the MMA issue).  For g below about -88 the quotient is -0,
// the limit of silu there.
MOE_DEVINL float silu_mul(float g, float u) { return __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u); }

MOE_DEVINL float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

MOE_DEVINL uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Byte offset of scale (row r, column c) in the tiled scale layout.
MOE_DEVINL int64_t tiled_sf_offset(int64_t r, int c, int K) {
  int64_t atom = (r >> 7) * (K >> 6) + (c >> 2);
  return atom * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// ----------------------------------------------------------------------------
// Shared memory, mbarriers
// ----------------------------------------------------------------------------
MOE_DEVINL uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

MOE_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
MOE_DEVINL void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

MOE_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
MOE_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) after timeout_ns, or early once *abort is set by another
// role of the same CTA.
MOE_DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Non-blocking test of the phase with the given parity (the thread is never suspended).
MOE_DEVINL bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait_bounded by spinning on test_wait: for a thread whose wake-up latency
// is on the critical path (a suspended try_wait can resume well after the phase
// completes).  Same bound and abort as mbar_wait_bounded.
MOE_DEVINL bool mbar_spin_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, volatile int* abort) {
  if (mbar_test_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// ----------------------------------------------------------------------------
// TMA and bulk copies (global -> shared, completion on an mbarrier)
// ----------------------------------------------------------------------------
MOE_DEVINL uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEVINL uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEVINL uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEVINL void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

MOE_DEVINL void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and the block-scaled MMA
// ----------------------------------------------------------------------------
MOE_DEVINL void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEVINL void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
MOE_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MOE_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] x B[smem]^T with e2m1 operands and ue4m3 scales per 16
// K-elements read from tensor memory (M = 128, N from the descriptor, K = 64).
MOE_DEVINL void mma_mxf4nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
                             uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// D (TMEM, FP32) (+)= A (smem, bf16, K-major) x B (smem, bf16, K-major)^T: one
// tcgen05.mma of kind::f16 (M = 128, K = 16); A and B are both bf16.
MOE_DEVINL void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
MOE_DEVINL void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Copies a 32-row x 16-byte shared-memory matrix into 4 TMEM columns of lanes
// 0-31, replicated into the lanes of all four warp quadrants.
MOE_DEVINL void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Each thread of the warp loads 32 consecutive 32-bit columns of its lane.
MOE_DEVINL void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
MOE_DEVINL void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Each thread of the warp stores 32 consecutive 32-bit columns of its lane.
MOE_DEVINL void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Each thread of the warp stores 16 consecutive 32-bit columns of its lane.
MOE_DEVINL void tmem_st_16cols(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// Each thread of the warp stores one 32-bit column of its lane.
MOE_DEVINL void tmem_st_1col(uint32_t taddr, uint32_t r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}
// Each thread of the warp stores 8 consecutive 32-bit columns of its lane.
MOE_DEVINL void tmem_st_8cols(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
MOE_DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format, version 1).
//   start: byte address; lbo/sbo: leading/stride byte offsets; layout:
//   0 = no swizzle, 2 = 128-byte swizzle.
MOE_DEVINL uint64_t smem_desc(uint32_t start, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor of kind::mxf4nvf4: e2m1 A and B (format 1), both
// K-major, ue4m3 scales (bit 23 = 0), dense, M = 128 (or m).
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int n, int m = 128) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// ----------------------------------------------------------------------------
// CTA pairs (tcgen05 cta_group::2).  Two CTAs of a cluster (ranks 2c and
// 2c + 1) form a pair; one thread of the even CTA issues MMAs with M = 256:
// A rows 0-127 from the even CTA's shared memory and rows 128-255 from the odd
// CTA's (same offset), B rows [0, N/2) from the even CTA's and [N/2, N) from
// the odd CTA's, the accumulator rows of each CTA in its own tensor memory.
// Every tcgen05 instruction of a kernel that uses pairs names cta_group::2:
// allocation and release are made by one warp of EACH CTA together.
// ----------------------------------------------------------------------------
MOE_DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
MOE_DEVINL uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
MOE_DEVINL uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of both CTAs arrives; returns once all have (release/acquire at cluster scope).
MOE_DEVINL void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Shared-memory address `addr` (of this CTA) mapped into CTA `rank` of the cluster.
MOE_DEVINL uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its cluster address (this CTA's or the peer's),
// with the default release semantics of an arrive (CTA scope): a cluster-scope
// release would make the arriving warp wait for all its earlier memory
// operations (an epilogue's global stores) to become visible cluster-wide.
// Tensor-memory operations before the arrive are ordered by the caller's
// tcgen05.fence::before_thread_sync, as for an arrive inside one CTA.
MOE_DEVINL void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
MOE_DEVINL void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEVINL void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The pair form of mma_mxf4nvf4 (M = 256 over the two CTAs), issued by one thread of the even CTA.
MOE_DEVINL void mma_mxf4nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                  uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// mma_mxf4nvf4_pair with the descriptors given as 32-bit halves: the high halves
// (stride, version, layout) are fixed for a kernel, so the issuing thread moves
// only the low halves (start addresses) and never does 64-bit arithmetic.
MOE_DEVINL void mma_mxf4nvf4_pair_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                     uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
      "mov.b64 ad, {%1, %2};\n\t"
      "mov.b64 bd, {%3, %4};\n\t"
      "setp.ne.b32 p, %8, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], ad, bd, %5, [%6], [%7], p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Arrives once on the mbarrier at the same shared-memory offset in each CTA of
// `cta_mask` when every tcgen05 operation issued so far by this thread has
// completed (the pair's MMAs write both CTAs' tensor memory).
MOE_DEVINL void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B (format 1), FP32 D
// (bits 4-5 = 1), both K-major, dense, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

}  // namespace moe

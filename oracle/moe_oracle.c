/*
 * moe_oracle.c -- plain CPU oracle for the NVFP4 Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never calls, links or loads
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA path.
 * It is deliberately slow: straight loops in the order the definitions give,
 * FP64 for every sum whose precision the method leaves open, FP32 exactly
 * where a floating-point result decides an integer (a routing slot, an e2m1
 * code, an e4m3 scale) so that both sides take the decision in the same
 * precision.
 *
 * What is computed, and where it is stated (page title, section):
 *  - "Cracking the SM120 Shared Memory Ceiling: A Deep Dive into CUTLASS Tile
 *    Configuration Debugging", section "The Shared Memory Calculation": FP4
 *    operands packed at 4 bits per element, one FP8 scale per 16 elements
 *    along K for both operands, FP32 accumulation, BF16 output; the same
 *    section prints a per-tile shared-memory model (smem_model_bytes below).
 *  - "The CUTLASS Tile That Wouldn't Fit: Debugging EP8 on Blackwell SM120",
 *    section "The Crash": the grouped GEMM multiplies e2m1 by e2m1 into bf16.
 *  - "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on
 *    Blackwell SM120", sections "The Broader Context" (256 experts, 8 active
 *    per token, 32x2048x6144 expert GEMMs at decode) and "Input Knowledge
 *    Required" (one GEMM per expert inside one grouped launch, with a problem
 *    size per expert).
 *  - "The Epilogue That Broke the Kernel: Tracing a CUTLASS Tile
 *    Configuration Failure on Blackwell GPUs", section "The Insight: FINALIZE
 *    vs NONE": NONE is a pass-through store of the GEMM result, FINALIZE does
 *    more work; "Cracking the SM120 Shared Memory Ceiling", "The Shared Memory
 *    Calculation", gives FINALIZE an FP32 accumulator plus a BF16 output.
 *
 * Readings taken where the pages are silent (each restated at its function):
 *  R1 routing: top-k of the FP32 logits, ties to the lower expert index, then a
 *     softmax over the k selected logits (max-subtracted, summed in slot order).
 *  R2 exp: Cody-Waite range reduction (x = n ln2 + r) and the degree-7 Taylor
 *     polynomial of e^r in Horner form with fused multiply-adds; results below
 *     e^-86 flush to zero.  Both sides implement this same published method so
 *     routing weights can be compared bit for bit.
 *  R3 permutation: stable counting sort of expanded index t*k+j by expert.
 *  R4 NVFP4 scales: decode multiplier s = amax/(6*448) per tensor (s = 1 when
 *     amax = 0); block scale sf = e4m3_rn_satfinite(amax_16 / (6 s)); codes
 *     q = e2m1_rn_satfinite(x * (1 / (e4m3(sf) * s))), zero when that product
 *     is zero; the value decoded is e2m1(q) * e4m3(sf) * s.
 *  R5 e2m1 rounding: nearest grid value, ties to the even code, magnitudes
 *     above 6 saturate, a result of magnitude 0 is encoded +0.
 *  R6 SiLU-mul: h = g / (1 + e^-g) * u with gate rows [0, I) and up rows
 *     [I, 2I) of the gate_up output; requantised with a given static scale.
 *  R7 FINALIZE: out[t] = sum_j w[t,j] * Y[row(t,j)], rounded once to bf16.
 *  R8 router logits: a bias-free linear gate, logits[t][e] = sum_h x[t][h] *
 *     w_gate[e][h] over bf16 inputs, summed in FP64 and rounded once to FP32.
 *
 * Parity status: every exported function is pinned by tests/test_oracle_*.py
 * against closed forms, library routines or brute force.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* FP4 e2m1 and FP8 e4m3 decode, from the bit definitions.             */
/* ------------------------------------------------------------------ */

/* e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is subnormal: 0.5 * m.  Otherwise (1 + m/2) * 2^(e-1). */
EXPORT double orc_e2m1_decode(uint8_t code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
  return s ? -mag : mag;
}

/* e4m3 (the "fn" variant: no infinities): bit 7 sign, bits 6..3 exponent
 * (bias 7), bits 2..0 mantissa.  Exponent 0 is subnormal: m/8 * 2^-6.
 * Exponent 15 with mantissa 7 is NaN; everything else is finite, max 448. */
EXPORT double orc_e4m3_decode(uint8_t code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? (m / 8.0) * ldexp(1.0, -6) : (1.0 + m / 8.0) * ldexp(1.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest representable e4m3 magnitude, ties to the even code, values at or
 * above the largest finite (448) saturate to it (the scale's "satfinite").
 * Plain search over the 127 finite non-negative codes. */
EXPORT uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs(a - orc_e4m3_decode((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) { best = c; best_d = d; }
  }
  if (a >= 448.0) best = 0x7E;
  if (best == 0) return 0;            /* +0 for any result of magnitude 0 */
  return (uint8_t)(best | (neg << 7));
}

/* Nearest e2m1 grid value (R5): ties to the even code, magnitudes above 6
 * saturate to 6, magnitude-0 results are +0.  Plain search over codes 0..7. */
EXPORT uint8_t orc_e2m1_encode(float x) {
  int neg = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 7; ++c) {
    double d = fabs(a - orc_e2m1_decode((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) { best = c; best_d = d; }
  }
  if (a >= 6.0) best = 7;
  if (best == 0) return 0;
  return (uint8_t)(best | (neg << 3));
}

/* ------------------------------------------------------------------ */
/* NVFP4 quantisation (R4).  Linear layouts:                            */
/*   codes[r][K/2]: element 2i in the low nibble, 2i+1 in the high one; */
/*   sf[r][K/16]:   e4m3 scale of elements [16c, 16c+16).               */
/* ------------------------------------------------------------------ */

EXPORT float orc_tensor_scale_from_amax(float amax) {
  if (amax == 0.0f) return 1.0f;
  volatile float denom = 2688.0f; /* 6 * 448, exact */
  return amax / denom;
}

EXPORT float orc_amax(const float* x, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > m) m = a;
  }
  return m;
}

/* Quantise one 16-element block with decode multiplier s (FP32 throughout). */
static void quantize_block(const float* x, float s, uint8_t* codes8, uint8_t* sf) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
  volatile float six_s = 6.0f * s;
  volatile float sf_f = amax / six_s;
  uint8_t sfc = orc_e4m3_encode(sf_f);
  volatile float d = (float)orc_e4m3_decode(sfc) * s;
  uint8_t q[16];
  if (d == 0.0f) {
    memset(q, 0, sizeof q);
  } else {
    volatile float r = 1.0f / d;
    for (int i = 0; i < 16; ++i) { volatile float v = x[i] * r; q[i] = orc_e2m1_encode(v); }
  }
  for (int i = 0; i < 8; ++i) codes8[i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
  *sf = sfc;
}

EXPORT int orc_quantize(const float* x, int64_t rows, int K, float s, uint8_t* codes, uint8_t* sf) {
  if (K % 16) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int c = 0; c < K / 16; ++c)
      quantize_block(x + r * K + 16 * c, s, codes + r * (K / 2) + 8 * c, sf + r * (K / 16) + c);
  return 0;
}

/* Dequantise rows of an NVFP4 tensor (linear layouts) into FP64, without the
 * per-tensor multiplier. */
EXPORT void orc_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int K, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t q = (k & 1) ? (byte >> 4) : (byte & 15);
      out[r * K + k] = orc_e2m1_decode(q) * orc_e4m3_decode(sf[r * (K / 16) + k / 16]);
    }
}

/* ------------------------------------------------------------------ */
/* exp (R2): Cody-Waite reduction + degree-7 Taylor, all FP32.         */
/* ------------------------------------------------------------------ */

EXPORT float orc_exp(float x) {
  /* LN2_HI = ln 2 rounded to FP32; LN2_LO = (ln 2 - LN2_HI) rounded to FP32;
   * C[k] = 1/k! rounded to FP32. */
  const float LOG2E = 0x1.715476p+0f;
  const float LN2_HI = 0x1.62e43p-1f;
  const float LN2_LO = -0x1.05c61p-29f;
  const float C[8] = {0x1p+0f, 0x1p+0f, 0x1p-1f, 0x1.555556p-3f,
                      0x1.555556p-5f, 0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f};
  if (!(x >= -86.0f)) return 0.0f; /* also NaN -> 0 */
  if (x > 88.0f) return INFINITY;
  volatile float t = x * LOG2E;
  float n = rintf(t); /* round half to even */
  float r = fmaf(-n, LN2_HI, x);
  r = fmaf(-n, LN2_LO, r);
  float p = C[7];
  for (int k = 6; k >= 0; --k) p = fmaf(p, r, C[k]);
  /* p * 2^n, exact: n in [-125, 127] keeps the result normal. */
  union { uint32_t u; float f; } two_n;
  two_n.u = (uint32_t)((int)n + 127) << 23;
  volatile float res = p * two_n.f;
  return res;
}

/* ------------------------------------------------------------------ */
/* Router logits (R8).  "Tracing the Failure: Debugging CUTLASS FP4     */
/* Tile Configurations on Blackwell SM120", "The Broader Context":      */
/* each token is scored against every expert before the top-k.          */
/* ------------------------------------------------------------------ */

/* x: [T][H], w: [E][H] (the bf16 values, widened to float); out: [T][E]. */
EXPORT void orc_router_logits(const float* x, const float* w, int T, int E, int H, float* out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += (double)x[(int64_t)t * H + h] * (double)w[(int64_t)e * H + h];
      out[(int64_t)t * E + e] = (float)acc;
    }
}

/* ------------------------------------------------------------------ */
/* Routing (R1) and permutation (R3).                                  */
/* ------------------------------------------------------------------ */

EXPORT int orc_route(const float* logits, int T, int E, int k, int32_t* topk_id, float* topk_w) {
  if (k < 1 || k > E) return -1;
  char* taken = (char*)malloc((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: ties keep the lower index */
      }
      taken[best] = 1;
      topk_id[(int64_t)t * k + j] = best;
    }
    float m = l[topk_id[(int64_t)t * k]];
    float ex[1024];
    volatile float sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      volatile float d = l[topk_id[(int64_t)t * k + j]] - m;
      ex[j] = orc_exp(d);
      sum = sum + ex[j];
    }
    for (int j = 0; j < k; ++j) { volatile float w = ex[j] / sum; topk_w[(int64_t)t * k + j] = w; }
  }
  free(taken);
  return 0;
}

EXPORT int orc_permute(const int32_t* topk_id, int T, int k, int E, int32_t* expert_offsets,
                       int32_t* perm_to_expanded, int32_t* expanded_to_perm) {
  int64_t R = (int64_t)T * k;
  int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  for (int e = 0; e <= E; ++e) expert_offsets[e] = 0;
  for (int64_t i = 0; i < R; ++i) expert_offsets[topk_id[i] + 1] += 1;
  for (int e = 0; e < E; ++e) expert_offsets[e + 1] += expert_offsets[e];
  for (int64_t i = 0; i < R; ++i) {
    int e = topk_id[i];
    int64_t p = expert_offsets[e] + fill[e]++;
    perm_to_expanded[p] = (int32_t)i;
    expanded_to_perm[i] = (int32_t)p;
  }
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Grouped GEMM: for every expert e and each of its rows r,            */
/*   Y[r][n] = a_scale * b_scale[e] * sum_k dq(A[r][k]) * dq(B[e][n][k])*/
/* in FP64, rows grouped by expert_offsets (linear layouts).           */
/* ------------------------------------------------------------------ */

EXPORT int orc_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf, double a_scale,
                            const uint8_t* b_codes, const uint8_t* b_sf, const float* b_scale,
                            const int32_t* expert_offsets, int E, int N, int K, double* out) {
  if (K % 16) return -1;
  for (int e = 0; e < E; ++e) {
    int64_t r0 = expert_offsets[e], r1 = expert_offsets[e + 1];
    if (r1 <= r0) continue;
    double* A = (double*)malloc(sizeof(double) * (size_t)(r1 - r0) * K);
    double* B = (double*)malloc(sizeof(double) * (size_t)N * K);
    orc_dequantize(a_codes + r0 * (K / 2), a_sf + r0 * (K / 16), r1 - r0, K, A);
    orc_dequantize(b_codes + (int64_t)e * N * (K / 2), b_sf + (int64_t)e * N * (K / 16), N, K, B);
    double alpha = a_scale * (double)b_scale[e];
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < r1 - r0; ++r)
      for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += A[r * K + k] * B[(int64_t)n * K + k];
        out[(r0 + r) * N + n] = alpha * acc;
      }
    free(A);
    free(B);
  }
  return 0;
}

/* One output element of the grouped GEMM (for sampled checks at full size). */
EXPORT double orc_grouped_gemm_element(const uint8_t* a_row_codes, const uint8_t* a_row_sf, double a_scale,
                                       const uint8_t* b_row_codes, const uint8_t* b_row_sf, double b_scale,
                                       int K) {
  double acc = 0.0;
  for (int k = 0; k < K; ++k) {
    uint8_t qa = (k & 1) ? (a_row_codes[k / 2] >> 4) : (a_row_codes[k / 2] & 15);
    uint8_t qb = (k & 1) ? (b_row_codes[k / 2] >> 4) : (b_row_codes[k / 2] & 15);
    acc += orc_e2m1_decode(qa) * orc_e4m3_decode(a_row_sf[k / 16]) *
           orc_e2m1_decode(qb) * orc_e4m3_decode(b_row_sf[k / 16]);
  }
  return a_scale * b_scale * acc;
}

/* ------------------------------------------------------------------ */
/* SiLU-mul (R6), FINALIZE (R7), bf16 rounding.                         */
/* ------------------------------------------------------------------ */

EXPORT void orc_silu_mul(const double* y1, int64_t rows, int I, double* h) {
  for (int64_t r = 0; r < rows; ++r)
    for (int i = 0; i < I; ++i) {
      double g = y1[r * 2 * I + i], u = y1[r * 2 * I + I + i];
      h[r * I + i] = g / (1.0 + exp(-g)) * u;
    }
}

/* Round an FP64 value to bf16 (round to nearest, ties to even) via FP32.
 * The FP64 -> FP32 step can double-round only where the FP64 value sits within
 * 2^-29 relative of a bf16 tie, far below every tolerance that uses this. */
EXPORT uint16_t orc_bf16_bits(double v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

EXPORT double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

EXPORT void orc_finalize(const double* y, const float* topk_w, const int32_t* row_of_expanded, int T, int k,
                         int N, double* out) {
  for (int t = 0; t < T; ++t)
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        int64_t i = (int64_t)t * k + j;
        acc += (double)topk_w[i] * y[(int64_t)row_of_expanded[i] * N + n];
      }
      out[(int64_t)t * N + n] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* The pages' shared-memory model for one SM120 CUTLASS tile ("Cracking */
/* the SM120 Shared Memory Ceiling", "The Shared Memory Calculation"):  */
/* A M*K/2 + B K*N/2 + scales (M + N)*K/16 per stage, plus an epilogue  */
/* staging tile of M*N*2 bytes (NONE) or M*N*4 bytes (FINALIZE).        */
/* ------------------------------------------------------------------ */

EXPORT int64_t orc_smem_model_bytes(int M, int N, int K, int stages, int finalize) {
  int64_t per_stage = (int64_t)M * K / 2 + (int64_t)K * N / 2 + (int64_t)M * (K / 16) + (int64_t)(K / 16) * N;
  int64_t epi = (int64_t)M * N * (finalize ? 4 : 2);
  return per_stage * stages + epi;
}

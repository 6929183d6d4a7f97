/*
 * nvfp4_moe.h -- C ABI of the GB300 (sm_103a) NVFP4 Mixture-of-Experts layer.
 *
 * The layer, as the pages state the problem: E experts with top-k routing per
 * token, hidden size H and intermediate size I; FP4 e2m1 operands with one FP8
 * e4m3 scale per 16 elements along K plus one FP32 scale per tensor; BF16
 * output.  Per token: route to k experts, run each expert's gate_up GEMM,
 * SiLU-mul, requantise to NVFP4, run its down GEMM, and FINALIZE the k expert
 * rows back into the token's BF16 row with the router weights.
 *   - "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on
 *     Blackwell SM120", "The Broader Context": 256 experts, 8 per token,
 *     decode expert GEMMs of about 32x2048x6144.
 *   - same page, "Input Knowledge Required": one GEMM per expert inside one
 *     grouped launch, with a problem size per expert.
 *   - "Cracking the SM120 Shared Memory Ceiling: A Deep Dive into CUTLASS Tile
 *     Configuration Debugging", "The Shared Memory Calculation": FP4 packed at
 *     4 bits, one FP8 scale per 16 elements along K for both operands.
 *   - "The CUTLASS Tile That Wouldn't Fit: Debugging EP8 on Blackwell SM120",
 *     "The Crash": e2m1 x e2m1 -> bf16 grouped GEMM.
 *   - "The Epilogue That Broke the Kernel: Tracing a CUTLASS Tile
 *     Configuration Failure on Blackwell GPUs", "The Insight: FINALIZE vs
 *     NONE": epilogue NONE stores the GEMM result, FINALIZE does more.
 *
 * Conventions for every call below.
 *   - Every pointer argument is a DEVICE pointer unless its comment says host.
 *     The caller allocates and owns all memory; the library never allocates.
 *     Where scratch is needed the caller passes a workspace of at least the
 *     size the matching *_workspace_size() query returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream).  Calls return after enqueueing; results are ready when the
 *     stream reaches them.
 *   - Errors are returned, never thrown.  Argument checks happen on the host
 *     before anything is launched; a call that returns an error has enqueued
 *     nothing.  Device-side bounded waits that give up record MOE_ERR_TIMEOUT
 *     in a device error word that moe_device_error() reads.
 *   - Raw bf16 values are passed as uint16_t bit patterns.
 *
 * Data layouts.
 *   NVFP4 codes: uint8 [rows][K/2], row-major, element 2i in the low nibble
 *     and 2i+1 in the high nibble of byte i.
 *   Linear scales: uint8 (e4m3) [rows][K/16], row-major.
 *   Tiled scales (what the GEMM reads): rows in blocks of 128, scale columns
 *     c = k/16 in groups of 4; each (row block, column group) is a 512-byte
 *     atom, atoms ordered row-block-major; inside an atom the scale of (r, c)
 *     sits at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.  Requires
 *     K % 64 == 0 and a row allocation that is a multiple of 128.
 *   Routed rows ("padded rows"): the R = T*k (token, slot) pairs sorted stably
 *     by expert; expert e owns rows [P_e, P_e + M_e) where M_e is its count
 *     and P_e = sum over e' < e of ceil(M_e' / 128) * 128.  The rows between
 *     P_e + M_e and P_{e+1} are padding: never read into any result.
 *   Blocked weights (what the GEMM reads for the expert weights; written by
 *     nvfp4_quantize with MOE_SF_BLOCKED): the E*N weight rows (N % 128 == 0)
 *     in 128-row tiles and K in 256-element tiles; tile (row tile t, K tile
 *     kt) is one 18432-byte block at byte ((t * KT) + kt) * 18432 with
 *     KT = ceil(K / 256).  Inside a block: bytes [0, 16384) hold the codes of
 *     the 128 rows, row rr at rr * 128, its 16-byte chunk c (K elements
 *     kt*256 + 32c .. +32) stored at chunk position c XOR (rr % 8) (the
 *     128-byte swizzle); bytes [16384, 18432) hold the tile's scales as four
 *     512-byte atoms (one per 64 K-elements) with the atom layout above.
 *     Chunks and atoms past K (a partial last K tile) are never read.
 *   Prepared rows: for the gate_up weights (N = 2I) the rows are interleaved
 *     in blocks of 64: prepared row 128*b + j is gate row 64*b + j and
 *     prepared row 128*b + 64 + j is up row 64*b + j (j < 64).  The down
 *     weights keep their row order.
 */
#ifndef NVFP4_MOE_H
#define NVFP4_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, non-positive or inconsistent size, k > E, ... */
  MOE_ERR_MISALIGNED = 2,  /* a pointer is not 16-byte aligned (TMA and vector access need it) */
  MOE_ERR_UNSUPPORTED = 3, /* shape outside what the kernels implement (K % 64, N % 128, E > 1024, ...) */
  MOE_ERR_RESOURCE = 4,    /* the tile configuration does not fit shared or tensor memory */
  MOE_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed (launch, attribute, tensor map) */
  MOE_ERR_TIMEOUT = 6,     /* a device-side bounded wait gave up (see moe_device_error) */
  MOE_ERR_WORKSPACE = 7    /* workspace pointer null or smaller than the size query asks for */
} moe_status;

enum { MOE_SF_LINEAR = 0, MOE_SF_TILED = 1, MOE_SF_BLOCKED = 2 };
enum { MOE_IN_BF16 = 0, MOE_IN_F32 = 1 };
enum { MOE_EPI_NONE = 0, MOE_EPI_SILU_MUL_QUANT = 1, MOE_EPI_FINALIZE = 2 };

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(int status);

/* ABI version of this header; bumped on any incompatible change (3: FINALIZE workspace query takes k;
 * 4: moe_router takes x_scale; 5: moe_finalize takes y_rows; 6: the forward layout has small_scratch). */
MOE_API int moe_abi_version(void);

/* Reads and clears the device error word written by bounded waits that gave
 * up: *code receives a moe_status (MOE_OK if none), *where a kernel-specific
 * location tag.  Synchronises the device.  Host pointers. */
MOE_API moe_status moe_device_error(int32_t* code, int32_t* where);

/* Bound, in nanoseconds, of every device-side wait of the grouped GEMM
 * (default 2 s; 0 restores the default).  A wait that runs out records
 * MOE_ERR_TIMEOUT and its kernel returns early. */
MOE_API void moe_set_wait_timeout_ns(uint64_t ns);

/* Test hooks: bit 0 makes the next grouped-GEMM launches skip filling their
 * first pipeline stage (and moe_router's first CTA skip its first), so the
 * bounded-wait path can be exercised without faulting anything; bit 1 makes
 * them keep the one-CTA 128-row tile where the CTA-pair tile would run, so
 * both kernels can be compared on one input;
 * bit 2 makes moe_forward (and its graph) use the staged kernels for layers
 * the single-launch path would take.  0 (the default) for normal operation. */
MOE_API void moe_debug_set_flags(int flags);

/* Bytes of a blocked weight buffer of `rows` rows (rows % 128 == 0) and K
 * columns (K % 64 == 0); 0 if the shape is not supported. */
MOE_API size_t moe_blocked_weight_bytes(int64_t rows, int K);

/* Upper bound, for the caller's allocation, of the padded routed rows of R
 * routed rows over E experts: R + 127 * min(E, R), rounded up to 128. */
MOE_API int64_t moe_padded_rows_max(int64_t routed_rows, int E);

/* ---------------------------------------------------------------------------
 * moe_route_permute -- top-k routing and the stable permutation by expert.
 *   "Tracing the Failure ...", "The Broader Context" (top-k of E experts per
 *   token) and "Input Knowledge Required" (rows grouped per expert).
 * For each token t: the k experts of largest logit (ties to the lower expert
 * index), in descending order, and router weights w = softmax of the k
 * selected logits (max-subtracted, exponentials summed in slot order, all
 * FP32, exp by Cody-Waite reduction and a degree-7 Taylor polynomial).  Then
 * the expanded items i = t*k + j are sorted stably by expert.
 *   logits            f32 [T][E]
 *   topk_id           i32 [T][k]   out
 *   topk_w            f32 [T][k]   out
 *   expert_offsets    i32 [E+1]    out: start of expert e among the R sorted items
 *   perm_to_expanded  i32 [R]      out: item i stored at sorted position p
 *   expanded_to_perm  i32 [R]      out: inverse of perm_to_expanded
 *   expanded_to_row   i32 [R]      out: padded routed row of item i
 *                                       (P_e + expanded_to_perm[i] - expert_offsets[e])
 *   ws / ws_bytes     workspace of moe_route_permute_workspace_size(T, E, k) bytes
 * Requires 1 <= k <= min(E, 32), E <= 1024, T >= 1.  Deterministic.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_route_permute_workspace_size(int T, int E, int k);
MOE_API moe_status moe_route_permute(const float* logits, int T, int E, int k, int32_t* topk_id, float* topk_w,
                             int32_t* expert_offsets, int32_t* perm_to_expanded, int32_t* expanded_to_perm,
                             int32_t* expanded_to_row, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_route_permute_static -- moe_route_permute without a workspace argument,
 * for callers that cannot allocate device memory: code running where an
 * allocation is not allowed or would stall it (cudaMalloc may wait for the
 * whole device to go idle), or a host whose device memory is all owned by
 * another allocator.  The pages have no counterpart of this call; it exists
 * for such callers only.
 * Same arguments, results and requirements as moe_route_permute, minus
 * ws/ws_bytes.  Its scratch is one fixed array of
 * moe_route_permute_static_scratch_bytes() bytes (1 MiB) in the library's
 * device memory, reserved on every GPU that loads the library until the
 * process exits; a call whose moe_route_permute_workspace_size(T, E, k)
 * exceeds it returns MOE_ERR_WORKSPACE without launching anything (shapes
 * outside the limits below get MOE_ERR_UNSUPPORTED first, as from
 * moe_route_permute; the size is checked before the pointers).  The call
 * allocates nothing.  Every call looks up the array's device address in the
 * current device's context (cudaGetSymbolAddress, which allocates nothing),
 * so the address never outlives a context; the first call on a device may
 * load the library's device code, so make it before any stream capture.
 * Every call shares the one array, so calls that
 * can overlap on the GPU (different streams, or different host threads) race
 * and must be serialised by the caller.  Nothing in the array needs clearing
 * between calls: the kernels write every scratch word before they read it.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_route_permute_static_scratch_bytes(void);
MOE_API moe_status moe_route_permute_static(const float* logits, int T, int E, int k, int32_t* topk_id, float* topk_w,
                                    int32_t* expert_offsets, int32_t* perm_to_expanded, int32_t* expanded_to_perm,
                                    int32_t* expanded_to_row, void* stream);

/* ---------------------------------------------------------------------------
 * moe_router -- the router in front of moe_route_permute: the logits GEMM
 *   logits[t][e] = sum_h x[t][h] * w_gate[e][h]
 * on the tensor cores (bf16 inputs, FP32 sums) with the top-k and softmax of
 * every token in the same kernel, then the stable permutation of
 * moe_route_permute (its selection rule and weights, bit for bit, on these
 * logits).  Three kernels per call.
 *   "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on
 *   Blackwell SM120", "The Broader Context" (each token scored against 256
 *   experts, 8 kept).  The pages give no gate formula: this is a bias-free
 *   linear gate.
 * The K = H sum is split into contiguous ranges whose FP32 partial sums are
 * added in range order, so the logits (and everything routed from them) are
 * the same on every call with the same inputs on the same device; they differ
 * from a sequential sum only by FP32 rounding order.  The number of ranges
 * (up to 16) follows from T, H and how many CTA clusters the device holds; a
 * call made while its stream is being captured, before any other call on that
 * device, takes at most 8.
 * Arguments (device pointers unless noted):
 *   x        bf16 [T][H] (raw bits), 16-byte aligned
 *   w_gate   bf16 [E][H], 16-byte aligned
 *   logits   f32 [T][E] out, or NULL (not written: the partial sums are
 *            added inside the router kernel and never leave the GPU's shared
 *            memory)
 *   x_scale  f32 [1] out, or NULL: the NVFP4 decode multiplier of x,
 *            s = max|x| / (6*448) (1 when x is all zero), with max|x| taken
 *            by the logits GEMM from the x tiles it loads anyway -- what
 *            nvfp4_quantize would compute as its dynamic scale, so a caller
 *            can quantise x with that static scale and skip its amax pass
 *   topk_id ... expanded_to_row   as moe_route_permute
 *   ws / ws_bytes  workspace of moe_router_workspace_size(T, E, H, k) bytes,
 *                  queried with the device that will run the call current
 * Requires 1 <= k <= min(E, 32), E <= 256, H a multiple of 64, T >= 1.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_router_workspace_size(int T, int E, int H, int k);
MOE_API moe_status moe_router(const uint16_t* x, const uint16_t* w_gate, int T, int E, int H, int k, float* logits,
                              float* x_scale, int32_t* topk_id, float* topk_w, int32_t* expert_offsets,
                              int32_t* perm_to_expanded, int32_t* expanded_to_perm, int32_t* expanded_to_row,
                              void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * nvfp4_quantize -- NVFP4 quantisation of rows of a bf16 or f32 matrix.
 *   "Cracking the SM120 Shared Memory Ceiling ...", "The Shared Memory
 *   Calculation" (4-bit values, one FP8 scale per 16 elements along K).
 * Decode multiplier per group of rows: s = amax/(6*448) (1 when amax = 0),
 * computed here when dynamic_scale != 0 and written to tensor_scale[g], else
 * read from tensor_scale[g].  Per 16-element block: scale
 * sf = e4m3_rn_satfinite(amax_16 / (6*s)); d = e4m3(sf)*s; codes
 * q = e2m1_rn_satfinite(x * (1/d)) (ties to even, magnitude-0 results +0),
 * all zero when d == 0.  The represented value is e2m1(q)*e4m3(sf)*s.
 *   x             [src_rows][K], bf16 bits (in_dtype MOE_IN_BF16) or f32
 *   groups        src_rows is split into `groups` equal consecutive groups, each
 *                 with its own scale (1 for an activation tensor, E for weights)
 *   tensor_scale  f32 [groups]: in (static) or out (dynamic)
 *   n_items       number of output rows to write
 *   src_div       item i reads source row i / src_div (1 = row i); when
 *                 src_div > 1 every source row must be read by exactly
 *                 src_div items (n_items == src_rows * src_div, src_div <= 32):
 *                 each source row is quantised once and written to all of them
 *   dst_row       i32 [n_items] or NULL: item i is written to output row
 *                 dst_row[i] (NULL: row i)
 *   codes         u8 [dst_rows_alloc][K/2]           out
 *                 (MOE_SF_BLOCKED: the blocked weight buffer, codes and
 *                 scales together, moe_blocked_weight_bytes(dst_rows_alloc, K))
 *   sf            u8, linear [dst_rows_alloc][K/16] or tiled over
 *                 dst_rows_alloc rows (sf_layout); unused (may be NULL) for
 *                 MOE_SF_BLOCKED                     out
 *   ws / ws_bytes workspace of nvfp4_quantize_workspace_size(groups) bytes
 * Requires K % 16 == 0 (K % 64 == 0 and dst_rows_alloc % 128 == 0 for tiled
 * and blocked),
 * src_rows % groups == 0.  Rows of the output not named by any item are left
 * untouched.  Deterministic, bit-exact with the definition above.
 * ------------------------------------------------------------------------- */
MOE_API size_t nvfp4_quantize_workspace_size(int groups);
MOE_API moe_status nvfp4_quantize(const void* x, int in_dtype, int64_t src_rows, int K, int groups, float* tensor_scale,
                          int dynamic_scale, int64_t n_items, int src_div, const int32_t* dst_row,
                          uint8_t* codes, uint8_t* sf, int sf_layout, int64_t dst_rows_alloc, void* ws,
                          size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_grouped_gemm_nvfp4 -- the expert-grouped block-scaled FP4 GEMM.
 *   "Tracing the Failure ...", "Input Knowledge Required" (one GEMM per expert
 *   in one grouped launch); "The CUTLASS Tile That Wouldn't Fit ...", "The
 *   Crash" (e2m1 x e2m1 -> bf16); "The Epilogue That Broke the Kernel ...",
 *   "The Insight: FINALIZE vs NONE" (epilogues).
 * For expert e and each of its routed rows r (padded-row layout, counts from
 * expert_offsets):
 *   Y[r][n] = a_scale[0] * b_scale[e] * sum_k dq(A[r][k]) * dq(B[e][n][k])
 * with FP32 accumulation on the tensor cores.  Epilogues:
 *   MOE_EPI_NONE: out = bf16 [a_rows_alloc][N], Y rounded to nearest even;
 *     padding rows untouched.
 *   MOE_EPI_SILU_MUL_QUANT (gate_up; B prepared with interleaved gate/up rows,
 *     N = 2I): h[r][i] = silu(Y_gate) * Y_up in FP32, then NVFP4-quantised
 *     with the static decode multiplier ep->h_scale into ep->h_codes
 *     [a_rows_alloc][I/2] and tiled ep->h_sf; ep->h_scale_out (device f32,
 *     optional) receives h_scale; ep->h_f32 (optional) receives the FP32 h.
 *     `out` is unused.
 *   MOE_EPI_FINALIZE (down): out = bf16 [ep->T][N],
 *     out[t][n] = sum_j topk_w[t][j] * Y[row of item t*k+j][n], summed in FP32
 *     and rounded once.  The sum is FP32 atomics in the epilogue (the order
 *     of the k terms is not fixed) into a T*N*4-byte workspace; when that
 *     exceeds 64 MiB the kernel takes the weight tiles in column chunks of
 *     at most 64 MiB of accumulator, so the atomics stay in L2.  Only when one
 *     128-column chunk is already larger (T > 131072) does the epilogue store
 *     each item's weighted row (k*T*N*4 bytes) and a second kernel sum the k
 *     rows in slot order.
 * Arguments:
 *   a_codes/a_sf  activations, padded-row layout, tiled scales, a_rows_alloc rows
 *   a_scale       f32 [1] decode multiplier of A
 *   b_blocked     prepared expert weights, blocked layout over E*N rows
 *   b_scale       f32 [E]
 *   expert_offsets i32 [E+1] (as moe_route_permute writes them)
 *   ep            host pointer to epilogue arguments (NULL for NONE)
 *   ws / ws_bytes workspace of moe_grouped_gemm_workspace_size(epilogue, T, k, N)
 *                 bytes (FINALIZE only; 0 otherwise)
 * Tiling: weight rows are the MMA M dimension and routed rows MMA N.  In the
 * decode regime (the allocation implies <= 48 routed rows per expert on
 * average) one CTA per SM takes 128 weight rows x up to 64 routed rows per
 * unit.  Otherwise, where N % 256 == 0, two CTAs of a cluster take 256 weight
 * rows x up to 192 routed rows per unit with M = 256 (tcgen05 CTA-pair) MMAs
 * (for FINALIZE, when a 256-column accumulator chunk of T rows fits 64 MiB);
 * else one CTA takes 128 weight rows x up to 128 routed rows.
 * Requires K % 64 == 0, N % 128 == 0,
 * E <= 1024, a_rows_alloc % 128 == 0, all pointers 16-byte aligned.
 * Device-side errors (read with moe_device_error): expert offsets that would
 * place a tile before row 0, past the a_rows_alloc rows or (FINALIZE) outside
 * the T*k routed items stop the launch with MOE_ERR_INVALID_ARG; other
 * inconsistent offsets give an undefined output without any access outside
 * the operands.  A wait past the bound set by moe_set_wait_timeout_ns reports
 * MOE_ERR_TIMEOUT.
 * ------------------------------------------------------------------------- */
typedef struct {
  /* MOE_EPI_SILU_MUL_QUANT */
  float h_scale;
  float* h_scale_out;
  uint8_t* h_codes;
  uint8_t* h_sf;
  float* h_f32;
  /* MOE_EPI_FINALIZE */
  const int32_t* perm_to_expanded;
  const float* topk_w;
  int32_t T;
  int32_t k;
} moe_epilogue_args;

MOE_API size_t moe_grouped_gemm_workspace_size(int epilogue, int T, int k, int N);
MOE_API moe_status moe_grouped_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                  const uint8_t* b_blocked, const float* b_scale,
                                  const int32_t* expert_offsets, int E, int64_t a_rows_alloc, int N, int K,
                                  int epilogue, const moe_epilogue_args* ep, void* out, void* ws, size_t ws_bytes,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * moe_finalize -- standalone FINALIZE: the router-weighted sum of each
 * token's k expert rows back into one BF16 row.
 *   "The Epilogue That Broke the Kernel ...", "The Insight: FINALIZE vs NONE";
 *   "Cracking the SM120 Shared Memory Ceiling ...", "The Shared Memory
 *   Calculation" (FP32 accumulator, BF16 output).
 *   out[t][n] = bf16_rn( sum_{j<k} topk_w[t][j] * y[row_of_item[t*k+j]][n] ),
 *   summed in FP32 in slot order (deterministic).
 *   y            bf16 [y_rows][N]
 *   topk_w       f32 [T][k]
 *   row_of_item  i32 [T*k]: the row of y holding item t*k+j (expanded_to_perm
 *                for an unpadded y, expanded_to_row for a padded one)
 *   out          bf16 [T][N]
 * Requires N % 8 == 0, y_rows >= 1.  A row_of_item entry outside [0, y_rows)
 * is not read: its term is left out and MOE_ERR_INVALID_ARG is recorded in the
 * device error word (moe_device_error, location 8).
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_finalize(const uint16_t* y, int64_t y_rows, const float* topk_w, const int32_t* row_of_item,
                                int T, int k, int N, uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * moe_fp4_mma_probe -- measurement aid: enqueues one launch that issues
 * `iters` back-to-back dense NVFP4 MMAs (the grouped GEMM's instruction,
 * M = 128, N = 256, K = 64, operands in shared memory, no global-memory
 * traffic) on each of `blocks` CTAs (0 = one per SM).  The caller times the
 * launch on `stream`; *flops_per_launch (host) receives the FLOPs it performs.
 * iters is at most 1,000,000 and at most one per 200 ns of the wait bound
 * (moe_set_wait_timeout_ns), so the launch's final wait cannot run out while
 * MMAs are still in flight; larger values return MOE_ERR_INVALID_ARG.
 * Gives the dense FP4 tensor rate the prefill roofline is measured against.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_fp4_mma_probe(int iters, int blocks, double* flops_per_launch, void* stream);

/* moe_fp4_mma_probe_pair -- the same measurement for the CTA-pair MMA form
 * (tcgen05 cta_group::2): `pairs` clusters of two CTAs (0 = as many as can be
 * resident at once), one thread of each pair issuing `iters` M = 256, N = 256,
 * K = 64 MMAs whose operand halves sit in the two CTAs' shared memory.  Same
 * limits on iters as moe_fp4_mma_probe; *flops_per_launch (host) receives the
 * FLOPs one launch performs. */
MOE_API moe_status moe_fp4_mma_probe_pair(int iters, int pairs, double* flops_per_launch, void* stream);

/* ---------------------------------------------------------------------------
 * moe_forward -- the fused MoE layer: route + permute, quantise x into the
 * routed rows, gate_up GEMM with SiLU-mul + requantise epilogue, down GEMM
 * with FINALIZE epilogue.  Same definitions as the calls above.
 *   x        bf16 [T][H]
 *   logits   f32 [T][E]
 *   w        host pointer to the prepared expert weights
 *   h_scale  static decode multiplier of the requantised intermediate (host value)
 *   out      bf16 [T][H]
 *   ws       workspace of moe_forward_workspace_size(T, E, k, H, I) bytes; its
 *            layout (moe_forward_workspace_layout) exposes the intermediates.
 * Requires H % 128 == 0, I % 64 == 0, plus the requirements above.
 * ------------------------------------------------------------------------- */
typedef struct {
  const uint8_t* w13;       /* blocked, E*2I rows x H, gate/up interleaved */
  const float* w13_scale;   /* [E] */
  const uint8_t* w2;        /* blocked, E*H rows x I */
  const float* w2_scale;    /* [E] */
} moe_weights;

/* Byte offsets of each intermediate inside the moe_forward workspace. */
typedef struct {
  size_t topk_id, topk_w, expert_offsets, perm_to_expanded, expanded_to_perm, expanded_to_row;
  size_t x_scale, x_codes, x_sf, h_scale, h_codes, h_sf, route_ws, quant_ws, gemm_ws;
  size_t small_scratch; /* 256 bytes reserved for the single-launch path; (size_t)-1 for layers it does not take */
  int64_t padded_rows; /* rows allocated for the routed-row buffers */
  size_t total;
} moe_forward_layout;

/* Small layers (T * k <= 64, E <= 64, H <= 1024, I <= 512, E * I <= 4096, and
 * no gate matrix) run as ONE kernel ("Tracing the Failure ...", "Conclusion":
 * persistent kernel designs against per-kernel overheads): one cluster of 16
 * CTAs (8 where 16 cannot be placed).  Every CTA routes every token itself and
 * takes x's amax itself; gate_up, SiLU-mul and the requantisation of h are
 * dealt out in (expert, 32 h columns) units; after the cluster barrier each CTA
 * runs down for its share of the output columns over every routed row and sums
 * each token's k slots in slot order into `out`.  Every intermediate of the
 * layout is written as the staged kernels write it: the routing and
 * permutation and the quantised x are the same bits, and h and out differ only
 * by the order of the FP32 sums in the contractions.  No state carries from one
 * launch to the next.
 * moe_forward_kernel_count: kernels one moe_forward call (or one replay of its
 * graph) launches for this shape, 0 for an invalid shape. */
MOE_API int moe_forward_kernel_count(int T, int E, int k, int H, int I);

MOE_API size_t moe_forward_workspace_size(int T, int E, int k, int H, int I);
MOE_API moe_status moe_forward_workspace_layout(int T, int E, int k, int H, int I, moe_forward_layout* layout);
MOE_API moe_status moe_forward(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k, int H,
                       int I, float h_scale, uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_forward_gated -- moe_forward with the router in front: the logits come
 * from moe_router (x . w_gate^T on the tensor cores), and the activation
 * quantiser takes x's decode multiplier from the router's logits GEMM, which
 * reads every element of x anyway, instead of a separate amax pass.
 * Same arguments as moe_forward with w_gate (bf16 [E][H], device, 16-byte
 * aligned) in place of the logits; requires E <= 256; ws_bytes >=
 * moe_forward_gated_workspace_size(...), whose first
 * moe_forward_workspace_size(...) bytes follow moe_forward_workspace_layout.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_forward_gated_workspace_size(int T, int E, int k, int H, int I);
MOE_API moe_status moe_forward_gated(const uint16_t* x, const uint16_t* w_gate, const moe_weights* w, int T, int E,
                                     int k, int H, int I, float h_scale, uint16_t* out, void* ws, size_t ws_bytes,
                                     void* stream);

/* ---------------------------------------------------------------------------
 * moe_forward_graph_* -- the whole layer as one CUDA graph.
 *   "Tracing the Failure ...", "Conclusion" names persistent kernel designs as
 *   the way past per-kernel overheads; "The Epilogue That Broke the Kernel
 *   ...", "The Broader Significance" names piecewise CUDA graphs.
 * moe_forward_graph_create checks its arguments like moe_forward, runs the
 * layer once eagerly (which computes `out` and prepares every kernel), then
 * captures moe_forward's launches into an executable graph.  The graph keeps
 * every pointer it was created with: refill x and logits in place and
 * relaunch; the workspace, weights and out must stay valid and must not be
 * used by anything else while a launch of the graph may run.  With
 * stage_events != 0 the graph records timing events between the four stages
 * (route+permute, quantise x, gate_up GEMM, down GEMM + FINALIZE), every step
 * in series; moe_forward_graph_stage_ms waits for the last launch and writes
 * the five durations in ms (the four stages, then the whole layer) to ms[5]
 * (host).  With stage_events == 0 two steps run on side branches of the graph:
 * the activation amax pass beside the routing, and the clearing of the
 * FINALIZE accumulator beside the gate_up GEMM.  The results are the same.
 * Creation makes CUDA objects (streams, events, the executable graph) but no
 * device buffers; destroy releases them.  *graph (host) receives the handle.
 * ------------------------------------------------------------------------- */
typedef struct moe_forward_graph moe_forward_graph;
MOE_API moe_status moe_forward_graph_create(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E,
                                    int k, int H, int I, float h_scale, uint16_t* out, void* ws, size_t ws_bytes,
                                    int stage_events, moe_forward_graph** graph);
MOE_API moe_status moe_forward_graph_launch(moe_forward_graph* graph, void* stream);
MOE_API moe_status moe_forward_graph_stage_ms(moe_forward_graph* graph, float* ms);

/* moe_forward_graph_run_host -- one step of the layer from and to HOST memory:
 * copies x_host (bf16 [T][H]) and logits_host (f32 [T][E]) into the device
 * buffers the graph was created with, replays the graph, and copies its output
 * into out_host (bf16 [T][H]), all enqueued on `stream` (asynchronous: the host
 * buffers must stay valid and unmodified until the stream reaches the end of
 * the call; page-locked buffers let the copies overlap other streams' work).
 * Two graphs, each with its own x, logits, out and workspace, can run steps
 * on two streams so that one step's copies overlap the other's layer. */
MOE_API moe_status moe_forward_graph_run_host(moe_forward_graph* graph, const uint16_t* x_host, const float* logits_host,
                                              uint16_t* out_host, void* stream);
MOE_API void moe_forward_graph_destroy(moe_forward_graph* graph);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_MOE_H */

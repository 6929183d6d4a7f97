// grouped_gemm.cu -- the expert-grouped NVFP4 GEMM on the 5th-generation
// tensor cores (tcgen05, kind::mxf4nvf4, e2m1 x e2m1 with ue4m3 scales per 16
// K-elements, FP32 accumulation in tensor memory).
//
// What it computes: "Tracing the Failure: Debugging CUTLASS FP4 Tile
// Configurations on Blackwell SM120", section "Input Knowledge Required" (one
// GEMM per expert inside a single grouped launch, one problem size per
// expert); "The CUTLASS Tile That Wouldn't Fit: Debugging EP8 on Blackwell
// SM120", section "The Crash" (e2m1 x e2m1 -> bf16); epilogues NONE and
// FINALIZE from "The Epilogue That Broke the Kernel: Tracing a CUTLASS Tile
// Configuration Failure on Blackwell GPUs", section "The Insight: FINALIZE vs
// NONE", plus the gate_up epilogue (SiLU-mul and NVFP4 requantisation).
//
// Design (GB300, one CTA per SM, persistent):
//   * Operand roles are swapped relative to the row-major problem: the 128
//     weight rows of a tile are the MMA M dimension and the expert's routed
//     rows (up to BN) are MMA N.  At decode an expert sees 4-64 rows, so every
//     weight tile is streamed from HBM once per BN routed rows and the tensor
//     core never computes padding rows of M.
//   * The routed-row tile BN is picked per launch from the rows-per-expert
//     regime: BN = 64 with 7 pipeline stages for decode, BN = 128 with 5
//     stages when experts see more rows (prefill).
//   * Work unit = (expert, BN-row block of its routed rows, 128-row weight
//     tile), full K.  Units are ordered expert-major so the CTAs running
//     together share each expert's token tile in L2.  CTA c takes units c,
//     c + grid, ...  A FINALIZE launch whose FP32 accumulator would not fit
//     in L2 walks the weight tiles in column chunks (every expert's units of
//     one chunk, then the next), so its atomics keep hitting L2.
//   * Weights are prepared in a blocked layout: per 128 rows x 256 K-elements
//     one contiguous 18 KB block holding the 128-byte-swizzled code tile (the
//     exact shared-memory image the MMA descriptor reads) and its four scale
//     atoms, so each pipeline stage of weights is ONE linear bulk copy that
//     streams a contiguous 18 KB run of HBM.
//   * Warp roles: warp 0 issues the copies (weights: bulk copy, evict-first;
//     routed rows: 2D tensor-map loads with 128-byte swizzle and a bulk copy
//     of their scale atoms, evict-last).  With one epilogue group warps 10-12
//     issue copies too, each one stage fill in four: one issuing thread gets
//     its bulk copies served one after another.  Warps 6-9 move each stage's
//     scale atoms from shared into tensor memory (tcgen05.st, one warp per lane
//     quadrant) and hand the MMA thread each unit's MMA N and scale column
//     offset with the unit's first stage.  Warp 1 owns tensor memory and
//     issues only the tcgen05.mma instructions and their commits; warps 2-5
//     drain the accumulator (tcgen05.ld) and run the epilogue.  A FINALIZE
//     launch at the 128-row tile has warps 10-13 as a second epilogue group
//     that drains every other unit, since one group could not keep up with
//     its atomics there.  A tcgen05.cp of the scales on the MMA thread would
//     serialise with the MMA that reads them: at decode that halved the
//     weight-streaming rate.  Several TMEM
//     accumulators (four for the 64-row tile, two for the 128-row one) let the
//     epilogue of one unit overlap the mainloops of the next ones; every
//     stage has its own TMEM scale slot, recycled by the same commit that
//     frees the stage.
//   * Every wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT in the
//     device error word, lets its own copies and MMAs finish, frees its tensor
//     memory and returns.
#include "common.cuh"

namespace moe {
moe_status launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t st);
moe_status launch_finalize_sum(const float* rows, int T, int k, int N, uint16_t* out, cudaStream_t st);

// FINALIZE accumulates with atomics into a [T][N] FP32 buffer.  The atomics stay
// in L2 while the part of that buffer being written fits comfortably there: the
// kernel walks the weight tiles in column chunks of `mt_chunk` 128-row tiles (all
// experts' units of one chunk before the next chunk), so the live part is
// T x 128*mt_chunk floats.  Returns the largest chunk (a divisor of N/128) whose
// live part is at most kFinalizeAtomicMaxBytes, or 0 when not even one tile
// column fits; the epilogue then stores each expanded item's weighted row and a
// second kernel sums the k rows of every token (deterministically, in slot order).
constexpr int64_t kFinalizeAtomicMaxBytes = 64ll << 20;
inline int finalize_mt_chunk(int T, int N) {
  const int MT = N / 128;
  for (int c = MT; c >= 1; --c)
    if (MT % c == 0 && static_cast<int64_t>(T) * c * 128 * 4 <= kFinalizeAtomicMaxBytes) return c;
  return 0;
}
inline bool finalize_gathers(int T, int N) { return finalize_mt_chunk(T, N) == 0; }

namespace {

constexpr int kBM = 128;                  // weight rows per tile (MMA M)
constexpr int kBK = 256;                  // K elements per stage (128 bytes per row)
constexpr int kWStageBytes = kBlockedTileBytes;  // 16 KB codes + 2 KB scale atoms
constexpr int kSfStageBytes = 4 * 512;    // scale atoms of the routed rows (one per 64-element K step)
constexpr int kExtraWarp = 10;           // warps 0-9: copies, MMA, epilogue 2-5, scale staging 6-9; then extras
constexpr int kMaxExperts = 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfSlotCols = 32;      // 16 columns weight scales + 16 columns routed-row scales
constexpr int kEpiStride = 130;           // floats per staged routed row (128 tile rows + 2: fewer bank conflicts)

// EG = epilogue warp groups.  With one group, four copy-issuing warps (0,
// 10-12) keep more bulk copies in flight.  Two groups are for a FINALIZE launch
// whose epilogue is slower than its mainloop (128 routed rows: short K = I
// units, an atomic per 4 outputs): warps 10-13 form a second group that takes
// every other unit, so two accumulators drain at once.  That configuration
// serves FINALIZE only, which needs no staging tile, and keeps one copy warp.
template <int BN, int EG>
struct Cfg {
  static constexpr int kEpiGroups = EG;
  static constexpr int kProducers = EG == 1 ? 4 : 1;
  static constexpr int kThreads = 32 * (kExtraWarp + (kProducers - 1) + 4 * (kEpiGroups - 1));
  static constexpr bool kFinalizeOnly = EG == 2;
  static constexpr int kStages = BN == 64 ? 7 : 5;
  static constexpr int kXStageBytes = BN * kBK / 2;
  static constexpr uint32_t kAccCols = BN;
  // Accumulator buffers: the epilogue of a unit may lag the mainloop by kAccBufs - 1 units
  // (decode units are short, so the 64-row tile keeps four).
  static constexpr int kAccBufs = BN == 64 ? 4 : 2;
  static constexpr uint32_t kSfTmemBase = kAccBufs * BN;
  static_assert(kSfTmemBase + kStages * kSfSlotCols <= kTmemCols, "tensor memory budget");
  // A producer waits on a stage's `empty` barrier by phase parity, so that barrier
  // must never be two phases behind the fill being waited for.  The producer's
  // previous fill (kProducers back) could only start once fill - kProducers - kStages
  // had been consumed; with kProducers <= kStages that covers fill - 2 * kStages.
  static_assert(kStages >= kProducers, "more producers than stages would alias barrier phases");
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int w = 0;
  static constexpr int x = w + kStages * kWStageBytes;
  static constexpr int sfx = x + kStages * kXStageBytes;
  static constexpr int epi = sfx + kStages * kSfStageBytes;  // float [32][kEpiStride] (SiLU staging tile)
  static constexpr int tok_t = epi + (kFinalizeOnly ? 0 : 32 * kEpiStride * 4);  // int [2][BN] (FINALIZE tables)
  static constexpr int tok_w = tok_t + 2 * BN * 4;           // float [2][BN]
  static constexpr int bars = tok_w + 2 * BN * 4;            // uint64 [3*kStages + 2*kAccBufs + 1]
  static constexpr int misc = bars + (3 * kStages + 2 * kAccBufs + 1) * 8;  // tmem base, abort flag
  static constexpr int last = misc + 16;                     // int [kProducers][kStages]
  static constexpr int info = last + kProducers * kStages * 4;  // int [kStages]: MMA N and scale column offset
  static constexpr int sched = info + kStages * 4;           // int [3][kMaxExperts+1]
  static constexpr int total = sched + 3 * (kMaxExperts + 1) * 4;
  static constexpr int smem_bytes = total + 1024;            // + alignment slack
  static_assert(smem_bytes <= 232448, "shared memory budget");
  static_assert(x % 1024 == 0 && kXStageBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct GemmParams {
  const uint8_t* w_blocked;   // prepared weights, blocked layout over E*N rows
  const uint8_t* x_sf;        // tiled scales of the routed rows
  const float* x_scale;       // [1]
  const float* w_scale;       // [E]
  const int32_t* expert_offsets;
  int E, N, K;
  int epilogue;
  void* out;                  // NONE: bf16 [rows][N]; FINALIZE: f32 [T][N] accumulator or [T*k][N] rows
  float h_scale;
  float* h_scale_out;
  uint8_t* h_codes;
  uint8_t* h_sf;
  float* h_f32;
  const int32_t* perm_to_expanded;
  const float* topk_w;
  int k;
  int T;
  int fin_gather;             // FINALIZE: 1 = store weighted rows per expanded item (summed later), 0 = atomics
  int mt_chunk;               // weight tiles per column chunk of the unit order (N/128 = one chunk)
  int64_t rows_alloc;         // rows of the routed-row operand (bounds every access to it)
  int64_t items;              // FINALIZE: T * k, the length of perm_to_expanded; otherwise unbounded
  int32_t* err;
  uint64_t timeout_ns;
  int debug_flags;            // bit 0: the producer skips the first stage (bounded-wait test hook)
};

struct Unit {
  int e, nb, nbe, mt, rows, n_mma, x_row, m_off;
  bool valid;  // false when the offsets place the unit outside the operands (the launch then stops)
};

// The expert owning unit u (start[e] <= u < start[e + 1]), searched from `e`, an
// expert at or before the owner: every role walks its units in increasing order,
// so the search gallops forward from the previous owner instead of bisecting all
// E experts.
MOE_DEVINL int find_expert_from(const int* start, int E, int u, int e) {
  int lo = e, step = 1, hi = e + 1;
  while (hi < E && start[hi] <= u) {
    lo = hi;
    step <<= 1;
    hi = lo + step;
  }
  if (hi > E) hi = E;  // start[E] = total units > u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// Unit u -> (column chunk c, expert e, weight tile mt, routed-row block nb):
// U units per chunk, ordered expert-major; inside an expert, weight tile by
// weight tile, with the expert's nbe routed-row blocks of one weight tile on
// consecutive units.  Consecutive units run on different CTAs at about the same
// time, so when a busy expert has several routed-row blocks, the CTAs reading
// one weight tile for its different blocks run together and share it in L2
// (the first read brings it from HBM).
template <int BN>
MOE_DEVINL Unit decode_unit(int u, const int* unit_start, const int* pad_start, const int* off, int E, int MTC, int U,
                            int64_t rows_alloc, int64_t items, int& e_hint) {
  Unit d;
  const int c = u / U;
  const int uc = u - c * U;
  if (unit_start[e_hint] > uc) e_hint = 0;  // a new column chunk starts over at expert 0
  d.e = e_hint = find_expert_from(unit_start, E, uc, e_hint);
  const int local = uc - unit_start[d.e];
  d.nbe = (unit_start[d.e + 1] - unit_start[d.e]) / MTC;
  const int mtl = local / d.nbe;
  d.nb = local - mtl * d.nbe;
  d.mt = c * MTC + mtl;
  const int m_e = off[d.e + 1] - off[d.e];
  d.rows = min(BN, m_e - d.nb * BN);
  d.n_mma = d.rows <= 32 ? 32 : (d.rows <= 64 ? 64 : 128);
  if (d.n_mma > BN) d.n_mma = BN;
  d.x_row = pad_start[d.e] + d.nb * BN;
  d.m_off = off[d.e] + d.nb * BN;
  // offsets as the routing writes them always pass; corrupted ones (decreasing,
  // negative, past the allocation or the item count) stop the launch instead of
  // reaching memory outside the operands
  d.valid = d.rows > 0 && d.x_row >= 0 && static_cast<int64_t>(d.x_row) + BN <= rows_alloc && d.m_off >= 0 &&
            static_cast<int64_t>(d.m_off) + d.rows <= items;
  return d;
}

// Named barrier 1 over the 128 epilogue threads.
// Named barrier over the 128 threads of epilogue group g (ids 1 and 3; 2 is the producers').
MOE_DEVINL void epi_bar(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + 2 * g) : "memory"); }

// True on every thread of epilogue group g if `pred` holds on any of them
// (that group's named barrier with an OR reduction).
MOE_DEVINL bool epi_any(int g, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(1 + 2 * g)
      : "memory");
  return r != 0;
}


// ---- epilogue bodies of one 32-column accumulator chunk (shared by both kernels) ----
// r: the chunk as loaded by tcgen05.ld (this thread's weight row, 32 routed rows);
// jn: routed rows of the chunk that exist.

// NONE: out[row0 + jj][col] = bf16(alpha * acc).
MOE_DEVINL void epi_chunk_none(const uint32_t (&r)[32], int jn, int64_t row0, int64_t col, int N, float alpha,
                               uint16_t* out) {
#pragma unroll
  for (int jj = 0; jj < 32; ++jj)
    if (jj < jn) out[(row0 + jj) * N + col] = float_to_bf16_bits(alpha * __uint_as_float(r[jj]));
}

// FINALIZE: 4x4 transposes inside each lane quad (two shuffle rounds) give lane
// 4g+i the four consecutive output columns 32q+4g .. +3 of routed rows i, i+4,
// ..., i+28 of the chunk: one 16-byte vector atomic (or store) per 4 outputs, a
// warp covering four 128-byte runs per instruction, with no shared-memory round
// trip or barrier.  acc_col: the accumulator at column (tile column + 32q +
// 4(lane/4)); tok/w: destination row and weight x alpha per routed row of the chunk.
MOE_DEVINL void epi_chunk_finalize(uint32_t (&r)[32], int lane, int jn, const int* tok, const float* w, float* acc_col,
                                   int N, bool gather) {
  const bool b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
#pragma unroll
  for (int sb = 0; sb < 8; ++sb) {
    float a0 = __uint_as_float(r[4 * sb]), a1 = __uint_as_float(r[4 * sb + 1]);
    float a2 = __uint_as_float(r[4 * sb + 2]), a3 = __uint_as_float(r[4 * sb + 3]);
    // rows {0,1} x cols {2,3} <-> rows {2,3} x cols {0,1}
    float t0 = __shfl_xor_sync(0xffffffffu, b1 ? a0 : a2, 2);
    float t1 = __shfl_xor_sync(0xffffffffu, b1 ? a1 : a3, 2);
    if (b1) { a0 = t0; a1 = t1; } else { a2 = t0; a3 = t1; }
    // then within each 2x2 block
    t0 = __shfl_xor_sync(0xffffffffu, b0 ? a0 : a1, 1);
    t1 = __shfl_xor_sync(0xffffffffu, b0 ? a2 : a3, 1);
    if (b0) { a0 = t0; a2 = t1; } else { a1 = t0; a3 = t1; }
    r[4 * sb] = __float_as_uint(a0);
    r[4 * sb + 1] = __float_as_uint(a1);
    r[4 * sb + 2] = __float_as_uint(a2);
    r[4 * sb + 3] = __float_as_uint(a3);
  }
#pragma unroll
  for (int sb = 0; sb < 8; ++sb) {
    const int jj = 4 * sb + (lane & 3);
    if (jj < jn) {
      const int t = tok[jj];
      if (t >= 0) {
        const float wt = w[jj];
        const float4 v = make_float4(wt * __uint_as_float(r[4 * sb]), wt * __uint_as_float(r[4 * sb + 1]),
                                     wt * __uint_as_float(r[4 * sb + 2]), wt * __uint_as_float(r[4 * sb + 3]));
        float4* dst = reinterpret_cast<float4*>(acc_col + static_cast<int64_t>(t) * N);
        if (gather)
          *dst = v;
        else
          atomicAdd(dst, v);
      }
    }
  }
}

// SILU_MUL_QUANT on a gate_up tile whose rows 0-63 are gate rows and rows
// 64-127 the matching up rows: the chunk (128 tile rows x 32 routed rows) is
// staged in shared memory, then each of the group's 128 threads (et) takes one
// routed row and one 16-wide block of the 64 outputs, so an NVFP4 block (amax,
// scale, codes) lives in one thread's registers.  row0: routed row of the
// chunk's first column; i_tile: the tile's first output column (64 per tile).
struct SiluOut {
  float h_scale;
  uint8_t* h_codes;
  uint8_t* h_sf;
  float* h_f32;
  int I;
};
MOE_DEVINL void epi_chunk_silu(const uint32_t (&r)[32], int m, int et, int eg, int jn, float alpha, float* s_epi_g,
                               int64_t row0, int i_tile, const SiluOut& o) {
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) s_epi_g[jj * kEpiStride + m] = alpha * __uint_as_float(r[jj]);
  epi_bar(eg);
  const int jj = et >> 2, blk = et & 3;
  if (jj < jn) {
    const float* gp = s_epi_g + jj * kEpiStride + 16 * blk;
    float h[16];
    float amax = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const float g = gp[t];
      h[t] = silu_mul(g, gp[64 + t]);
      amax = fmaxf(amax, fabsf(h[t]));
    }
    float recip;
    const uint32_t sfb = nvfp4_block_scale(amax, o.h_scale, &recip);
    const uint32_t lo = nvfp4_codes8(h, recip), hi = nvfp4_codes8(h + 8, recip);
    const int64_t row = row0 + jj;
    const int i0 = i_tile + 16 * blk;
    *reinterpret_cast<uint2*>(o.h_codes + row * (o.I / 2) + i0 / 2) = make_uint2(lo, hi);
    o.h_sf[tiled_sf_offset(row, i0 / 16, o.I)] = static_cast<uint8_t>(sfb);
    if (o.h_f32) {
      float4* dst = reinterpret_cast<float4*>(o.h_f32 + row * o.I + i0);
#pragma unroll
      for (int t = 0; t < 4; ++t) dst[t] = make_float4(h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]);
    }
  }
  epi_bar(eg);
}

template <int BN, int EG>
__global__ void __launch_bounds__(Cfg<BN, EG>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xt,
                        const GemmParams p) {
  using C = Cfg<BN, EG>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_w = smem + C::w;
  uint8_t* s_x = smem + C::x;
  uint8_t* s_sfx = smem + C::sfx;
  float* s_epi = reinterpret_cast<float*>(smem + C::epi);
  int* s_tok_t = reinterpret_cast<int*>(smem + C::tok_t);
  float* s_tok_w = reinterpret_cast<float*>(smem + C::tok_w);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* empty = full + S;
  uint64_t* sf_ready = empty + S;
  uint64_t* acc_full = sf_ready + S;
  uint64_t* acc_empty = acc_full + C::kAccBufs;
  uint64_t* mma_done = acc_empty + C::kAccBufs;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::misc + 4);
  int* s_info = reinterpret_cast<int*>(smem + C::info);
  int* unit_start = reinterpret_cast<int*>(smem + C::sched);
  int* pad_start = unit_start + (kMaxExperts + 1);
  int* off = pad_start + (kMaxExperts + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, N = p.N, K = p.K;
  if (C::kFinalizeOnly && p.epilogue != MOE_EPI_FINALIZE) {  // the host never launches this; no smem tile for it
    if (threadIdx.x == 0) record_error(p.err, MOE_ERR_INVALID_ARG, 9);
    return;
  }
  const int MT = N / kBM;
  const int MTC = p.mt_chunk;
  const int KT = (K + kBK - 1) / kBK;

  // ---- prologue: barriers, tensor memory, work list --------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); mbar_init(&sf_ready[s], 4); }
    for (int b = 0; b < C::kAccBufs; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 128); }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0) {
    // unit_start[e]: first unit of expert e; pad_start[e]: first padded row (128-row padding).
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int units = 0, pads = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int m = __ldg(p.expert_offsets + e + 1) - __ldg(p.expert_offsets + e);
      units += ((m + BN - 1) / BN) * MTC;
      pads += ((m + 127) / 128) * 128;
    }
    int iu = units, ip = pads;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yu = __shfl_up_sync(0xffffffffu, iu, o), yp = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) { iu += yu; ip += yp; }
    }
    int ru = iu - units, rp = ip - pads;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int o0 = __ldg(p.expert_offsets + e), o1 = __ldg(p.expert_offsets + e + 1);
      unit_start[e] = ru;
      pad_start[e] = rp;
      off[e] = o0;
      ru += ((o1 - o0 + BN - 1) / BN) * MTC;
      rp += ((o1 - o0 + 127) / 128) * 128;
    }
    if (lane == 31) {
      unit_start[E] = iu;
      pad_start[E] = ip;
      off[E] = __ldg(p.expert_offsets + E);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int U = unit_start[E];
  const int total_units = U * (MT / MTC);

  if (warp == 0 || (C::kProducers > 1 && warp >= kExtraWarp)) {
    // ---------------- producers ----------------
    // Stage fill i (counted over this CTA's units and K steps) is issued by
    // producer i % kProducers: bulk copies from one issuing thread are served
    // one after another, so several issuing warps keep more of them in flight
    // (the weight and token tiles of a compute-bound unit are mostly L2 hits).
    constexpr int kProducers = C::kProducers;
    const int pid = warp == 0 ? 0 : warp - kExtraWarp + 1;
    int* s_last = reinterpret_cast<int*>(smem + C::last);  // [kProducers][S] last fill index per stage
    if (lane == 0) {
      // a weight tile with one reader (an expert with one routed-row block) at
      // evict-first; one that the expert's other blocks read at the same time
      // at normal priority, so those reads hit L2
      const uint64_t pol_w1 = l2_policy_evict_first(), pol_wn = l2_policy_evict_normal();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int fill = 0;
      for (int s = 0; s < S; ++s) s_last[pid * S + s] = -1;
      bool skip_once = pid == 0 && (p.debug_flags & 1) != 0;
      int e_hint = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit d = decode_unit<BN>(u, unit_start, pad_start, off, E, MTC, U, p.rows_alloc, p.items, e_hint);
        if (!d.valid) {  // offsets that place a unit outside the routed-row allocation: stop the launch
          if (!*s_abort) record_error(p.err, MOE_ERR_INVALID_ARG, 5);
          *s_abort = 1;
          break;
        }
        const uint8_t* w_src = p.w_blocked + static_cast<int64_t>(d.e * MT + d.mt) * KT * kWStageBytes;
        const uint8_t* sfx_src = p.x_sf + static_cast<int64_t>(d.x_row / 128) * (K / 64) * 512;
        const uint64_t pol_w = d.nbe > 1 ? pol_wn : pol_w1;
        for (int kt = 0; kt < KT; ++kt, ++fill) {
          if (fill % kProducers == pid) {
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, p.timeout_ns, s_abort)) {
              if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 1);
              *s_abort = 1;
              ok = false;
              break;
            }
            const int steps = min(4, (K - kt * kBK) / 64);
            if (skip_once) {
              skip_once = false;  // test hook: this stage is never filled
            } else {
              const uint32_t bytes = kWStageBytes + d.n_mma * (kBK / 2) + steps * 512;
              mbar_arrive_expect_tx(&full[stage], bytes);
              bulk_load(s_w + stage * kWStageBytes, w_src + static_cast<int64_t>(kt) * kWStageBytes, kWStageBytes,
                        &full[stage], pol_w);
              if (d.n_mma == BN) {
                // a full tile: one box of BN rows (tm_xt)
                tma_load_2d(s_x + stage * C::kXStageBytes, &tm_xt, &full[stage], kt * (kBK / 2), d.x_row, pol_x);
              } else {
                for (int q = 0; q < d.n_mma / 32; ++q)
                  tma_load_2d(s_x + stage * C::kXStageBytes + q * 32 * (kBK / 2), &tm_x, &full[stage],
                              kt * (kBK / 2), d.x_row + 32 * q, pol_x);
              }
              bulk_load(s_sfx + stage * kSfStageBytes, sfx_src + kt * 4 * 512, steps * 512, &full[stage], pol_x);
              s_last[pid * S + stage] = fill;
            }
          }
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
    }
    // Let every copy this CTA started land before the CTA can exit: once all
    // producers are past their loops, wait for the last fill of every stage
    // (an earlier fill of a stage has landed before a later one can start).
    __syncwarp();
    asm volatile("bar.sync 2, %0;" ::"r"(kProducers * 32) : "memory");
    if (pid == 0 && lane == 0) {
      int zero = 0;
      for (int s = 0; s < S; ++s) {
        int last = -1;
        for (int q = 0; q < kProducers; ++q) last = max(last, s_last[q * S + s]);
        if (last >= 0)
          mbar_wait_bounded(&full[s], static_cast<uint32_t>(last / S) & 1u, p.timeout_ns,
                            reinterpret_cast<volatile int*>(&zero));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool ok = true;
      // Every instruction on this thread delays the next MMA issue, and at a
      // 128-row tile the tensor core finishes an MMA about as fast as one is
      // issued: descriptors are precomputed, the four MMAs of a stage unrolled,
      // and one barrier wait covers two stages (the staging warps complete the
      // stages in order, so the later stage being ready implies the earlier).
      const uint64_t adesc0 = smem_desc(smem_u32(s_w), 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_u32(s_x), 16, 1024, 2);
      // The unit's MMA N and scale column offset come from the staging warps with
      // the unit's first stage (s_info): decoding the unit here would put a chain
      // of dependent shared-memory loads on this thread once per unit.
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++acc_i) {
        const int b = acc_i % C::kAccBufs;
        if (!mbar_wait_bounded(&acc_empty[b], ((acc_i / C::kAccBufs) & 1) ^ 1u, p.timeout_ns, s_abort)) {
          if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 2);
          *s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * C::kAccCols;
        uint32_t idesc = 0, sfx_col_off = 0;
        for (int kt = 0; kt < KT; ++kt) {
          if ((kt & 1) == 0) {
            // sf_ready implies full: the staging warps saw the stage's copies land.
            int ws = stage;
            uint32_t wph = phase;
            if (kt + 1 < KT && ++ws == S) { ws = 0; wph ^= 1u; }
            if (!mbar_wait_bounded(&sf_ready[ws], wph, p.timeout_ns, s_abort)) {
              if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 3);
              *s_abort = 1;
              ok = false;
              break;
            }
            tc_fence_after();
            if (kt == 0) {
              const int info = s_info[stage];
              idesc = idesc_mxf4nvf4(info & 0xFFFF);
              sfx_col_off = static_cast<uint32_t>(info >> 16);
            }
          }
          const uint32_t sf_col = tmem_base + C::kSfTmemBase + stage * kSfSlotCols;
          // start-address field of the descriptors: byte address / 16
          const uint64_t adesc = adesc0 + static_cast<uint64_t>((stage * kWStageBytes) >> 4);
          const uint64_t bdesc = bdesc0 + static_cast<uint64_t>((stage * C::kXStageBytes) >> 4);
          if (kt * kBK + kBK <= K) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              mma_mxf4nvf4(d_tmem, adesc + 2 * g, bdesc + 2 * g, idesc, sf_col + 4 * g,
                           sf_col + 16 + 4 * g + sfx_col_off, (kt | g) != 0);
          } else {
            const int steps = (K - kt * kBK) / 64;
            for (int g = 0; g < steps; ++g)
              mma_mxf4nvf4(d_tmem, adesc + 2 * g, bdesc + 2 * g, idesc, sf_col + 4 * g,
                           sf_col + 16 + 4 * g + sfx_col_off, (kt | g) != 0);
          }
          mma_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[b]);
      }
      // Every MMA and scale copy this thread issued has completed once this arrives.
      mma_commit(mma_done);
      int zero = 0;
      mbar_wait_bounded(mma_done, 0, p.timeout_ns, reinterpret_cast<volatile int*>(&zero));
    }
  } else if (warp >= 6 && warp < kExtraWarp) {
    // ---------------- scale staging warps 6..9 ----------------
    // The block-scaled MMA reads its scales from tensor memory.  Each of these
    // warps (one per TMEM lane quadrant) writes the stage's 32 scale columns
    // into its quadrant: columns 0-15 the weight atoms of the 4 K steps,
    // columns 16-31 the routed-row atoms, each atom's 32 rows of 16 bytes in
    // lanes 0-31 of every quadrant.  Keeping these stores off the MMA thread
    // leaves it nothing to issue but the MMAs themselves.
    const uint32_t quad_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    int stage = 0;
    uint32_t phase = 0;
    int e_hint = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const Unit d = decode_unit<BN>(u, unit_start, pad_start, off, E, MTC, U, p.rows_alloc, p.items, e_hint);
      if (!d.valid) {
        if (lane == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_INVALID_ARG, 5);
          *s_abort = 1;
        }
        break;
      }
      for (int kt = 0; kt < KT; ++kt) {
        const bool got = mbar_wait_bounded(&full[stage], phase, p.timeout_ns, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) {
            if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 7);
            *s_abort = 1;
          }
          ok = false;
          break;
        }
        const uint8_t* sfw = s_w + stage * kWStageBytes + 16384 + lane * 16;
        const uint8_t* sfx = s_sfx + stage * kSfStageBytes + lane * 16;
        uint32_t v[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 a = *reinterpret_cast<const uint4*>(sfw + 512 * g);
          const uint4 b = *reinterpret_cast<const uint4*>(sfx + 512 * g);
          v[4 * g] = a.x; v[4 * g + 1] = a.y; v[4 * g + 2] = a.z; v[4 * g + 3] = a.w;
          v[16 + 4 * g] = b.x; v[16 + 4 * g + 1] = b.y; v[16 + 4 * g + 2] = b.z; v[16 + 4 * g + 3] = b.w;
        }
        tmem_st_32cols(tmem_base + quad_lane + C::kSfTmemBase + stage * kSfSlotCols, v);
        tmem_st_wait();
        tc_fence_before();
        // the unit's MMA N and the routed rows' scale column offset within each atom
        // ((x_row % 128) / 32) for the MMA thread, published with the unit's first stage
        if (kt == 0 && warp == 6 && lane == 0) s_info[stage] = d.n_mma | (((d.x_row & 127) >> 5) << 16);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[stage]);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    const int m = 32 * q + lane;       // weight row of the tile owned by this thread
    const int eg = warp >= kExtraWarp ? 1 : 0;                          // epilogue group
    const int et = eg ? threadIdx.x - 32 * kExtraWarp : threadIdx.x - 64;  // 0..127 within the group
    float* s_epi_g = s_epi;  // only the one-group configuration stages tiles (SiLU)
    const float x_scale = __ldg(p.x_scale);
    if (p.epilogue == MOE_EPI_SILU_MUL_QUANT && p.h_scale_out && blockIdx.x == 0 && eg == 0 && et == 0)
      *p.h_scale_out = p.h_scale;
    int acc_i = 0;
    int e_hint = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++acc_i) {
      const Unit d = decode_unit<BN>(u, unit_start, pad_start, off, E, MTC, U, p.rows_alloc, p.items, e_hint);
      if (!d.valid) {
        if (et == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_INVALID_ARG, 5);
          *s_abort = 1;
        }
        break;
      }
      if (acc_i % C::kEpiGroups != eg) continue;  // the other group drains this unit
      const int b = acc_i % C::kAccBufs;
      const float alpha = x_scale * __ldg(p.w_scale + d.e);
      int* tok_tab = s_tok_t + (acc_i & 1) * BN;
      float* w_tab = s_tok_w + (acc_i & 1) * BN;
      if (p.epilogue == MOE_EPI_FINALIZE) {
        // Token table of this unit: routed row et -> destination row (token, or
        // expanded item when gathering) and router weight x alpha, built before the
        // accumulator wait so that its dependent global loads overlap the mainloop.
        // With one group it is double-buffered (the barrier after the previous
        // unit's table orders the reads of this buffer two units back before this
        // write); with two, each group's buffer is released by the barrier that
        // ends the group's previous unit.
        if (et < d.rows) {
          const int ex = __ldg(p.perm_to_expanded + d.m_off + et);
          const bool in_range = ex >= 0 && ex < p.T * p.k;
          if (!in_range) record_error(p.err, MOE_ERR_INVALID_ARG, 6);
          tok_tab[et] = in_range ? (p.fin_gather ? ex : ex / p.k) : -1;
          w_tab[et] = in_range ? __ldg(p.topk_w + ex) * alpha : 0.0f;
        }
      }
      const bool got = mbar_wait_bounded(&acc_full[b], (acc_i / C::kAccBufs) & 1, p.timeout_ns, s_abort);
      // The four warps of the group decide together, so none is left waiting on a
      // named barrier that the others have abandoned; the barrier also publishes
      // the token table to the group.
      if (epi_any(eg, !got)) {
        if (et == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 4);
          *s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * C::kAccCols;
      const SiluOut so{p.h_scale, p.h_codes, p.h_sf, p.h_f32, N / 2};
      for (int j0 = 0; j0 < d.rows; j0 += 32) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + j0, r);
        tmem_ld_wait();
        const int jn = min(32, d.rows - j0);
        if (p.epilogue == MOE_EPI_NONE) {
          epi_chunk_none(r, jn, d.x_row + j0, static_cast<int64_t>(d.mt) * kBM + m, N, alpha,
                         static_cast<uint16_t*>(p.out));
        } else if (p.epilogue == MOE_EPI_FINALIZE) {
          epi_chunk_finalize(r, lane, jn, tok_tab + j0, w_tab + j0,
                             static_cast<float*>(p.out) + static_cast<int64_t>(d.mt) * kBM + 32 * q + 4 * (lane >> 2),
                             N, p.fin_gather != 0);
        } else {
          epi_chunk_silu(r, m, et, eg, jn, alpha, s_epi_g, d.x_row + j0, d.mt * 64, so);
        }
      }
      // with two groups, this group's next unit rewrites the same token table
      if (C::kEpiGroups > 1 && p.epilogue == MOE_EPI_FINALIZE) epi_bar(eg);
      tc_fence_before();
      mbar_arrive(&acc_empty[b]);
    }
  }
  // (control reaches here on every path)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ===========================================================================
// CTA-pair kernel (prefill regime): tcgen05 cta_group::2.
//
// Two CTAs of a cluster form a pair that computes one unit = (expert, up to
// 192 of its routed rows, 256 weight rows) with M = 256 MMAs: CTA r holds
// weight tile 2*mt2 + r (128 rows, MMA M half r) and routed rows [n/2*r,
// n/2*(r+1)) of the unit (MMA N half r); one thread of the even CTA issues
// the MMAs, which read both CTAs' shared memory and write each CTA's
// accumulator rows into its own tensor memory.  Per SM this doubles the work
// of one MMA instruction (128 x 192 x 64 against 128 x 128 x 64 for the
// one-CTA tile) and brings the bytes each SM moves from L2 per FLOP to 0.6 of
// the one-CTA tile's: a 34 KB stage feeds 12.6 MFLOP per SM where the
// one-CTA tile's 37 KB stage fed 8.4.
// Tensor memory of each CTA: two 192-column accumulators (the epilogue of one
// unit overlaps the mainloop of the next) and three 40-column scale slots, 504
// of the 512 columns.  The MMA reads weight row r's scales from lane r % 128
// only (column scale address + r / 32), but every lane quadrant of the
// accumulator reads the scales of every routed row: those sit in all four
// quadrants (column scale address + n / 32 holds routed rows 32c..32c+31 in
// lanes 0-31 of each quadrant).  A slot: 16 columns of weight scales (4 per K
// step) and 24 of routed-row scales (6 per K step, 192 rows).  A slot is
// reused three fills later, once the MMAs of that fill have completed (the
// empty barrier of its stage); the MMA thread waits for each stage's scales on
// its own, so two stages stay queued in the tensor pipe while the slot of the
// next one is refilled.
// Roles per CTA: warps 0 and 10-11 (10-12) issue copies (each CTA its own halves),
// warp 1 owns tensor memory (in the even CTA its lane 0 issues the MMAs),
// two sets of four warps (6-9 and the CTA's last four) take alternate stage
// fills, stage their scales into their own CTA's tensor memory and tell the
// even CTA, warps 2-5 (and 12-15) drain the accumulator and run the epilogue.
// Signals between the CTAs: the MMA thread's commits arrive on both CTAs'
// stage-empty and accumulator-full barriers (one multicast commit each); the
// staging and epilogue warps of both CTAs arrive on the even CTA's
// scales-ready and accumulator-empty barriers.
// ===========================================================================
constexpr int kPairBN = 192;               // routed rows per pair unit (MMA N)
constexpr int kPairStages = 6;
constexpr int kPairMaxExperts = 512;       // larger launches take the one-CTA kernel
constexpr int kPairEpiRows = 16;           // routed rows per SiLU staging round
constexpr int kPairSlots = 3;              // tensor-memory scale slots
constexpr uint32_t kPairSlotCols = 40;     // 16 weight-scale + 24 routed-row-scale columns

// EG = epilogue warp groups.  With two groups, three copy warps (0, 10, 11) keep
// the CTA at 20 warps; with one, four copy warps (0, 10-12) make 17.
template <int EG>
struct PairCfg {
  static constexpr int kProducers = EG == 2 ? 3 : 4;
  static constexpr int kThreads = 32 * (kExtraWarp + (kProducers - 1) + 4 * (EG - 1) + 4);
  static constexpr int kEpi1Warp = kExtraWarp + kProducers - 1;  // first warp of epilogue group 1
  static constexpr int kStage1Warp = kEpi1Warp + 4 * (EG - 1);   // first warp of the second staging set
  static constexpr int kXStageBytes = (kPairBN / 2) * (kBK / 2);  // this CTA's half of the routed rows
  static constexpr int kSfxStageBytes = 2 * kSfStageBytes;        // scales of up to two 128-row blocks
  static constexpr int kAccBufs = 2;
  static constexpr uint32_t kSfTmemBase = kAccBufs * kPairBN;
  static_assert(kSfTmemBase + kPairSlots * kPairSlotCols <= kTmemCols, "tensor memory budget");
  static_assert(kPairStages >= kProducers, "more producers than stages would alias barrier phases");
  static constexpr int w = 0;
  static constexpr int x = w + kPairStages * kWStageBytes;
  static constexpr int sfx = x + kPairStages * kXStageBytes;
  // SiLU staging, float [EG][kPairEpiRows][kEpiStride]; a FINALIZE launch (which stages nothing) keeps
  // its token tables in the same bytes: int [EG][2][kPairBN] then float [EG][2][kPairBN]
  static constexpr int epi = sfx + kPairStages * kSfxStageBytes;
  static constexpr int epi_bytes = EG * kPairEpiRows * kEpiStride * 4;
  static constexpr int tok_t = epi;
  static constexpr int tok_w = tok_t + EG * 2 * kPairBN * 4;
  static_assert(EG * 2 * kPairBN * 8 <= epi_bytes, "token tables fit the staging bytes");
  static constexpr int bars = epi + epi_bytes;                         // uint64 [3*S + 2*kAccBufs + 1]
  static constexpr int misc = bars + (3 * kPairStages + 2 * kAccBufs + 1) * 8;
  static constexpr int last = misc + 16;                               // int [kProducers][S]
  static constexpr int info = last + kProducers * kPairStages * 4;     // int [S]
  static constexpr int sched = info + kPairStages * 4;                 // int [2][kPairMaxExperts+1]
  static constexpr int total = sched + 2 * (kPairMaxExperts + 1) * 4;
  static constexpr int smem_bytes = total + 1024;
  static_assert(smem_bytes <= 232448, "shared memory budget");
  static_assert(x % 1024 == 0 && kXStageBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct PairUnit {
  int e, nb, mt2, rows, n_mma, x_row, m_off;
  bool valid;
};

// Pair unit u -> (column chunk, expert e, weight tile pair mt2, 192-row block nb);
// the same order as decode_unit with MTC weight tile pairs per chunk.
MOE_DEVINL PairUnit decode_pair_unit(int u, const int* unit_start, const int* pad_start, const int32_t* off, int E,
                                     int MTC, int U, int64_t rows_alloc, int64_t items, int& e_hint) {
  PairUnit d;
  const int c = u / U;
  const int uc = u - c * U;
  if (unit_start[e_hint] > uc) e_hint = 0;
  d.e = e_hint = find_expert_from(unit_start, E, uc, e_hint);
  const int local = uc - unit_start[d.e];
  const int nbe = (unit_start[d.e + 1] - unit_start[d.e]) / MTC;
  const int mtl = local / nbe;
  d.nb = local - mtl * nbe;
  d.mt2 = c * MTC + mtl;
  const int o0 = __ldg(off + d.e);  // expert offsets straight from global memory (L1-cached)
  const int m_e = __ldg(off + d.e + 1) - o0;
  d.rows = min(kPairBN, m_e - d.nb * kPairBN);
  d.n_mma = (d.rows + 31) & ~31;
  d.x_row = pad_start[d.e] + d.nb * kPairBN;
  d.m_off = o0 + d.nb * kPairBN;
  d.valid = d.rows > 0 && d.x_row >= 0 && static_cast<int64_t>(d.x_row) + d.n_mma <= rows_alloc && d.m_off >= 0 &&
            static_cast<int64_t>(d.m_off) + d.rows <= items;
  return d;
}

// epi_chunk_silu through a 16-row staging buffer: the chunk's 32 routed rows in
// two rounds of 16 (threads et < 64 compute in each round).
MOE_DEVINL void epi_chunk_silu16(const uint32_t (&r)[32], int m, int et, int eg, int jn, float alpha, float* s_epi_g,
                                 int64_t row0, int i_tile, const SiluOut& o) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) s_epi_g[jj * kEpiStride + m] = alpha * __uint_as_float(r[16 * half + jj]);
    epi_bar(eg);
    const int jj = et >> 2, blk = et & 3;
    if (et < 64 && 16 * half + jj < jn) {
      const float* gp = s_epi_g + jj * kEpiStride + 16 * blk;
      float h[16];
      float amax = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float g = gp[t];
        h[t] = silu_mul(g, gp[64 + t]);
        amax = fmaxf(amax, fabsf(h[t]));
      }
      float recip;
      const uint32_t sfb = nvfp4_block_scale(amax, o.h_scale, &recip);
      const uint32_t lo = nvfp4_codes8(h, recip), hi = nvfp4_codes8(h + 8, recip);
      const int64_t row = row0 + 16 * half + jj;
      const int i0 = i_tile + 16 * blk;
      *reinterpret_cast<uint2*>(o.h_codes + row * (o.I / 2) + i0 / 2) = make_uint2(lo, hi);
      o.h_sf[tiled_sf_offset(row, i0 / 16, o.I)] = static_cast<uint8_t>(sfb);
      if (o.h_f32) {
        float4* dst = reinterpret_cast<float4*>(o.h_f32 + row * o.I + i0);
#pragma unroll
        for (int t = 0; t < 4; ++t) dst[t] = make_float4(h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]);
      }
    }
    epi_bar(eg);
  }
}

template <int EG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<EG>::kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_x16, const __grid_constant__ CUtensorMap tm_x96,
                             const GemmParams p) {
  using C = PairCfg<EG>;
  constexpr int S = kPairStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_w = smem + C::w;
  uint8_t* s_x = smem + C::x;
  uint8_t* s_sfx = smem + C::sfx;
  float* s_epi = reinterpret_cast<float*>(smem + C::epi);
  int* s_tok_t = reinterpret_cast<int*>(smem + C::tok_t);
  float* s_tok_w = reinterpret_cast<float*>(smem + C::tok_w);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* empty = full + S;
  uint64_t* sf_ready = empty + S;
  uint64_t* acc_full = sf_ready + S;
  uint64_t* acc_empty = acc_full + C::kAccBufs;
  uint64_t* mma_done = acc_empty + C::kAccBufs;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::misc + 4);
  int* s_info = reinterpret_cast<int*>(smem + C::info);
  int* unit_start = reinterpret_cast<int*>(smem + C::sched);
  int* pad_start = unit_start + (kPairMaxExperts + 1);
  const int32_t* off = p.expert_offsets;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x()), npairs = static_cast<int>(cluster_count_x());
  const int E = p.E, N = p.N, K = p.K;
  const int MT = N / kBM;
  const int MTC = p.mt_chunk;  // weight tile pairs per column chunk
  const int KT = (K + kBK - 1) / kBK;

  // ---- prologue ----------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); mbar_init(&sf_ready[s], 8); }
    for (int b = 0; b < C::kAccBufs; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 8); }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {  // the pair's tensor memory: one warp of each CTA allocates together
    tmem_alloc_pair(s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int units = 0, pads = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int m = __ldg(p.expert_offsets + e + 1) - __ldg(p.expert_offsets + e);
      units += ((m + kPairBN - 1) / kPairBN) * MTC;
      pads += ((m + 127) / 128) * 128;
    }
    int iu = units, ip = pads;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yu = __shfl_up_sync(0xffffffffu, iu, o), yp = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) { iu += yu; ip += yp; }
    }
    int ru = iu - units, rp = ip - pads;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int o0 = __ldg(p.expert_offsets + e), o1 = __ldg(p.expert_offsets + e + 1);
      unit_start[e] = ru;
      pad_start[e] = rp;
      ru += ((o1 - o0 + kPairBN - 1) / kPairBN) * MTC;
      rp += ((o1 - o0 + 127) / 128) * 128;
    }
    if (lane == 31) {
      unit_start[E] = iu;
      pad_start[E] = ip;
    }
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs: barriers initialised, tensor memory allocated, schedule built
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int U = unit_start[E];
  const int total_units = U * ((MT / 2) / MTC);

  if (warp == 0 || (warp >= kExtraWarp && warp < kExtraWarp + C::kProducers - 1)) {
    // ---------------- producers (each CTA loads its own halves) ----------------
    const int pid = warp == 0 ? 0 : warp - kExtraWarp + 1;
    int* s_last = reinterpret_cast<int*>(smem + C::last);
    if (lane == 0) {
      // Each weight tile pair is read by the pairs working on the expert's other routed-row
      // blocks at about the same time, so weights stay in L2 at normal priority (measured:
      // gate_up 1.66 -> 1.63 ms at 16384 tokens), except under FINALIZE, whose FP32 atomics need
      // L2 for the live accumulator chunk (there evict-first measured faster, 1.52 -> 1.50 ms);
      // routed rows, read once per weight tile pair, at evict-last.
      const uint64_t pol_w = p.epilogue == MOE_EPI_FINALIZE ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int fill = 0;
      for (int s = 0; s < S; ++s) s_last[pid * S + s] = -1;
      bool skip_once = pid == 0 && (p.debug_flags & 1) != 0;
      int e_hint = 0;
      bool ok = true;
      for (int u = pair; ok && u < total_units; u += npairs) {
        const PairUnit d = decode_pair_unit(u, unit_start, pad_start, off, E, MTC, U, p.rows_alloc, p.items, e_hint);
        if (!d.valid) {
          if (!*s_abort) record_error(p.err, MOE_ERR_INVALID_ARG, 5);
          *s_abort = 1;
          break;
        }
        const int mt = 2 * d.mt2 + static_cast<int>(rank);
        const uint8_t* w_src = p.w_blocked + static_cast<int64_t>(d.e * MT + mt) * KT * kWStageBytes;
        const int half = d.n_mma / 2;
        const int xr = d.x_row + static_cast<int>(rank) * half;
        const int b0 = d.x_row >> 7, b1 = (d.x_row + d.n_mma - 1) >> 7;
        const uint8_t* sf0 = p.x_sf + static_cast<int64_t>(b0) * (K / 64) * 512;
        for (int kt = 0; kt < KT; ++kt, ++fill) {
          if (fill % C::kProducers == pid) {
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, p.timeout_ns, s_abort)) {
              if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 11);
              *s_abort = 1;
              ok = false;
              break;
            }
            const int steps = min(4, (K - kt * kBK) / 64);
            if (skip_once) {
              skip_once = false;
            } else {
              const uint32_t bytes = kWStageBytes + half * (kBK / 2) + (b1 > b0 ? 2 : 1) * steps * 512;
              mbar_arrive_expect_tx(&full[stage], bytes);
              bulk_load(s_w + stage * kWStageBytes, w_src + static_cast<int64_t>(kt) * kWStageBytes, kWStageBytes,
                        &full[stage], pol_w);
              uint8_t* xdst = s_x + stage * C::kXStageBytes;
              if (half == kPairBN / 2) {
                tma_load_2d(xdst, &tm_x96, &full[stage], kt * (kBK / 2), xr, pol_x);
              } else {
                for (int q = 0; q < half / 16; ++q)
                  tma_load_2d(xdst + q * 16 * (kBK / 2), &tm_x16, &full[stage], kt * (kBK / 2), xr + 16 * q, pol_x);
              }
              uint8_t* sdst = s_sfx + stage * C::kSfxStageBytes;
              bulk_load(sdst, sf0 + kt * 4 * 512, steps * 512, &full[stage], pol_x);
              if (b1 > b0)
                bulk_load(sdst + kSfStageBytes, sf0 + static_cast<int64_t>(K / 64) * 512 + kt * 4 * 512, steps * 512,
                          &full[stage], pol_x);
              s_last[pid * S + stage] = fill;
            }
          }
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
    }
    __syncwarp();
    asm volatile("bar.sync 2, %0;" ::"r"(C::kProducers * 32) : "memory");
    if (pid == 0 && lane == 0) {
      int zero = 0;
      for (int s = 0; s < S; ++s) {
        int last = -1;
        for (int q = 0; q < C::kProducers; ++q) last = max(last, s_last[q * S + s]);
        if (last >= 0)
          mbar_wait_bounded(&full[s], static_cast<uint32_t>(last / S) & 1u, p.timeout_ns,
                            reinterpret_cast<volatile int*>(&zero));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA, one thread) ----------------
    // This one thread issues every MMA of the pair.  The tensor core queues only a
    // stage's last MMA or two, so whatever this thread does between the last MMA of
    // one stage and the first of the next leaves the tensor core idle: the next
    // stage's bookkeeping and a non-blocking check of its scales-ready barrier are
    // done between this stage's MMA issues (where the thread waits for queue room
    // anyway), leaving only the commit and a fence in the gap.  Descriptors move as
    // 32-bit low halves (the high halves are fixed for the kernel).
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool ok = true;
      const uint64_t adesc0 = smem_desc(smem_u32(s_w), 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_u32(s_x), 16, 1024, 2);
      const uint32_t a_lo0 = static_cast<uint32_t>(adesc0), a_hi = static_cast<uint32_t>(adesc0 >> 32);
      const uint32_t b_lo0 = static_cast<uint32_t>(bdesc0), b_hi = static_cast<uint32_t>(bdesc0 >> 32);
      constexpr uint32_t kAStep = kWStageBytes >> 4, kBStep = C::kXStageBytes >> 4;  // descriptor units per stage
      uint32_t a_lo = a_lo0, b_lo = b_lo0;
      const uint32_t sf_base = tmem_base + C::kSfTmemBase;
      const uint32_t sf_last = sf_base + (kPairSlots - 1) * kPairSlotCols;
      uint32_t sfc = sf_base;
      const int KF = K / kBK;                      // full 256-element K stages
      const int k_tail = (K - KF * kBK) / 64;      // MMAs of a partial last stage (0-3)
      const int n_st = KF + (k_tail > 0 ? 1 : 0);
      for (int u = pair; ok && u < total_units; u += npairs, ++acc_i) {
        const int b = acc_i % C::kAccBufs;
        if (!mbar_wait_bounded(&acc_empty[b], ((acc_i / C::kAccBufs) & 1) ^ 1u, p.timeout_ns, s_abort)) {
          if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 12);
          *s_abort = 1;
          break;
        }
        const uint32_t d_tmem = tmem_base + b * kPairBN;
        // first stage of the unit (starts the accumulator), and a unit of one partial stage
        if (!mbar_spin_bounded(&sf_ready[stage], phase, p.timeout_ns, s_abort)) {
          if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 13);
          *s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_mxf4nvf4(s_info[stage], 256);
        int kt = 0;
        bool next_ready = false;  // the next stage's scales-ready phase already seen complete
        while (true) {
          // stage kt's scales are ready (and fenced); issue its MMAs
          const int n = kt < KF ? 4 : k_tail;
          const uint32_t a_n = a_lo + kAStep, b_n = b_lo + kBStep;  // next stage's values, worked out in the
          const int st_n = stage + 1 == S ? 0 : stage + 1;          // shadow of the MMA issues below
          const uint32_t ph_n = stage + 1 == S ? phase ^ 1u : phase;
          const uint32_t sfc_n = sfc == sf_last ? sf_base : sfc + kPairSlotCols;
          const bool more = kt + 1 < n_st;
          if (n == 4) {
            mma_mxf4nvf4_pair_lo(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, sfc, sfc + 16, kt != 0 ? 1u : 0u);
            mma_mxf4nvf4_pair_lo(d_tmem, a_lo + 2, a_hi, b_lo + 2, b_hi, idesc, sfc + 4, sfc + 22, 1u);
            if (more) next_ready = mbar_test_wait(&sf_ready[st_n], ph_n);
            mma_mxf4nvf4_pair_lo(d_tmem, a_lo + 4, a_hi, b_lo + 4, b_hi, idesc, sfc + 8, sfc + 28, 1u);
            mma_mxf4nvf4_pair_lo(d_tmem, a_lo + 6, a_hi, b_lo + 6, b_hi, idesc, sfc + 12, sfc + 34, 1u);
          } else {
            for (int g = 0; g < n; ++g)
              mma_mxf4nvf4_pair_lo(d_tmem, a_lo + 2 * g, a_hi, b_lo + 2 * g, b_hi, idesc, sfc + 4 * g,
                                   sfc + 16 + 6 * g, (kt | g) != 0 ? 1u : 0u);
            if (more) next_ready = mbar_test_wait(&sf_ready[st_n], ph_n);
          }
          mma_commit_pair(&empty[stage], 0x3);
          stage = st_n;
          phase = ph_n;
          sfc = sfc_n;
          a_lo = stage == 0 ? a_lo0 : a_n;
          b_lo = stage == 0 ? b_lo0 : b_n;
          if (!more) break;
          ++kt;
          if (!next_ready && !mbar_spin_bounded(&sf_ready[stage], phase, p.timeout_ns, s_abort)) {
            if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 13);
            *s_abort = 1;
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (!ok) break;
        mma_commit_pair(&acc_full[b], 0x3);
      }
      mma_commit_pair(mma_done, 0x3);
      int zero = 0;
      mbar_wait_bounded(mma_done, 0, p.timeout_ns, reinterpret_cast<volatile int*>(&zero));
    }
  } else if ((warp >= 6 && warp < kExtraWarp) || warp >= C::kStage1Warp) {
    // ---------------- scale staging: two sets of four warps (6..9 and the last four) ----------------
    // Each set takes every other fill: a staging warp's turn (wait, loads, tensor-memory
    // stores, their completion, fence, arrive) takes longer than the tensor core needs for
    // a stage, so two sets alternate.
    // Per fill, the 40 columns of the fill's slot in this warp's lane quadrant:
    // columns 4g..4g+3 the weight scales of K step g (only this quadrant's own
    // column is read by the MMA: weight row r's scales come from quadrant r/32),
    // columns 16+6g..16+6g+5 the routed-row scales of K step g, column c holding
    // routed rows 32c..32c+31 of the unit in lanes 0-31 of every quadrant.
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const uint32_t quad_lane = (32u * quad) << 16;
    const uint32_t sf_ready_even = map_shared_rank(smem_u32(sf_ready), 0);
    const int set = warp >= C::kStage1Warp ? 1 : 0;
    const bool info_warp = warp == (set ? C::kStage1Warp : 6);  // quadrant 0 of the set: publishes unit info
    int stage = 0;
    uint32_t phase = 0;
    int fill = 0;
    int e_hint = 0;
    bool ok = true;
    for (int u = pair; ok && u < total_units; u += npairs) {
      const PairUnit d = decode_pair_unit(u, unit_start, pad_start, off, E, MTC, U, p.rows_alloc, p.items, e_hint);
      if (!d.valid) {
        if (lane == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_INVALID_ARG, 5);
          *s_abort = 1;
        }
        break;
      }
      // the unit starts 0 or 64 rows into a 128-row scale block: routed row 32c of the unit is
      // column (o + c) % 4 of block (o + c) / 4, o = (x_row % 128) / 32
      const bool mid = (d.x_row & 127) != 0;
      for (int kt = 0; kt < KT; ++kt, ++fill) {
        if ((fill & 1) != set) {  // the other set's fill
          if (++stage == S) { stage = 0; phase ^= 1u; }
          continue;
        }
        bool got = mbar_wait_bounded(&full[stage], phase, p.timeout_ns, s_abort);
        // The scales go into registers before the wait for the slot, so only the stores
        // and the hand-off follow the slot's release (the MMAs of fill - 3 completing).
        uint32_t a[4], v[24];
        if (__all_sync(0xffffffffu, got)) {
          const uint8_t* sfw = s_w + stage * kWStageBytes + 16384 + lane * 16 + 4 * quad;
          const uint8_t* sfx = s_sfx + stage * C::kSfxStageBytes + lane * 16;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            a[g] = *reinterpret_cast<const uint32_t*>(sfw + 512 * g);
            const uint4 b0 = *reinterpret_cast<const uint4*>(sfx + 512 * g);
            const uint4 b1 = *reinterpret_cast<const uint4*>(sfx + kSfStageBytes + 512 * g);
            v[6 * g + 0] = mid ? b0.z : b0.x;
            v[6 * g + 1] = mid ? b0.w : b0.y;
            v[6 * g + 2] = mid ? b1.x : b0.z;
            v[6 * g + 3] = mid ? b1.y : b0.w;
            v[6 * g + 4] = mid ? b1.z : b1.x;
            v[6 * g + 5] = mid ? b1.w : b1.y;
          }
          if (fill >= kPairSlots) {
            // the slot's previous fill (fill - kPairSlots) must be consumed by its MMAs
            const int pf = fill - kPairSlots;
            got = mbar_wait_bounded(&empty[pf % S], static_cast<uint32_t>(pf / S) & 1u, p.timeout_ns, s_abort);
          }
        }
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) {
            if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 14);
            *s_abort = 1;
          }
          ok = false;
          break;
        }
        // weight scales: only this quadrant's own column of each K step (4g + quad) is read;
        // routed-row scales: all 24 columns (every quadrant reads every routed row's scales)
        const uint32_t slot = tmem_base + quad_lane + C::kSfTmemBase + (fill % kPairSlots) * kPairSlotCols;
#pragma unroll
        for (int g = 0; g < 4; ++g) tmem_st_1col(slot + 4 * g + quad, a[g]);
        tmem_st_16cols(slot + 16, v);
        tmem_st_8cols(slot + 32, v + 16);
        tmem_st_wait();
        tc_fence_before();
        if (kt == 0 && info_warp && lane == 0) s_info[stage] = d.n_mma;
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(sf_ready_even + stage * 8);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ---------------- epilogue warps 2..5 (and 12..15) ----------------
    const int q = warp & 3;
    const int m = 32 * q + lane;
    const int eg = warp >= C::kEpi1Warp ? 1 : 0;
    const int et = eg ? threadIdx.x - 32 * C::kEpi1Warp : threadIdx.x - 64;
    float* s_epi_g = s_epi + eg * kPairEpiRows * kEpiStride;
    const uint32_t acc_empty_even = map_shared_rank(smem_u32(acc_empty), 0);
    const float x_scale = __ldg(p.x_scale);
    if (p.epilogue == MOE_EPI_SILU_MUL_QUANT && p.h_scale_out && blockIdx.x == 0 && eg == 0 && et == 0)
      *p.h_scale_out = p.h_scale;
    const SiluOut so{p.h_scale, p.h_codes, p.h_sf, p.h_f32, N / 2};
    int acc_i = 0;
    int e_hint = 0;
    for (int u = pair; u < total_units; u += npairs, ++acc_i) {
      const PairUnit d = decode_pair_unit(u, unit_start, pad_start, off, E, MTC, U, p.rows_alloc, p.items, e_hint);
      if (!d.valid) {
        if (et == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_INVALID_ARG, 5);
          *s_abort = 1;
        }
        break;
      }
      if (acc_i % EG != eg) continue;
      const int b = acc_i % C::kAccBufs;
      const int mt = 2 * d.mt2 + static_cast<int>(rank);
      const float alpha = x_scale * __ldg(p.w_scale + d.e);
      // token table double-buffered per group: this group's unit before last read the other half
      // (the barrier after the previous unit's table orders those reads before this write).  It is
      // built before the accumulator wait, so its dependent global loads overlap the mainloop.
      int* tok_tab = s_tok_t + (eg * 2 + ((acc_i / EG) & 1)) * kPairBN;
      float* w_tab = s_tok_w + (eg * 2 + ((acc_i / EG) & 1)) * kPairBN;
      if (p.epilogue == MOE_EPI_FINALIZE) {
        for (int i = et; i < d.rows; i += 128) {
          const int ex = __ldg(p.perm_to_expanded + d.m_off + i);
          const bool in_range = ex >= 0 && ex < p.T * p.k;
          if (!in_range) record_error(p.err, MOE_ERR_INVALID_ARG, 6);
          tok_tab[i] = in_range ? (p.fin_gather ? ex : ex / p.k) : -1;
          w_tab[i] = in_range ? __ldg(p.topk_w + ex) * alpha : 0.0f;
        }
      }
      const bool got = mbar_wait_bounded(&acc_full[b], (acc_i / C::kAccBufs) & 1, p.timeout_ns, s_abort);
      // the OR-reduction barrier also publishes the token table to the whole group
      if (epi_any(eg, !got)) {
        if (et == 0) {
          if (!*s_abort) record_error(p.err, MOE_ERR_TIMEOUT, 15);
          *s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * kPairBN;
      for (int j0 = 0; j0 < d.rows; j0 += 32) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + j0, r);
        tmem_ld_wait();
        if (j0 + 32 >= d.rows) {
          // the accumulator is fully read: hand it back to the MMA thread before the last chunk's math
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_even + b * 8);
        }
        const int jn = min(32, d.rows - j0);
        if (p.epilogue == MOE_EPI_NONE) {
          epi_chunk_none(r, jn, d.x_row + j0, static_cast<int64_t>(mt) * kBM + m, N, alpha,
                         static_cast<uint16_t*>(p.out));
        } else if (p.epilogue == MOE_EPI_FINALIZE) {
          epi_chunk_finalize(r, lane, jn, tok_tab + j0, w_tab + j0,
                             static_cast<float*>(p.out) + static_cast<int64_t>(mt) * kBM + 32 * q + 4 * (lane >> 2),
                             N, p.fin_gather != 0);
        } else {
          epi_chunk_silu16(r, m, et, eg, jn, alpha, s_epi_g, d.x_row + j0, mt * 64, so);
        }
      }
    }
  }
  // (control reaches here on every path)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!leader && lane == 0) {
      // the even CTA's MMAs write this CTA's tensor memory: wait for the last of them
      int zero = 0;
      mbar_wait_bounded(mma_done, 0, p.timeout_ns, reinterpret_cast<volatile int*>(&zero));
    }
    __syncwarp();
  }
  tc_fence_before();
  cluster_sync_all();  // neither CTA frees its tensor memory or exits while the pair may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace
}  // namespace moe

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace moe {
namespace {

// 2D map over a [rows][row_bytes] byte matrix, boxes of 128 bytes x box_rows,
// 128-byte swizzle (the layout the tcgen05 K-major descriptors expect).
bool make_code_map(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EG>
moe_status prepare_gemm() {
  return cudaFuncSetAttribute(grouped_gemm_kernel<BN, EG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<BN, EG>::smem_bytes) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_RESOURCE;
}

template <int BN, int EG>
moe_status launch_gemm(const CUtensorMap& tm_x, const CUtensorMap& tm_xt, const GemmParams& p, int64_t max_units,
                       cudaStream_t st) {
  using C = Cfg<BN, EG>;
  int grid = num_sms();
  if (grid < 1) return MOE_ERR_CUDA;
  if (max_units < grid) grid = static_cast<int>(max_units);
  grouped_gemm_kernel<BN, EG><<<grid, C::kThreads, C::smem_bytes, st>>>(tm_x, tm_xt, p);
  return check_launch();
}

template <int EG>
moe_status prepare_pair() {
  return cudaFuncSetAttribute(grouped_gemm_pair_kernel<EG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PairCfg<EG>::smem_bytes) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_RESOURCE;
}

// CTA pairs the current device can hold at once with this configuration (each CTA
// takes a whole SM's shared memory); looked up once per device.
template <int EG>
int resident_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(PairCfg<EG>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<EG>::smem_bytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<EG>, &cfg) != cudaSuccess) return 0;
  cached[dev] = n;
  return n;
}

template <int EG>
moe_status launch_pair(const CUtensorMap& tm16, const CUtensorMap& tm96, const GemmParams& p, int64_t max_units,
                       cudaStream_t st) {
  int pairs = resident_pairs<EG>();
  if (pairs < 1) return MOE_ERR_RESOURCE;
  if (max_units < pairs) pairs = static_cast<int>(max_units);
  grouped_gemm_pair_kernel<EG><<<2 * pairs, PairCfg<EG>::kThreads, PairCfg<EG>::smem_bytes, st>>>(tm16, tm96, p);
  return check_launch();
}

// FINALIZE column chunk of the pair kernel, in weight tile pairs: the largest
// divisor of N/256 whose live accumulator (T x 256*chunk floats) stays within
// kFinalizeAtomicMaxBytes; 0 if not even one pair fits.
int finalize_pair_chunk(int T, int N) {
  const int MT2 = N / 256;
  for (int c = MT2; c >= 1; --c)
    if (MT2 % c == 0 && static_cast<int64_t>(T) * c * 256 * 4 <= kFinalizeAtomicMaxBytes) return c;
  return 0;
}

}  // namespace

int& gemm_debug_flags() {
  static int flags = 0;
  return flags;
}

// Routed-row tile of a launch from the rows-per-expert regime: the average
// rows per expert the allocation implies (a_rows_alloc exceeds the routed rows
// by at most 127 per expert).
int gemm_tile_rows(int64_t a_rows_alloc, int E) {
  const int64_t excess = 127ll * E;
  const int64_t avg = a_rows_alloc > excess ? (a_rows_alloc - excess) / E : 0;
  return avg <= 48 ? 64 : 128;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_grouped_gemm_workspace_size(int epilogue, int T, int k, int N) {
  if (epilogue != MOE_EPI_FINALIZE) return 0;
  if (T < 1 || N < 1 || k < 1) return 0;
  size_t b = static_cast<size_t>(T) * N * sizeof(float);
  if (finalize_gathers(T, N)) b *= static_cast<size_t>(k);
  return ((b + 255) / 256) * 256;
}

namespace moe {

size_t finalize_accumulator_bytes(int T, int N) {
  if (T < 1 || N < 1 || finalize_gathers(T, N)) return 0;
  return static_cast<size_t>(T) * N * sizeof(float);
}

moe_status grouped_gemm_enqueue(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                const uint8_t* b_blocked, const float* b_scale, const int32_t* expert_offsets, int E,
                                int64_t a_rows_alloc, int N, int K, int epilogue, const moe_epilogue_args* ep,
                                void* out, void* ws, size_t ws_bytes, bool clear_accumulator, cudaStream_t st) {
  if (!a_codes || !a_sf || !a_scale || !b_blocked || !b_scale || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (E < 1 || a_rows_alloc < 1 || N < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (epilogue != MOE_EPI_NONE && epilogue != MOE_EPI_SILU_MUL_QUANT && epilogue != MOE_EPI_FINALIZE)
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || K % 64 || N % kBM || a_rows_alloc % 128) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(E) * N > 0x7FFFFFFF || a_rows_alloc > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(a_codes) || !aligned16(a_sf) || !aligned16(b_blocked)) return MOE_ERR_MISALIGNED;
  GemmParams p{};
  p.w_blocked = b_blocked;
  p.x_sf = a_sf;
  p.x_scale = a_scale;
  p.w_scale = b_scale;
  p.expert_offsets = expert_offsets;
  p.E = E;
  p.N = N;
  p.K = K;
  p.epilogue = epilogue;
  if (epilogue == MOE_EPI_NONE) {
    if (!out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(out)) return MOE_ERR_MISALIGNED;
    p.out = out;
  } else if (epilogue == MOE_EPI_SILU_MUL_QUANT) {
    if (!ep || !ep->h_codes || !ep->h_sf) return MOE_ERR_INVALID_ARG;
    if (!(ep->h_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ep->h_codes) || !aligned16(ep->h_sf)) return MOE_ERR_MISALIGNED;
    p.h_scale = ep->h_scale;
    p.h_scale_out = ep->h_scale_out;
    p.h_codes = ep->h_codes;
    p.h_sf = ep->h_sf;
    p.h_f32 = ep->h_f32;
  } else {
    if (!ep || !ep->perm_to_expanded || !ep->topk_w || !out || ep->T < 1 || ep->k < 1) return MOE_ERR_INVALID_ARG;
    if (!aligned16(out)) return MOE_ERR_MISALIGNED;
    if (!ws || ws_bytes < moe_grouped_gemm_workspace_size(epilogue, ep->T, ep->k, N)) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
    p.out = ws;
    p.perm_to_expanded = ep->perm_to_expanded;
    p.topk_w = ep->topk_w;
    p.k = ep->k;
    p.T = ep->T;
    p.fin_gather = finalize_gathers(ep->T, N) ? 1 : 0;
    if (!p.fin_gather) p.mt_chunk = finalize_mt_chunk(ep->T, N);
  }
  p.rows_alloc = a_rows_alloc;
  p.items = epilogue == MOE_EPI_FINALIZE ? static_cast<int64_t>(ep->T) * ep->k : INT64_MAX;
  p.err = device_error_word();
  p.timeout_ns = wait_timeout_ns();
  p.debug_flags = gemm_debug_flags();
  if (!p.err) return MOE_ERR_CUDA;

  const int bn = gemm_tile_rows(a_rows_alloc, E);
  // The prefill regime runs on CTA pairs (256 weight rows x up to 192 routed rows per unit) where N is a
  // multiple of 256 and, for FINALIZE, a 256-column accumulator chunk stays within the atomic budget.
  // Debug flag bit 1 keeps the one-CTA 128-row tile (so tests can compare both kernels on one input).
  bool pair = bn == 128 && N % 256 == 0 && E <= kPairMaxExperts && (p.debug_flags & 2) == 0;
  if (pair && epilogue == MOE_EPI_FINALIZE && finalize_pair_chunk(ep->T, N) == 0) pair = false;
  if (pair) p.mt_chunk = epilogue == MOE_EPI_FINALIZE ? finalize_pair_chunk(ep->T, N) : N / 256;
  else if (p.mt_chunk == 0) p.mt_chunk = N / kBM;
  // two epilogue groups pay off where FINALIZE outlasts the mainloop (128-row tiles); at decode the
  // weight stream dominates and four copy warps are worth more (measured: 0.303 vs 0.319 ms, C4 down)
  const bool two_groups = bn == 128 && epilogue == MOE_EPI_FINALIZE;
  const int64_t max_units = pair ? ((a_rows_alloc + kPairBN - 1) / kPairBN) * (N / 256)
                                 : ((a_rows_alloc + bn - 1) / bn) * (N / kBM);
  if (max_units > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  // routed-row tiles come as 32-row boxes, or as one box when a unit fills the whole tile (one-CTA
  // kernel); as 16-row boxes or one 96-row box per CTA (pair kernel)
  CUtensorMap tm_x, tm_xt;
  if (!make_code_map(&tm_x, a_codes, static_cast<uint64_t>(a_rows_alloc), K / 2, pair ? 16 : 32))
    return MOE_ERR_CUDA;
  if (!make_code_map(&tm_xt, a_codes, static_cast<uint64_t>(a_rows_alloc), K / 2, pair ? kPairBN / 2 : bn))
    return MOE_ERR_CUDA;
  {
    const moe_status ps = pair ? (epilogue == MOE_EPI_NONE ? prepare_pair<1>() : prepare_pair<2>())
                          : bn == 64 ? prepare_gemm<64, 1>()
                          : two_groups ? prepare_gemm<128, 2>()
                                       : prepare_gemm<128, 1>();
    if (ps != MOE_OK) return ps;
  }
  if (clear_accumulator && epilogue == MOE_EPI_FINALIZE && !p.fin_gather) {
    if (cudaMemsetAsync(ws, 0, static_cast<size_t>(ep->T) * N * sizeof(float), st) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  moe_status s = pair ? (epilogue == MOE_EPI_NONE ? launch_pair<1>(tm_x, tm_xt, p, max_units, st)
                                                  : launch_pair<2>(tm_x, tm_xt, p, max_units, st))
                 : bn == 64  ? launch_gemm<64, 1>(tm_x, tm_xt, p, max_units, st)
                 : two_groups ? launch_gemm<128, 2>(tm_x, tm_xt, p, max_units, st)
                              : launch_gemm<128, 1>(tm_x, tm_xt, p, max_units, st);
  if (s != MOE_OK) return s;
  if (epilogue == MOE_EPI_FINALIZE) {
    if (p.fin_gather)
      return launch_finalize_sum(static_cast<const float*>(ws), ep->T, ep->k, N, static_cast<uint16_t*>(out), st);
    return launch_f32_to_bf16(static_cast<const float*>(ws), static_cast<uint16_t*>(out),
                              static_cast<int64_t>(ep->T) * N, st);
  }
  return MOE_OK;
}

}  // namespace moe

extern "C" moe_status moe_grouped_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                             const uint8_t* b_blocked, const float* b_scale,
                                             const int32_t* expert_offsets, int E, int64_t a_rows_alloc, int N, int K,
                                             int epilogue, const moe_epilogue_args* ep, void* out, void* ws,
                                             size_t ws_bytes, void* stream) {
  return grouped_gemm_enqueue(a_codes, a_sf, a_scale, b_blocked, b_scale, expert_offsets, E, a_rows_alloc, N, K,
                              epilogue, ep, out, ws, ws_bytes, true, static_cast<cudaStream_t>(stream));
}

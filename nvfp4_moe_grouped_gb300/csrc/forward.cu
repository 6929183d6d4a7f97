// forward.cu -- moe_forward: the whole MoE layer as one call on one stream.
//
//   route + permute -> quantise x into the routed rows (dynamic per-tensor
//   scale) -> gate_up grouped GEMM with the SiLU-mul + NVFP4 requantise
//   epilogue -> down grouped GEMM with the FINALIZE epilogue (router-weighted
//   sum back into BF16 token rows).
// Every intermediate lives in the caller's workspace at the offsets
// moe_forward_workspace_layout reports.
#include "common.cuh"

namespace moe {
int32_t* route_pad_offsets(void* ws, int T, int E, int k);
int& gemm_debug_flags();
bool small_layer_eligible(int T, int E, int k, int H, int I);
size_t small_layer_scratch_bytes(int T, int k, int I);
moe_status small_layer_enqueue(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k,
                               int H, int I, float h_scale, uint16_t* out, int32_t* topk_id, float* topk_w,
                               int32_t* offs, int32_t* p2e, int32_t* e2p, int32_t* e2r, float* x_scale,
                               uint8_t* x_codes, uint8_t* x_sf, float* hs, uint8_t* h_codes, uint8_t* h_sf,
                               void* scratch, cudaStream_t st);
bool route_one_chunk(int T, int E, int k);
}

using namespace moe;

namespace {
size_t align256(size_t b) { return ((b + 255) / 256) * 256; }
}

extern "C" moe_status moe_forward_workspace_layout(int T, int E, int k, int H, int I, moe_forward_layout* L) {
  if (!L || T < 1 || E < 1 || k < 1 || k > E || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(T) * k;
  const int64_t P = moe_padded_rows_max(R, E);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += align256(bytes); return at; };
  L->topk_id = take(R * 4);
  L->topk_w = take(R * 4);
  L->expert_offsets = take((E + 1) * 4);
  L->perm_to_expanded = take(R * 4);
  L->expanded_to_perm = take(R * 4);
  L->expanded_to_row = take(R * 4);
  L->x_scale = take(4);
  L->x_codes = take(static_cast<size_t>(P) * H / 2);
  L->x_sf = take(static_cast<size_t>(P) * H / 16);
  L->h_scale = take(4);
  L->h_codes = take(static_cast<size_t>(P) * I / 2);
  L->h_sf = take(static_cast<size_t>(P) * I / 16);
  L->route_ws = take(moe_route_permute_workspace_size(T, E, k));
  L->quant_ws = take(nvfp4_quantize_workspace_size(1));
  L->gemm_ws = take(moe_grouped_gemm_workspace_size(MOE_EPI_FINALIZE, T, k, H));
  L->small_scratch = small_layer_eligible(T, E, k, H, I) ? take(small_layer_scratch_bytes(T, k, I)) : SIZE_MAX;
  L->padded_rows = P;
  L->total = o;
  return MOE_OK;
}

// The single-launch path (small_layer.cu) serves small layers fed logits,
// unless debug flag bit 2 keeps the staged kernels.
namespace {
bool use_small_layer(int T, int E, int k, int H, int I) {
  return small_layer_eligible(T, E, k, H, I) && (gemm_debug_flags() & 4) == 0;
}
}  // namespace

extern "C" int moe_forward_kernel_count(int T, int E, int k, int H, int I) {
  if (T < 1 || E < 1 || k < 1 || k > E || H < 1 || I < 1) return 0;
  if (use_small_layer(T, E, k, H, I)) return 1;
  // routing (one kernel when every item fits one chunk, else top-k, scan and scatter), the
  // activation amax and quantiser, the two GEMMs, and the FINALIZE closing pass
  return (route_one_chunk(T, E, k) ? 1 : 3) + 2 + 2 + 1;
}

extern "C" size_t moe_forward_workspace_size(int T, int E, int k, int H, int I) {
  moe_forward_layout L;
  if (moe_forward_workspace_layout(T, E, k, H, I, &L) != MOE_OK) return 0;
  return L.total;
}

// moe_forward_gated: moe_forward's workspace, then the router's.
extern "C" size_t moe_forward_gated_workspace_size(int T, int E, int k, int H, int I) {
  const size_t base = moe_forward_workspace_size(T, E, k, H, I);
  const size_t rws = moe_router_workspace_size(T, E, H, k);
  if (base == 0 || rws == 0) return 0;
  return base + align256(rws);
}

namespace {

// Checks everything the stage calls would check, so moe_forward either fails
// before enqueueing anything or enqueues the whole layer.
moe_status forward_check(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k, int H,
                         int I, float h_scale, const uint16_t* out, const void* ws, size_t ws_bytes,
                         moe_forward_layout* L) {
  if (!x || !logits || !w || !out) return MOE_ERR_INVALID_ARG;
  if (!w->w13 || !w->w13_scale || !w->w2 || !w->w2_scale) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || k < 1 || k > E || H < 1 || I < 1 || !(h_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (H % 128 || I % 64 || E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * k > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  moe_status s = moe_forward_workspace_layout(T, E, k, H, I, L);
  if (s != MOE_OK) return s;
  if (!ws || ws_bytes < L->total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws) || !aligned16(x) || !aligned16(out) || !aligned16(w->w13) || !aligned16(w->w2))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

// The layer's four stages; when `ev` is given, ev[i] is recorded (as an external
// event, visible to timing even inside a captured graph) after stage i.  With
// `w_gate` the first stage is moe_router (logits GEMM, routing, and x's decode
// multiplier from the GEMM's own pass over x) and the quantiser takes that
// multiplier as a static scale; otherwise the logits are an input.
// With `side` (a second stream, used while capturing the layer's graph) two
// steps leave the chain: the activation quantiser's amax pass runs beside the
// routing (it reads only x), and the FINALIZE accumulator is cleared beside the
// gate_up GEMM; jev[0..3] are the events of those forks and joins.
// `external` is set while the layer is being captured into a graph.
moe_status forward_stages(const uint16_t* x, const float* logits, const uint16_t* w_gate, const moe_weights* w,
                          int T, int E, int k, int H, int I, float h_scale, uint16_t* out, void* ws,
                          const moe_forward_layout& L, cudaStream_t stream, cudaEvent_t* ev, bool external,
                          cudaStream_t side = nullptr, cudaEvent_t* jev = nullptr) {
  char* base = static_cast<char*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(base + off); };
  auto mark = [&](int i) -> moe_status {
    if (!ev) return MOE_OK;
    cudaError_t e = external ? cudaEventRecordWithFlags(ev[i], stream, cudaEventRecordExternal)
                             : cudaEventRecord(ev[i], stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  };
  const int64_t R = static_cast<int64_t>(T) * k;
  int32_t* topk_id = static_cast<int32_t*>(at(L.topk_id));
  float* topk_w = static_cast<float*>(at(L.topk_w));
  int32_t* offs = static_cast<int32_t*>(at(L.expert_offsets));
  int32_t* p2e = static_cast<int32_t*>(at(L.perm_to_expanded));
  int32_t* e2p = static_cast<int32_t*>(at(L.expanded_to_perm));
  int32_t* e2r = static_cast<int32_t*>(at(L.expanded_to_row));
  float* x_scale = static_cast<float*>(at(L.x_scale));
  uint8_t* x_codes = static_cast<uint8_t*>(at(L.x_codes));
  uint8_t* x_sf = static_cast<uint8_t*>(at(L.x_sf));
  float* hs = static_cast<float*>(at(L.h_scale));
  uint8_t* h_codes = static_cast<uint8_t*>(at(L.h_codes));
  uint8_t* h_sf = static_cast<uint8_t*>(at(L.h_sf));
  auto fork = [&](cudaEvent_t e, cudaStream_t from, cudaStream_t to) -> moe_status {
    return cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess ? MOE_OK
                                                                                                  : MOE_ERR_CUDA;
  };
  const bool par = side != nullptr && jev != nullptr;
  const bool amax_beside = par && !w_gate;  // with w_gate the router's GEMM supplies x's multiplier
  moe_status s = mark(0);
  if (s != MOE_OK) return s;
  if (!w_gate && L.small_scratch != SIZE_MAX && use_small_layer(T, E, k, H, I)) {
    // the whole layer in one launch (its time is all in the first stage)
    s = small_layer_enqueue(x, logits, w, T, E, k, H, I, h_scale, out, topk_id, topk_w, offs, p2e, e2p, e2r,
                            x_scale, x_codes, x_sf, hs, h_codes, h_sf, at(L.small_scratch), stream);
    for (int i = 1; i <= 4 && s == MOE_OK; ++i) s = mark(i);
    return s;
  }
  if (amax_beside) {
    if ((s = fork(jev[0], stream, side)) != MOE_OK) return s;
    s = quantize_amax_enqueue(x, MOE_IN_BF16, T, H, 1, static_cast<uint32_t*>(at(L.quant_ws)), side);
    if (s != MOE_OK || cudaEventRecord(jev[1], side) != cudaSuccess) return s != MOE_OK ? s : MOE_ERR_CUDA;
  }
  if (w_gate) {
    s = moe_router(x, w_gate, T, E, H, k, nullptr, x_scale, topk_id, topk_w, offs, p2e, e2p, e2r, at(L.total),
                   moe_router_workspace_size(T, E, H, k), stream);
  } else {
    s = moe_route_permute(logits, T, E, k, topk_id, topk_w, offs, p2e, e2p, e2r, at(L.route_ws),
                          moe_route_permute_workspace_size(T, E, k), stream);
  }
  if (s != MOE_OK || (s = mark(1)) != MOE_OK) return s;
  if (amax_beside && cudaStreamWaitEvent(stream, jev[1], 0) != cudaSuccess) return MOE_ERR_CUDA;
  s = quantize_enqueue(x, MOE_IN_BF16, T, H, 1, x_scale, w_gate ? 0 : (amax_beside ? 2 : 1), R, k, e2r, x_codes,
                       x_sf, MOE_SF_TILED, L.padded_rows, at(L.quant_ws), nvfp4_quantize_workspace_size(1), stream);
  if (s != MOE_OK || (s = mark(2)) != MOE_OK) return s;
  const size_t acc_bytes = finalize_accumulator_bytes(T, H);
  const bool clear_beside = par && acc_bytes > 0;
  if (clear_beside) {
    if ((s = fork(jev[2], stream, side)) != MOE_OK) return s;
    if (cudaMemsetAsync(at(L.gemm_ws), 0, acc_bytes, side) != cudaSuccess ||
        cudaEventRecord(jev[3], side) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  moe_epilogue_args ep{};
  ep.h_scale = h_scale;
  ep.h_scale_out = hs;
  ep.h_codes = h_codes;
  ep.h_sf = h_sf;
  s = grouped_gemm_enqueue(x_codes, x_sf, x_scale, w->w13, w->w13_scale, offs, E, L.padded_rows, 2 * I, H,
                           MOE_EPI_SILU_MUL_QUANT, &ep, nullptr, nullptr, 0, true, stream);
  if (s != MOE_OK || (s = mark(3)) != MOE_OK) return s;
  if (clear_beside && cudaStreamWaitEvent(stream, jev[3], 0) != cudaSuccess) return MOE_ERR_CUDA;
  moe_epilogue_args ep2{};
  ep2.perm_to_expanded = p2e;
  ep2.topk_w = topk_w;
  ep2.T = T;
  ep2.k = k;
  s = grouped_gemm_enqueue(h_codes, h_sf, hs, w->w2, w->w2_scale, offs, E, L.padded_rows, H, I, MOE_EPI_FINALIZE,
                           &ep2, out, at(L.gemm_ws), moe_grouped_gemm_workspace_size(MOE_EPI_FINALIZE, T, k, H),
                           !clear_beside, stream);
  if (s != MOE_OK) return s;
  return mark(4);
}

}  // namespace

extern "C" moe_status moe_forward(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k,
                                  int H, int I, float h_scale, uint16_t* out, void* ws, size_t ws_bytes,
                                  void* stream) {
  moe_forward_layout L;
  moe_status s = forward_check(x, logits, w, T, E, k, H, I, h_scale, out, ws, ws_bytes, &L);
  if (s != MOE_OK) return s;
  return forward_stages(x, logits, nullptr, w, T, E, k, H, I, h_scale, out, ws, L, static_cast<cudaStream_t>(stream),
                        nullptr, false);
}

extern "C" moe_status moe_forward_gated(const uint16_t* x, const uint16_t* w_gate, const moe_weights* w, int T,
                                        int E, int k, int H, int I, float h_scale, uint16_t* out, void* ws,
                                        size_t ws_bytes, void* stream) {
  if (!w_gate) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate)) return MOE_ERR_MISALIGNED;
  if (E > 256) return MOE_ERR_UNSUPPORTED;
  moe_forward_layout L;
  // forward_check validates everything but the logits, which this call computes
  moe_status s = forward_check(x, reinterpret_cast<const float*>(w_gate), w, T, E, k, H, I, h_scale, out, ws, ws_bytes,
                               &L);
  if (s != MOE_OK) return s;
  if (ws_bytes < moe_forward_gated_workspace_size(T, E, k, H, I)) return MOE_ERR_WORKSPACE;
  return forward_stages(x, nullptr, w_gate, w, T, E, k, H, I, h_scale, out, ws, L, static_cast<cudaStream_t>(stream),
                        nullptr, false);
}

// ---------------------------------------------------------------------------
// The layer as one CUDA graph: captured once, replayed with one launch.
// ---------------------------------------------------------------------------
struct moe_forward_graph {
  cudaGraphExec_t exec = nullptr;
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  bool timed = false;
  // the device buffers the graph was captured with, for moe_forward_graph_run_host
  void* x = nullptr;
  void* logits = nullptr;
  void* out = nullptr;
  size_t x_bytes = 0, logits_bytes = 0, out_bytes = 0;
};

namespace {
void graph_release(moe_forward_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  for (auto& e : g->ev)
    if (e) cudaEventDestroy(e);
  delete g;
}
}  // namespace

extern "C" moe_status moe_forward_graph_create(const uint16_t* x, const float* logits, const moe_weights* w, int T,
                                               int E, int k, int H, int I, float h_scale, uint16_t* out, void* ws,
                                               size_t ws_bytes, int stage_events, moe_forward_graph** graph) {
  if (!graph) return MOE_ERR_INVALID_ARG;
  *graph = nullptr;
  moe_forward_layout L;
  moe_status s = forward_check(x, logits, w, T, E, k, H, I, h_scale, out, ws, ws_bytes, &L);
  if (s != MOE_OK) return s;
  if (!device_error_word() || num_sms() < 1) return MOE_ERR_CUDA;
  moe_forward_graph* g = new moe_forward_graph();
  g->timed = stage_events != 0;
  g->x = const_cast<uint16_t*>(x);
  g->logits = const_cast<float*>(logits);
  g->out = out;
  g->x_bytes = static_cast<size_t>(T) * H * sizeof(uint16_t);
  g->logits_bytes = static_cast<size_t>(T) * E * sizeof(float);
  g->out_bytes = static_cast<size_t>(T) * H * sizeof(uint16_t);
  cudaStream_t st = nullptr, side = nullptr;
  cudaEvent_t jev[4] = {nullptr, nullptr, nullptr, nullptr};
  cudaGraph_t raw = nullptr;
  auto release_capture_objects = [&]() {
    for (auto& e : jev)
      if (e) { cudaEventDestroy(e); e = nullptr; }
    if (side) { cudaStreamDestroy(side); side = nullptr; }
    if (st) { cudaStreamDestroy(st); st = nullptr; }
  };
  auto fail = [&](moe_status code) {
    if (raw) cudaGraphDestroy(raw);
    release_capture_objects();
    graph_release(g);
    return code;
  };
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return fail(MOE_ERR_CUDA);
  // The untimed graph takes the amax pass and the accumulator clear off the
  // chain (forward_stages); the timed one keeps every step between its stage
  // events.
  if (!g->timed) {
    if (cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) != cudaSuccess) return fail(MOE_ERR_CUDA);
    for (auto& e : jev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return fail(MOE_ERR_CUDA);
  }
  if (g->timed)
    for (auto& e : g->ev)
      if (cudaEventCreate(&e) != cudaSuccess) return fail(MOE_ERR_CUDA);
  // One eager pass first: every host-side preparation (kernel attributes, cached
  // device addresses) happens outside the capture.
  s = forward_stages(x, logits, nullptr, w, T, E, k, H, I, h_scale, out, ws, L, st, nullptr, false);
  if (s != MOE_OK) return fail(s);
  if (cudaStreamSynchronize(st) != cudaSuccess) return fail(MOE_ERR_CUDA);
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return fail(MOE_ERR_CUDA);
  s = forward_stages(x, logits, nullptr, w, T, E, k, H, I, h_scale, out, ws, L, st, g->timed ? g->ev : nullptr, true,
                     side, g->timed ? nullptr : jev);
  cudaError_t ce = cudaStreamEndCapture(st, &raw);
  if (s != MOE_OK) return fail(s);
  if (ce != cudaSuccess || !raw) return fail(MOE_ERR_CUDA);
  if (cudaGraphInstantiate(&g->exec, raw, 0) != cudaSuccess) return fail(MOE_ERR_CUDA);
  cudaGraphDestroy(raw);
  raw = nullptr;
  release_capture_objects();
  *graph = g;
  return MOE_OK;
}

extern "C" moe_status moe_forward_graph_launch(moe_forward_graph* graph, void* stream) {
  if (!graph || !graph->exec) return MOE_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_forward_graph_run_host(moe_forward_graph* graph, const uint16_t* x_host,
                                                 const float* logits_host, uint16_t* out_host, void* stream) {
  if (!graph || !graph->exec || !x_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(graph->x, x_host, graph->x_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(graph->logits, logits_host, graph->logits_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaGraphLaunch(graph->exec, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(out_host, graph->out, graph->out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status moe_forward_graph_stage_ms(moe_forward_graph* graph, float* ms) {
  if (!graph || !ms) return MOE_ERR_INVALID_ARG;
  if (!graph->timed) return MOE_ERR_INVALID_ARG;
  if (cudaEventSynchronize(graph->ev[4]) != cudaSuccess) return MOE_ERR_CUDA;
  for (int i = 0; i < 4; ++i)
    if (cudaEventElapsedTime(&ms[i], graph->ev[i], graph->ev[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaEventElapsedTime(&ms[4], graph->ev[0], graph->ev[4]) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" void moe_forward_graph_destroy(moe_forward_graph* graph) { graph_release(graph); }

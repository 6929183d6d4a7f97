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
  L->padded_rows = P;
  L->total = o;
  return MOE_OK;
}

extern "C" size_t moe_forward_workspace_size(int T, int E, int k, int H, int I) {
  moe_forward_layout L;
  if (moe_forward_workspace_layout(T, E, k, H, I, &L) != MOE_OK) return 0;
  return L.total;
}

extern "C" moe_status moe_forward(const uint16_t* x, const float* logits, const moe_weights* w, int T, int E, int k,
                                  int H, int I, float h_scale, uint16_t* out, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!x || !logits || !w || !out) return MOE_ERR_INVALID_ARG;
  if (!w->w13 || !w->w13_scale || !w->w2 || !w->w2_scale) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || k < 1 || k > E || H < 1 || I < 1 || !(h_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (H % 128 || I % 64) return MOE_ERR_UNSUPPORTED;
  moe_forward_layout L;
  moe_status s = moe_forward_workspace_layout(T, E, k, H, I, &L);
  if (s != MOE_OK) return s;
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  char* base = static_cast<char*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(base + off); };
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

  s = moe_route_permute(logits, T, E, k, topk_id, topk_w, offs, p2e, e2p, e2r, at(L.route_ws),
                        moe_route_permute_workspace_size(T, E, k), stream);
  if (s != MOE_OK) return s;
  s = nvfp4_quantize(x, MOE_IN_BF16, T, H, 1, x_scale, 1, R, k, e2r, x_codes, x_sf, MOE_SF_TILED, L.padded_rows,
                     at(L.quant_ws), nvfp4_quantize_workspace_size(1), stream);
  if (s != MOE_OK) return s;
  moe_epilogue_args ep{};
  ep.h_scale = h_scale;
  ep.h_scale_out = hs;
  ep.h_codes = h_codes;
  ep.h_sf = h_sf;
  s = moe_grouped_gemm_nvfp4(x_codes, x_sf, x_scale, w->w13, w->w13_scale, offs, E, L.padded_rows,
                             2 * I, H, MOE_EPI_SILU_MUL_QUANT, &ep, nullptr, nullptr, 0, stream);
  if (s != MOE_OK) return s;
  moe_epilogue_args ep2{};
  ep2.perm_to_expanded = p2e;
  ep2.topk_w = topk_w;
  ep2.T = T;
  ep2.k = k;
  return moe_grouped_gemm_nvfp4(h_codes, h_sf, hs, w->w2, w->w2_scale, offs, E, L.padded_rows, H, I,
                                MOE_EPI_FINALIZE, &ep2, out, at(L.gemm_ws),
                                moe_grouped_gemm_workspace_size(MOE_EPI_FINALIZE, T, k, H), stream);
}

// route_permute_static.cu -- moe_route_permute for callers that cannot
// allocate device memory.
//
// Some callers cannot provide a workspace: code that runs where allocation is
// not allowed or not wanted (cudaMalloc may wait for the whole device to go
// idle, which breaks a latency budget or a caller's own stream ordering), or a
// host whose device memory is owned entirely by another allocator.  This entry
// point gives them routing and permutation with no workspace argument: its
// scratch is a fixed array in the library's own device memory, reserved on
// every GPU that loads the library for as long as the process lives.
#include "common.cuh"

namespace moe {
namespace {

// Largest workspace the static scratch can stand in for: 1 MiB.  That covers
// e.g. T = 16384 tokens with E = 256 experts and k = 8.
constexpr size_t kStaticScratchBytes = 1u << 20;

static __device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

// Device address of g_route_scratch in the current device's context.  Host
// code must not pass the symbol itself to a kernel: on the host it names a
// stand-in object, not device memory.  The lookup allocates nothing and is
// cheap, so it runs on every call: a cached address could outlive its context
// (cudaDeviceReset, or another context made current on the same device).
void* static_scratch_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_permute_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" moe_status moe_route_permute_static(const float* logits, int T, int E, int k, int32_t* topk_id,
                                               float* topk_w, int32_t* expert_offsets, int32_t* perm_to_expanded,
                                               int32_t* expanded_to_perm, int32_t* expanded_to_row, void* stream) {
  if (T < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  // the shape limits of moe_route_permute come first, so an unsupported shape gets the same status here
  if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * k > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  // then the size (before the pointers: a caller's oversized problem is reported as such)
  const size_t need = moe_route_permute_workspace_size(T, E, k);
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = static_scratch_address();
  if (!scratch) return MOE_ERR_CUDA;
  // The routing kernels overwrite every scratch word they read before reading
  // it, so nothing has to be cleared between calls.
  return moe_route_permute(logits, T, E, k, topk_id, topk_w, expert_offsets, perm_to_expanded, expanded_to_perm,
                           expanded_to_row, scratch, kStaticScratchBytes, stream);
}

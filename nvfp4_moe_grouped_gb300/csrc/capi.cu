// capi.cu -- the C ABI's housekeeping: status names, the device error word of
// the bounded waits, the wait bound, the debug hook, device properties.
#include "common.cuh"

namespace moe {
namespace {

// {code, where} of the first bounded wait that gave up since the last read.
__device__ int32_t g_device_error[2];

uint64_t g_timeout_ns = 2000000000ull;  // 2 s: far beyond any legitimate wait

}  // namespace

// Device address of g_device_error in the current device's context, looked up
// on every call (cheap, allocates nothing): a cached address could outlive its
// context after cudaDeviceReset or under another context on the same device.
int32_t* device_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
  return static_cast<int32_t*>(p);
}

uint64_t wait_timeout_ns() { return g_timeout_ns; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

moe_status check_launch() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

int& gemm_debug_flags();

}  // namespace moe

using namespace moe;

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case MOE_ERR_RESOURCE: return "tile configuration does not fit shared or tensor memory";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

extern "C" int moe_abi_version(void) { return 6; }

extern "C" moe_status moe_device_error(int32_t* code, int32_t* where) {
  if (!code || !where) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_device_error, sizeof h) != cudaSuccess) return MOE_ERR_CUDA;
  const int32_t zero[2] = {0, 0};
  if (cudaMemcpyToSymbol(g_device_error, zero, sizeof zero) != cudaSuccess) return MOE_ERR_CUDA;
  *code = h[0];
  *where = h[1];
  return MOE_OK;
}

extern "C" void moe_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns = ns ? ns : 2000000000ull; }

extern "C" void moe_debug_set_flags(int flags) { gemm_debug_flags() = flags; }

extern "C" int64_t moe_padded_rows_max(int64_t routed_rows, int E) {
  if (routed_rows < 0 || E < 1) return 0;
  int64_t extra = 127 * (routed_rows < E ? routed_rows : static_cast<int64_t>(E));
  int64_t rows = routed_rows + extra;
  rows = ((rows + 127) / 128) * 128;
  return rows < 128 ? 128 : rows;
}

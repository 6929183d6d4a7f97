// cublaslt_fp4.cu -- a timing comparison for the dense NVFP4 GEMM: the same
// contraction D = A . B^T (A [M][K], B [N][K] e2m1 codes with one e4m3 scale per
// 16 elements along K, FP32 accumulation, bf16 output) run through cuBLASLt's
// block-scaled FP4 matmul, as a library reference beside the repository's own
// tcgen05 kernel.  Built as a separate shared library (it links cuBLASLt; the
// layer's library depends on the driver only) and used by the benchmark alone.
//
// "Tracing the Failure: Debugging CUTLASS FP4 Tile Configurations on Blackwell
// SM120", section "The Broader Context": the dense FP4 GEMM on very large
// matrices as a measurement of its own.  Only the time is of interest here, so
// the operands hold a fixed pattern (codes 0x22 = 1.0 in both nibbles, scales
// 0x38 = 1.0).
#include <cublasLt.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

struct Buffers {
  void *a = nullptr, *b = nullptr, *sa = nullptr, *sb = nullptr, *d = nullptr, *ws = nullptr;
  ~Buffers() {
    for (void* p : {a, b, sa, sb, d, ws})
      if (p) cudaFree(p);
  }
};

// Bytes allocated for a VEC16_UE4M3 scale tensor of `rows` rows of K elements:
// tiles of 128 rows x 4 scale columns (64 K-elements), so both extents round
// up, plus 1 MiB of slack so that no reading of the layout rule can run past
// the allocation.
size_t scale_bytes(int rows, int K) {
  const size_t r = (static_cast<size_t>(rows) + 127) / 128 * 128;
  const size_t c = (static_cast<size_t>(K) / 16 + 3) / 4 * 4;
  return r * c + (1u << 20);
}

int fail(char* msg, int len, const char* what, int code) {
  if (msg && len > 0) snprintf(msg, static_cast<size_t>(len), "%s (status %d)", what, code);
  return code == 0 ? -1 : code;
}

}  // namespace

// Times `iters` cuBLASLt NVFP4 GEMMs of M x N x K after `warmup` untimed ones.
// Returns 0 with the mean milliseconds per GEMM in *ms, or a non-zero status
// with a one-line reason in msg (cuBLASLt offering no algorithm for the shape
// on this GPU included).  Allocates and frees its own device buffers.
extern "C" __attribute__((visibility("default"))) int nvfp4_cublaslt_gemm_time(int M, int N, int K, int warmup,
                                                                               int iters, float* ms, char* msg,
                                                                               int msg_len) {
  if (M < 1 || N < 1 || K < 32 || K % 32 || iters < 1 || warmup < 0 || !ms) return fail(msg, msg_len, "bad arguments", 1);
  Buffers buf;
  const size_t a_bytes = static_cast<size_t>(M) * K / 2, b_bytes = static_cast<size_t>(N) * K / 2;
  const size_t ws_bytes = 64u << 20;
  if (cudaMalloc(&buf.a, a_bytes) || cudaMalloc(&buf.b, b_bytes) || cudaMalloc(&buf.sa, scale_bytes(M, K)) ||
      cudaMalloc(&buf.sb, scale_bytes(N, K)) || cudaMalloc(&buf.d, static_cast<size_t>(M) * N * 2) ||
      cudaMalloc(&buf.ws, ws_bytes))
    return fail(msg, msg_len, "cudaMalloc failed", 2);
  cudaMemset(buf.a, 0x22, a_bytes);
  cudaMemset(buf.b, 0x22, b_bytes);
  cudaMemset(buf.sa, 0x38, scale_bytes(M, K));
  cudaMemset(buf.sb, 0x38, scale_bytes(N, K));

  cublasLtHandle_t lt = nullptr;
  cublasStatus_t st = cublasLtCreate(&lt);
  if (st != CUBLAS_STATUS_SUCCESS) return fail(msg, msg_len, "cublasLtCreate failed", static_cast<int>(st));
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  int rc = 0;
  do {
    if ((st = cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F)) != CUBLAS_STATUS_SUCCESS) {
      rc = fail(msg, msg_len, "matmul descriptor", static_cast<int>(st));
      break;
    }
    // column-major terms: D [M][N] (ld M) = op(A) op(B), op(A) = A^T with A stored K x M (ld K), B stored
    // K x N (ld K): both operands K-contiguous, the form block-scaled FP4 requires
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    const int32_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta));
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb));
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &mode, sizeof(mode));
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &mode, sizeof(mode));
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &buf.sa, sizeof(buf.sa));
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &buf.sb, sizeof(buf.sb));
    if (cublasLtMatrixLayoutCreate(&la, CUDA_R_4F_E2M1, K, M, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&lb, CUDA_R_4F_E2M1, K, N, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&ld, CUDA_R_16BF, M, N, M) != CUBLAS_STATUS_SUCCESS) {
      rc = fail(msg, msg_len, "matrix layouts", 3);
      break;
    }
    cublasLtMatmulPreferenceCreate(&pref);
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof(ws_bytes));
    cublasLtMatmulHeuristicResult_t heur = {};
    int found = 0;
    st = cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, ld, ld, pref, 1, &heur, &found);
    if (st != CUBLAS_STATUS_SUCCESS || found < 1) {
      rc = fail(msg, msg_len, "no cuBLASLt algorithm for this FP4 shape", st != CUBLAS_STATUS_SUCCESS ? static_cast<int>(st) : 4);
      break;
    }
    const float alpha = 1.0f, beta = 0.0f;
    cudaStream_t s = nullptr;
    auto run = [&]() {
      return cublasLtMatmul(lt, op, &alpha, buf.a, la, buf.b, lb, &beta, buf.d, ld, buf.d, ld, &heur.algo, buf.ws,
                            ws_bytes, s);
    };
    for (int i = 0; i < warmup && st == CUBLAS_STATUS_SUCCESS; ++i) st = run();
    if (st != CUBLAS_STATUS_SUCCESS || cudaStreamSynchronize(s) != cudaSuccess) {
      rc = fail(msg, msg_len, "cublasLtMatmul failed", static_cast<int>(st));
      break;
    }
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0, s);
    for (int i = 0; i < iters && st == CUBLAS_STATUS_SUCCESS; ++i) st = run();
    cudaEventRecord(e1, s);
    cudaEventSynchronize(e1);
    float t = 0.0f;
    cudaEventElapsedTime(&t, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != CUBLAS_STATUS_SUCCESS) {
      rc = fail(msg, msg_len, "cublasLtMatmul failed", static_cast<int>(st));
      break;
    }
    *ms = t / static_cast<float>(iters);
    if (msg && msg_len > 0) snprintf(msg, static_cast<size_t>(msg_len), "ok");
  } while (false);
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (ld) cublasLtMatrixLayoutDestroy(ld);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  cublasLtDestroy(lt);
  return rc;
}

// kernel_api.cu — the kernel-level entry points of ttt_kernels.h.
#include <cstring>

#include "../../include/ttt.h"
#include "../../include/ttt_kernels.h"
#include "kernels.h"

namespace {
int* g_err = nullptr;  // device error word shared by kernel-level launches
int ensure_err() {
  if (g_err) return 0;
  if (cudaMalloc(&g_err, sizeof(int)) != cudaSuccess) return TTT_ERR_OOM;
  return cudaMemset(g_err, 0, sizeof(int)) == cudaSuccess ? 0 : TTT_ERR_CUDA;
}
}  // namespace

extern "C" int ttt_kernel_gemm(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                               const void* B, int64_t ldb, int32_t b_mn, const void* B2, float* C,
                               int64_t ldc, int32_t impl, void* stream) {
  if (!A || !B || !C || M < 0 || N < 0 || K < 1 || (N & 1) || (ldc & 1)) return TTT_ERR_INVALID;
  if (ensure_err()) return TTT_ERR_OOM;
  cudaStream_t st = (cudaStream_t)stream;
  ttt::Epi e;
  memset(&e, 0, sizeof(e));
  e.kind = ttt::EPI_STORE;
  e.out_f32 = 1;
  e.out = C;
  e.ldo = ldc;
  if (impl == 0 || impl == 1) {
    ttt::GemmArgs<ttt::bf16> g{M, N, K, (const ttt::bf16*)A, lda, a_mn, (const ttt::bf16*)B, ldb, b_mn, e,
                               (const ttt::bf16*)B2};
    if (impl == 0) {
      if (ttt::gemm_tc_init()) return TTT_ERR_CUDA;
      int dev = 0, sms = 148;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      int rc = ttt::gemm_tc(g, sms, g_err, st);
      if (rc == (int)cudaErrorNotSupported || rc == (int)cudaErrorInvalidValue) return TTT_ERR_SHAPE;
      return rc ? TTT_ERR_CUDA : 0;
    }
    ttt::gemm_simt<ttt::bf16>(g, st);
  } else if (impl == 2) {
    ttt::GemmArgs<float> g{M, N, K, (const float*)A, lda, a_mn, (const float*)B, ldb, b_mn, e, (const float*)B2};
    ttt::gemm_simt<float>(g, st);
  } else {
    return TTT_ERR_INVALID;
  }
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
}

extern "C" int ttt_kernel_error(void) {
  if (ensure_err()) return TTT_ERR_OOM;
  if (cudaDeviceSynchronize() != cudaSuccess) return TTT_ERR_CUDA;
  int h = 0;
  cudaMemcpy(&h, g_err, sizeof(int), cudaMemcpyDeviceToHost);
  cudaMemset(g_err, 0, sizeof(int));
  return h;
}

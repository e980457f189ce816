// gemm_simt.cu — plain fp32-FMA tiled GEMM with the shared epilogues.
// It serves the fp32 check mode (no tensor cores, no tf32) and is the
// reference the tensor-core GEMM is unit-tested against on the GPU.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace ttt {

namespace {
constexpr int SBM = 64, SBN = 64, SBK = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(int M, int N, int K, const T* __restrict__ A,
                                                        int64_t lda, int a_mn, const T* __restrict__ B,
                                                        int64_t ldb, int b_mn, Epi e,
                                                        const T* __restrict__ B2) {
  __shared__ float As[SBK][SBM + 4];
  __shared__ float Bs[SBK][SBN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * SBM, n0 = blockIdx.x * SBN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  const int nk = (K + SBK - 1) / SBK;
  for (int kb = 0; kb < (B2 ? 2 * nk : nk); ++kb) {
    const int k0 = (kb % nk) * SBK;
    const T* Bc = kb < nk ? B : B2;
    // 64x16 tiles: 1024 elements each, 4 per thread
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      int idx = tid + it * 256;
      int mm, kk;
      if (a_mn) { mm = idx % SBM; kk = idx / SBM; } else { kk = idx % SBK; mm = idx / SBK; }
      int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < M && gk < K) v = to_f<T>(a_mn ? A[(int64_t)gk * lda + gm] : A[(int64_t)gm * lda + gk]);
      As[kk][mm] = v;
      int nn;
      if (b_mn) { nn = idx % SBN; kk = idx / SBN; } else { kk = idx % SBK; nn = idx / SBK; }
      int gn = n0 + nn;
      gk = k0 + kk;
      float w = 0.f;
      if (gn < N && gk < K) w = to_f<T>(b_mn ? Bc[(int64_t)gk * ldb + gn] : Bc[(int64_t)gn * ldb + gk]);
      Bs[kk][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      int n = n0 + tx * 4 + j;
      if (n < N) epi_pair<T>(e, m, n, acc[i][j], acc[i][j + 1]);
    }
  }
}
}  // namespace

template <typename T>
void gemm_simt(const GemmArgs<T>& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return;
  if (g.groups > 1) {
    // grouped product: one launch per group, on its rows and its B
    for (int gi = 0; gi < g.groups; ++gi) {
      GemmArgs<T> s = g;
      const int64_t r0 = (int64_t)gi * g.group_rows;
      s.M = (int)std::min<int64_t>(g.group_rows, g.M - r0);
      if (s.M <= 0) break;
      s.A = g.a_mn ? g.A + r0 : g.A + r0 * g.lda;
      s.B = g.B + gi * g.group_stride;
      s.B2 = g.B2 ? g.B2 + gi * g.group_stride : nullptr;
      s.e = epi_rows_from<T>(g.e, r0);
      s.groups = 1;
      gemm_simt<T>(s, st);
    }
    return;
  }
  dim3 grid((g.N + SBN - 1) / SBN, (g.M + SBM - 1) / SBM);
  gemm_simt_kernel<T><<<grid, 256, 0, st>>>(g.M, g.N, g.K, g.A, g.lda, g.a_mn, g.B, g.ldb, g.b_mn, g.e, g.B2);
}

template void gemm_simt<float>(const GemmArgs<float>&, cudaStream_t);
template void gemm_simt<bf16>(const GemmArgs<bf16>&, cudaStream_t);

}  // namespace ttt

// gemv.cu — the one-row product of a decode step (M = 1):
//
//   C[0, n] = x . B[n]  (+ x . B2[n]),   B, B2 [N][K] bf16 (row pitch ldb)
//
// followed by the column-pair epilogue of the GEMMs (epi_pair: residual,
// RoPE into the key/value ring, SwiGLU, store) or by the greedy pick
// (EPI_ARGMAX).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace ttt {

namespace {

// One-row product (M = 1, a decode step): C[0, n] = x . B[n] (+ x . B2[n]).
// The work is streaming B from HBM once, so it runs on SIMT cores rather
// than on 128-row tensor-core tiles: one warp per two adjacent output
// columns, 16-byte loads along K, a warp reduction, then the epilogue of
// the column pair (the same epi_pair as the GEMM's ragged-column path).
__device__ __forceinline__ float dot8(uint4 a, uint4 b) {
  const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = unbf2(ua[i]), fb = unbf2(ub[i]);
    s = fmaf(fa.x, fb.x, s);
    s = fmaf(fa.y, fb.y, s);
  }
  return s;
}

// KS warps share one column pair, each over a K range of its own, and their
// sums are added in a fixed order (KS > 1 when there are too few column
// pairs to give every SM several blocks).
template <bool DUAL, int KS>
__global__ void __launch_bounds__(256) gemv_row_kernel(const bf16* __restrict__ x, const bf16* __restrict__ B,
                                                       const bf16* __restrict__ B2, int N, int K, int64_t ldb,
                                                       Epi e) {
  constexpr int RP = 8 / KS;  // column pairs per block
  __shared__ float red[8][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rp = warp / KS, ks = warp % KS;
  const int n = 2 * (blockIdx.x * RP + rp);
  const int kchunk = ((K / 8 + KS - 1) / KS) * 8;
  const int k0 = ks * kchunk, k1 = min(K, k0 + kchunk);
  float a0 = 0.f, a1 = 0.f;
  // the first PRE weight chunks are loaded before waiting on the kernel
  // that writes x (weights are not written by the kernels this one may
  // overlap under programmatic launch)
  constexpr int PRE = 4;
  constexpr int NB = DUAL ? 4 : 2;
  uint4 wp[PRE][NB];
  const bf16* b0 = B + (int64_t)n * ldb;
  const bf16* b1 = b0 + ldb;
  if (n < N) {
#pragma unroll
    for (int i = 0; i < PRE; ++i) {
      const int k = k0 + lane * 8 + 256 * i;
      if (k < k1) {
        wp[i][0] = __ldg(reinterpret_cast<const uint4*>(b0 + k));
        wp[i][1] = __ldg(reinterpret_cast<const uint4*>(b1 + k));
        if (DUAL) {
          wp[i][NB - 2] = __ldg(reinterpret_cast<const uint4*>(B2 + (int64_t)n * ldb + k));
          wp[i][NB - 1] = __ldg(reinterpret_cast<const uint4*>(B2 + (int64_t)(n + 1) * ldb + k));
        }
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  if (n < N) {
#pragma unroll
    for (int i = 0; i < PRE; ++i) {
      const int k = k0 + lane * 8 + 256 * i;
      if (k < k1) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + k);
        a0 += dot8(xv, wp[i][0]);
        a1 += dot8(xv, wp[i][1]);
        if (DUAL) {
          a0 += dot8(xv, wp[i][NB - 2]);
          a1 += dot8(xv, wp[i][NB - 1]);
        }
      }
    }
#pragma unroll 4
    for (int k = k0 + lane * 8 + 256 * PRE; k < k1; k += 256) {
      const uint4 xv = *reinterpret_cast<const uint4*>(x + k);
      a0 += dot8(xv, __ldg(reinterpret_cast<const uint4*>(b0 + k)));
      a1 += dot8(xv, __ldg(reinterpret_cast<const uint4*>(b1 + k)));
      if (DUAL) {
        a0 += dot8(xv, __ldg(reinterpret_cast<const uint4*>(B2 + (int64_t)n * ldb + k)));
        a1 += dot8(xv, __ldg(reinterpret_cast<const uint4*>(B2 + (int64_t)(n + 1) * ldb + k)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a0 += __shfl_xor_sync(0xffffffffu, a0, o);
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
  }
  bool mine = lane == 0 && n < N;  // this thread holds the pair's sums
  if (KS > 1) {
    if (lane == 0) {
      red[warp][0] = a0;
      red[warp][1] = a1;
    }
    __syncthreads();
    mine = mine && ks == 0;
    if (mine) {
      a0 = a1 = 0.f;
#pragma unroll
      for (int t = 0; t < KS; ++t) {
        a0 += red[warp + t][0];
        a1 += red[warp + t][1];
      }
    }
  }
  if (e.kind != EPI_ARGMAX) {
    if (mine) epi_pair<bf16>(e, 0, n, a0, a1);
    return;
  }
  // greedy pick: the block's best key, then one atomic per block
  __shared__ unsigned long long skey[8];
  if (lane == 0) {
    const unsigned long long k0 = mine ? argmax_key(a0, n) : 0ull, k1 = mine ? argmax_key(a1, n + 1) : 0ull;
    skey[warp] = k0 > k1 ? k0 : k1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long k = 0ull;
#pragma unroll
    for (int w = 0; w < 8; ++w) k = skey[w] > k ? skey[w] : k;
    if (k) atomicMax((unsigned long long*)e.out, k);
  }
}

template <bool DUAL>
void launch_gemv(const GemmArgs<bf16>& g, int num_sms, cudaStream_t st) {
  // enough blocks for about four per SM
  const int64_t want = 4ll * num_sms;
  int ks = 1;
  while (ks < 8 && (int64_t)(g.N / 2) * ks / 8 < want) ks *= 2;
  const int rp = 8 / ks;
  const int blocks = (g.N / 2 + rp - 1) / rp;
  switch (ks) {
    case 1: launch_k(gemv_row_kernel<DUAL, 1>, blocks, 256, 0, st, g.A, g.B, g.B2, g.N, g.K, g.ldb, g.e); break;
    case 2: launch_k(gemv_row_kernel<DUAL, 2>, blocks, 256, 0, st, g.A, g.B, g.B2, g.N, g.K, g.ldb, g.e); break;
    case 4: launch_k(gemv_row_kernel<DUAL, 4>, blocks, 256, 0, st, g.A, g.B, g.B2, g.N, g.K, g.ldb, g.e); break;
    default: launch_k(gemv_row_kernel<DUAL, 8>, blocks, 256, 0, st, g.A, g.B, g.B2, g.N, g.K, g.ldb, g.e); break;
  }
}

}  // namespace

bool gemv_supported(const GemmArgs<bf16>& g) {
  auto a16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  return g.M == 1 && !g.a_mn && !g.b_mn && (g.N & 1) == 0 && (g.K & 7) == 0 && (g.ldb & 7) == 0 && a16(g.A) &&
         a16(g.B) && (!g.B2 || a16(g.B2));
}

int gemv_row(const GemmArgs<bf16>& g, int num_sms, cudaStream_t st) {
  if (g.B2)
    launch_gemv<true>(g, num_sms, st);
  else
    launch_gemv<false>(g, num_sms, st);
  return 0;
}

}  // namespace ttt

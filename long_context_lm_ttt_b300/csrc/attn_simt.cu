// attn_simt.cu — sliding-window causal attention, forward and chunk-local
// backward, one warp per (row, head) with fp32 arithmetic.  Used by the fp32
// check mode and as the GPU-side reference of the tensor-core kernels.
//
// Query at absolute position t (row r = t - pos0 of the chunk) attends to
// keys j with t - W < j <= t; key j lives in ring slot j mod R of its KV
// head (query head h reads KV head h / (H/Hkv)).  Keys before the chunk are
// constants: the backward produces dq over the whole window but dk, dv only
// for the chunk's own keys.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int MAXD = 8;  // head_dim <= 256

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <typename T>
__global__ void __launch_bounds__(128) attn_fwd_simt_kernel(AttnArgs a) {
  __shared__ float qs[4][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp;
  if (r >= a.n) return;
  const int h = blockIdx.y, hd = a.hd, group = a.H / a.Hkv, kvh = h / group;
  const int64_t pos = a.pos0 + r;
  const int64_t ldq = (int64_t)a.H * hd;
  const T* q = (const T*)a.q + r * ldq + h * hd;
  for (int d = lane; d < hd; d += 32) qs[warp][d] = to_f<T>(q[d]);
  __syncwarp();
  const float scale = rsqrtf((float)hd);
  const T* K = (const T*)a.kring + (int64_t)kvh * a.R * hd;
  const T* V = (const T*)a.vring + (int64_t)kvh * a.R * hd;
  const int64_t jlo = pos - a.W + 1 > 0 ? pos - a.W + 1 : 0;
  float m = -INFINITY, l = 0.f, acc[MAXD];
#pragma unroll
  for (int i = 0; i < MAXD; ++i) acc[i] = 0.f;
  for (int64_t jb = jlo; jb <= pos; jb += 32) {
    const int64_t j = jb + lane;
    float s = -INFINITY;
    if (j <= pos) {
      const T* kr = K + (j % a.R) * hd;
      float dot = 0.f;
      for (int d = 0; d < hd; ++d) dot = fmaf(qs[warp][d], to_f<T>(kr[d]), dot);
      s = dot * scale;
    }
    const float mn = fmaxf(m, warp_max(s));
    const float p = (j <= pos) ? expf(s - mn) : 0.f;
    const float al = expf(m - mn);
    l = l * al + warp_sum(p);
#pragma unroll
    for (int i = 0; i < MAXD; ++i) acc[i] *= al;
    const int cnt = (int)((pos - jb + 1) < 32 ? (pos - jb + 1) : 32);
    for (int t = 0; t < cnt; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
      const T* vr = V + ((jb + t) % a.R) * hd;
#pragma unroll
      for (int i = 0; i < MAXD; ++i) {
        const int d = lane + 32 * i;
        if (d < hd) acc[i] = fmaf(pt, to_f<T>(vr[d]), acc[i]);
      }
    }
    m = mn;
  }
  T* o = (T*)a.o + r * ldq + h * hd;
  const float il = 1.0f / l;
#pragma unroll
  for (int i = 0; i < MAXD; ++i) {
    const int d = lane + 32 * i;
    if (d < hd) o[d] = from_f<T>(acc[i] * il);
  }
  if (lane == 0) a.lse[(int64_t)h * a.ld_lse + r] = m + logf(l);
}

// D[h][r] = sum_d dO[r,h,d] * O[r,h,d]
template <typename T>
__global__ void attn_bwd_prep_kernel(AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp;
  if (r >= a.n) return;
  const int h = blockIdx.y, hd = a.hd;
  const int64_t off = r * (int64_t)a.H * hd + h * hd;
  const T* dO = (const T*)a.dout + off;
  const T* O = (const T*)a.out + off;
  float s = 0.f;
  for (int d = lane; d < hd; d += 32) s = fmaf(to_f<T>(dO[d]), to_f<T>(O[d]), s);
  s = warp_sum(s);
  if (lane == 0) a.Dsum[(int64_t)h * a.ld_lse + r] = s;
}

// dq over the whole window of each query
template <typename T>
__global__ void __launch_bounds__(128) attn_bwd_dq_simt_kernel(AttnArgs a) {
  __shared__ float qs[4][256];
  __shared__ float gs[4][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp;
  if (r >= a.n) return;
  const int h = blockIdx.y, hd = a.hd, group = a.H / a.Hkv, kvh = h / group;
  const int64_t pos = a.pos0 + r;
  const int64_t ldq = (int64_t)a.H * hd;
  const T* q = (const T*)a.q + r * ldq + h * hd;
  const T* dO = (const T*)a.dout + r * ldq + h * hd;
  for (int d = lane; d < hd; d += 32) {
    qs[warp][d] = to_f<T>(q[d]);
    gs[warp][d] = to_f<T>(dO[d]);
  }
  __syncwarp();
  const float scale = rsqrtf((float)hd);
  const float lse = a.lse[(int64_t)h * a.ld_lse + r];
  const float Dt = a.Dsum[(int64_t)h * a.ld_lse + r];
  const T* K = (const T*)a.kring + (int64_t)kvh * a.R * hd;
  const T* V = (const T*)a.vring + (int64_t)kvh * a.R * hd;
  const int64_t jlo = pos - a.W + 1 > 0 ? pos - a.W + 1 : 0;
  float acc[MAXD];
#pragma unroll
  for (int i = 0; i < MAXD; ++i) acc[i] = 0.f;
  for (int64_t jb = jlo; jb <= pos; jb += 32) {
    const int64_t j = jb + lane;
    float ds = 0.f;
    if (j <= pos) {
      const T* kr = K + (j % a.R) * hd;
      const T* vr = V + (j % a.R) * hd;
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < hd; ++d) {
        s = fmaf(qs[warp][d], to_f<T>(kr[d]), s);
        dp = fmaf(gs[warp][d], to_f<T>(vr[d]), dp);
      }
      const float p = expf(s * scale - lse);
      ds = p * (dp - Dt) * scale;
    }
    const int cnt = (int)((pos - jb + 1) < 32 ? (pos - jb + 1) : 32);
    for (int t = 0; t < cnt; ++t) {
      const float dst = __shfl_sync(0xffffffffu, ds, t);
      const T* kr = K + ((jb + t) % a.R) * hd;
#pragma unroll
      for (int i = 0; i < MAXD; ++i) {
        const int d = lane + 32 * i;
        if (d < hd) acc[i] = fmaf(dst, to_f<T>(kr[d]), acc[i]);
      }
    }
  }
  const int64_t ldg = (int64_t)(a.H + 2 * a.Hkv) * hd;
  T* dq = (T*)a.dqkv + r * ldg + h * hd;
#pragma unroll
  for (int i = 0; i < MAXD; ++i) {
    const int d = lane + 32 * i;
    if (d < hd) dq[d] = from_f<T>(acc[i]);
  }
}

// dk, dv of the chunk's own keys, summed over the heads of the KV group
template <typename T>
__global__ void __launch_bounds__(128) attn_bwd_dkv_simt_kernel(AttnArgs a) {
  __shared__ float ks[4][256];
  __shared__ float vs[4][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rj = blockIdx.x * 4 + warp;
  if (rj >= a.n) return;
  const int kvh = blockIdx.y, hd = a.hd, group = a.H / a.Hkv;
  const int64_t slot = (a.pos0 + rj) % a.R;
  const T* kr = (const T*)a.kring + ((int64_t)kvh * a.R + slot) * hd;
  const T* vr = (const T*)a.vring + ((int64_t)kvh * a.R + slot) * hd;
  for (int d = lane; d < hd; d += 32) {
    ks[warp][d] = to_f<T>(kr[d]);
    vs[warp][d] = to_f<T>(vr[d]);
  }
  __syncwarp();
  const float scale = rsqrtf((float)hd);
  const int64_t ldq = (int64_t)a.H * hd;
  const int tmax = (rj + a.W - 1) < (a.n - 1) ? (rj + a.W - 1) : (a.n - 1);
  float dk[MAXD], dv[MAXD];
#pragma unroll
  for (int i = 0; i < MAXD; ++i) dk[i] = dv[i] = 0.f;
  for (int g = 0; g < group; ++g) {
    const int h = kvh * group + g;
    for (int tb = rj; tb <= tmax; tb += 32) {
      const int t = tb + lane;
      float ds = 0.f, p = 0.f;
      if (t <= tmax) {
        const T* q = (const T*)a.q + t * ldq + h * hd;
        const T* dO = (const T*)a.dout + t * ldq + h * hd;
        float s = 0.f, dp = 0.f;
        for (int d = 0; d < hd; ++d) {
          s = fmaf(to_f<T>(q[d]), ks[warp][d], s);
          dp = fmaf(to_f<T>(dO[d]), vs[warp][d], dp);
        }
        p = expf(s * scale - a.lse[(int64_t)h * a.ld_lse + t]);
        ds = p * (dp - a.Dsum[(int64_t)h * a.ld_lse + t]) * scale;
      }
      const int cnt = (tmax - tb + 1) < 32 ? (tmax - tb + 1) : 32;
      for (int u = 0; u < cnt; ++u) {
        const float dsu = __shfl_sync(0xffffffffu, ds, u);
        const float pu = __shfl_sync(0xffffffffu, p, u);
        const T* q = (const T*)a.q + (tb + u) * ldq + h * hd;
        const T* dO = (const T*)a.dout + (tb + u) * ldq + h * hd;
#pragma unroll
        for (int i = 0; i < MAXD; ++i) {
          const int d = lane + 32 * i;
          if (d < hd) {
            dk[i] = fmaf(dsu, to_f<T>(q[d]), dk[i]);
            dv[i] = fmaf(pu, to_f<T>(dO[d]), dv[i]);
          }
        }
      }
    }
  }
  const int64_t ldg = (int64_t)(a.H + 2 * a.Hkv) * hd;
  T* dkp = (T*)a.dqkv + rj * ldg + (int64_t)a.H * hd + kvh * hd;
  T* dvp = (T*)a.dqkv + rj * ldg + (int64_t)(a.H + a.Hkv) * hd + kvh * hd;
#pragma unroll
  for (int i = 0; i < MAXD; ++i) {
    const int d = lane + 32 * i;
    if (d < hd) {
      dkp[d] = from_f<T>(dk[i]);
      dvp[d] = from_f<T>(dv[i]);
    }
  }
}

}  // namespace

template <typename T>
void attn_fwd_simt(const AttnArgs& a, cudaStream_t st) {
  if (a.n <= 0) return;
  dim3 grid((a.n + 3) / 4, a.H);
  attn_fwd_simt_kernel<T><<<grid, 128, 0, st>>>(a);
}

template <typename T>
void attn_bwd_simt(const AttnArgs& a, cudaStream_t st) {
  if (a.n <= 0) return;
  dim3 grid((a.n + 3) / 4, a.H);
  attn_bwd_prep_kernel<T><<<grid, 128, 0, st>>>(a);
  attn_bwd_dq_simt_kernel<T><<<grid, 128, 0, st>>>(a);
  dim3 grid_kv((a.n + 3) / 4, a.Hkv);
  attn_bwd_dkv_simt_kernel<T><<<grid_kv, 128, 0, st>>>(a);
}

template void attn_fwd_simt<float>(const AttnArgs&, cudaStream_t);
template void attn_fwd_simt<bf16>(const AttnArgs&, cudaStream_t);
template void attn_bwd_simt<float>(const AttnArgs&, cudaStream_t);
template void attn_bwd_simt<bf16>(const AttnArgs&, cudaStream_t);

}  // namespace ttt

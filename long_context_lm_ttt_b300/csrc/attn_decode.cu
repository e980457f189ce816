// attn_decode.cu — sliding-window attention of ONE query position (a decode
// step), split over the key range so that the whole GPU streams the window.
//
//   o_h = sum_j softmax_j(q_h . k_j / sqrt(hd)) v_j,   j in [max(0, t-W+1), t]
//
// attn_decode_part_kernel: one CTA per (KV head, key slice).  Its four warps
// take every fourth tile of 32 keys of the slice; the G = H / Hkv query
// heads of the KV group share each key and value row read.  For the scores
// lane j reads key j of the tile (its whole row, 16 bytes at a time), so a
// warp has 32 rows in flight; for P.V lane i holds hd / 32 consecutive
// output dimensions and the probabilities come by shuffle.  Each warp keeps
// an online softmax per query head (running max, sum, unnormalised
// output), updated once per tile; the CTA folds its warps together and
// writes (max, sum, output) of the slice.
// attn_decode_combine_kernel: one CTA per query head folds the slices and
// writes o (row 0) and the log-sum-exp.
// Scores use log2 units (q.k * log2(e) / sqrt(hd)) and exp2f throughout.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace ttt {

namespace {

constexpr int kDecWarps = 4;
constexpr int kMaxGroup = 8;  // query heads per KV head
constexpr int kMaxEpl = 8;    // dimensions per lane (hd <= 256)

template <typename T, int EPL>
__global__ void __launch_bounds__(kDecWarps * 32)
    attn_decode_part_kernel(const T* __restrict__ q, const T* __restrict__ kring, const T* __restrict__ vring,
                            int H, int Hkv, int W, int R, int64_t pos, int splits, float scale_log2,
                            float* __restrict__ part) {
  constexpr int hd = EPL * 32;
  const int kvh = blockIdx.x, sp = blockIdx.y;
  const int G = H / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t j_lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
  const int64_t cnt = pos - j_lo + 1;
  const int64_t s0 = j_lo + cnt * sp / splits, s1 = j_lo + cnt * (sp + 1) / splits;

  // the group's query rows, scaled into log2 units, shared by every lane
  __shared__ float sq[kMaxGroup][hd];
  for (int i = threadIdx.x; i < G * hd; i += blockDim.x)
    sq[i / hd][i % hd] = to_f<T>(q[(int64_t)kvh * G * hd + i]) * scale_log2;
  __syncthreads();

  float m[kMaxGroup], l[kMaxGroup], acc[kMaxGroup][EPL];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
  }
  // tiles of 32 keys: lane j scores key kb + j over the whole head
  // dimension, then the lanes own EPL output dimensions for P.V
  for (int64_t kb = s0 + 32 * warp; kb < s1; kb += 32 * kDecWarps) {
    const int64_t k = kb + lane;
    const bool valid = k < s1;
    float sc[kMaxGroup];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) sc[g] = 0.f;
    if (valid) {
      const T* kr = kring + ((int64_t)kvh * R + k % R) * hd;
#pragma unroll
      for (int c = 0; c < hd; c += 16 / (int)sizeof(T)) {
        float kv[16 / sizeof(T)];
        if constexpr (sizeof(T) == 2) {
          const uint4 u = *reinterpret_cast<const uint4*>(kr + c);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 f = unbf2(w4[t]);
            kv[2 * t] = f.x;
            kv[2 * t + 1] = f.y;
          }
        } else {
          const float4 f = *reinterpret_cast<const float4*>(kr + c);
          kv[0] = f.x;
          kv[1] = f.y;
          kv[2] = f.z;
          kv[3] = f.w;
        }
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) {
          if (g >= G) break;
#pragma unroll
          for (int t = 0; t < (int)(16 / sizeof(T)); ++t) sc[g] = fmaf(sq[g][c + t], kv[t], sc[g]);
        }
      }
    }
    float p[kMaxGroup];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g >= G) break;
      const float s = valid ? sc[g] : -INFINITY;
      float mt = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float mn = fmaxf(m[g], mt);
      const float alpha = exp2f(m[g] - mn);  // 0 while m is -inf
      p[g] = exp2f(s - mn);
      float ps = p[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[g] = l[g] * alpha + ps;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] *= alpha;
      m[g] = mn;
    }
    const int nk = s1 - kb < 32 ? (int)(s1 - kb) : 32;
#pragma unroll 4
    for (int jj = 0; jj < nk; ++jj) {
      const T* vr = vring + ((int64_t)kvh * R + (kb + jj) % R) * hd + lane * EPL;
      float vv[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) vv[e] = to_f<T>(vr[e]);
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g >= G) break;
        const float pj = __shfl_sync(0xffffffffu, p[g], jj);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pj, vv[e], acc[g][e]);
      }
    }
  }
  // fold the four warps: per (query head, dimension)
  __shared__ float sm[kDecWarps][kMaxGroup], sl[kDecWarps][kMaxGroup];
  __shared__ float sa[kDecWarps][kMaxGroup][hd];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g >= G) break;
    if (lane == 0) {
      sm[warp][g] = m[g];
      sl[warp][g] = l[g];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) sa[warp][g][lane * EPL + e] = acc[g][e];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * (hd + 2); idx += blockDim.x) {
    const int g = idx / (hd + 2), e = idx % (hd + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm[w][g]);
    float v = 0.f;
    if (e == hd) {
      v = M;
    } else if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = exp2f(sm[w][g] - M);
        v += f * (e == hd + 1 ? sl[w][g] : sa[w][g][e]);
      }
    }
    part[((int64_t)(kvh * G + g) * splits + sp) * (hd + 2) + e] = v;
  }
}

// One CTA per query head: warp 0 reduces the slices' maxima and sums (two
// slices per lane), leaving each slice's weight exp2(m_s - M) in shared
// memory; then every thread sums its output dimensions over the slices with
// independent loads.
template <typename T>
__global__ void attn_decode_combine_kernel(const float* __restrict__ part, int hd, int splits, T* __restrict__ o,
                                           float* __restrict__ lse, int ld_lse) {
  __shared__ float wsh[kMaxDecodeSplits];
  __shared__ float sML[2];
  const int h = blockIdx.x;
  const int64_t st = hd + 2;
  const float* ph = part + (int64_t)h * splits * st;
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    const float m0 = l < splits ? ph[l * st + hd] : -INFINITY;
    const float m1 = l + 32 < splits ? ph[(l + 32) * st + hd] : -INFINITY;
    float M = fmaxf(m0, m1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
    const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
    float L = (w0 > 0.f ? w0 * ph[l * st + hd + 1] : 0.f) + (w1 > 0.f ? w1 * ph[(l + 32) * st + hd + 1] : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (l < splits) wsh[l] = w0;
    if (l + 32 < splits) wsh[l + 32] = w1;
    if (l == 0) {
      sML[0] = M;
      sML[1] = L;
    }
  }
  __syncthreads();
  const float M = sML[0], L = sML[1];
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  for (int e = threadIdx.x; e < hd; e += blockDim.x) {
    float a = 0.f;
#pragma unroll 8
    for (int s2 = 0; s2 < splits; ++s2) {
      const float w = wsh[s2];
      if (w > 0.f) a = fmaf(w, ph[s2 * st + e], a);
    }
    o[(int64_t)h * hd + e] = from_f<T>(a * inv);
  }
  if (threadIdx.x == 0 && lse) lse[(int64_t)h * ld_lse] = (M + log2f(L)) * 0.69314718055994531f;
}

template <typename T, int EPL>
void launch_part(const AttnArgs& a, int splits, float* part, cudaStream_t st) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.hd);
  attn_decode_part_kernel<T, EPL><<<dim3(a.Hkv, splits), kDecWarps * 32, 0, st>>>(
      (const T*)a.q, (const T*)a.kring, (const T*)a.vring, a.H, a.Hkv, a.W, a.R, a.pos0, splits, scale_log2, part);
}

}  // namespace

bool attn_decode_supported(const AttnArgs& a) {
  // the kernels read query, key and value rows with 16-byte vector loads
  const bool aligned =
      (((uintptr_t)a.q | (uintptr_t)a.kring | (uintptr_t)a.vring | (uintptr_t)a.o) & 15) == 0;
  return a.n == 1 && a.hd % 32 == 0 && a.hd / 32 <= kMaxEpl && a.H % a.Hkv == 0 && a.H / a.Hkv <= kMaxGroup &&
         aligned;
}

int attn_decode_splits(const AttnArgs& a, int num_sms) {
  const int64_t keys = std::min<int64_t>(a.pos0 + 1, a.W);
  // two CTAs per SM over the KV heads, at least 32 keys per slice
  int s = (2 * num_sms + a.Hkv - 1) / a.Hkv;
  const int64_t by_keys = (keys + 31) / 32;
  if (s > by_keys) s = (int)by_keys;
  return s < 1 ? 1 : (s > kMaxDecodeSplits ? kMaxDecodeSplits : s);
}

template <typename T>
void attn_decode(const AttnArgs& a, int splits, float* part, cudaStream_t st) {
  switch (a.hd / 32) {
    case 1: launch_part<T, 1>(a, splits, part, st); break;
    case 2: launch_part<T, 2>(a, splits, part, st); break;
    case 3: launch_part<T, 3>(a, splits, part, st); break;
    case 4: launch_part<T, 4>(a, splits, part, st); break;
    case 5: launch_part<T, 5>(a, splits, part, st); break;
    case 6: launch_part<T, 6>(a, splits, part, st); break;
    case 7: launch_part<T, 7>(a, splits, part, st); break;
    default: launch_part<T, 8>(a, splits, part, st); break;
  }
  attn_decode_combine_kernel<T><<<a.H, a.hd, 0, st>>>(part, a.hd, splits, (T*)a.o, a.lse, a.ld_lse);
}

template void attn_decode<bf16>(const AttnArgs&, int, float*, cudaStream_t);
template void attn_decode<float>(const AttnArgs&, int, float*, cudaStream_t);

}  // namespace ttt

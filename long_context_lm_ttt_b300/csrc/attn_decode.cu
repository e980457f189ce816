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
//
// bf16 (the model's precision) takes attn_decode_bulk_kernel instead: one
// CTA per (KV head, key slice) as above, but the slice's key and value rows
// come into shared memory by 1-D bulk copies (contiguous ring rows, at
// most two pieces where the ring wraps), P keys per pass in three buffers,
// so that a CTA has 96 KB of the window in flight from its first cycle.
// Its eight warps take groups of 8 keys of a pass in turn; lane i owns
// hd / 32 consecutive dimensions of q, of the key and value rows and of the
// output.  A group's 8 scores are summed over the warp by a transposed
// butterfly (each exchange halves the keys a lane keeps: 9 shuffles per
// query head instead of 40), and its probabilities reach every lane
// through shared memory.  The last CTA of a KV head to finish
// (a counter per KV head) folds that head group's slices, in slice order,
// and leaves the counter at zero for the next launch.
// Scores use log2 units (q.k * log2(e) / sqrt(hd)) and exp2f throughout.
// The query position comes either as a value or from a device word, so that
// one captured launch serves every decode step.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "bounds.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace ttt {

TTT_BOUNDS_UNIT(attn_decode)

namespace {

constexpr int kDecWarps = 4;
constexpr int kMaxGroup = 8;  // query heads per KV head
constexpr int kMaxEpl = 8;    // dimensions per lane (hd <= 256)

template <typename T, int EPL>
__global__ void __launch_bounds__(kDecWarps * 32)
    attn_decode_part_kernel(const T* __restrict__ q, const T* __restrict__ kring, const T* __restrict__ vring,
                            int H, int Hkv, int W, int R, int64_t pos, const int64_t* __restrict__ pos_dev,
                            int splits, float scale_log2, float* __restrict__ part) {
  constexpr int hd = EPL * 32;
  const int kvh = blockIdx.x, sp = blockIdx.y;
  const int G = H / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (pos_dev) pos = *pos_dev;
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

enum : int { ERR_DEC_WAIT = 301, ERR_DEC_DRAIN = 302 };

// keys per pass: at most 16 KB of key rows (and as many of value rows), a
// multiple of 32 so that each warp's quarter is whole groups of 8 keys
template <int EPL>
constexpr int dec_pass_keys() {
  return (8192 / (EPL * 32)) / 32 * 32;
}
constexpr int kDecBufs = 3;  // passes in flight per CTA
template <int EPL>
constexpr int dec_smem_bytes() {
  return kDecBufs * 2 * dec_pass_keys<EPL>() * EPL * 32 * 2;  // buffers x (K, V)
}

// EPL consecutive bf16 of shared memory as floats (4-byte loads when EPL is
// even, so the address is 4-byte aligned)
template <int EPL>
__device__ __forceinline__ void load_dims(const bf16* p, float (&v)[EPL]) {
  if constexpr (EPL % 2 == 0) {
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const float2 f = unbf2(*reinterpret_cast<const uint32_t*>(p + e));
      v[e] = f.x;
      v[e + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = __bfloat162float(p[e]);
  }
}

constexpr int kBulkWarps = 8;

// GM: the register arrays' size in query heads (G <= GM)
template <int EPL, int GM>
__global__ void __launch_bounds__(kBulkWarps * 32, 2)
    attn_decode_bulk_kernel(const bf16* __restrict__ q, const bf16* __restrict__ kring,
                            const bf16* __restrict__ vring, int H, int Hkv, int W, int R, int64_t pos,
                            const int64_t* __restrict__ pos_dev, int splits, float scale_log2, float* part,
                            int* count, bf16* __restrict__ o, float* __restrict__ lse, int ld_lse, int* err) {
  constexpr int hd = EPL * 32;
  constexpr int P = dec_pass_keys<EPL>();
  constexpr uint32_t ROW = hd * 2;    // bytes of one key or value row
  extern __shared__ __align__(128) uint8_t dsm[];
  bf16* sk = reinterpret_cast<bf16*>(dsm);  // [kDecBufs][P][hd]
  bf16* sv = sk + kDecBufs * P * hd;        // [kDecBufs][P][hd]
  __shared__ __align__(8) uint64_t bar[kDecBufs];
  __shared__ int abort_flag, last;
  __shared__ __align__(16) float sprob[kBulkWarps][GM][8];  // a group's probabilities, per warp
  const int kvh = blockIdx.x, sid = blockIdx.y;  // KV head, key slice
  const int G = H / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < kDecBufs; ++b) tc::mbar_init(tc::smem_u32(&bar[b]), 1);
    tc::fence_mbar_init();
    abort_flag = 0;
  }
  // q, the newest key and value rows and the position come from the
  // kernels before this one
  pdl_wait();
  pdl_trigger();
  if (pos_dev) pos = *pos_dev;
  const int64_t j_lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
  const int64_t cnt = pos - j_lo + 1;
  const int64_t s0 = j_lo + cnt * sid / splits, s1 = j_lo + cnt * (sid + 1) / splits;
  const int npass = (int)((s1 - s0 + P - 1) / P);
  __syncthreads();
  // pass ps: keys [s0 + ps P, ...) into buffer ps % kDecBufs (thread 0 only)
  auto issue = [&](int ps) {
    const int buf = ps % kDecBufs;
    const int64_t k0 = s0 + (int64_t)ps * P;
    const int n = (int)(s1 - k0 < P ? s1 - k0 : P);
    const uint32_t b = tc::smem_u32(&bar[buf]);
    tc::mbar_arrive_expect_tx(b, 2u * n * ROW);
    const int slot = (int)(k0 % R);
    const int n1 = n < R - slot ? n : R - slot;
    const int64_t g0 = ((int64_t)kvh * R + slot) * hd;
    // the debug build checks that both parts lie inside the head's ring and
    // the pass buffer (the 16-byte rule of the copies holds by construction:
    // rows of hd * 2 bytes, hd a multiple of 32, 16-byte aligned rings)
    if (!(TTT_IN(KB_ATTN_DECODE, kvh, Hkv) && TTT_IN(KB_ATTN_DECODE, slot, R) &&
          TTT_IN(KB_ATTN_DECODE, slot + n1 - 1, R) && TTT_IN(KB_ATTN_DECODE, n - 1, P) &&
          TTT_IN(KB_ATTN_DECODE, n - n1, slot + 1))) {
      *(volatile int*)&abort_flag = 1;
      return;
    }
    tc::bulk_load_1d(tc::smem_u32(sk + (int64_t)buf * P * hd), kring + g0, n1 * ROW, b);
    tc::bulk_load_1d(tc::smem_u32(sv + (int64_t)buf * P * hd), vring + g0, n1 * ROW, b);
    if (n > n1) {  // the ring wraps inside the pass
      const int64_t g1 = (int64_t)kvh * R * hd;
      tc::bulk_load_1d(tc::smem_u32(sk + ((int64_t)buf * P + n1) * hd), kring + g1, (n - n1) * ROW, b);
      tc::bulk_load_1d(tc::smem_u32(sv + ((int64_t)buf * P + n1) * hd), vring + g1, (n - n1) * ROW, b);
    }
  };
  if (threadIdx.x == 0)
    for (int ps = 0; ps < kDecBufs && ps < npass; ++ps) issue(ps);

  // the lane's dimensions of the group's query rows, in log2 units
  float qr[GM][EPL];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      qr[g][e] = g < G ? __bfloat162float(q[((int64_t)kvh * G + g) * hd + lane * EPL + e]) * scale_log2 : 0.f;
  }
  float m[GM], l[GM], acc[GM][EPL];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
  }

  int done = 0;  // passes whose copies have landed
  bool aborted = false;
  for (int ps = 0; ps < npass; ++ps) {
    const int buf = ps % kDecBufs;
    const bool ok =
        tc::mbar_wait(tc::smem_u32(&bar[buf]), (ps / kDecBufs) & 1, err, ERR_DEC_WAIT, (volatile int*)&abort_flag);
    if (!__syncthreads_and(ok)) {  // every thread leaves the loop together
      aborted = true;
      break;
    }
    done = ps + 1;
    const int64_t k0 = s0 + (int64_t)ps * P;
    const int n = (int)(s1 - k0 < P ? s1 - k0 : P);
    const bf16* kt = sk + (int64_t)buf * P * hd;
    const bf16* vt = sv + (int64_t)buf * P * hd;
    // groups of 8 keys: warp w takes groups w, w + kBulkWarps, ... of the pass
    for (int k8 = warp * 8; k8 < n; k8 += 8 * kBulkWarps) {
      const int nk = n - k8 < 8 ? n - k8 : 8;
      // partial dot products over the lane's dimensions
      float v[GM][8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float kv[EPL];
        if (j < nk) {
          load_dims<EPL>(kt + (int64_t)(k8 + j) * hd + lane * EPL, kv);
        } else {
#pragma unroll
          for (int e = 0; e < EPL; ++e) kv[e] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) d = fmaf(qr[g][e], kv[e], d);
          v[g][j] = d;
        }
      }
      // transposed butterfly over the warp: each exchange halves the keys a
      // lane keeps, so 8 sums take 4 + 2 + 1 + 2 shuffles; afterwards lane
      // L holds in v[g][0] the score of key jl (bits 4, 3, 2 of L)
      const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
      const int jl = (b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0);
      const bool valid = jl < nk;
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g >= G) break;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float snd = b4 ? v[g][i] : v[g][i + 4], kp = b4 ? v[g][i + 4] : v[g][i];
          v[g][i] = kp + __shfl_xor_sync(0xffffffffu, snd, 16);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float snd = b3 ? v[g][i] : v[g][i + 2], kp = b3 ? v[g][i + 2] : v[g][i];
          v[g][i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
        }
        {
          const float snd = b2 ? v[g][0] : v[g][1], kp = b2 ? v[g][1] : v[g][0];
          v[g][0] = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
        }
        v[g][0] += __shfl_xor_sync(0xffffffffu, v[g][0], 2);
        v[g][0] += __shfl_xor_sync(0xffffffffu, v[g][0], 1);
        // online softmax over the group's keys (one per 4-lane set)
        const float sc = valid ? v[g][0] : -INFINITY;
        float mt = sc;
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float mn = fmaxf(m[g], mt);
        const float alpha = exp2f(m[g] - mn);  // 0 while m is -inf
        const float p = valid ? exp2f(sc - mn) : 0.f;
        float ps_ = p;
        ps_ += __shfl_xor_sync(0xffffffffu, ps_, 4);
        ps_ += __shfl_xor_sync(0xffffffffu, ps_, 8);
        ps_ += __shfl_xor_sync(0xffffffffu, ps_, 16);
        l[g] = l[g] * alpha + ps_;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[g][e] *= alpha;
        m[g] = mn;
        if ((lane & 3) == 0) sprob[warp][g][jl] = p;
      }
      __syncwarp();
      float pr[GM][8];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g >= G) break;
        const float4 a = *reinterpret_cast<const float4*>(&sprob[warp][g][0]);
        const float4 b = *reinterpret_cast<const float4*>(&sprob[warp][g][4]);
        pr[g][0] = a.x; pr[g][1] = a.y; pr[g][2] = a.z; pr[g][3] = a.w;
        pr[g][4] = b.x; pr[g][5] = b.y; pr[g][6] = b.z; pr[g][7] = b.w;
      }
      __syncwarp();  // sp is rewritten by the next group
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < nk) {
          float vv[EPL];
          load_dims<EPL>(vt + (int64_t)(k8 + j) * hd + lane * EPL, vv);
#pragma unroll
          for (int g = 0; g < GM; ++g) {
            if (g >= G) break;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pr[g][j], vv[e], acc[g][e]);
          }
        }
      }
    }
    __syncthreads();  // every warp is done with the buffer
    if (threadIdx.x == 0 && ps + kDecBufs < npass) issue(ps + kDecBufs);
  }
  if (aborted) {
    // a wait gave up: let the copies already issued land (bounded) before
    // the CTA's shared memory goes away, write no slice, but still count
    // the CTA so that the counter returns to zero
    if (threadIdx.x == 0) {
      for (int ps = done; ps < npass && ps < done + kDecBufs; ++ps) {
        const uint32_t b = tc::smem_u32(&bar[ps % kDecBufs]);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(b, (ps / kDecBufs) & 1)) {
          if (clock64() - t0 > tc::kWaitClocks) {
            atomicCAS(err, 0, ERR_DEC_DRAIN);
            break;
          }
        }
      }
    }
    if (threadIdx.x == 0 && atomicAdd(&count[kvh], 1) == splits - 1) count[kvh] = 0;
    __syncthreads();
    return;
  }
  // fold the warps (the key buffers are free now) and write the slice:
  // rows of PS floats (16-byte aligned), the output, then max and sum
  constexpr int PS = hd + 4;
  float* sa = reinterpret_cast<float*>(dsm);  // [kBulkWarps][GM][hd]
  __shared__ float sm[kBulkWarps][GM], sl[kBulkWarps][GM];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    if (g >= G) break;
    if (lane == 0) {
      sm[warp][g] = m[g];
      sl[warp][g] = l[g];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) sa[(warp * GM + g) * hd + lane * EPL + e] = acc[g][e];
  }
  __syncthreads();
  float* pg = part + (int64_t)kvh * G * splits * PS;  // the head group's slices [G][splits][PS]
  for (int idx = threadIdx.x; idx < G * (hd + 2); idx += blockDim.x) {
    const int g = idx / (hd + 2), e = idx % (hd + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kBulkWarps; ++w) M = fmaxf(M, sm[w][g]);
    float v = 0.f;
    if (e == hd) {
      v = M;
    } else if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kBulkWarps; ++w) {
        const float f = exp2f(sm[w][g] - M);
        v += f * (e == hd + 1 ? sl[w][g] : sa[(w * GM + g) * hd + e]);
      }
    }
    pg[((int64_t)g * splits + sid) * PS + e] = v;
  }
  // the last CTA of this KV head folds the head group's slices
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&count[kvh], 1) == splits - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // weights exp2(m_t - M) of the slices (0 for empty ones) and the sums,
  // one warp per query head; then every thread folds 4 dimensions of one
  // head over all slices with 16-byte loads, many in flight
  float* sw = reinterpret_cast<float*>(dsm);  // [G][kMaxDecodeSplits]
  __shared__ float sM[kMaxGroup], sL[kMaxGroup];
  for (int g = warp; g < G; g += kBulkWarps) {
    const float* ph = pg + (int64_t)g * splits * PS + hd;
    float2 ml0 = make_float2(-INFINITY, 0.f), ml1 = make_float2(-INFINITY, 0.f);
    if (lane < splits) ml0 = __ldcg(reinterpret_cast<const float2*>(ph + (int64_t)lane * PS));
    if (lane + 32 < splits) ml1 = __ldcg(reinterpret_cast<const float2*>(ph + (int64_t)(lane + 32) * PS));
    float M = fmaxf(ml0.x, ml1.x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w0 = ml0.x == -INFINITY ? 0.f : exp2f(ml0.x - M);
    const float w1 = ml1.x == -INFINITY ? 0.f : exp2f(ml1.x - M);
    float L = w0 * ml0.y + w1 * ml1.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    sw[g * kMaxDecodeSplits + lane] = w0;
    sw[g * kMaxDecodeSplits + lane + 32] = w1;
    if (lane == 0) {
      sM[g] = M;
      sL[g] = L;
    }
  }
  __syncthreads();
  constexpr int QD = hd / 4;
  for (int it = threadIdx.x; it < G * QD; it += blockDim.x) {
    const int g = it / QD, qd = it % QD;
    const float* pq = pg + (int64_t)g * splits * PS + 4 * qd;
    const float* wg = sw + g * kMaxDecodeSplits;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 16
    for (int t = 0; t < splits; ++t) {
      const float w = wg[t];
      const float4 v = __ldcg(reinterpret_cast<const float4*>(pq + (int64_t)t * PS));
      a.x = fmaf(w, v.x, a.x);
      a.y = fmaf(w, v.y, a.y);
      a.z = fmaf(w, v.z, a.z);
      a.w = fmaf(w, v.w, a.w);
    }
    const float L = sL[g];
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    bf16* og = o + ((int64_t)kvh * G + g) * hd + 4 * qd;
    og[0] = __float2bfloat16_rn(a.x * inv);
    og[1] = __float2bfloat16_rn(a.y * inv);
    og[2] = __float2bfloat16_rn(a.z * inv);
    og[3] = __float2bfloat16_rn(a.w * inv);
  }
  if (threadIdx.x < G && lse)
    lse[((int64_t)kvh * G + threadIdx.x) * ld_lse] = (sM[threadIdx.x] + log2f(sL[threadIdx.x])) * 0.69314718055994531f;
  if (threadIdx.x == 0) count[kvh] = 0;  // ready for the next launch
}

template <typename T, int EPL>
void launch_part(const AttnArgs& a, int splits, float* part, cudaStream_t st) {
  part += kDecCounters;  // the slices follow the counters
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.hd);
  attn_decode_part_kernel<T, EPL><<<dim3(a.Hkv, splits), kDecWarps * 32, 0, st>>>(
      (const T*)a.q, (const T*)a.kring, (const T*)a.vring, a.H, a.Hkv, a.W, a.R, a.pos0, a.pos_dev, splits, scale_log2, part);
}

template <int EPL, int GM>
int launch_bulk(const AttnArgs& a, int splits, float* part, int* err, cudaStream_t st) {
  static std::atomic<uint64_t> raised{0};
  auto kern = attn_decode_bulk_kernel<EPL, GM>;
  constexpr int smem = dec_smem_bytes<EPL>();
  if (raise_smem_limit(raised, kern, smem) != cudaSuccess) return -1;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.hd);
  int* count = reinterpret_cast<int*>(part);
  return launch_k(kern, dim3(a.Hkv, splits), kBulkWarps * 32, smem, st, (const bf16*)a.q, (const bf16*)a.kring,
                  (const bf16*)a.vring, a.H, a.Hkv, a.W, a.R, a.pos0, a.pos_dev, splits, scale_log2,
                  part + kDecCounters, count, (bf16*)a.o, a.lse, a.ld_lse, err) != cudaSuccess;
}
template <int EPL>
int launch_bulk_g(const AttnArgs& a, int splits, float* part, int* err, cudaStream_t st) {
  const int G = a.H / a.Hkv;
  if (G <= 2) return launch_bulk<EPL, 2>(a, splits, part, err, st);
  if (G == 3) return launch_bulk<EPL, 3>(a, splits, part, err, st);
  if (G == 4) return launch_bulk<EPL, 4>(a, splits, part, err, st);
  return launch_bulk<EPL, 8>(a, splits, part, err, st);
}

}  // namespace

bool attn_decode_supported(const AttnArgs& a) {
  // the kernels read query, key and value rows with 16-byte vector loads
  const bool aligned =
      (((uintptr_t)a.q | (uintptr_t)a.kring | (uintptr_t)a.vring | (uintptr_t)a.o) & 15) == 0;
  return a.n == 1 && a.hd % 32 == 0 && a.hd / 32 <= kMaxEpl && a.H % a.Hkv == 0 && a.H / a.Hkv <= kMaxGroup &&
         a.Hkv <= kDecCounters && aligned;
}

int attn_decode_splits(const AttnArgs& a, int num_sms) {
  // a position read on the device may be any: plan for a full window (the
  // slices past the last key come out empty and the fold skips them)
  const int64_t keys = a.pos_dev ? (int64_t)a.W : std::min<int64_t>(a.pos0 + 1, a.W);
  // two CTAs per SM over the KV heads (what the bulk kernel's registers
  // and 96 KB of buffers allow: one wave), at least 32 keys per slice
  int s = 2 * num_sms / a.Hkv;
  const int64_t by_keys = (keys + 31) / 32;
  if (s > by_keys) s = (int)by_keys;
  return s < 1 ? 1 : (s > kMaxDecodeSplits ? kMaxDecodeSplits : s);
}

int64_t attn_decode_scratch_elems(int H, int hd) {
  return kDecCounters + (int64_t)H * kMaxDecodeSplits * (hd + 4);
}

template <typename T>
int attn_decode(const AttnArgs& a, int splits, float* part, int* err, cudaStream_t st) {
  if constexpr (sizeof(T) == 2) {
    switch (a.hd / 32) {
      case 1: return launch_bulk_g<1>(a, splits, part, err, st);
      case 2: return launch_bulk_g<2>(a, splits, part, err, st);
      case 3: return launch_bulk_g<3>(a, splits, part, err, st);
      case 4: return launch_bulk_g<4>(a, splits, part, err, st);
      case 5: return launch_bulk_g<5>(a, splits, part, err, st);
      case 6: return launch_bulk_g<6>(a, splits, part, err, st);
      case 7: return launch_bulk_g<7>(a, splits, part, err, st);
      default: return launch_bulk_g<8>(a, splits, part, err, st);
    }
  }
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
  attn_decode_combine_kernel<T><<<a.H, a.hd, 0, st>>>(part + kDecCounters, a.hd, splits, (T*)a.o, a.lse, a.ld_lse);
  return 0;
}

template int attn_decode<bf16>(const AttnArgs&, int, float*, int*, cudaStream_t);
template int attn_decode<float>(const AttnArgs&, int, float*, int*, cudaStream_t);

}  // namespace ttt

// kernels.cu — the row-wise and element-wise kernels of the inner loop:
// embedding gather, RMSNorm forward/backward, RoPE tables and the inverse
// rotation of gradients, next-token targets, the vocabulary-slab softmax
// statistics of the streamed cross-entropy, its finalisation, the
// deterministic chunk-loss reduction, and weight packing.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ttt {

namespace {

constexpr int RB = 256;  // threads per row block

struct AddOp {
  __device__ float operator()(float a, float b) const { return a + b; }
  __device__ static float identity() { return 0.f; }
};
struct MaxOp {
  __device__ float operator()(float a, float b) const { return fmaxf(a, b); }
  __device__ static float identity() { return -INFINITY; }
};

// deterministic block reduction (fixed tree)
template <typename Op>
__device__ __forceinline__ float block_reduce(float v, Op op, float* sh) {
  const float ident = Op::identity();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  if (wid == 0) {
    v = lane < nw ? sh[lane] : ident;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sh[0] = v;
  }
  __syncthreads();
  float r = sh[0];
  __syncthreads();
  return r;
}

template <typename T>
__global__ void embed_kernel(const int32_t* __restrict__ tok, int d, const T* __restrict__ E,
                             float* __restrict__ x, int V, int* err_tok) {
  const int r = blockIdx.x;
  int64_t id = tok[r];
  if (id < 0 || id >= V) {      // out-of-range id: flag it, read row 0 instead
    if (threadIdx.x == 0) atomicOr(err_tok, 1);
    id = 0;
  }
  for (int c = threadIdx.x; c < d; c += blockDim.x) x[(int64_t)r * d + c] = to_f<T>(E[id * d + c]);
}

template <typename T>
__global__ void rmsnorm_fwd_kernel(const float* __restrict__ x, const float* __restrict__ g, int d,
                                   float eps, T* __restrict__ out, float* __restrict__ rr) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const float* xr = x + (int64_t)r * d;
  float s = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) s = fmaf(xr[c], xr[c], s);
  s = block_reduce(s, AddOp(), sh);
  const float rinv = 1.0f / sqrtf(s / (float)d + eps);
  for (int c = threadIdx.x; c < d; c += blockDim.x)
    out[(int64_t)r * d + c] = from_f<T>(g[c] * xr[c] * rinv);
  if (threadIdx.x == 0) rr[r] = rinv;
}

template <typename T>
__global__ void rmsnorm_bwd_kernel(const float* __restrict__ x, const float* __restrict__ g,
                                   const float* __restrict__ rr, const float* __restrict__ dy,
                                   const float* __restrict__ resid, int d, float* __restrict__ out,
                                   T* __restrict__ out_t) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const int64_t o = (int64_t)r * d;
  float s = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) s = fmaf(x[o + c] * g[c], dy[o + c], s);
  s = block_reduce(s, AddOp(), sh) / (float)d;
  const float ri = rr[r];
  const float r3 = ri * ri * ri;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float v = ri * g[c] * dy[o + c] - r3 * x[o + c] * s;
    if (resid) v += resid[o + c];
    out[o + c] = v;
    if (out_t) out_t[o + c] = from_f<T>(v);
  }
}

__global__ void rope_table_kernel(int64_t pos0, int n, int hd, double theta, float2* cs) {
  const int half = hd >> 1;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  const int r = idx / half, i = idx % half;
  const double inv = pow(theta, -(2.0 * (double)i) / (double)hd);
  const double ang = (double)(pos0 + r) * inv;
  double sn, cn;
  sincos(ang, &sn, &cn);
  cs[idx] = make_float2((float)cn, (float)sn);
}

template <typename T>
__global__ void rope_bwd_kernel(T* dqkv, int n, int ld, int n_rot_heads, int hd, const float2* cs) {
  const int half = hd >> 1;
  const int64_t total = (int64_t)n * n_rot_heads * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / (n_rot_heads * half));
    const int rem = (int)(idx % (n_rot_heads * half));
    const int h = rem / half, i = rem % half;
    T* p = dqkv + (int64_t)r * ld + h * hd + 2 * i;
    float2 v = load2<T>(p);
    const float2 c = cs[(int64_t)r * half + i];
    store2<T>(p, v.x * c.x + v.y * c.y, v.y * c.x - v.x * c.y);
  }
}

__global__ void targets_kernel(const int32_t* tok, int64_t T, int64_t pos0, int n, int32_t* tgt, int V,
                               int* err_tok) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n) return;
  const int64_t t = pos0 + r + 1;
  int y = t < T ? tok[t] : -1;
  if (y >= V || (t < T && y < 0)) {
    atomicOr(err_tok, 1);
    y = -1;
  }
  tgt[r] = y;
}

template <typename T>
__global__ void ce_slab_stats_kernel(const float* __restrict__ z, int64_t ldz, int nv,
                                     T* __restrict__ p, int64_t ldp, float* m_run, float* l_run,
                                     float* alpha, float* beta, int first) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const float* zr = z + (int64_t)r * ldz;
  float m = -INFINITY;
  for (int c = threadIdx.x; c < nv; c += blockDim.x) m = fmaxf(m, zr[c]);
  m = block_reduce(m, MaxOp(), sh);
  float l = 0.f;
  T* pr = p + (int64_t)r * ldp;
  for (int c = threadIdx.x; c < nv; c += blockDim.x) {
    const float e = expf(zr[c] - m);
    l += e;
    pr[c] = from_f<T>(e);
  }
  l = block_reduce(l, AddOp(), sh);
  if (threadIdx.x == 0) {
    if (first) {
      m_run[r] = m;
      l_run[r] = l;
      alpha[r] = 0.f;
      beta[r] = 1.f;
    } else {
      const float mo = m_run[r];
      const float mn = fmaxf(mo, m);
      const float a = expf(mo - mn), b = expf(m - mn);
      l_run[r] = l_run[r] * a + l * b;
      m_run[r] = mn;
      alpha[r] = a;
      beta[r] = b;
    }
  }
}

template <typename T>
__global__ void ce_finalize_kernel(const float* m_run, const float* l_run, const float* ztgt,
                                   const int32_t* tgt, float inv_ntgt, const float* __restrict__ dh_acc,
                                   const T* __restrict__ Wlm, int d, float* __restrict__ dhf,
                                   float* loss_row) {
  const int r = blockIdx.x;
  const int64_t o = (int64_t)r * d;
  const int y = tgt[r];
  if (y < 0) {
    for (int c = threadIdx.x; c < d; c += blockDim.x) dhf[o + c] = 0.f;
    if (threadIdx.x == 0) loss_row[r] = 0.f;
    return;
  }
  const float l = l_run[r];
  const float il = 1.0f / l;
  const T* wy = Wlm + (int64_t)y * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x)
    dhf[o + c] = (dh_acc[o + c] * il - to_f<T>(wy[c])) * inv_ntgt;
  if (threadIdx.x == 0) loss_row[r] = m_run[r] + logf(l) - ztgt[r];
}

__global__ void loss_reduce_kernel(const float* loss_row, int n, float inv_ntgt, float* out, int chunk,
                                   int* err_chunk) {
  __shared__ float sh[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += loss_row[i];
  s = block_reduce(s, AddOp(), sh);
  if (threadIdx.x == 0) {
    const float v = s * inv_ntgt;
    out[chunk] = v;
    if (!isfinite(v)) atomicMin(err_chunk, chunk);
  }
}

__device__ __forceinline__ int64_t map_row(int64_t r, int mode, int hd) {
  switch (mode) {
    case 1: {
      const int64_t h = r / hd, i = r % hd, half = hd / 2;
      return h * hd + (i < half ? 2 * i : 2 * (i - half) + 1);
    }
    case 2: return 2 * r;
    case 3: return 2 * r + 1;
    default: return r;
  }
}

template <typename T>
__global__ void pack_kernel(const float* __restrict__ src, int64_t rows, int64_t cols, int mode, int hd,
                            T* __restrict__ dst) {
  const int64_t total = rows * cols;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / cols, c = idx % cols;
    dst[map_row(r, mode, hd) * cols + c] = from_f<T>(src[idx]);
  }
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, int64_t n, bf16* __restrict__ dst) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

__global__ void split_bf16_kernel(const float* __restrict__ w, int64_t n, bf16* __restrict__ hi,
                                  bf16* __restrict__ lo) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bf16 h = __float2bfloat16_rn(w[i]);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(w[i] - __bfloat162float(h));
  }
}

inline int grid_for(int64_t total, int threads) {
  int64_t g = (total + threads - 1) / threads;
  return (int)(g > 148 * 32 ? 148 * 32 : (g < 1 ? 1 : g));
}

}  // namespace

template <typename T>
void launch_embed(const int32_t* tok, int n, const T* E, int d, float* x, int V, int* err_tok,
                  cudaStream_t st) {
  if (n > 0) embed_kernel<T><<<n, RB, 0, st>>>(tok, d, E, x, V, err_tok);
}
template <typename T>
void launch_rmsnorm_fwd(const float* x, const float* g, int n, int d, float eps, T* out, float* r,
                        cudaStream_t st) {
  if (n > 0) rmsnorm_fwd_kernel<T><<<n, RB, 0, st>>>(x, g, d, eps, out, r);
}
template <typename T>
void launch_rmsnorm_bwd(const float* x, const float* g, const float* r, const float* dy,
                        const float* resid, int n, int d, float* out, T* out_t, cudaStream_t st) {
  if (n > 0) rmsnorm_bwd_kernel<T><<<n, RB, 0, st>>>(x, g, r, dy, resid, d, out, out_t);
}
void launch_rope_table(int64_t pos0, int n, int hd, float theta, float2* cs, cudaStream_t st) {
  const int total = n * (hd / 2);
  if (total > 0) rope_table_kernel<<<(total + 255) / 256, 256, 0, st>>>(pos0, n, hd, (double)theta, cs);
}
template <typename T>
void launch_rope_bwd(T* dqkv, int n, int ld, int n_rot_heads, int hd, const float2* cs, cudaStream_t st) {
  const int64_t total = (int64_t)n * n_rot_heads * (hd / 2);
  if (total > 0) rope_bwd_kernel<T><<<grid_for(total, 256), 256, 0, st>>>(dqkv, n, ld, n_rot_heads, hd, cs);
}
void launch_targets(const int32_t* tok, int64_t T, int64_t pos0, int n, int32_t* tgt, int V, int* err_tok,
                    cudaStream_t st) {
  if (n > 0) targets_kernel<<<(n + 255) / 256, 256, 0, st>>>(tok, T, pos0, n, tgt, V, err_tok);
}
template <typename T>
void launch_ce_slab_stats(const float* z, int64_t ldz, int n, int nv, T* p, int64_t ldp, float* m_run,
                          float* l_run, float* alpha, float* beta, int first, cudaStream_t st) {
  if (n > 0) ce_slab_stats_kernel<T><<<n, RB, 0, st>>>(z, ldz, nv, p, ldp, m_run, l_run, alpha, beta, first);
}
template <typename T>
void launch_ce_finalize(int n, const float* m_run, const float* l_run, const float* ztgt,
                        const int32_t* tgt, float inv_ntgt, const float* dh_acc, const T* Wlm, int d,
                        float* dhf, float* loss_row, cudaStream_t st) {
  if (n > 0)
    ce_finalize_kernel<T><<<n, RB, 0, st>>>(m_run, l_run, ztgt, tgt, inv_ntgt, dh_acc, Wlm, d, dhf, loss_row);
}
void launch_loss_reduce(const float* loss_row, int n, float inv_ntgt, float* out, int chunk, int* err_chunk,
                        cudaStream_t st) {
  loss_reduce_kernel<<<1, RB, 0, st>>>(loss_row, n, inv_ntgt, out, chunk, err_chunk);
}
template <typename T>
void launch_pack(const float* src, int64_t rows, int64_t cols, int mode, int hd, T* dst, cudaStream_t st) {
  const int64_t total = rows * cols;
  if (total > 0) pack_kernel<T><<<grid_for(total, 256), 256, 0, st>>>(src, rows, cols, mode, hd, dst);
}
void launch_split_bf16(const float* w, int64_t n, bf16* hi, bf16* lo, cudaStream_t st) {
  if (n > 0) split_bf16_kernel<<<grid_for(n, 256), 256, 0, st>>>(w, n, hi, lo);
}
void launch_f32_to_bf16(const float* src, int64_t n, bf16* dst, cudaStream_t st) {
  if (n > 0) f32_to_bf16_kernel<<<grid_for(n, 256), 256, 0, st>>>(src, n, dst);
}

#define INST(T)                                                                                         \
  template void launch_embed<T>(const int32_t*, int, const T*, int, float*, int, int*, cudaStream_t);               \
  template void launch_rmsnorm_fwd<T>(const float*, const float*, int, int, float, T*, float*,          \
                                      cudaStream_t);                                                    \
  template void launch_rmsnorm_bwd<T>(const float*, const float*, const float*, const float*,           \
                                      const float*, int, int, float*, T*, cudaStream_t);                \
  template void launch_rope_bwd<T>(T*, int, int, int, int, const float2*, cudaStream_t);                \
  template void launch_ce_slab_stats<T>(const float*, int64_t, int, int, T*, int64_t, float*, float*,   \
                                        float*, float*, int, cudaStream_t);                             \
  template void launch_ce_finalize<T>(int, const float*, const float*, const float*, const int32_t*,    \
                                      float, const float*, const T*, int, float*, float*, cudaStream_t); \
  template void launch_pack<T>(const float*, int64_t, int64_t, int, int, T*, cudaStream_t);
INST(float)
INST(bf16)
#undef INST

}  // namespace ttt

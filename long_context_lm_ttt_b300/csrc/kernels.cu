// kernels.cu — the row-wise and element-wise kernels of the inner loop:
// embedding gather, RMSNorm forward/backward, RoPE tables and the inverse
// rotation of gradients, next-token targets, the vocabulary-slab softmax
// statistics of the streamed cross-entropy, its finalisation, the
// deterministic chunk-loss reduction, and weight packing.
#include <math.h>
#include <stdint.h>

#include "bounds.cuh"
#include "common.cuh"
#include "kernels.h"

namespace ttt {

TTT_BOUNDS_UNIT(kernels)

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
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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

__global__ void rope_table_kernel(int64_t pos0, const int64_t* pos_dev, int n, int hd, double theta, float2* cs) {
  pdl_wait();
  pdl_trigger();
  const int half = hd >> 1;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  if (pos_dev) pos0 = *pos_dev;
  const int r = idx / half, i = idx % half;
  const double inv = pow(theta, -(2.0 * (double)i) / (double)hd);
  const double ang = (double)(pos0 + r) * inv;
  double sn, cn;
  sincos(ang, &sn, &cn);
  cs[idx] = make_float2((float)cn, (float)sn);
}

template <typename T>
__global__ void rope_bwd_kernel(T* dqkv, int n, int ld, int n_rot_heads, int hd, const float2* cs) {
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  if (dh_acc)
    for (int c = threadIdx.x; c < d; c += blockDim.x)
      dhf[o + c] = (dh_acc[o + c] * il - to_f<T>(wy[c])) * inv_ntgt;
  if (threadIdx.x == 0) loss_row[r] = m_run[r] + logf(l) - ztgt[r];
}

__global__ void loss_reduce_kernel(const float* loss_row, int n, float inv_ntgt, float* out, int chunk,
                                   int* err_chunk) {
  pdl_wait();
  pdl_trigger();
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

__global__ void decode_begin_kernel(DecodeState* s, int64_t pos, int r, const int32_t* given, int n_given,
                                    int32_t* out, unsigned long long* pick) {
  if (threadIdx.x != 0) return;
  *pick = 0ull;
  s->pos = pos;
  s->given = given;
  s->out = out;
  s->r = r;
  s->i = 0;
  s->n_given = n_given;
  s->tok = given[0];
}

__global__ void decode_tail_kernel(DecodeState* s, const float* __restrict__ x, float* __restrict__ xdec, int d,
                                   int32_t* dtok, unsigned long long* pick, int b) {
  pdl_wait();
  pdl_trigger();
  const int r = s->r;
  // the step's row of the chunk buffers (the debug build checks it; every
  // thread takes the same branch)
  const bool row_ok = TTT_IN(KB_DECODE_TAIL, r, b);
  if (row_ok)
    for (int c = threadIdx.x; c < d; c += blockDim.x) xdec[(int64_t)r * d + c] = x[c];
  __syncthreads();  // every thread has read r before it moves on
  if (threadIdx.x == 0 && row_ok) {
    const int i = s->i, tok = s->tok;
    const int nxt = i + 1 < s->n_given ? s->given[i + 1] : argmax_col(*pick);
    *pick = 0ull;
    dtok[r] = tok;
    dtok[r + 1] = nxt;
    s->out[i] = tok;
    s->tok = nxt;
    s->pos += 1;
    s->i = i + 1;
    s->r = r + 1 == b ? 0 : r + 1;
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

__global__ void split_bf16_kernel(const float* __restrict__ w, int64_t n, bf16* __restrict__ hi,
                                  bf16* __restrict__ lo) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bf16 h = __float2bfloat16_rn(w[i]);
    hi[i] = h;
    if (lo) lo[i] = __float2bfloat16_rn(w[i] - __bfloat162float(h));
  }
}

// ---------------------------------------------------------------------------
// Vectorised row kernels for the bf16 path: 16-byte loads, the row held in
// registers (one read of each input), VPT float4 per thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint2 pack4_bf16(float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

template <int VPT>
__global__ void __launch_bounds__(256) rmsnorm_fwd_vec_kernel(const float* __restrict__ x, const float* __restrict__ g,
                                                              int d, float eps, bf16* __restrict__ out,
                                                              float* __restrict__ rr) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)r * d);
  const float4* gr = reinterpret_cast<const float4*>(g);
  const int nq = d >> 2;
  float4 v[VPT];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int q = threadIdx.x + 256 * i;
    v[i] = q < nq ? xr[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    s = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, fmaf(v[i].z, v[i].z, fmaf(v[i].w, v[i].w, s))));
  }
  s = block_reduce(s, AddOp(), sh);
  const float rinv = 1.0f / sqrtf(s / (float)d + eps);
  uint2* o = reinterpret_cast<uint2*>(out + (int64_t)r * d);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int q = threadIdx.x + 256 * i;
    if (q < nq) {
      const float4 gg = gr[q];
      o[q] = pack4_bf16(make_float4(gg.x * v[i].x * rinv, gg.y * v[i].y * rinv, gg.z * v[i].z * rinv,
                                    gg.w * v[i].w * rinv));
    }
  }
  if (threadIdx.x == 0) rr[r] = rinv;
}

// out = resid + r (g dy) - r^3 x mean(x g dy); out_t = bf16(out)
template <int VPT>
__global__ void __launch_bounds__(256) rmsnorm_bwd_vec_kernel(const float* __restrict__ x, const float* __restrict__ g,
                                                              const float* __restrict__ rr, const float* __restrict__ dy,
                                                              const float* __restrict__ resid, int d,
                                                              float* __restrict__ out, bf16* __restrict__ out_t) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const int64_t o = (int64_t)r * d;
  const float4* xr = reinterpret_cast<const float4*>(x + o);
  const float4* dr = reinterpret_cast<const float4*>(dy + o);
  const float4* gr = reinterpret_cast<const float4*>(g);
  const int nq = d >> 2;
  float4 xv[VPT], gd[VPT];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int q = threadIdx.x + 256 * i;
    if (q < nq) {
      xv[i] = xr[q];
      const float4 gg = gr[q], dd = dr[q];
      gd[i] = make_float4(gg.x * dd.x, gg.y * dd.y, gg.z * dd.z, gg.w * dd.w);
    } else {
      xv[i] = gd[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    s = fmaf(xv[i].x, gd[i].x, fmaf(xv[i].y, gd[i].y, fmaf(xv[i].z, gd[i].z, fmaf(xv[i].w, gd[i].w, s))));
  }
  s = block_reduce(s, AddOp(), sh) / (float)d;
  const float ri = rr[r];
  const float c3 = ri * ri * ri * s;
  float4* outr = reinterpret_cast<float4*>(out + o);
  const float4* rs = reinterpret_cast<const float4*>(resid ? resid + o : nullptr);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int q = threadIdx.x + 256 * i;
    if (q < nq) {
      float4 v = make_float4(ri * gd[i].x - c3 * xv[i].x, ri * gd[i].y - c3 * xv[i].y, ri * gd[i].z - c3 * xv[i].z,
                             ri * gd[i].w - c3 * xv[i].w);
      if (rs) {
        const float4 t = rs[q];
        v.x += t.x;
        v.y += t.y;
        v.z += t.z;
        v.w += t.w;
      }
      outr[q] = v;
      if (out_t) reinterpret_cast<uint2*>(out_t + o)[q] = pack4_bf16(v);
    }
  }
}

// Streamed softmax statistics of one vocabulary slab: max, sum of exp, and
// P = exp(z - max) in bf16.  1024 threads per row, float4 loads; the second
// pass re-reads the slab, which is resident in L2.
__global__ void __launch_bounds__(1024) ce_slab_stats_vec_kernel(const float* __restrict__ z, int64_t ldz, int nv,
                                                                 bf16* __restrict__ p, int64_t ldp, float* m_run,
                                                                 float* l_run, float* alpha, float* beta, int first) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const float4* zr = reinterpret_cast<const float4*>(z + (int64_t)r * ldz);
  uint2* pr = reinterpret_cast<uint2*>(p + (int64_t)r * ldp);
  const int nq = nv >> 2;
  float m = -INFINITY;
  for (int q = threadIdx.x; q < nq; q += blockDim.x) {
    const float4 v = zr[q];
    m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
  }
  m = block_reduce(m, MaxOp(), sh);
  const float L2E = 1.4426950408889634f;
  const float nm = -m * L2E;
  float l = 0.f;
  for (int q = threadIdx.x; q < nq; q += blockDim.x) {
    const float4 v = zr[q];
    // exp(z - m) = 2^(z log2(e) - m log2(e))
    float4 e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(fmaf(v.x, L2E, nm)));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(fmaf(v.y, L2E, nm)));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.z) : "f"(fmaf(v.z, L2E, nm)));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.w) : "f"(fmaf(v.w, L2E, nm)));
    l += (e.x + e.y) + (e.z + e.w);
    pr[q] = pack4_bf16(e);
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

inline int grid_for(int64_t total, int threads) {
  int64_t g = (total + threads - 1) / threads;
  return (int)(g > 148 * 32 ? 148 * 32 : (g < 1 ? 1 : g));
}

}  // namespace

static thread_local bool t_pdl = false;
void set_pdl(bool on) { t_pdl = on; }
bool pdl_enabled() { return t_pdl; }

template <typename T>
void launch_embed(const int32_t* tok, int n, const T* E, int d, float* x, int V, int* err_tok,
                  cudaStream_t st) {
  if (n > 0) launch_k(embed_kernel<T>, n, RB, 0, st, tok, d, E, x, V, err_tok);
}
static inline bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

template <typename T>
void launch_rmsnorm_fwd(const float* x, const float* g, int n, int d, float eps, T* out, float* r,
                        cudaStream_t st) {
  if (n <= 0) return;
  if constexpr (sizeof(T) == 2) {
    if (d % 4 == 0 && d <= 4 * 256 * 4 && al16(x) && al16(g) && ((uintptr_t)out & 7) == 0) {
      const int vpt = (d / 4 + 255) / 256;
      auto k = vpt <= 1 ? rmsnorm_fwd_vec_kernel<1>
               : vpt <= 2 ? rmsnorm_fwd_vec_kernel<2>
               : vpt <= 3 ? rmsnorm_fwd_vec_kernel<3>
                          : rmsnorm_fwd_vec_kernel<4>;
      launch_k(k, n, 256, 0, st, x, g, d, eps, (bf16*)out, r);
      return;
    }
  }
  launch_k(rmsnorm_fwd_kernel<T>, n, RB, 0, st, x, g, d, eps, out, r);
}
template <typename T>
void launch_rmsnorm_bwd(const float* x, const float* g, const float* r, const float* dy,
                        const float* resid, int n, int d, float* out, T* out_t, cudaStream_t st) {
  if (n <= 0) return;
  if constexpr (sizeof(T) == 2) {
    if (d % 4 == 0 && d <= 3 * 256 * 4 && al16(x) && al16(g) && al16(dy) && al16(out) &&
        (!resid || al16(resid)) && ((uintptr_t)out_t & 7) == 0) {
      const int vpt = (d / 4 + 255) / 256;
      if (vpt <= 1) launch_k(rmsnorm_bwd_vec_kernel<1>, n, 256, 0, st, x, g, r, dy, resid, d, out, (bf16*)out_t);
      else if (vpt <= 2) launch_k(rmsnorm_bwd_vec_kernel<2>, n, 256, 0, st, x, g, r, dy, resid, d, out, (bf16*)out_t);
      else launch_k(rmsnorm_bwd_vec_kernel<3>, n, 256, 0, st, x, g, r, dy, resid, d, out, (bf16*)out_t);
      return;
    }
  }
  launch_k(rmsnorm_bwd_kernel<T>, n, RB, 0, st, x, g, r, dy, resid, d, out, out_t);
}
void launch_rope_table(int64_t pos0, int n, int hd, float theta, float2* cs, cudaStream_t st,
                       const int64_t* pos_dev) {
  const int total = n * (hd / 2);
  if (total > 0) launch_k(rope_table_kernel, (total + 255) / 256, 256, 0, st, pos0, pos_dev, n, hd, (double)theta, cs);
}
void launch_decode_begin(DecodeState* s, int64_t pos, int r, const int32_t* given, int n_given, int32_t* out,
                         unsigned long long* pick, cudaStream_t st) {
  decode_begin_kernel<<<1, 32, 0, st>>>(s, pos, r, given, n_given, out, pick);
}
void launch_decode_tail(DecodeState* s, const float* x, float* xdec, int d, int32_t* dtok, unsigned long long* pick,
                        int b, cudaStream_t st) {
  launch_k(decode_tail_kernel, 1, 256, 0, st, s, x, xdec, d, dtok, pick, b);
}
template <typename T>
void launch_rope_bwd(T* dqkv, int n, int ld, int n_rot_heads, int hd, const float2* cs, cudaStream_t st) {
  const int64_t total = (int64_t)n * n_rot_heads * (hd / 2);
  if (total > 0) launch_k(rope_bwd_kernel<T>, grid_for(total, 256), 256, 0, st, dqkv, n, ld, n_rot_heads, hd, cs);
}
void launch_targets(const int32_t* tok, int64_t T, int64_t pos0, int n, int32_t* tgt, int V, int* err_tok,
                    cudaStream_t st) {
  if (n > 0) launch_k(targets_kernel, (n + 255) / 256, 256, 0, st, tok, T, pos0, n, tgt, V, err_tok);
}
template <typename T>
void launch_ce_slab_stats(const float* z, int64_t ldz, int n, int nv, T* p, int64_t ldp, float* m_run,
                          float* l_run, float* alpha, float* beta, int first, cudaStream_t st) {
  if (n <= 0) return;
  if constexpr (sizeof(T) == 2) {
    if (nv % 4 == 0 && ldz % 4 == 0 && ldp % 4 == 0 && al16(z) && ((uintptr_t)p & 7) == 0) {
      launch_k(ce_slab_stats_vec_kernel, n, 1024, 0, st, z, ldz, nv, (bf16*)p, ldp, m_run, l_run, alpha, beta, first);
      return;
    }
  }
  launch_k(ce_slab_stats_kernel<T>, n, RB, 0, st, z, ldz, nv, p, ldp, m_run, l_run, alpha, beta, first);
}
template <typename T>
void launch_ce_finalize(int n, const float* m_run, const float* l_run, const float* ztgt,
                        const int32_t* tgt, float inv_ntgt, const float* dh_acc, const T* Wlm, int d,
                        float* dhf, float* loss_row, cudaStream_t st) {
  if (n > 0)
    launch_k(ce_finalize_kernel<T>, n, RB, 0, st, m_run, l_run, ztgt, tgt, inv_ntgt, dh_acc, Wlm, d, dhf, loss_row);
}
void launch_loss_reduce(const float* loss_row, int n, float inv_ntgt, float* out, int chunk, int* err_chunk,
                        cudaStream_t st) {
  launch_k(loss_reduce_kernel, 1, RB, 0, st, loss_row, n, inv_ntgt, out, chunk, err_chunk);
}
template <typename T>
void launch_pack(const float* src, int64_t rows, int64_t cols, int mode, int hd, T* dst, cudaStream_t st) {
  const int64_t total = rows * cols;
  if (total > 0) pack_kernel<T><<<grid_for(total, 256), 256, 0, st>>>(src, rows, cols, mode, hd, dst);
}
void launch_split_bf16(const float* w, int64_t n, bf16* hi, bf16* lo, cudaStream_t st) {
  if (n > 0) split_bf16_kernel<<<grid_for(n, 256), 256, 0, st>>>(w, n, hi, lo);
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

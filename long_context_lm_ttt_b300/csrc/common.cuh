// common.cuh — shared device helpers of the TTT kernels: element types,
// the GEMM epilogue descriptor, and the epilogue arithmetic applied to each
// pair of adjacent accumulator columns.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ttt {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// element conversions (round to nearest even for bf16)
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

template <typename T> __device__ __forceinline__ void store2(T* p, float a, float b);
template <> __device__ __forceinline__ void store2<float>(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
template <> __device__ __forceinline__ void store2<bf16>(bf16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}
template <typename T> __device__ __forceinline__ float2 load2(const T* p);
template <> __device__ __forceinline__ float2 load2<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <> __device__ __forceinline__ float2 load2<bf16>(const bf16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Programmatic dependent launch.  A kernel launched with it (launch_k with
// launches marked by set_pdl) may begin while the previous kernel on its
// stream still runs.  It calls pdl_wait() before touching anything that
// kernel or an earlier one writes (the wait returns at once after an
// ordinary launch), and pdl_trigger() after that wait, which lets the next
// such kernel begin: so at most two kernels of a chain overlap, and
// everything two or more kernels back has completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// GEMM:  C[m, n] = sum_k A(m, k) * B(n, k)
//   A(m,k) = a_mn ? A[k*lda + m] : A[m*lda + k]
//   B(n,k) = b_mn ? B[k*ldb + n] : B[n*ldb + k]
// The accumulator (fp32) goes through one of the epilogues below; every
// epilogue works on column pairs (n even, n+1), so N must be even.
// ---------------------------------------------------------------------------
enum EpiKind : int {
  EPI_STORE = 0,      // out[m, n] = acc                      (out fp32 or T)
  EPI_RESID = 1,      // out[m, n] = resid[m, n] + acc        (fp32)
  EPI_QKV = 2,        // RoPE on q/k pairs, q -> out, k/v -> key/value ring
  EPI_SWIGLU = 3,     // (g, u) pair -> a = silu(g) u; optional stash of (g, u)
  EPI_SWIGLU_BWD = 4, // da -> (dg, du) using the stashed (g, u)
  EPI_SGD = 5,        // w32 -= lr * acc; w16 = rn(w32); w16lo = rn(w32 - w16)
  EPI_CE_Z = 6,       // z slab (fp32) + pick the target logit
  EPI_CE_ACC = 7,     // acc_out = acc_out * alpha[m] + acc * beta[m]
  EPI_ARGMAX = 8,     // out (uint64 per row) = max of argmax_key(acc, n): the greedy pick
};

// The greedy pick as one 64-bit key, so that an atomic max finds it: the
// logit's bits made order-preserving as an unsigned word (high half; -0
// taken as +0) and the complement of its column (low half), so the largest
// key is the largest logit at its smallest column.  NaN never wins (key 0);
// argmax_col() turns a key back into the column (0 when nothing won).
__device__ __forceinline__ unsigned long long argmax_key(float v, int n) {
  if (v != v) return 0ull;
  const uint32_t b = v == 0.f ? 0u : __float_as_uint(v);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (uint32_t)~(uint32_t)n;
}
__device__ __forceinline__ int argmax_col(unsigned long long key) {
  return key == 0ull ? 0 : (int)~(uint32_t)(key & 0xffffffffull);
}

struct Epi {
  int kind;
  int out_f32;            // EPI_STORE: 1 = fp32 output, 0 = element type T
  void* out;              // output matrix
  int64_t ldo;
  const float* resid;     // EPI_RESID
  int64_t ldr;
  // EPI_QKV
  int n_q, n_kv, hd;      // heads of q, heads of k/v, head dim
  int64_t pos0;           // absolute position of row 0
  const int64_t* pos_dev; // non-null: row 0's position is read here instead
                          // (decode steps replayed from one captured graph)
  int ring;               // ring slots R
  void* kring;            // [n_kv][R][hd]
  void* vring;
  const float2* rope_cs;  // [rows][hd/2] (cos, sin) of the rows' positions
  // rows of several sequences stacked (seg_rows > 0): row m is row
  // m % seg_rows of sequence m / seg_rows, whose rings start ring_seq
  // elements after the previous sequence's; positions and the RoPE table
  // are those of the row within its sequence
  int seg_rows;
  int64_t ring_seq;
  // EPI_SWIGLU / EPI_SWIGLU_BWD
  void* stash;            // (g, u) interleaved [rows][2*d_ff]
  int64_t ld_stash;
  // EPI_SGD
  float* w32;
  void* w16;              // may be null (fp32 mode: w32 is the weight)
  void* w16lo;            // may be null: low half of the compensated pair
  float lr;
  // EPI_CE_Z
  const int32_t* tgt;     // target id per row (-1: none)
  float* ztgt;
  int64_t col0;           // vocab index of column 0
  // EPI_CE_ACC
  const float* alpha;
  const float* beta;
  int first;              // 1: ignore the old content of out
  // set by the tensor-core launcher: every pointer and row pitch the
  // epilogue touches allows 16-byte vector access (epi_row32 below)
  int vec;
};

// Apply the epilogue to columns (n, n+1) of row m.  T is the element type of
// the activations (float in check mode, bf16 otherwise).
template <typename T>
__device__ __forceinline__ void epi_pair(const Epi& e, int m, int n, float v0, float v1) {
  switch (e.kind) {
    case EPI_STORE: {
      if (e.out_f32) store2<float>((float*)e.out + (int64_t)m * e.ldo + n, v0, v1);
      else store2<T>((T*)e.out + (int64_t)m * e.ldo + n, v0, v1);
    } break;
    case EPI_RESID: {
      float2 r = load2<float>(e.resid + (int64_t)m * e.ldr + n);
      store2<float>((float*)e.out + (int64_t)m * e.ldo + n, r.x + v0, r.y + v1);
    } break;
    case EPI_QKV: {
      const int hd = e.hd;
      const int qcols = e.n_q * hd;
      const int kcols = e.n_kv * hd;
      const int mr = e.seg_rows ? m % e.seg_rows : m;                       // row within its sequence
      const int64_t rs = e.seg_rows ? (int64_t)(m / e.seg_rows) * e.ring_seq : 0;  // its rings
      if (n < qcols + kcols) {
        const float2 cs = e.rope_cs[(int64_t)mr * (hd >> 1) + ((n % hd) >> 1)];
        const float a = v0 * cs.x - v1 * cs.y;
        const float b = v1 * cs.x + v0 * cs.y;
        if (n < qcols) {
          store2<T>((T*)e.out + (int64_t)m * e.ldo + n, a, b);
        } else {
          const int c = n - qcols;
          const int64_t slot = ((e.pos_dev ? *e.pos_dev : e.pos0) + mr) % e.ring;
          store2<T>((T*)e.kring + rs + ((int64_t)(c / hd) * e.ring + slot) * hd + (c % hd), a, b);
        }
      } else {
        const int c = n - qcols - kcols;
        const int64_t slot = ((e.pos_dev ? *e.pos_dev : e.pos0) + mr) % e.ring;
        store2<T>((T*)e.vring + rs + ((int64_t)(c / hd) * e.ring + slot) * hd + (c % hd), v0, v1);
      }
    } break;
    case EPI_SWIGLU: {
      const float a = v0 * sigmoidf_(v0) * v1;
      ((T*)e.out)[(int64_t)m * e.ldo + (n >> 1)] = from_f<T>(a);
      if (e.stash) store2<T>((T*)e.stash + (int64_t)m * e.ld_stash + n, v0, v1);
    } break;
    case EPI_SWIGLU_BWD: {
      // columns n, n+1 are d_ff indices f, f+1; outputs go to 2f .. 2f+3
      const T* st = (const T*)e.stash + (int64_t)m * e.ld_stash + 2 * n;
      float2 gu0 = load2<T>(st), gu1 = load2<T>(st + 2);
      float s0 = sigmoidf_(gu0.x), s1 = sigmoidf_(gu1.x);
      float dg0 = v0 * gu0.y * s0 * (1.0f + gu0.x * (1.0f - s0));
      float du0 = v0 * gu0.x * s0;
      float dg1 = v1 * gu1.y * s1 * (1.0f + gu1.x * (1.0f - s1));
      float du1 = v1 * gu1.x * s1;
      T* o = (T*)e.out + (int64_t)m * e.ldo + 2 * n;
      store2<T>(o, dg0, du0);
      store2<T>(o + 2, dg1, du1);
    } break;
    case EPI_SGD: {
      float* w = e.w32 + (int64_t)m * e.ldo + n;
      float2 cur = load2<float>(w);
      cur.x -= e.lr * v0;
      cur.y -= e.lr * v1;
      store2<float>(w, cur.x, cur.y);
      if (e.w16) {
        const __nv_bfloat162 hi = __floats2bfloat162_rn(cur.x, cur.y);
        *reinterpret_cast<__nv_bfloat162*>((bf16*)e.w16 + (int64_t)m * e.ldo + n) = hi;
        if (e.w16lo) {
          const float2 hf = __bfloat1622float2(hi);
          store2<bf16>((bf16*)e.w16lo + (int64_t)m * e.ldo + n, cur.x - hf.x, cur.y - hf.y);
        }
      }
    } break;
    case EPI_CE_Z: {
      store2<float>((float*)e.out + (int64_t)m * e.ldo + n, v0, v1);
      const int64_t t = (int64_t)e.tgt[m] - e.col0;
      if (t == n) e.ztgt[m] = v0;
      else if (t == n + 1) e.ztgt[m] = v1;
    } break;
    case EPI_ARGMAX: {
      const unsigned long long k0 = argmax_key(v0, n), k1 = argmax_key(v1, n + 1);
      atomicMax((unsigned long long*)e.out + m, k0 > k1 ? k0 : k1);
    } break;
    case EPI_CE_ACC: {
      float* o = (float*)e.out + (int64_t)m * e.ldo + n;
      const float be = e.beta[m];
      if (e.first) {
        store2<float>(o, v0 * be, v1 * be);
      } else {
        const float al = e.alpha[m];
        float2 c = load2<float>(o);
        store2<float>(o, c.x * al + v0 * be, c.y * al + v1 * be);
      }
    } break;
    default: break;
  }
}

// ---------------------------------------------------------------------------
// Row-chunk form of the epilogues for the tensor-core GEMM: one thread owns
// one output row and applies the epilogue to 32 consecutive accumulator
// columns [col0, col0+32) at once, with 16-byte loads and stores.  The
// operand the epilogue reads besides the accumulator (its "source": the
// residual, the fp32 master weight, the running dh, the (g, u) stash, or
// the RoPE (cos, sin) pairs) is exactly 128 bytes per row chunk; it is
// fetched by epi_src_load ahead of use so the load latency overlaps the
// previous chunk.  Requires e.vec, col0 + 32 <= N and, for EPI_QKV,
// hd % 32 == 0 (a chunk never straddles two heads); otherwise the caller
// falls back to epi_pair.  bf16 activations only.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void stg16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ uint32_t bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unbf2(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(h);
}

__device__ __forceinline__ bool epi_has_src(const Epi& e) {
  switch (e.kind) {
    case EPI_RESID:
    case EPI_SGD:
    case EPI_SWIGLU_BWD:
      return true;
    case EPI_CE_ACC:
      return !e.first;
    case EPI_QKV:
      return true;
    default:
      return false;
  }
}

__device__ __forceinline__ void epi_src_load(const Epi& e, int m, int col0, uint4 (&src)[8]) {
  const uint8_t* p = nullptr;
  switch (e.kind) {
    case EPI_RESID: p = (const uint8_t*)(e.resid + (int64_t)m * e.ldr + col0); break;
    case EPI_SGD: p = (const uint8_t*)(e.w32 + (int64_t)m * e.ldo + col0); break;
    case EPI_CE_ACC: p = (const uint8_t*)((const float*)e.out + (int64_t)m * e.ldo + col0); break;
    case EPI_SWIGLU_BWD: p = (const uint8_t*)((const bf16*)e.stash + (int64_t)m * e.ld_stash + 2 * col0); break;
    case EPI_QKV: {
      const int hd = e.hd;
      if (col0 >= (e.n_q + e.n_kv) * hd) return;  // values: no rotation
      const int mr = e.seg_rows ? m % e.seg_rows : m;
      p = (const uint8_t*)(e.rope_cs + (int64_t)mr * (hd >> 1) + ((col0 % hd) >> 1));
    } break;
    default: return;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) src[i] = ldg16(p + 16 * i);
}

__device__ __forceinline__ void epi_row32(const Epi& e, int m, int col0, const float (&v)[32],
                                          const uint4 (&src)[8]) {
  const float* sf = reinterpret_cast<const float*>(src);      // 32 fp32 sources
  const uint32_t* su = reinterpret_cast<const uint32_t*>(src);
  switch (e.kind) {
    case EPI_STORE: {
      if (e.out_f32) {
        float* o = (float*)e.out + (int64_t)m * e.ldo + col0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          stg16(o + 4 * i, make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                      __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])));
      } else {
        bf16* o = (bf16*)e.out + (int64_t)m * e.ldo + col0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          stg16(o + 8 * i, make_uint4(bf2(v[8 * i], v[8 * i + 1]), bf2(v[8 * i + 2], v[8 * i + 3]),
                                      bf2(v[8 * i + 4], v[8 * i + 5]), bf2(v[8 * i + 6], v[8 * i + 7])));
      }
    } break;
    case EPI_RESID: {
      float* o = (float*)e.out + (int64_t)m * e.ldo + col0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        stg16(o + 4 * i, make_uint4(__float_as_uint(sf[4 * i] + v[4 * i]), __float_as_uint(sf[4 * i + 1] + v[4 * i + 1]),
                                    __float_as_uint(sf[4 * i + 2] + v[4 * i + 2]),
                                    __float_as_uint(sf[4 * i + 3] + v[4 * i + 3])));
    } break;
    case EPI_QKV: {
      const int hd = e.hd;
      const int qcols = e.n_q * hd, kcols = e.n_kv * hd;
      float r[32];
      if (col0 < qcols + kcols) {
        const float2* cs = reinterpret_cast<const float2*>(src);
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          r[2 * p] = v[2 * p] * cs[p].x - v[2 * p + 1] * cs[p].y;
          r[2 * p + 1] = v[2 * p + 1] * cs[p].x + v[2 * p] * cs[p].y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = v[k];
      }
      bf16* o;
      if (col0 < qcols) {
        o = (bf16*)e.out + (int64_t)m * e.ldo + col0;
      } else {
        const bool is_k = col0 < qcols + kcols;
        const int c = col0 - (is_k ? qcols : qcols + kcols);
        const int mr = e.seg_rows ? m % e.seg_rows : m;
        const int64_t rs = e.seg_rows ? (int64_t)(m / e.seg_rows) * e.ring_seq : 0;
        const int64_t slot = ((e.pos_dev ? *e.pos_dev : e.pos0) + mr) % e.ring;
        o = (bf16*)(is_k ? e.kring : e.vring) + rs + ((int64_t)(c / hd) * e.ring + slot) * hd + (c % hd);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        stg16(o + 8 * i, make_uint4(bf2(r[8 * i], r[8 * i + 1]), bf2(r[8 * i + 2], r[8 * i + 3]),
                                    bf2(r[8 * i + 4], r[8 * i + 5]), bf2(r[8 * i + 6], r[8 * i + 7])));
    } break;
    case EPI_SWIGLU: {
      float a[16];
#pragma unroll
      for (int p = 0; p < 16; ++p) a[p] = v[2 * p] * sigmoidf_(v[2 * p]) * v[2 * p + 1];
      bf16* o = (bf16*)e.out + (int64_t)m * e.ldo + (col0 >> 1);
      stg16(o, make_uint4(bf2(a[0], a[1]), bf2(a[2], a[3]), bf2(a[4], a[5]), bf2(a[6], a[7])));
      stg16(o + 8, make_uint4(bf2(a[8], a[9]), bf2(a[10], a[11]), bf2(a[12], a[13]), bf2(a[14], a[15])));
      if (e.stash) {
        bf16* st = (bf16*)e.stash + (int64_t)m * e.ld_stash + col0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          stg16(st + 8 * i, make_uint4(bf2(v[8 * i], v[8 * i + 1]), bf2(v[8 * i + 2], v[8 * i + 3]),
                                       bf2(v[8 * i + 4], v[8 * i + 5]), bf2(v[8 * i + 6], v[8 * i + 7])));
      }
    } break;
    case EPI_SWIGLU_BWD: {
      // columns are d_ff indices f; the stash holds (g, u) at 2f, 2f+1 and
      // the outputs (dg, du) go to the same places of out
      uint32_t r[32];
#pragma unroll
      for (int f = 0; f < 32; ++f) {
        const float2 gu = unbf2(su[f]);
        const float sg = sigmoidf_(gu.x);
        const float dg = v[f] * gu.y * sg * (1.0f + gu.x * (1.0f - sg));
        const float du = v[f] * gu.x * sg;
        r[f] = bf2(dg, du);
      }
      bf16* o = (bf16*)e.out + (int64_t)m * e.ldo + 2 * col0;
#pragma unroll
      for (int i = 0; i < 8; ++i) stg16(o + 8 * i, make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]));
    } break;
    case EPI_SGD: {
      float w[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) w[k] = sf[k] - e.lr * v[k];
      float* wp = e.w32 + (int64_t)m * e.ldo + col0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        stg16(wp + 4 * i, make_uint4(__float_as_uint(w[4 * i]), __float_as_uint(w[4 * i + 1]),
                                     __float_as_uint(w[4 * i + 2]), __float_as_uint(w[4 * i + 3])));
      if (e.w16) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          hi[p] = bf2(w[2 * p], w[2 * p + 1]);
          const float2 hf = unbf2(hi[p]);
          lo[p] = bf2(w[2 * p] - hf.x, w[2 * p + 1] - hf.y);
        }
        bf16* hp = (bf16*)e.w16 + (int64_t)m * e.ldo + col0;
#pragma unroll
        for (int i = 0; i < 4; ++i) stg16(hp + 8 * i, make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]));
        if (e.w16lo) {
          bf16* lp = (bf16*)e.w16lo + (int64_t)m * e.ldo + col0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            stg16(lp + 8 * i, make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]));
        }
      }
    } break;
    case EPI_CE_Z: {
      float* o = (float*)e.out + (int64_t)m * e.ldo + col0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        stg16(o + 4 * i, make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                    __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])));
      const int64_t t = (int64_t)e.tgt[m] - e.col0 - col0;
      if (t >= 0 && t < 32) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k == t) e.ztgt[m] = v[k];
      }
    } break;
    case EPI_CE_ACC: {
      float* o = (float*)e.out + (int64_t)m * e.ldo + col0;
      const float be = e.beta[m];
      const float al = e.first ? 0.f : e.alpha[m];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = e.first ? v[4 * i + k] * be : sf[4 * i + k] * al + v[4 * i + k] * be;
        stg16(o + 4 * i, make_uint4(__float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]),
                                    __float_as_uint(r[3])));
      }
    } break;
    default: break;
  }
}

}  // namespace ttt

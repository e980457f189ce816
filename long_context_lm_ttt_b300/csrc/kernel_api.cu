// kernel_api.cu — the kernel-level entry points of ttt_kernels.h.
#include <climits>
#include <cstring>

#include "../../include/ttt.h"
#include "../../include/ttt_kernels.h"
#include "bounds.cuh"
#include "kernels.h"

namespace ttt {
// code of a bounded wait of ttt_kernel_attn_bwd_noalloc that gave up on the
// current device, cleared by the read (noalloc.cu)
int noalloc_take_wait_error();
}  // namespace ttt

namespace {
constexpr int kDevs = 64;
// device error word shared by the kernel-level launches, one per device;
// g_err names the current device's word after ensure_err()
int* g_err_of[kDevs] = {};
int* g_err = nullptr;
int ensure_err() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return TTT_ERR_CUDA;
  if (!g_err_of[dev]) {
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) return TTT_ERR_OOM;
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return TTT_ERR_CUDA;
    g_err_of[dev] = p;
  }
  g_err = g_err_of[dev];
  return 0;
}
}  // namespace

extern "C" int ttt_kernel_gemm(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                               const void* B, int64_t ldb, int32_t b_mn, const void* B2, float* C,
                               int64_t ldc, int32_t impl, void* stream) {
  if (!A || !B || !C || M < 0 || N < 0 || K < 1 || (N & 1) || (ldc & 1)) return TTT_ERR_INVALID;
  if (int r = ensure_err()) return r;
  cudaStream_t st = (cudaStream_t)stream;
  ttt::Epi e;
  memset(&e, 0, sizeof(e));
  e.kind = ttt::EPI_STORE;
  e.out_f32 = 1;
  e.out = C;
  e.ldo = ldc;
  if (impl == 0 || impl == 1 || impl == 3 || impl == 4) {
    ttt::GemmArgs<ttt::bf16> g{M, N, K, (const ttt::bf16*)A, lda, a_mn, (const ttt::bf16*)B, ldb, b_mn, e,
                               (const ttt::bf16*)B2, nullptr, 0};
    if (impl != 1) {
      g.pair = impl == 3 ? 0 : (impl == 4 ? 1 : -1);
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

extern "C" int ttt_kernel_gemm_grouped(int32_t groups, int32_t group_rows, int32_t N, int32_t K, const void* A,
                                       int64_t lda, const void* B, int64_t ldb, int32_t b_mn, int64_t group_stride,
                                       const void* B2, float* C, int64_t ldc, int32_t impl, void* stream) {
  if (!A || !B || !C || groups < 1 || group_rows < 1 || N < 0 || K < 1 || (N & 1) || (ldc & 1) ||
      group_stride < 0)
    return TTT_ERR_INVALID;
  if (impl != 0 && impl != 1 && impl != 3 && impl != 4) return TTT_ERR_INVALID;
  if (int r = ensure_err()) return r;
  cudaStream_t st = (cudaStream_t)stream;
  ttt::Epi e;
  memset(&e, 0, sizeof(e));
  e.kind = ttt::EPI_STORE;
  e.out_f32 = 1;
  e.out = C;
  e.ldo = ldc;
  const int64_t M = (int64_t)groups * group_rows;
  if (M > INT32_MAX) return TTT_ERR_SHAPE;
  ttt::GemmArgs<ttt::bf16> g{(int)M, N, K, (const ttt::bf16*)A, lda, 0, (const ttt::bf16*)B, ldb, b_mn, e,
                             (const ttt::bf16*)B2, nullptr, 0};
  g.groups = groups;
  g.group_rows = group_rows;
  g.group_stride = group_stride;
  if (impl == 1) {
    ttt::gemm_simt<ttt::bf16>(g, st);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
  }
  g.pair = impl == 3 ? 0 : (impl == 4 ? 1 : -1);
  if (ttt::gemm_tc_init()) return TTT_ERR_CUDA;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int rc = ttt::gemm_tc(g, sms, g_err, st);
  if (rc == (int)cudaErrorNotSupported || rc == (int)cudaErrorInvalidValue) return TTT_ERR_SHAPE;
  return rc ? TTT_ERR_CUDA : 0;
}

extern "C" int ttt_kernel_gemm_sgd(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                                   const void* B, int64_t ldb, int32_t b_mn, float* w32, void* w16, void* w16lo,
                                   int64_t ldw, float lr, int32_t impl, void* stream) {
  if (!A || !B || !w32 || M < 0 || N < 0 || K < 1 || (N & 1) || (ldw & 1) || ldw < N) return TTT_ERR_INVALID;
  if (impl < 0 || impl > 3) return TTT_ERR_INVALID;
  if (int r = ensure_err()) return r;
  cudaStream_t st = (cudaStream_t)stream;
  ttt::Epi e;
  memset(&e, 0, sizeof(e));
  e.kind = ttt::EPI_SGD;
  e.w32 = w32;
  e.w16 = w16;
  e.w16lo = w16lo;
  e.ldo = ldw;
  e.lr = lr;
  ttt::GemmArgs<ttt::bf16> g{M, N, K, (const ttt::bf16*)A, lda, a_mn, (const ttt::bf16*)B, ldb, b_mn, e,
                             nullptr, nullptr, 0};
  if (impl != 1) {
    g.pair = impl == 2 ? 0 : (impl == 3 ? 1 : -1);
    if (ttt::gemm_tc_init()) return TTT_ERR_CUDA;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int rc = ttt::gemm_tc(g, sms, g_err, st);
    if (rc == (int)cudaErrorNotSupported || rc == (int)cudaErrorInvalidValue) return TTT_ERR_SHAPE;
    return rc ? TTT_ERR_CUDA : 0;
  }
  ttt::gemm_simt<ttt::bf16>(g, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
}

static int attn_check(int32_t impl, int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W, int32_t R,
                      int32_t max_impl = 1) {
  if (impl < 0 || impl > max_impl) return TTT_ERR_INVALID;
  if (n < 0 || H < 1 || Hkv < 1 || H % Hkv || hd < 2 || (hd & 1) || hd > 256 || W < 1 || R < 1)
    return TTT_ERR_INVALID;
  if ((int64_t)R < (int64_t)W + n - 1) return TTT_ERR_SHAPE;
  return 0;
}

static ttt::AttnArgs attn_args(int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W, int32_t R, int64_t pos0,
                               const void* q, const void* kring, const void* vring, void* o, float* lse,
                               int32_t ld_lse) {
  ttt::AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.kring = kring;
  a.vring = vring;
  a.o = o;
  a.lse = lse;
  a.ld_lse = ld_lse;
  a.n = n;
  a.H = H;
  a.Hkv = Hkv;
  a.hd = hd;
  a.W = W;
  a.R = R;
  a.pos0 = pos0;
  return a;
}

extern "C" int ttt_kernel_attn_fwd(int32_t impl, int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W,
                                   int32_t R, int64_t pos0, const void* q, const void* kring, const void* vring,
                                   void* o, float* lse, int32_t ld_lse, void* stream) {
  int rc = attn_check(impl, n, H, Hkv, hd, W, R, 4);
  if (rc) return rc;
  if (!q || !kring || !vring || !o || !lse || ld_lse < n) return TTT_ERR_INVALID;
  ttt::AttnArgs a = attn_args(n, H, Hkv, hd, W, R, pos0, q, kring, vring, o, lse, ld_lse);
  // shape and alignment of the one-query kernel, checked before any device work
  if (impl == 4 && !ttt::attn_decode_supported(a)) return TTT_ERR_SHAPE;
  if (int r = ensure_err()) return r;
  cudaStream_t st = (cudaStream_t)stream;
  if (impl == 4) {
    // one query position (a decode step): the key range split over the GPU
    // slice scratch per device, grown as needed and kept for the process
    static float* part_of[kDevs] = {};
    static size_t elems_of[kDevs] = {};
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return TTT_ERR_CUDA;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t need = (size_t)ttt::attn_decode_scratch_elems(H, hd);
    if (elems_of[dev] < need) {
      if (part_of[dev]) cudaFree(part_of[dev]);
      part_of[dev] = nullptr;
      elems_of[dev] = 0;
      if (cudaMalloc(&part_of[dev], need * sizeof(float)) != cudaSuccess) return TTT_ERR_OOM;
      // the per-KV-head counters at the start begin at zero
      if (cudaMemset(part_of[dev], 0, need * sizeof(float)) != cudaSuccess) return TTT_ERR_CUDA;
      elems_of[dev] = need;
    }
    float* part = part_of[dev];
    if (ttt::attn_decode<ttt::bf16>(a, ttt::attn_decode_splits(a, sms), part, g_err, st)) return TTT_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
  }
  if (impl == 0 || impl == 2 || impl == 3) {
    if (!ttt::attn_tc_supported(a)) return TTT_ERR_SHAPE;
    if (impl == 0) {
      // scratch that lets the kernel split key ranges, per device: grown on
      // demand, kept for later calls (calls on one device must not overlap)
      static float* ws_of[kDevs] = {};
      static int64_t elems_of[kDevs] = {};
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return TTT_ERR_CUDA;
      const int64_t need = (int64_t)3 * ((int64_t)n * H * hd + (int64_t)2 * n * H);
      if (need > elems_of[dev]) {
        if (ws_of[dev]) cudaFree(ws_of[dev]);
        ws_of[dev] = nullptr;
        elems_of[dev] = 0;
        if (cudaMalloc(&ws_of[dev], need * sizeof(float)) != cudaSuccess) return TTT_ERR_OOM;
        elems_of[dev] = need;
      }
      a.ws = ws_of[dev];
      a.ws_elems = elems_of[dev];
    }
    rc = ttt::attn_fwd_tc(a, g_err, st, impl == 0 ? 0 : (impl == 2 ? 1 : 2));
    return rc ? TTT_ERR_CUDA : 0;
  }
  ttt::attn_fwd_simt<ttt::bf16>(a, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
}

extern "C" int ttt_kernel_attn_bwd(int32_t impl, int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W,
                                   int32_t R, int64_t pos0, const void* q, const void* kring, const void* vring,
                                   const void* o, const float* lse, int32_t ld_lse, const void* dout, float* dsum,
                                   void* dqkv, void* stream) {
  int rc = attn_check(impl, n, H, Hkv, hd, W, R);
  if (rc) return rc;
  if (!q || !kring || !vring || !o || !lse || !dout || !dsum || !dqkv || ld_lse < n) return TTT_ERR_INVALID;
  if (int r = ensure_err()) return r;
  ttt::AttnArgs a = attn_args(n, H, Hkv, hd, W, R, pos0, q, kring, vring, nullptr, const_cast<float*>(lse),
                              ld_lse);
  a.out = o;
  a.dout = dout;
  a.Dsum = dsum;
  a.dqkv = dqkv;
  cudaStream_t st = (cudaStream_t)stream;
  if (impl == 0) {
    // scratch for this entry point, per device: grown on demand, kept for
    // later calls (calls on one device must not overlap)
    static float* ws_of[kDevs] = {};
    static int64_t elems_of[kDevs] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return TTT_ERR_CUDA;
    const int64_t need = ttt::attn_bwd_tc_ws_elems(n, H, hd, 0);
    if (need > elems_of[dev]) {
      if (ws_of[dev]) cudaFree(ws_of[dev]);
      ws_of[dev] = nullptr;
      elems_of[dev] = 0;
      if (cudaMalloc(&ws_of[dev], need * sizeof(float)) != cudaSuccess) return TTT_ERR_OOM;
      elems_of[dev] = need;
    }
    a.ws = ws_of[dev];
    a.ws_elems = elems_of[dev];
    if (!ttt::attn_bwd_tc_supported(a)) return TTT_ERR_SHAPE;
    rc = ttt::attn_bwd_tc(a, g_err, st);
    if (rc == (int)cudaErrorNotSupported) return TTT_ERR_SHAPE;
    return rc ? TTT_ERR_CUDA : 0;
  }
  ttt::attn_bwd_simt<ttt::bf16>(a, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
}

namespace {
// one thread waits on an mbarrier expecting one arrival that never comes
__global__ void wait_selftest_kernel(long long budget, int* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a)
        : "memory");
    if (ok) return;
    if (clock64() - t0 > budget) {
      atomicCAS(err, 0, 199);
      return;
    }
  }
}
}  // namespace

extern "C" int ttt_kernel_wait_selftest(int64_t clocks, void* stream) {
  if (clocks < 1 || clocks > 2000000000LL) return TTT_ERR_INVALID;
  if (int r = ensure_err()) return r;
  wait_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>((long long)clocks, g_err);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
}

namespace ttt {
TTT_BOUNDS_UNIT(kernel_api)
namespace {
// evaluates one range check and touches no memory: the debug build records
// (KB_SELFTEST, index, limit) when index lies outside [0, limit)
__global__ void bounds_selftest_kernel(long long index, long long limit) {
  if (!TTT_IN(KB_SELFTEST, index, limit)) return;
}
}  // namespace
}  // namespace ttt

extern "C" int ttt_kernel_bounds_checked(void) { return ttt::kBoundsChecked ? 1 : 0; }

extern "C" int ttt_kernel_bounds_selftest(int64_t index, int64_t limit, void* stream) {
  ttt::bounds_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>((long long)index, (long long)limit);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TTT_ERR_CUDA;
}

extern "C" int ttt_kernel_bounds(int32_t* kernel, int64_t* index, int64_t* limit) {
  if (cudaDeviceSynchronize() != cudaSuccess) return TTT_ERR_CUDA;
  ttt::BoundsRecord r;
  if (ttt::bounds_fetch_all(&r)) return TTT_ERR_CUDA;
  if (kernel) *kernel = r.kernel;
  if (index) *index = r.index;
  if (limit) *limit = r.limit;
  return r.count;
}

extern "C" int ttt_kernel_error(void) {
  if (int r = ensure_err()) return r;
  if (cudaDeviceSynchronize() != cudaSuccess) return TTT_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, g_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TTT_ERR_CUDA;
  if (cudaMemset(g_err, 0, sizeof(int)) != cudaSuccess) return TTT_ERR_CUDA;
  const int h2 = ttt::noalloc_take_wait_error();
  return h != 0 ? h : h2;
}

// noalloc.cu — the attention backward of ttt_kernel_attn_bwd (tensor cores)
// with its scratch in a fixed device array instead of memory from
// cudaMalloc, for callers that must not allocate.
//
// Who cannot allocate: code whose device memory is owned by a framework's
// caching allocator or by a fixed budget (a cudaMalloc outside it can fail
// once that allocator holds the free memory, and escapes its accounting),
// and real-time callers that plan every byte before they start and may not
// block in the driver's allocator in the middle of a step.
//
// The scratch is a file-scope __device__ array of kMaxScratchFloats fp32
// values (32 MiB).  A device context that loads this module reserves it
// until the process exits: with lazy module loading (the CUDA default) that
// happens at the first use of the module on the device, with eager loading
// (CUDA_MODULE_LOADING=EAGER) when the context is created.  Host code cannot
// use the array's name as a device address (in host code it names a
// host-side stand-in), so the first call on each device looks up the real
// address with cudaGetSymbolAddress, with that device current, and caches
// it; that first call should therefore come before any stream capture.  All
// calls share the array and it keeps the last call's contents: nothing in it
// needs to start at zero (every value the reductions read was written
// earlier in the same call), and calls that overlap on the GPU (different
// streams, or different host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ttt.h"
#include "../../include/ttt_kernels.h"
#include "kernels.h"

namespace {

constexpr int64_t kMaxScratchFloats = 8ll << 20;  // 32 MiB of fp32
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_scratch[kMaxScratchFloats];
// code of a bounded device-side wait that gave up; read and cleared by
// ttt_kernel_error()
static __device__ int g_wait_error;

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};
int* g_err_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int ttt_kernel_attn_bwd_noalloc(int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W, int32_t R,
                                           int64_t pos0, const void* q, const void* kring, const void* vring,
                                           const void* o, const float* lse, int32_t ld_lse, const void* dout,
                                           float* dsum, void* dqkv, void* stream) {
  if (n < 0 || H < 1 || Hkv < 1 || H % Hkv || hd < 2 || (hd & 1) || hd > 256 || W < 1 || R < 1)
    return TTT_ERR_INVALID;
  if (!q || !kring || !vring || !o || !lse || !dout || !dsum || !dqkv || ld_lse < n) return TTT_ERR_INVALID;
  if ((int64_t)R < (int64_t)W + n - 1) return TTT_ERR_SHAPE;
  if (n == 0) return TTT_OK;
  // the backward needs two fp32 planes of n x H x hd (per-head dk and dv);
  // more room only lets the dq kernel split key ranges
  const int64_t plane = (int64_t)n * H * hd;
  if (2 * plane > kMaxScratchFloats) return TTT_ERR_SHAPE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TTT_ERR_CUDA;
  float* ws = nullptr;
  int* err = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      void* e = nullptr;
      if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return TTT_ERR_CUDA;
      if (cudaGetSymbolAddress(&e, g_wait_error) != cudaSuccess || !e) return TTT_ERR_CUDA;
      g_scratch_ptr[dev] = (float*)p;
      g_err_ptr[dev] = (int*)e;
    }
    ws = g_scratch_ptr[dev];
    err = g_err_ptr[dev];
  }

  ttt::AttnArgs a{};
  a.q = q;
  a.kring = kring;
  a.vring = vring;
  a.lse = const_cast<float*>(lse);
  a.ld_lse = ld_lse;
  a.n = n;
  a.H = H;
  a.Hkv = Hkv;
  a.hd = hd;
  a.W = W;
  a.R = R;
  a.pos0 = pos0;
  a.out = o;
  a.dout = dout;
  a.Dsum = dsum;
  a.dqkv = dqkv;
  a.ws = ws;
  a.ws_elems = kMaxScratchFloats;
  if (!ttt::attn_bwd_tc_supported(a)) return TTT_ERR_SHAPE;
  const int rc = ttt::attn_bwd_tc(a, err, (cudaStream_t)stream);
  if (rc == (int)cudaErrorNotSupported) return TTT_ERR_SHAPE;
  return rc ? TTT_ERR_CUDA : TTT_OK;
}

namespace ttt {
// The wait code of the device that is current, read and cleared with plain
// copies (nothing allocated).  0 when the entry point never ran on it.
int noalloc_take_wait_error() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int* e = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    e = g_err_ptr[dev];
  }
  if (!e) return 0;
  int h = 0;
  if (cudaMemcpy(&h, e, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TTT_ERR_CUDA;
  if (h != 0 && cudaMemset(e, 0, sizeof(int)) != cudaSuccess) return TTT_ERR_CUDA;
  return h;
}
}  // namespace ttt

// bounds.cuh — range checks of the debug build (nvcc -DTTT_DEBUG_BOUNDS,
// `python -m long_context_lm_ttt_b300.build --debug-bounds`, which writes
// libttt_debug.so beside libttt.so).
//
// TTT_IN(kernel, i, n) is true when 0 <= i < n.  In the debug build a false
// check records the first violation of its translation unit (kernel id,
// index, limit, and a count of all violations) in a device record, and the
// caller skips the access it guards: nothing traps, and no thread leaves a
// kernel early past a barrier its block still waits on.  A copy engine
// operation that is skipped raises the kernel's abort flag, so the other
// roles leave their bounded waits at once.  In the normal build every
// check is the constant true and the kernels are unchanged.
//
// The host reads and clears the records of every translation unit through
// bounds_fetch_all(); ttt_kernel_bounds() and the context calls report them.
#pragma once
#include <stdint.h>

#include <cuda_runtime.h>

namespace ttt {

struct BoundsRecord {
  int kernel;        // id of the first failed check (0: none)
  int count;         // failed checks since the last read
  long long index;   // the index of the first one
  long long limit;   // and its limit
};

// kernel ids of the checks (0 = none)
enum BoundsKernel : int {
  KB_DECODE_TAIL = 1,   // the decode step's row of the chunk buffers
  KB_ATTN_DECODE = 2,   // one-query attention: key/value slices of the ring
  KB_ATTN_FWD_TC = 3,   // tensor-core attention kernels: tile copies
  KB_ATTN_FWD2_TC = 4,
  KB_ATTN_DQ_TC = 5,
  KB_ATTN_DKV_TC = 6,
  KB_SELFTEST = 7,      // ttt_kernel_bounds_selftest
};

inline const char* bounds_kernel_name(int id) {
  switch (id) {
    case KB_DECODE_TAIL: return "decode_tail";
    case KB_ATTN_DECODE: return "attn_decode";
    case KB_ATTN_FWD_TC: return "attn_fwd_tc";
    case KB_ATTN_FWD2_TC: return "attn_fwd2_tc";
    case KB_ATTN_DQ_TC: return "attn_dq_tc";
    case KB_ATTN_DKV_TC: return "attn_dkv_tc";
    case KB_SELFTEST: return "selftest";
    default: return "none";
  }
}

#ifdef TTT_DEBUG_BOUNDS
constexpr bool kBoundsChecked = true;
__device__ __forceinline__ bool bounds_ok_(BoundsRecord* rec, int kid, long long i, long long n) {
  if (i >= 0 && i < n) return true;
  if (atomicAdd(&rec->count, 1) == 0) {
    rec->kernel = kid;
    rec->index = i;
    rec->limit = n;
  }
  return false;
}
// one record per translation unit, and the host function that reads and
// clears it on the current device
#define TTT_BOUNDS_UNIT(name)                                                      \
  namespace {                                                                      \
  __device__ ::ttt::BoundsRecord g_bounds;                                         \
  }                                                                                \
  int bounds_fetch_##name(::ttt::BoundsRecord* out) {                              \
    const ::ttt::BoundsRecord zero = {0, 0, 0, 0};                                 \
    cudaError_t e = cudaMemcpyFromSymbol(out, g_bounds, sizeof(*out));             \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bounds, &zero, sizeof(zero));   \
    return (int)e;                                                                 \
  }
#define TTT_IN(kid, i, n) ::ttt::bounds_ok_(&g_bounds, (kid), (long long)(i), (long long)(n))
#else
constexpr bool kBoundsChecked = false;
#define TTT_BOUNDS_UNIT(name)                                \
  int bounds_fetch_##name(::ttt::BoundsRecord* out) {        \
    *out = ::ttt::BoundsRecord{0, 0, 0, 0};                  \
    return 0;                                                \
  }
#define TTT_IN(kid, i, n) true
#endif

int bounds_fetch_kernels(BoundsRecord* out);
int bounds_fetch_attn_decode(BoundsRecord* out);
int bounds_fetch_attn_tc(BoundsRecord* out);
int bounds_fetch_kernel_api(BoundsRecord* out);

// every unit's record, merged (the first unit with a violation names it,
// counts add up) and cleared; returns a cudaError_t
inline int bounds_fetch_all(BoundsRecord* out) {
  *out = BoundsRecord{0, 0, 0, 0};
  int (*const fetch[])(BoundsRecord*) = {bounds_fetch_kernels, bounds_fetch_attn_decode, bounds_fetch_attn_tc,
                                         bounds_fetch_kernel_api};
  for (auto f : fetch) {
    BoundsRecord r;
    const int e = f(&r);
    if (e) return e;
    if (r.count > 0 && out->count == 0) {
      out->kernel = r.kernel;
      out->index = r.index;
      out->limit = r.limit;
    }
    out->count += r.count;
  }
  return 0;
}

}  // namespace ttt

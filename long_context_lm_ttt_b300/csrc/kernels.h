// kernels.h — host-side launchers of every kernel of the inner loop.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace ttt {

// cudaFuncSetAttribute acts on the current device only.  `done` remembers
// the devices (bit d for device d < 64) on which `kern`'s dynamic shared
// memory limit is already raised to `bytes`; devices beyond 64 are set on
// every call.
template <typename K>
inline cudaError_t raise_smem_limit(std::atomic<uint64_t>& done, K kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load() & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit);
  return e;
}

// While set (per host thread), the launchers of the kernels a decode step
// issues (one-row products, RMSNorm forward, embedding, RoPE table,
// one-query attention, step tail) mark their launches for programmatic
// dependent launch; those kernels call pdl_wait() / pdl_trigger().
void set_pdl(bool on);
bool pdl_enabled();
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  c.attrs = at;
  c.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&c, kern, static_cast<KArgs>(args)...);
}

template <typename T>
struct GemmArgs {
  int M, N, K;
  const T* A;
  int64_t lda;
  int a_mn;
  const T* B;
  int64_t ldb;
  int b_mn;
  Epi e;
  const T* B2;  // optional second B (same layout): C = A B^T + A B2^T
  // optional fp32 scratch: lets the tensor-core GEMM split K across CTAs
  // (partial sums here, then a fixed-order reduction applies the epilogue)
  float* ws = nullptr;
  int64_t ws_elems = 0;
  // tensor-core GEMM CTAs: 0 = one persistent CTA per SM; otherwise at most
  // this many (a large value gives one CTA per tile)
  int grid_cap = 0;
  // tensor-core GEMM tiles: -1 = chosen by the planner, 0 = 128-row tiles on
  // one CTA, 1 = 256-row tiles on a CTA pair (cta_group::2)
  int pair = -1;
  // grouped product (groups > 1): rows [g * group_rows, (g + 1) * group_rows)
  // of A and of the output use the B (and B2) of group g, which starts
  // g * group_stride elements after B (B2); one weight set per sequence
  int groups = 1;
  int group_rows = 0;
  int64_t group_stride = 0;
};

// The epilogue of rows [r0, ...) of a product seen as a product of its own:
// every row-indexed pointer of e moved down r0 rows (T: the element type of
// bf16/fp32 activations).  Covers the epilogues grouped products use.
template <typename T>
inline Epi epi_rows_from(const Epi& e, int64_t r0) {
  Epi o = e;
  switch (e.kind) {
    case EPI_STORE:
      o.out = e.out_f32 ? (void*)((float*)e.out + r0 * e.ldo) : (void*)((T*)e.out + r0 * e.ldo);
      break;
    case EPI_RESID:
      o.out = (float*)e.out + r0 * e.ldo;
      o.resid = e.resid + r0 * e.ldr;
      break;
    case EPI_SWIGLU:
      o.out = (T*)e.out + r0 * e.ldo;
      if (e.stash) o.stash = (T*)e.stash + r0 * e.ld_stash;
      break;
    case EPI_SWIGLU_BWD:
      o.out = (T*)e.out + r0 * e.ldo;
      o.stash = (T*)e.stash + r0 * e.ld_stash;
      break;
    default:
      break;
  }
  return o;
}

// SIMT fp32-accumulate GEMM (check mode; reference for the tensor-core one)
template <typename T> void gemm_simt(const GemmArgs<T>& g, cudaStream_t st);

// tcgen05 / TMA GEMM (bf16 in, fp32 accumulate).  Returns a cudaError_t
// (cudaErrorNotSupported when the shape cannot be described by TMA).
// *kernels (optional) receives the number of kernels launched (2 with a
// split-K reduction).
// one-row product (M = 1) streamed from HBM on SIMT cores (gemv.cu): K-major
// operands, N even, K a multiple of 8, 16-byte aligned x, B, B2 and row
// pitch; the epilogue of g.e per column pair, or EPI_ARGMAX
bool gemv_supported(const GemmArgs<bf16>& g);
int gemv_row(const GemmArgs<bf16>& g, int num_sms, cudaStream_t st);
int gemm_tc(const GemmArgs<bf16>& g, int num_sms, int* dev_err, cudaStream_t st, int* kernels = nullptr);
int gemm_tc_init();

// --- element-wise / row kernels (kernels.cu) -------------------------------
template <typename T>
void launch_embed(const int32_t* tok, int n, const T* E, int d, float* x, int V, int* err_tok,
                  cudaStream_t st);
template <typename T>
void launch_rmsnorm_fwd(const float* x, const float* g, int n, int d, float eps, T* out, float* r,
                        cudaStream_t st);
// out = resid + rmsnorm_bwd(x, g, r, dy); also out_t = (T)out when out_t != null
template <typename T>
void launch_rmsnorm_bwd(const float* x, const float* g, const float* r, const float* dy,
                        const float* resid, int n, int d, float* out, T* out_t, cudaStream_t st);
// RoPE table of positions pos0 .. pos0+n-1 (pos0 read from *pos_dev when
// that is non-null)
void launch_rope_table(int64_t pos0, int n, int hd, float theta, float2* cs, cudaStream_t st,
                       const int64_t* pos_dev = nullptr);
template <typename T>
void launch_rope_bwd(T* dqkv, int n, int ld, int n_rot_heads, int hd, const float2* cs,
                     cudaStream_t st);
void launch_targets(const int32_t* tok, int64_t T, int64_t pos0, int n, int32_t* tgt, int V,
                    int* err_tok, cudaStream_t st);

// State of a decode call kept in device memory, so that every step can
// replay the same captured launches: the step's position and input token,
// its row within the chunk being filled, its index within the call, and
// where the given tokens come from and the inputs go to.
struct DecodeState {
  int64_t pos;            // absolute position of the step's token
  const int32_t* given;   // tokens given by the caller (n_given of them)
  int32_t* out;           // out[i] = input token of step i
  int32_t r;              // row of the chunk the step fills
  int32_t i;              // step index within the call
  int32_t n_given;
  int32_t tok;            // input token of the step
};
// start of a call: pos, r, the given tokens (given[0] is the first input);
// clears the greedy-pick key
void launch_decode_begin(DecodeState* s, int64_t pos, int r, const int32_t* given, int n_given, int32_t* out,
                         unsigned long long* pick, cudaStream_t st);
// end of a step: xdec[r] = x (d floats, the first fast block's input row),
// tok row r and the next input (given[i + 1] if there is one, else the
// column of the greedy-pick key *pick, which is then cleared) into dtok[r],
// dtok[r + 1], out[i] = the step's input, then the state moves to the next
// position (r wraps to 0 after row b - 1)
void launch_decode_tail(DecodeState* s, const float* x, float* xdec, int d, int32_t* dtok, unsigned long long* pick,
                        int b, cudaStream_t st);
template <typename T>
void launch_ce_slab_stats(const float* z, int64_t ldz, int n, int nv, T* p, int64_t ldp,
                          float* m_run, float* l_run, float* alpha, float* beta, int first,
                          cudaStream_t st);
template <typename T>
void launch_ce_finalize(int n, const float* m_run, const float* l_run, const float* ztgt,
                        const int32_t* tgt, float inv_ntgt, const float* dh_acc, const T* Wlm,
                        int d, float* dhf, float* loss_row, cudaStream_t st);
void launch_loss_reduce(const float* loss_row, int n, float inv_ntgt, float* out, int chunk,
                        int* err_chunk, cudaStream_t st);
// pack an fp32 [rows, cols] matrix into T with a row permutation:
// dst[(row_map(r)) * cols + c] = src[r * cols + c]
//   mode 0: identity, 1: rope pair interleave within heads of size hd
//   (i < hd/2 -> 2i, else 2(i-hd/2)+1), 2: interleave into even rows
//   (r -> 2r), 3: interleave into odd rows (r -> 2r+1)
template <typename T>
void launch_pack(const float* src, int64_t rows, int64_t cols, int mode, int hd, T* dst,
                 cudaStream_t st);
// hi = rn(w), lo = rn(w - hi): a bf16 pair whose sum carries ~16 mantissa
// bits (lo may be null: hi alone)
void launch_split_bf16(const float* w, int64_t n, bf16* hi, bf16* lo, cudaStream_t st);

// --- attention (attn_simt.cu / attn_mma.cu) --------------------------------
struct AttnArgs {
  const void* q;      // [n, H*hd] (pair-interleaved RoPE layout)
  const void* kring;  // [Hkv][R][hd]
  const void* vring;
  void* o;            // [n, H*hd]
  float* lse;         // [H][ld_lse]
  int ld_lse;
  int n, H, Hkv, hd, W, R;
  int64_t pos0;
  // non-null: pos0 is read from this device word instead (decode kernel only)
  const int64_t* pos_dev;
  // backward
  const void* dout;   // [n, H*hd]
  const void* out;    // forward output o
  float* Dsum;        // [H][ld_lse]
  void* dqkv;         // [n, (H+2Hkv)*hd]: dq | dk | dv
  float* ws;          // fp32 scratch of the tensor-core backward
  int64_t ws_elems;   //   (attn_bwd_tc_ws_elems() of the shape)
  // tensor-core backward: the chunk's RoPE table [n][hd/2] of (cos, sin);
  // when set, dq and dk leave the kernels already rotated back (the
  // transpose of the forward rotation), so no separate pass is needed
  const float2* rope_cs;
  // tensor-core backward: with side set, the dk/dv kernels run on that
  // stream beside the dq kernels (side_ev[0] forks it after the shared
  // prep, side_ev[1] joins it back), when the scratch also holds the dk/dv
  // partials next to dq's
  cudaStream_t side;
  cudaEvent_t side_ev[2];
};
template <typename T> void attn_fwd_simt(const AttnArgs& a, cudaStream_t st);
// one query position (n == 1, a decode step): key range split into `splits`
// slices (at most kMaxDecodeSplits) folded through fp32 scratch `part` of
// attn_decode_scratch_elems() values: kDecCounters counters (one per KV
// head; zero them once after allocating, the kernels leave them at zero,
// and their place does not depend on the shape, so one scratch serves
// every shape), then the slices; hd a multiple of 32 up to 256, at most 8
// query heads per KV head, at most kDecCounters KV heads.  A bounded wait
// that gives up writes its code into *err.  Returns non-zero if a kernel
// attribute could not be set.
constexpr int kMaxDecodeSplits = 64;
constexpr int kDecCounters = 256;
bool attn_decode_supported(const AttnArgs& a);
int attn_decode_splits(const AttnArgs& a, int num_sms);
int64_t attn_decode_scratch_elems(int H, int hd);
template <typename T> int attn_decode(const AttnArgs& a, int splits, float* part, int* err, cudaStream_t st);
template <typename T> void attn_bwd_simt(const AttnArgs& a, cudaStream_t st);
// tcgen05 kernels (bf16); attn_tc_supported() tells whether the shape and
// alignment fit them (64 <= hd <= 128, hd % 16 == 0, R % 128 == 0).  They
// return a cudaError_t; device-side bounded waits that give up write a code
// into *err.
bool attn_tc_supported(const AttnArgs& a);
// variant 0: choose by size; 1: one 128-row tile per CTA (two CTAs per
// SM); 2: two tiles per CTA with P kept in tensor memory.  With scratch
// (a.ws, at least 3 x (n H hd + 2 n H) floats) variant 2 may split each
// tile pair's key range into parts merged by a second kernel.  *kernels
// (optional) receives the number of kernels launched.
int attn_fwd_tc(const AttnArgs& a, int* err, cudaStream_t st, int variant = 0, int* kernels = nullptr);
int attn_bwd_tc(const AttnArgs& a, int* err, cudaStream_t st);
// the backward additionally needs chunk starts at multiples of 64 and scratch
bool attn_bwd_tc_supported(const AttnArgs& a);
// fp32 elements of scratch attn_bwd_tc needs for a chunk of n rows with the
// given heads (an upper bound over all chunk positions)
int64_t attn_bwd_tc_ws_elems(int n, int H, int hd, int num_sms);

}  // namespace ttt

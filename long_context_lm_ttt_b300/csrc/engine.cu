// engine.cu — the inner loop behind the C ABI of ttt.h.
//
// One context owns, on one GPU:
//   * the weights in the working type T (bf16, or fp32 in check mode), with
//     q/k rows of every head reordered so that RoPE pairs (i, i+hd/2) become
//     adjacent columns (2i, 2i+1) — attention only sees q.k products, which
//     this shared reordering leaves unchanged — and gate/up rows interleaved
//     (gate f -> row 2f, up f -> row 2f+1) so SwiGLU pairs are adjacent too;
//   * fp32 masters of the fast weights (the MLPs of the last n_ttt_layers
//     blocks) and a copy of their initial values for ttt_reset;
//   * per layer a key/value ring (position p in slot p mod R_l), constant in
//     the sequence length: R >= W+b-1 slots for the fast blocks, R_s >=
//     W+S-1 for the static ones;
//   * the activations of one chunk for the fast blocks (the backward needs
//     them all) and one scratch set of S rows for the static blocks.
//
// The static blocks [0, L-n_ttt_layers) never change, so their outputs do
// not depend on any test-time update: ttt_prefill runs them over
// super-chunks of S tokens (a multiple of b) with large-M GEMMs, then runs
// the chunk loop (fast blocks forward, cross-entropy, backward, SGD) over
// the chunks of that super-chunk.  Every value is the one the chunk-by-chunk
// order produces; only the batching of the frozen part differs.
// The residual stream, norm statistics, softmax statistics and all
// gradients that cross kernels in fp32 stay fp32; matrices fed to GEMMs are
// in T.
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <string>
#include <thread>
#include <vector>

#include "../../include/ttt.h"
#include "bounds.cuh"
#include "kernels.h"

namespace ttt {

static thread_local std::string g_create_error;

// ---------------------------------------------------------------------------
struct DeviceArena {
  std::vector<void*> ptrs;
  size_t total = 0;
  cudaError_t alloc(void** p, size_t bytes) {
    *p = nullptr;
    if (bytes == 0) bytes = 16;
    bytes = (bytes + 255) & ~size_t(255);
    cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) {
      ptrs.push_back(*p);
      total += bytes;
    }
    return e;
  }
  ~DeviceArena() {
    for (void* p : ptrs) cudaFree(p);
  }
};

static bool is_device_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

struct Status {
  int code = TTT_OK;
  std::string msg;
};

#define CU_TRY(expr)                                                                         \
  do {                                                                                       \
    cudaError_t e_ = (expr);                                                                 \
    if (e_ != cudaSuccess) {                                                                 \
      err = std::string(#expr) + ": " + cudaGetErrorString(e_);                              \
      return e_ == cudaErrorMemoryAllocation ? TTT_ERR_OOM : TTT_ERR_CUDA;                   \
    }                                                                                        \
  } while (0)

// programmatic dependent launch for the launches issued while in scope
struct PdlScope {
  explicit PdlScope(bool on) { set_pdl(on); }
  ~PdlScope() { set_pdl(false); }
};

// ---------------------------------------------------------------------------
struct EngineBase {
  ttt_config cfg;
  std::string err;
  int R = 0, R_s = 0, S_bulk = 0, qkv_cols = 0, Vs = 0, num_sms = 148;
  // sequences the context holds (ttt_config.n_seq): each has its own fast
  // weights and key/value rings; every activation buffer holds ns blocks
  // of rows, one per sequence, stacked
  int ns = 1;
  int64_t pos = 0;
  bool used = false;
  bool use_tc_gemm = false, use_tc_attn = false, use_tc_attn_bwd = false;
  virtual int init(const ttt_weights* w, cudaStream_t st) = 0;
  virtual int prefill(const int32_t* tok, int64_t T, float* losses, cudaStream_t st) = 0;
  virtual int logits(const int32_t* cont, int n, float* out, cudaStream_t st) = 0;
  virtual int decode(const int32_t* tokens, int64_t n_given, int64_t n_steps, int32_t* tokens_out, float* losses,
                     cudaStream_t st) = 0;
  // decode state: rows of the current chunk already decoded
  int dec_fill = 0;
  bool dec_graph_off = false;  // capture failed once (or asked): issue steps directly
  // programmatic dependent launch in ttt_prefill's chunk loop: off by
  // default (measured slower at 3B / 128K: 2.10 s against 2.06 s per
  // sequence; kernels waiting at their dependency hold the SMs the
  // overlapped bulk pass fills otherwise)
  bool pdl_prefill = false;
  // the chunk loop's weight updates on their own stream (ttt_prefill)
  bool sgd_side_ok = true;
  // programmatic dependent launch inside decode steps (off under profiling:
  // the events between launches would serialise them anyway)
  bool pdl_ok = true;
  virtual int get_fast(int block, int which, float* dst, cudaStream_t st) = 0;
  virtual int reset(cudaStream_t st) = 0;

  // --- optional per-launch timing (ttt_profile) ---------------------------
  // Each profiled launch is bracketed by two events on its own stream; the
  // events are resolved after the call's final synchronisation.
  enum ProfCls {
    P_GEMM_FWD, P_GEMM_LMHEAD, P_GEMM_BWD, P_GEMM_SGD, P_ATTN_FWD, P_ATTN_BWD, P_ROW,
    P_GEMM_FWD_BULK, P_ATTN_FWD_BULK, P_N
  };
  struct ProfRec {
    int cls, nk;
    cudaEvent_t a, b;
    double flops, bytes;
  };
  bool prof_on = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_next = 0;
  std::vector<ProfRec> prof_recs;
  ttt_kernel_stat prof_stat[P_N];
  static const char* prof_name(int c) {
    static const char* n[P_N] = {"gemm_fwd", "gemm_lm_head", "gemm_bwd_dx", "gemm_dw_sgd", "attn_fwd",
                                 "attn_bwd", "rowwise", "gemm_fwd_bulk", "attn_fwd_bulk"};
    return n[c];
  }
  void prof_clear() {
    memset(prof_stat, 0, sizeof(prof_stat));
    for (int c = 0; c < P_N; ++c) snprintf(prof_stat[c].name, sizeof(prof_stat[c].name), "%s", prof_name(c));
    prof_recs.clear();
    ev_next = 0;
  }
  cudaEvent_t prof_event() {
    if (ev_next == ev_pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      ev_pool.push_back(e);
    }
    return ev_pool[ev_next++];
  }
  // nk: kernels the launch function issues
  template <typename F>
  void prof(int cls, double flops, double bytes, cudaStream_t st, F&& launch, int nk = 1) {
    prof(cls, flops, bytes, st, launch, [nk] { return nk; });
  }
  // nk(): kernels the launch issued, asked after it ran
  template <typename F, typename G>
  void prof(int cls, double flops, double bytes, cudaStream_t st, F&& launch, G&& nk) {
    if (!prof_on) {
      launch();
      return;
    }
    cudaEvent_t a = prof_event(), b = prof_event();
    if (a) cudaEventRecord(a, st);
    launch();
    if (b) cudaEventRecord(b, st);
    if (a && b) prof_recs.push_back({cls, nk(), a, b, flops, bytes});
  }
  // after a synchronisation: fold the recorded pairs into prof_stat
  void prof_collect() {
    for (const ProfRec& r : prof_recs) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      ttt_kernel_stat& k = prof_stat[r.cls];
      k.launches += r.nk;
      k.ms += ms;
      k.flops += r.flops;
      k.bytes += r.bytes;
    }
    prof_recs.clear();
    ev_next = 0;
  }
  virtual ~EngineBase() {
    for (cudaEvent_t e : ev_pool) cudaEventDestroy(e);
  }
};

template <typename T>
struct Engine : EngineBase {
  static constexpr bool kBF16 = sizeof(T) == 2;
  DeviceArena mem;
  ~Engine() override {
    cudaDeviceSynchronize();
    for (cudaEvent_t e : {ev_fork, ev_a[0], ev_a[1], ev_b[0], ev_b[1], ev_join_a, ev_join_b, ev_sgd_fork,
                          ev_sgd_join[0], ev_sgd_join[1], ev_dkv[0], ev_dkv[1]})
      if (e) cudaEventDestroy(e);
    if (sd) cudaStreamDestroy(sd);
    if (sa) cudaStreamDestroy(sa);
    if (sb) cudaStreamDestroy(sb);
    if (sc) cudaStreamDestroy(sc);
    for (cudaGraphExec_t& g : dec_graph)
      if (g) cudaGraphExecDestroy(g);
    if (cap_st) cudaStreamDestroy(cap_st);
  }

  struct Layer {
    float *g_attn = nullptr, *g_mlp = nullptr;
    T *wqkv = nullptr, *wo = nullptr, *wgu = nullptr, *wd = nullptr;
    float *wgu32 = nullptr, *wd32 = nullptr;            // fast layers: fp32 value
    T *wgu_lo = nullptr, *wd_lo = nullptr;              // bf16: w ~ hi + lo (null: hi alone)
    float *wgu32_init = nullptr, *wd32_init = nullptr;  // for ttt_reset
    T *kring = nullptr, *vring = nullptr;
    int R = 0;  // ring slots
    int64_t ring_elems = 0;  // one sequence's ring (keys or values): Hkv * R * hd
    // fast blocks: one sequence's gate/up and down weights (the stride of
    // the ns copies every fast-weight array holds)
    int64_t gu_elems = 0, d_elems = 0;
    // dual_mlp, fast blocks: the static second MLP (after the fast one)
    float* g_mlp2 = nullptr;
    T *wgu2 = nullptr, *wd2 = nullptr;
  };
  struct Stash {
    float* x = nullptr;  // layer input (fp32)
    T* xn = nullptr;
    float* r1 = nullptr;
    T* q = nullptr;
    T* o = nullptr;
    float* lse = nullptr;
    float* h = nullptr;
    T* hn = nullptr;
    float* r2 = nullptr;
    T* gu = nullptr;
    T* a = nullptr;
    int ld_lse = 0;
    // dual_mlp, fast blocks: input and norm statistics of the static second
    // MLP and its (gate, up) pairs
    float* h2 = nullptr;
    float* r3 = nullptr;
    T* gu2 = nullptr;
  };
  std::vector<Layer> layers;
  std::vector<Stash> fstash;  // fast blocks
  Stash sstash;               // static blocks, one chunk (ttt_logits)
  Stash bstash;               // static blocks, one super-chunk (ttt_prefill)
  float* bx[2] = {nullptr, nullptr};  // residual stream of the bulk pass
  // Double-buffered by super-chunk parity: the bulk pass over super-chunk
  // k+1 (low-priority stream sa) runs while the chunk loop consumes
  // super-chunk k (high-priority stream sb).
  float* x_lo_buf[2] = {nullptr, nullptr};      // input of the first fast block, S rows
  float2* cs_bulk_buf[2] = {nullptr, nullptr};  // RoPE table of the super-chunk
  float* x_lo = nullptr;                        // buffers of the span being processed
  float2* cs_bulk = nullptr;
  cudaStream_t sa = nullptr, sb = nullptr;
  // the chunk loop's weight updates run on sc, beside the backward of the
  // layers below (ttt_prefill only; see backward()), at the chunk loop's
  // priority: a chunk's backward ends waiting for its last updates
  cudaStream_t sc = nullptr;
  cudaEvent_t ev_sgd_fork = nullptr, ev_sgd_join[2] = {nullptr, nullptr};
  // and the attention backward's dk/dv kernels on sd, beside its dq kernels
  cudaStream_t sd = nullptr;
  cudaEvent_t ev_dkv[2] = {nullptr, nullptr};
  bool sgd_side = false;
  cudaEvent_t ev_fork = nullptr, ev_a[2] = {nullptr, nullptr}, ev_b[2] = {nullptr, nullptr},
              ev_join_a = nullptr, ev_join_b = nullptr;
  int grid_cap = 0;  // CTA cap of tensor-core GEMMs (0: one per SM, persistent)
  const float2* cs_cur = nullptr;  // RoPE table of the chunk being processed
  T *E = nullptr, *Wlm = nullptr;
  float* g_final = nullptr;
  float* xlow[2] = {nullptr, nullptr};
  std::vector<float*> xs;  // inputs of the fast blocks, then the final stream
  int32_t *tgt = nullptr, *tok_stage = nullptr;
  float2* cs = nullptr;
  T* hf = nullptr;
  float* rf = nullptr;
  float *z_slab = nullptr, *m_run = nullptr, *l_run = nullptr, *alpha = nullptr, *beta = nullptr,
        *ztgt = nullptr, *dh_acc = nullptr, *dhf = nullptr, *loss_row = nullptr;
  T* p_slab = nullptr;
  float *dy = nullptr, *dhn = nullptr, *dh = nullptr, *dxn = nullptr, *Dsum = nullptr;
  T *dy_t = nullptr, *dgu = nullptr, *dh_t = nullptr, *dO = nullptr, *dqkv = nullptr;
  // second copies of dy_t and dgu: layers alternate between the two, so a
  // layer's weight updates (on sc) may still read theirs during the next
  // layer's backward (allocated for ttt_prefill with 2+ fast blocks)
  T *dy_t2 = nullptr, *dgu2 = nullptr;
  // dual_mlp: the static MLP's normed input and activation (forward
  // temporaries) and the gradient at its input (backward)
  T *hn2 = nullptr, *a2 = nullptr, *dy2_t = nullptr;
  float* dy2 = nullptr;
  float* losses_stage = nullptr;
  float* logits_stage = nullptr;
  // decode (allocated on first use): the fast blocks' input rows of the
  // current chunk, its tokens (b + 1: the last is the next input) and the
  // tokens of one call
  float* xdec = nullptr;
  int32_t* dtok = nullptr;
  int32_t* dec_out = nullptr;
  float* dec_part = nullptr;  // one-query attention slices (set while decoding)
  float* dec_buf = nullptr;
  // a decode step's position, row and tokens live in device memory
  // (dstate) so that one captured graph per step kind (given next token,
  // greedy) replays every step; dpos is set while such a step is issued
  DecodeState* dstate = nullptr;
  unsigned long long* dec_pick = nullptr;  // greedy-pick key (argmax_key)
  const int64_t* dpos = nullptr;
  cudaGraphExec_t dec_graph[2] = {nullptr, nullptr};
  cudaStream_t cap_st = nullptr;
  int gemm_cls = -1;          // profile class of the next GEMMs, if set
  int* dev_err = nullptr;  // [0] first non-finite chunk, [1] bad token, [2] kernel check
  float* stage32 = nullptr;
  size_t stage32_elems = 0;
  float* attn_ws = nullptr;  // scratch of the tensor-core attention backward
  int64_t attn_ws_elems = 0;
  float* gemm_ws = nullptr;  // split-K partial sums of the tensor-core GEMMs
  int64_t gemm_ws_elems = 0;

  template <typename U>
  int A(U** p, size_t elems) {
    cudaError_t e = mem.alloc((void**)p, elems * sizeof(U));
    if (e != cudaSuccess) {
      err = "cudaMalloc(" + std::to_string(elems * sizeof(U)) + " bytes): " + cudaGetErrorString(e);
      cudaGetLastError();
      return TTT_ERR_OOM;
    }
    return TTT_OK;
  }
#define A_TRY(p, n)            \
  do {                         \
    int rc_ = A(&(p), (n));    \
    if (rc_) return rc_;       \
  } while (0)

  // copy an fp32 [rows, cols] tensor (host or device) into dst (type U) with
  // the row mapping `mode` of launch_pack
  template <typename U>
  int upload(const float* src, int64_t rows, int64_t cols, int mode, U* dst, cudaStream_t st) {
    if (!src) {
      err = "null weight pointer";
      return TTT_ERR_INVALID;
    }
    const float* s = src;
    if (!is_device_ptr(src)) {
      CU_TRY(cudaMemcpyAsync(stage32, src, rows * cols * sizeof(float), cudaMemcpyHostToDevice, st));
      s = stage32;
    }
    launch_pack<U>(s, rows, cols, mode, cfg.head_dim, dst, st);
    if (!is_device_ptr(src)) CU_TRY(cudaStreamSynchronize(st));  // stage reused next call
    CU_TRY(cudaGetLastError());
    return TTT_OK;
  }

  int init(const ttt_weights* w, cudaStream_t st) override {
    const int L = cfg.n_layers, d = cfg.d_model, H = cfg.n_heads, Hkv = cfg.n_kv_heads,
              hd = cfg.head_dim, ff = cfg.d_ff, V = cfg.vocab, b = cfg.chunk, Lt = cfg.n_ttt_layers;
    const int64_t Hhd = (int64_t)H * hd;
    int dev = 0;
    CU_TRY(cudaGetDevice(&dev));
    CU_TRY(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
    {
      // vocabulary slab of the streamed cross-entropy: a whole number of
      // 256-column tiles such that the slab's logits GEMM over b rows fills
      // whole waves of SMs, about 16-24K columns
      auto gcd = [](int a, int c) {
        while (c) {
          const int t = a % c;
          a = c;
          c = t;
        }
        return a;
      };
      const int num_m = (ns * b + 127) / 128;
      const int per = num_sms / gcd(num_sms, num_m);  // n-tiles per whole number of waves
      const int k = std::max(1, 20480 / (per * 256));
      Vs = (int)std::min<int64_t>(V, (int64_t)per * k * 256);
    }
    stage32_elems = std::max<int64_t>((int64_t)V * d, (int64_t)2 * ff * d);
    A_TRY(stage32, stage32_elems);
    A_TRY(E, (size_t)V * d);
    A_TRY(Wlm, (size_t)V * d);
    A_TRY(g_final, d);
    int rc;
    if ((rc = upload<T>(w->tok_embed, V, d, 0, E, st))) return rc;
    if ((rc = upload<T>(w->lm_head, V, d, 0, Wlm, st))) return rc;
    if ((rc = upload<float>(w->final_norm, 1, d, 0, g_final, st))) return rc;
    layers.resize(L);
    for (int l = 0; l < L; ++l) {
      Layer& y = layers[l];
      const bool fast = l >= L - Lt;
      const int copies = fast ? ns : 1;  // fast weights: one copy per sequence
      y.gu_elems = (int64_t)2 * ff * d;
      y.d_elems = (int64_t)d * ff;
      A_TRY(y.g_attn, d);
      A_TRY(y.g_mlp, d);
      A_TRY(y.wqkv, (size_t)qkv_cols * d);
      A_TRY(y.wo, (size_t)d * Hhd);
      A_TRY(y.wgu, (size_t)copies * y.gu_elems);
      A_TRY(y.wd, (size_t)copies * y.d_elems);
      y.R = fast ? R : R_s;
      y.ring_elems = (int64_t)Hkv * y.R * hd;
      A_TRY(y.kring, (size_t)ns * y.ring_elems);
      A_TRY(y.vring, (size_t)ns * y.ring_elems);
      CU_TRY(cudaMemsetAsync(y.kring, 0, sizeof(T) * (size_t)ns * y.ring_elems, st));
      CU_TRY(cudaMemsetAsync(y.vring, 0, sizeof(T) * (size_t)ns * y.ring_elems, st));
      if (!w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo || !w->mlp_norm || !w->w_gate ||
          !w->w_up || !w->w_down) {
        err = "null per-layer weight array";
        return TTT_ERR_INVALID;
      }
      if ((rc = upload<float>(w->attn_norm[l], 1, d, 0, y.g_attn, st))) return rc;
      if ((rc = upload<float>(w->mlp_norm[l], 1, d, 0, y.g_mlp, st))) return rc;
      if ((rc = upload<T>(w->wq[l], Hhd, d, 1, y.wqkv, st))) return rc;
      if ((rc = upload<T>(w->wk[l], (int64_t)Hkv * hd, d, 1, y.wqkv + Hhd * d, st))) return rc;
      if ((rc = upload<T>(w->wv[l], (int64_t)Hkv * hd, d, 0, y.wqkv + (Hhd + (int64_t)Hkv * hd) * d, st)))
        return rc;
      if ((rc = upload<T>(w->wo[l], d, Hhd, 0, y.wo, st))) return rc;
      if ((rc = upload<T>(w->w_gate[l], ff, d, 2, y.wgu, st))) return rc;
      if ((rc = upload<T>(w->w_up[l], ff, d, 3, y.wgu, st))) return rc;
      if ((rc = upload<T>(w->w_down[l], d, ff, 0, y.wd, st))) return rc;
      if (fast) {
        if (kBF16) {
          A_TRY(y.wgu32, (size_t)ns * y.gu_elems);
          A_TRY(y.wd32, (size_t)ns * y.d_elems);
          if ((rc = upload<float>(w->w_gate[l], ff, d, 2, y.wgu32, st))) return rc;
          if ((rc = upload<float>(w->w_up[l], ff, d, 3, y.wgu32, st))) return rc;
          if ((rc = upload<float>(w->w_down[l], d, ff, 0, y.wd32, st))) return rc;
          if (!cfg.fast_bf16_single) {
            A_TRY(y.wgu_lo, (size_t)ns * y.gu_elems);
            A_TRY(y.wd_lo, (size_t)ns * y.d_elems);
          }
        } else {
          y.wgu32 = (float*)y.wgu;
          y.wd32 = (float*)y.wd;
        }
        A_TRY(y.wgu32_init, (size_t)y.gu_elems);
        A_TRY(y.wd32_init, (size_t)y.d_elems);
        CU_TRY(cudaMemcpyAsync(y.wgu32_init, y.wgu32, sizeof(float) * y.gu_elems, cudaMemcpyDeviceToDevice, st));
        CU_TRY(cudaMemcpyAsync(y.wd32_init, y.wd32, sizeof(float) * y.d_elems, cudaMemcpyDeviceToDevice, st));
        // every sequence starts from the same initial fast weights
        for (int q = 1; q < ns; ++q) {
          CU_TRY(cudaMemcpyAsync(y.wgu32 + q * y.gu_elems, y.wgu32_init, sizeof(float) * y.gu_elems,
                                 cudaMemcpyDeviceToDevice, st));
          CU_TRY(cudaMemcpyAsync(y.wd32 + q * y.d_elems, y.wd32_init, sizeof(float) * y.d_elems,
                                 cudaMemcpyDeviceToDevice, st));
        }
        if (kBF16) {
          launch_split_bf16(y.wgu32, ns * y.gu_elems, (bf16*)y.wgu, (bf16*)y.wgu_lo, st);
          launch_split_bf16(y.wd32, ns * y.d_elems, (bf16*)y.wd, (bf16*)y.wd_lo, st);
        }
        if (cfg.dual_mlp) {
          if (!w->mlp2_norm || !w->w_gate2 || !w->w_up2 || !w->w_down2) {
            err = "dual_mlp needs mlp2_norm, w_gate2, w_up2 and w_down2";
            return TTT_ERR_INVALID;
          }
          A_TRY(y.g_mlp2, d);
          A_TRY(y.wgu2, (size_t)2 * ff * d);
          A_TRY(y.wd2, (size_t)d * ff);
          if ((rc = upload<float>(w->mlp2_norm[l], 1, d, 0, y.g_mlp2, st))) return rc;
          if ((rc = upload<T>(w->w_gate2[l], ff, d, 2, y.wgu2, st))) return rc;
          if ((rc = upload<T>(w->w_up2[l], ff, d, 3, y.wgu2, st))) return rc;
          if ((rc = upload<T>(w->w_down2[l], d, ff, 0, y.wd2, st))) return rc;
        }
      }
    }
    // activations of one chunk
    auto alloc_stash = [&](Stash& s, bool fast, int rows) -> int {
      A_TRY(s.xn, (size_t)rows * d);
      A_TRY(s.r1, rows);
      A_TRY(s.q, (size_t)rows * Hhd);
      A_TRY(s.o, (size_t)rows * Hhd);
      A_TRY(s.lse, (size_t)H * rows);
      A_TRY(s.h, (size_t)rows * d);
      A_TRY(s.hn, (size_t)rows * d);
      A_TRY(s.r2, rows);
      A_TRY(s.a, (size_t)rows * ff);
      if (fast) A_TRY(s.gu, (size_t)rows * 2 * ff);
      if (fast && cfg.dual_mlp) {
        A_TRY(s.h2, (size_t)rows * d);
        A_TRY(s.r3, rows);
        A_TRY(s.gu2, (size_t)rows * 2 * ff);
      }
      s.ld_lse = rows;
      return TTT_OK;
    };
    const int rows = ns * b;  // chunk rows of all sequences
    if ((rc = alloc_stash(sstash, false, b))) return rc;
    if (L - Lt > 0) {
      if ((rc = alloc_stash(bstash, false, ns * S_bulk))) return rc;
      A_TRY(bx[0], (size_t)ns * S_bulk * d);
      A_TRY(bx[1], (size_t)ns * S_bulk * d);
    }
    for (int k = 0; k < 2; ++k) {
      A_TRY(x_lo_buf[k], (size_t)ns * S_bulk * d);
      A_TRY(cs_bulk_buf[k], (size_t)S_bulk * (hd / 2));
    }
    x_lo = x_lo_buf[0];
    cs_bulk = cs_bulk_buf[0];
    {
      int lo_pri = 0, hi_pri = 0;
      CU_TRY(cudaDeviceGetStreamPriorityRange(&lo_pri, &hi_pri));
      CU_TRY(cudaStreamCreateWithPriority(&sa, cudaStreamNonBlocking, lo_pri));
      CU_TRY(cudaStreamCreateWithPriority(&sb, cudaStreamNonBlocking, hi_pri));
      CU_TRY(cudaStreamCreateWithPriority(&sc, cudaStreamNonBlocking, hi_pri));
      CU_TRY(cudaStreamCreateWithPriority(&sd, cudaStreamNonBlocking, hi_pri));
      for (cudaEvent_t* e : {&ev_fork, &ev_a[0], &ev_a[1], &ev_b[0], &ev_b[1], &ev_join_a, &ev_join_b, &ev_sgd_fork,
                             &ev_sgd_join[0], &ev_sgd_join[1], &ev_dkv[0], &ev_dkv[1]})
        CU_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    }
    fstash.resize(Lt);
    xs.resize(Lt + 1);
    for (int i = 0; i <= Lt; ++i) A_TRY(xs[i], (size_t)rows * d);
    for (int i = 0; i < Lt; ++i) {
      if ((rc = alloc_stash(fstash[i], true, rows))) return rc;
      fstash[i].x = xs[i];
    }
    A_TRY(xlow[0], (size_t)b * d);
    A_TRY(xlow[1], (size_t)b * d);
    A_TRY(tgt, rows);
    A_TRY(tok_stage, (size_t)ns * std::max<int64_t>(cfg.max_tokens, b));
    A_TRY(cs, (size_t)b * (hd / 2));
    A_TRY(hf, (size_t)rows * d);
    A_TRY(rf, rows);
    A_TRY(z_slab, (size_t)rows * Vs);
    A_TRY(p_slab, (size_t)rows * Vs);
    A_TRY(m_run, rows);
    A_TRY(l_run, rows);
    A_TRY(alpha, rows);
    A_TRY(beta, rows);
    A_TRY(ztgt, rows);
    A_TRY(dh_acc, (size_t)rows * d);
    A_TRY(dhf, (size_t)rows * d);
    A_TRY(loss_row, rows);
    A_TRY(dy, (size_t)rows * d);
    A_TRY(dy_t, (size_t)rows * d);
    A_TRY(dgu, (size_t)rows * 2 * ff);
    if (Lt > 1 && !cfg.dual_mlp) {
      A_TRY(dy_t2, (size_t)rows * d);
      A_TRY(dgu2, (size_t)rows * 2 * ff);
    }
    A_TRY(dhn, (size_t)rows * d);
    A_TRY(dh, (size_t)rows * d);
    A_TRY(dh_t, (size_t)rows * d);
    A_TRY(dO, (size_t)rows * Hhd);
    A_TRY(dqkv, (size_t)rows * qkv_cols);
    A_TRY(dxn, (size_t)rows * d);
    A_TRY(Dsum, (size_t)H * rows);
    if (cfg.dual_mlp && Lt > 0) {
      A_TRY(hn2, (size_t)rows * d);
      A_TRY(a2, (size_t)rows * ff);
      A_TRY(dy2, (size_t)rows * d);
      A_TRY(dy2_t, (size_t)rows * d);
    }
    if (kBF16 && use_tc_gemm) {
      gemm_ws_elems = (int64_t)4 * rows * std::max<int64_t>(std::max<int64_t>(d, qkv_cols), Hhd);
      A_TRY(gemm_ws, (size_t)gemm_ws_elems);
    }
    if (kBF16 && use_tc_attn_bwd) {
      attn_ws_elems = attn_bwd_tc_ws_elems(b, H, hd, num_sms);
      A_TRY(attn_ws, (size_t)attn_ws_elems);
    }
    A_TRY(losses_stage, (size_t)ns * ((cfg.max_tokens + b - 1) / b + 1));
    A_TRY(dev_err, 4);
    CU_TRY(cudaStreamSynchronize(st));
    return TTT_OK;
  }

  // -------------------------------------------------------------------------
  // groups > 1: a grouped product, rows [q * M / groups, ...) against the
  // weights B + q * group_stride (one fast-weight set per sequence)
  void gemm(int M, int N, int K, const T* A_, int64_t lda, int a_mn, const T* B_, int64_t ldb,
            int b_mn, const Epi& e, cudaStream_t st, int* rc, const T* B2 = nullptr, int groups = 1,
            int64_t group_stride = 0) {
    // the split-K scratch belongs to the chunk loop; the bulk pass (grid_cap
    // set, other stream) never splits
    GemmArgs<T> g{M, N, K, A_, lda, a_mn, B_, ldb, b_mn, e, B2, grid_cap ? nullptr : gemm_ws,
                  grid_cap ? 0 : gemm_ws_elems, grid_cap};
    if (groups > 1) {
      g.groups = groups;
      g.group_rows = M / groups;
      g.group_stride = group_stride;
    }
    int cls = P_GEMM_FWD;
    double out_b = (double)M * N * (e.kind == EPI_STORE && !e.out_f32 ? sizeof(T) : 4);
    switch (e.kind) {
      case EPI_RESID: out_b *= 2; break;                              // residual read + write
      case EPI_CE_Z: case EPI_CE_ACC: cls = P_GEMM_LMHEAD; out_b *= 2; break;
      case EPI_SWIGLU_BWD: cls = P_GEMM_BWD; out_b = (double)M * N * 4 * sizeof(T); break;
      case EPI_STORE: cls = P_GEMM_BWD; break;
      case EPI_SGD: cls = P_GEMM_SGD; out_b = (double)M * N * (8 + (e.w16lo ? 2 : 1) * sizeof(T)); break;
      case EPI_SWIGLU: out_b = (double)M * N * sizeof(T) * (e.stash ? 1.5 : 0.5); break;
      default: break;
    }
    // the forward products of the frozen blocks' bulk pass (more rows than a
    // chunk) form their own class
    if (cls == P_GEMM_FWD && M > cfg.chunk) cls = P_GEMM_FWD_BULK;
    if (gemm_cls >= 0) cls = gemm_cls;
    const double flops = 2.0 * M * N * K;
    const double bytes = (double)sizeof(T) * ((double)M * K + (double)N * K) + out_b;
    int nk = 1;
    prof(cls, flops, bytes, st, [&] {
      if constexpr (kBF16) {
        if (use_tc_gemm) {
          int r = gemm_tc(g, num_sms, dev_err + 2, st, &nk);
          if (r != 0 && *rc == TTT_OK) {
            *rc = TTT_ERR_SHAPE;
            err = "tensor-core GEMM rejected M=" + std::to_string(M) + " N=" + std::to_string(N) +
                  " K=" + std::to_string(K) + " (" + cudaGetErrorString((cudaError_t)r) + ")";
          }
          return;
        }
      }
      gemm_simt<T>(g, st);
    }, [&] { return nk; });
  }
  // algorithmic attention work of a chunk of n queries starting at pos0:
  // unmasked (query, key) pairs and the pairs whose key is in the chunk
  void attn_pairs(int64_t pos0, int n, double* pairs, double* local) const {
    const int64_t W = cfg.window;
    double p = 0, q = 0;
    for (int r = 0; r < n; ++r) {
      const int64_t t = pos0 + r;
      p += (double)std::min<int64_t>(t + 1, W);
      q += (double)std::min<int64_t>(r + 1, W);
    }
    *pairs = p;
    *local = q;
  }
  static Epi epi(int kind) {
    Epi e;
    memset(&e, 0, sizeof(e));
    e.kind = kind;
    return e;
  }
  // attention of sequence q (rows [q n, q n + n) of the stash) at positions
  // s .. s + n - 1, against its own key/value ring
  AttnArgs attn_args(const Stash& S, const Layer& y, int64_t s, int n, int q = 0) {
    const int64_t Hhd = (int64_t)cfg.n_heads * cfg.head_dim;
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.q = S.q + (int64_t)q * n * Hhd;
    a.kring = y.kring + (int64_t)q * y.ring_elems;
    a.vring = y.vring + (int64_t)q * y.ring_elems;
    a.o = S.o + (int64_t)q * n * Hhd;
    a.lse = S.lse + (int64_t)q * n;
    a.ld_lse = S.ld_lse;
    a.n = n;
    a.H = cfg.n_heads;
    a.Hkv = cfg.n_kv_heads;
    a.hd = cfg.head_dim;
    a.W = cfg.window;
    a.R = y.R;
    a.pos0 = s;
    a.pos_dev = dpos;
    return a;
  }
  void attn_fwd(const AttnArgs& a, cudaStream_t st, int* rc) {
    double P, Pl;
    attn_pairs(a.pos0, a.n, &P, &Pl);
    const double hdH = (double)a.H * a.hd;
    const double kv = (double)std::min<int64_t>(a.pos0 + a.n, (int64_t)a.W + a.n - 1) * a.Hkv * a.hd;
    const double bytes = sizeof(T) * (2.0 * a.n * hdH + 2.0 * kv) + 4.0 * a.n * a.H;
    int nk = 1;
    prof(a.n > cfg.chunk ? P_ATTN_FWD_BULK : P_ATTN_FWD, 4.0 * hdH * P, bytes, st, [&] {
      // a decode step: one query, the window split over the whole GPU
      if (dec_part && a.n == 1 && attn_decode_supported(a)) {
        if (attn_decode<T>(a, attn_decode_splits(a, num_sms), dec_part, dev_err + 2, st) && *rc == TTT_OK) {
          *rc = TTT_ERR_CUDA;
          err = "one-query attention: kernel attribute not set";
        }
        return;
      }
      if constexpr (kBF16) {
        if (use_tc_attn && attn_tc_supported(a)) {
          // the chunk loop's forward may split key ranges through the
          // attention scratch; the bulk pass (grid_cap set, other stream)
          // never touches it
          AttnArgs as = a;
          if (!grid_cap && attn_ws) {
            as.ws = attn_ws;
            as.ws_elems = attn_ws_elems;
          }
          int r = attn_fwd_tc(as, dev_err + 2, st, 0, &nk);
          if (r != 0 && *rc == TTT_OK) {
            *rc = TTT_ERR_SHAPE;
            err = "tensor-core attention forward rejected the shape";
          }
          return;
        }
      }
      attn_fwd_simt<T>(a, st);
    }, [&] { return nk; });
  }
  // returns true when dq and dk left the kernels already rotated back by
  // the RoPE table a.rope_cs (tensor-core path)
  bool attn_bwd(const AttnArgs& a, cudaStream_t st, int* rc) {
    double P, Pl;
    attn_pairs(a.pos0, a.n, &P, &Pl);
    const double hdH = (double)a.H * a.hd;
    const double kv = (double)std::min<int64_t>(a.pos0 + a.n, (int64_t)a.W + a.n - 1) * a.Hkv * a.hd;
    const double bytes = sizeof(T) * (4.0 * a.n * hdH + 2.0 * kv + (double)a.n * qkv_cols) + 8.0 * a.n * a.H;
    const bool tc = kBF16 && use_tc_attn_bwd && attn_bwd_tc_supported(a);
    prof(P_ATTN_BWD, 6.0 * hdH * P + 4.0 * hdH * Pl, bytes, st, [&] {
      if constexpr (kBF16) {
        if (tc) {
          int r = attn_bwd_tc(a, dev_err + 2, st);
          if (r != 0 && *rc == TTT_OK) {
            *rc = TTT_ERR_SHAPE;
            err = "tensor-core attention backward rejected the shape";
          }
          return;
        }
      }
      attn_bwd_simt<T>(a, st);
    }, tc ? 5 : 3);
    return tc && a.rope_cs != nullptr;
  }
  // row-wise kernels: bytes moved, no tensor work
  template <typename F>
  void row(double bytes, cudaStream_t st, F&& launch) {
    prof(P_ROW, 0.0, bytes, st, launch);
  }

  // one decoder block over the rows of nseq sequences, n rows each, at
  // positions s..s+n-1 (RoPE table cs_), from x_in to x_out, keeping its
  // intermediates in S.  Products with static weights take all rows in one
  // launch; attention runs per sequence; the fast MLP's products are
  // grouped, one weight set per sequence.
  void block_fwd(int l, Stash& S, const float* x_in, float* x_out, const float2* cs_, int64_t s, int n,
                 cudaStream_t st, int* rc, int nseq = 1) {
    const int d = cfg.d_model, H = cfg.n_heads, hd = cfg.head_dim, ff = cfg.d_ff;
    const bool fast = l >= cfg.n_layers - cfg.n_ttt_layers;
    const int64_t Hhd = (int64_t)H * hd;
    const int rows = nseq * n;
    Layer& y = layers[l];
    row((double)rows * d * (4 + sizeof(T)), st, [&] { launch_rmsnorm_fwd<T>(x_in, y.g_attn, rows, d, cfg.norm_eps, S.xn, S.r1, st); });
    Epi e = epi(EPI_QKV);
    e.out = S.q;
    e.ldo = Hhd;
    e.n_q = H;
    e.n_kv = cfg.n_kv_heads;
    e.hd = hd;
    e.pos0 = s;
    e.pos_dev = dpos;
    e.ring = y.R;
    e.kring = y.kring;
    e.vring = y.vring;
    e.rope_cs = cs_;
    if (nseq > 1) {
      e.seg_rows = n;
      e.ring_seq = y.ring_elems;
    }
    gemm(rows, qkv_cols, d, S.xn, d, 0, y.wqkv, d, 0, e, st, rc);
    for (int q = 0; q < nseq; ++q) attn_fwd(attn_args(S, y, s, n, q), st, rc);
    e = epi(EPI_RESID);
    e.out = S.h;
    e.ldo = d;
    e.resid = x_in;
    e.ldr = d;
    gemm(rows, d, (int)Hhd, S.o, Hhd, 0, y.wo, Hhd, 0, e, st, rc);
    row((double)rows * d * (4 + sizeof(T)), st, [&] { launch_rmsnorm_fwd<T>(S.h, y.g_mlp, rows, d, cfg.norm_eps, S.hn, S.r2, st); });
    e = epi(EPI_SWIGLU);
    e.out = S.a;
    e.ldo = ff;
    e.stash = fast ? S.gu : nullptr;
    e.ld_stash = 2 * (int64_t)ff;
    // fast weights in bf16 mode: the pair hi + lo of the master, so updates
    // below one bf16 ulp still reach the forward, or with fast_bf16_single
    // the bf16 copy alone (the low halves are null then)
    const int grp = fast ? nseq : 1;
    gemm(rows, 2 * ff, d, S.hn, d, 0, y.wgu, d, 0, e, st, rc, y.wgu_lo, grp, y.gu_elems);
    const bool dual = fast && cfg.dual_mlp;
    e = epi(EPI_RESID);
    e.out = dual ? S.h2 : x_out;
    e.ldo = d;
    e.resid = S.h;
    e.ldr = d;
    gemm(rows, d, ff, S.a, ff, 0, y.wd, ff, 0, e, st, rc, y.wd_lo, grp, y.d_elems);
    if (dual) {
      // the static second MLP: x_out = h2 + Wd2 (silu(Wg2 n(h2)) * Wu2 n(h2))
      row((double)rows * d * (4 + sizeof(T)), st, [&] { launch_rmsnorm_fwd<T>(S.h2, y.g_mlp2, rows, d, cfg.norm_eps, hn2, S.r3, st); });
      e = epi(EPI_SWIGLU);
      e.out = a2;
      e.ldo = ff;
      e.stash = S.gu2;
      e.ld_stash = 2 * (int64_t)ff;
      gemm(rows, 2 * ff, d, hn2, d, 0, y.wgu2, d, 0, e, st, rc);
      e = epi(EPI_RESID);
      e.out = x_out;
      e.ldo = d;
      e.resid = S.h2;
      e.ldr = d;
      gemm(rows, d, ff, a2, ff, 0, y.wd2, ff, 0, e, st, rc);
    }
  }

  // static blocks over a super-chunk [s0, s0+n): embedding, blocks
  // [0, L-n_ttt_layers); leaves the input of the first fast block in x_lo
  // and the super-chunk's RoPE table in cs_bulk
  // (buffers x_lo_buf[buf], cs_bulk_buf[buf]).  Its GEMMs launch one CTA per
  // tile instead of one persistent CTA per SM, so that SMs free up often
  // for the chunk loop running concurrently on the other stream.
  //
  // With ns sequences the super-chunk's rows are those of every sequence,
  // n rows each, stacked; tok holds the sequences' tokens tok_ld apart.
  void static_fwd(const int32_t* tok, int64_t tok_ld, int64_t s0, int n, int buf, cudaStream_t st, int* rc) {
    const int d = cfg.d_model, hd = cfg.head_dim, lo = cfg.n_layers - cfg.n_ttt_layers;
    // the bulk pass's kernels launch plainly: launched early, they would
    // hold SMs (waiting on their predecessor) that the chunk loop needs
    const bool pdl_was = pdl_enabled();
    set_pdl(false);
    float2* cs_ = cs_bulk_buf[buf];
    float* xl = x_lo_buf[buf];
    row((double)n * hd * 4, st, [&] { launch_rope_table(s0, n, hd, cfg.rope_theta, cs_, st); });
    float* x = lo == 0 ? xl : bx[0];
    for (int q = 0; q < ns; ++q)
      row((double)n * d * (4 + sizeof(T)), st, [&] {
        launch_embed<T>(tok + q * tok_ld + s0, n, E, d, x + (int64_t)q * n * d, cfg.vocab, dev_err + 1, st);
      });
    grid_cap = INT_MAX;
    for (int l = 0; l < lo; ++l) {
      float* x_out = l + 1 == lo ? xl : bx[(l + 1) & 1];
      block_fwd(l, bstash, x, x_out, cs_, s0, n, st, rc, ns);
      x = x_out;
    }
    grid_cap = 0;
    set_pdl(pdl_was);
  }

  // fast blocks of positions [s, s+n) from x_in (the output of the static
  // blocks), then the final norm: leaves the normed hidden state in hf and
  // its statistics in rf
  // (nseq sequences: x_in holds their rows stacked, n each)
  void fast_fwd(const float* x_in, const float2* cs_, int64_t s, int n, cudaStream_t st, int* rc, int nseq = 1) {
    const int L = cfg.n_layers, d = cfg.d_model, Lt = cfg.n_ttt_layers, lo = L - Lt;
    const int rows = nseq * n;
    cs_cur = cs_;
    if (Lt > 0) fstash[0].x = const_cast<float*>(x_in);
    const float* x = x_in;
    for (int l = lo; l < L; ++l) {
      float* x_out = xs[l + 1 - lo];
      block_fwd(l, fstash[l - lo], x, x_out, cs_, s, n, st, rc, nseq);
      x = x_out;
    }
    row((double)rows * d * (4 + sizeof(T)), st, [&] { launch_rmsnorm_fwd<T>(x, g_final, rows, d, cfg.norm_eps, hf, rf, st); });
  }

  // every block for a span of at most b positions (ttt_logits)
  void forward_all(const int32_t* tok, int64_t s, int n, cudaStream_t st, int* rc) {
    const int d = cfg.d_model, hd = cfg.head_dim, lo = cfg.n_layers - cfg.n_ttt_layers;
    row((double)n * hd * 4, st, [&] { launch_rope_table(s, n, hd, cfg.rope_theta, cs, st, dpos); });
    float* x = xlow[0];
    row((double)n * d * (4 + sizeof(T)), st, [&] { launch_embed<T>(tok, n, E, d, x, cfg.vocab, dev_err + 1, st); });
    for (int l = 0; l < lo; ++l) {
      float* x_out = xlow[(l + 1) & 1];
      block_fwd(l, sstash, x, x_out, cs, s, n, st, rc);
      x = x_out;
    }
    fast_fwd(x, cs, s, n, st, rc);
  }

  // streamed lm_head + cross-entropy: loss of chunk c into losses[c] and the
  // gradient w.r.t. the final normed hidden state into dhf (fp32)
  // need_grad = false (no fast blocks): the loss only, no d hidden
  // nseq sequences: tok and losses of sequence q start q * tok_ld and
  // q * loss_ld elements in; the hidden rows are stacked, n per sequence
  void cross_entropy(const int32_t* tok, int64_t n_tok, int64_t s, int n, int n_tgt, float* losses, int c,
                     cudaStream_t st, int* rc, bool need_grad = true, int nseq = 1, int64_t tok_ld = 0,
                     int64_t loss_ld = 0) {
    const int d = cfg.d_model, V = cfg.vocab;
    const int n1 = n;  // rows of one sequence
    for (int q = 0; q < nseq; ++q)
      row((double)n1 * 8, st, [&] { launch_targets(tok + q * tok_ld, n_tok, s, n1, tgt + (int64_t)q * n1, V, dev_err + 1, st); });
    n = nseq * n1;  // every row from here on
    for (int v0 = 0; v0 < V; v0 += Vs) {
      const int nv = std::min(Vs, V - v0);
      const int first = v0 == 0;
      Epi e = epi(EPI_CE_Z);
      e.out = z_slab;
      e.ldo = Vs;
      e.tgt = tgt;
      e.ztgt = ztgt;
      e.col0 = v0;
      gemm(n, nv, d, hf, d, 0, Wlm + (int64_t)v0 * d, d, 0, e, st, rc);
      row((double)n * nv * (4 + sizeof(T)), st, [&] { launch_ce_slab_stats<T>(z_slab, Vs, n, nv, p_slab, Vs, m_run, l_run, alpha, beta, first, st); });
      if (!need_grad) continue;
      e = epi(EPI_CE_ACC);
      e.out = dh_acc;
      e.ldo = d;
      e.alpha = alpha;
      e.beta = beta;
      e.first = first;
      gemm(n, d, nv, p_slab, Vs, 0, Wlm + (int64_t)v0 * d, d, 1, e, st, rc);
    }
    const float inv = 1.0f / (float)n_tgt;
    row((double)n * d * (8 + sizeof(T)), st, [&] {
      launch_ce_finalize<T>(n, m_run, l_run, ztgt, tgt, inv, need_grad ? dh_acc : nullptr, Wlm, d, dhf, loss_row, st);
    });
    for (int q = 0; q < nseq; ++q)
      row((double)n1 * 4, st, [&] { launch_loss_reduce(loss_row + (int64_t)q * n1, n1, inv, losses + q * loss_ld, c, dev_err, st); });
  }

  // backward of the chunk loss into the fast MLPs, with the SGD step fused
  // into the weight-gradient GEMMs.  Every read of a fast weight (da, dhn)
  // happens before that weight's update in stream order.
  // nseq sequences: rows stacked, n per sequence; the fast MLPs' input
  // gradients are grouped products and each sequence takes its own SGD step
  void backward(int64_t s, int n, cudaStream_t st, int* rc, int nseq = 1) {
    const int L = cfg.n_layers, d = cfg.d_model, H = cfg.n_heads, Hkv = cfg.n_kv_heads,
              hd = cfg.head_dim, ff = cfg.d_ff, Lt = cfg.n_ttt_layers;
    const int lo = L - Lt;
    const int64_t Hhd = (int64_t)H * hd;
    const int rows = nseq * n;
    // With sgd_side, each layer's weight updates run on sc (see below).
    // deep: dy_t and dgu alternate between two buffers by layer, so the
    // updates of layer l may run on through layer l - 1's backward, and the
    // chunk loop waits for them only before layer l - 1's last norm backward
    // writes their dy_t buffer again; otherwise it waits before layer l's.
    const bool side = sgd_side && !prof_on;
    const bool deep = side && dy_t2 && dgu2;
    T* const dyt[2] = {dy_t, deep ? dy_t2 : dy_t};
    T* const dgub[2] = {dgu, deep ? dgu2 : dgu};
    int cur = 0;                         // this layer's dy_t / dgu buffer
    bool pending[2] = {false, false};    // updates on sc not yet waited for, by buffer
    row((double)rows * d * (12 + sizeof(T)), st, [&] { launch_rmsnorm_bwd<T>(xs[Lt], g_final, rf, dhf, nullptr, rows, d, dy, dyt[cur], st); });
    for (int l = L - 1; l >= lo; --l) {
      Stash& S = fstash[l - lo];
      Layer& y = layers[l];
      T* const dgu_l = dgub[cur];
      // gradient at the fast MLP's output: dy, or with dual_mlp the one at
      // the static second MLP's input h2 = dy + n'(h2)^T ([dg2 du2] [Wg2; Wu2])
      float* gy = dy;
      T* gy_t = dyt[cur];
      if (cfg.dual_mlp) {
        Epi e2 = epi(EPI_SWIGLU_BWD);
        e2.out = dgu_l;
        e2.ldo = 2 * (int64_t)ff;
        e2.stash = S.gu2;
        e2.ld_stash = 2 * (int64_t)ff;
        gemm(rows, ff, d, dyt[cur], d, 0, y.wd2, ff, 1, e2, st, rc);
        e2 = epi(EPI_STORE);
        e2.out_f32 = 1;
        e2.out = dhn;
        e2.ldo = d;
        gemm(rows, d, 2 * ff, dgu_l, 2 * (int64_t)ff, 0, y.wgu2, d, 1, e2, st, rc);
        row((double)rows * d * (16 + sizeof(T)), st, [&] { launch_rmsnorm_bwd<T>(S.h2, y.g_mlp2, S.r3, dhn, dy, rows, d, dy2, dy2_t, st); });
        gy = dy2;
        gy_t = dy2_t;
      }
      // da = dy Wd  ->  (dg, du) with the stashed (g, u)
      Epi e = epi(EPI_SWIGLU_BWD);
      e.out = dgu_l;
      e.ldo = 2 * (int64_t)ff;
      e.stash = S.gu;
      e.ld_stash = 2 * (int64_t)ff;
      gemm(rows, ff, d, gy_t, d, 0, y.wd, ff, 1, e, st, rc, nullptr, nseq, y.d_elems);
      if (l > lo) {
        // dhn = [dg du] [Wg; Wu]
        e = epi(EPI_STORE);
        e.out_f32 = 1;
        e.out = dhn;
        e.ldo = d;
        gemm(rows, d, 2 * ff, dgu_l, 2 * (int64_t)ff, 0, y.wgu, d, 1, e, st, rc, nullptr, nseq, y.gu_elems);
      }
      // per sequence: Wd -= lr dy^T a ;  [Wg;Wu] -= lr [dg du]^T hn.
      // Nothing after this point reads this layer's fast weights, so with
      // sgd_side the updates run on sc beside the layer's remaining backward
      // (norm, o-proj and attention backward, the QKV product), whose
      // partial waves leave SMs free; they read only dy_t / dy2_t, dgu and
      // the stash, which nothing rewrites before the wait described above.
      // One CTA per tile, so that the chunk loop's own CTAs get SMs back
      // soon.
      cudaStream_t su = side ? sc : st;
      if (side) {
        cudaEventRecord(ev_sgd_fork, st);
        cudaStreamWaitEvent(sc, ev_sgd_fork, 0);
        grid_cap = INT_MAX;
      }
      for (int q = 0; q < nseq; ++q) {
        const int64_t r0 = (int64_t)q * n;
        e = epi(EPI_SGD);
        e.w32 = y.wd32 + q * y.d_elems;
        e.w16 = kBF16 ? (void*)(y.wd + q * y.d_elems) : nullptr;
        e.w16lo = y.wd_lo ? y.wd_lo + q * y.d_elems : nullptr;
        e.ldo = ff;
        e.lr = cfg.lr;
        gemm(d, ff, n, gy_t + r0 * d, d, 1, S.a + r0 * ff, ff, 1, e, su, rc);
        e.w32 = y.wgu32 + q * y.gu_elems;
        e.w16 = kBF16 ? (void*)(y.wgu + q * y.gu_elems) : nullptr;
        e.w16lo = y.wgu_lo ? y.wgu_lo + q * y.gu_elems : nullptr;
        e.ldo = d;
        gemm(2 * ff, d, n, dgu_l + r0 * 2 * ff, 2 * (int64_t)ff, 1, S.hn + r0 * d, d, 1, e, su, rc);
      }
      if (side) {
        grid_cap = 0;
        cudaEventRecord(ev_sgd_join[cur], sc);
        pending[cur] = true;
      }
      if (l == lo) {
        for (int k = 0; k < 2; ++k)
          if (pending[k]) cudaStreamWaitEvent(st, ev_sgd_join[k], 0);
        break;
      }
      // through the MLP norm and the residual
      row((double)rows * d * (16 + sizeof(T)), st, [&] { launch_rmsnorm_bwd<T>(S.h, y.g_mlp, S.r2, dhn, gy, rows, d, dh, dh_t, st); });
      // dO = dh Wo
      e = epi(EPI_STORE);
      e.out = dO;
      e.ldo = Hhd;
      gemm(rows, (int)Hhd, d, dh_t, d, 0, y.wo, Hhd, 1, e, st, rc);
      for (int q = 0; q < nseq; ++q) {
        const int64_t r0 = (int64_t)q * n;
        AttnArgs a = attn_args(S, y, s, n, q);
        a.dout = dO + r0 * Hhd;
        a.out = S.o + r0 * Hhd;
        a.Dsum = Dsum + r0;
        a.dqkv = dqkv + r0 * qkv_cols;
        a.ws = attn_ws;
        a.ws_elems = attn_ws_elems;
        a.rope_cs = cs_cur;
        if (side) {  // ttt_prefill's chunk loop: dk/dv beside dq
          a.side = sd;
          a.side_ev[0] = ev_dkv[0];
          a.side_ev[1] = ev_dkv[1];
        }
        // the tensor-core backward rotates dq, dk back as it writes them
        if (!attn_bwd(a, st, rc))
          row((double)n * (H + Hkv) * hd * 2 * sizeof(T), st, [&] {
            launch_rope_bwd<T>(dqkv + r0 * qkv_cols, n, qkv_cols, H + Hkv, hd, cs_cur, st);
          });
      }
      // dxn = [dq dk dv] Wqkv
      e = epi(EPI_STORE);
      e.out_f32 = 1;
      e.out = dxn;
      e.ldo = d;
      gemm(rows, d, qkv_cols, dqkv, qkv_cols, 0, y.wqkv, d, 1, e, st, rc);
      // the next layer's dy_t buffer: its last reader (updates of the layer
      // above, deep, or of this layer) must be done
      const int nxt = deep ? 1 - cur : cur;
      if (pending[nxt]) {
        cudaStreamWaitEvent(st, ev_sgd_join[nxt], 0);
        pending[nxt] = false;
      }
      row((double)rows * d * (16 + sizeof(T)), st, [&] { launch_rmsnorm_bwd<T>(S.x, y.g_attn, S.r1, dxn, dh, rows, d, dy, dyt[nxt], st); });
      cur = nxt;
    }
  }

  int finish(cudaStream_t st, const char* what) {
    CU_TRY(cudaGetLastError());
    int h_err[3];
    CU_TRY(cudaMemcpyAsync(h_err, dev_err, sizeof(h_err), cudaMemcpyDeviceToHost, st));
    CU_TRY(cudaStreamSynchronize(st));
    if (prof_on) prof_collect();
    if (kBoundsChecked) {
      // the debug build's range checks (every stream's work has joined st)
      CU_TRY(cudaDeviceSynchronize());
      BoundsRecord br;
      CU_TRY((cudaError_t)bounds_fetch_all(&br));
      if (br.count > 0) {
        err = std::string(what) + ": range check failed in " + bounds_kernel_name(br.kernel) + " (index " +
              std::to_string(br.index) + " outside [0, " + std::to_string(br.limit) + "), " +
              std::to_string(br.count) + " failed checks)";
        return TTT_ERR_INTERNAL;
      }
    }
    if (h_err[2] != 0) {
      err = std::string(what) + ": a device-side check failed (code " + std::to_string(h_err[2]) + ")";
      return TTT_ERR_INTERNAL;
    }
    if (h_err[1] != 0) {
      err = std::string(what) + ": token id outside [0, vocab)";
      return TTT_ERR_INVALID;
    }
    if (h_err[0] != INT_MAX) {
      err = std::string(what) + ": non-finite loss at chunk " + std::to_string(h_err[0]);
      return TTT_ERR_NONFINITE;
    }
    return TTT_OK;
  }
  int clear_err(cudaStream_t st) {
    int h_err[4] = {INT_MAX, 0, 0, 0};
    CU_TRY(cudaMemcpyAsync(dev_err, h_err, sizeof(h_err), cudaMemcpyHostToDevice, st));
    return TTT_OK;
  }

  int prefill(const int32_t* tok, int64_t n_tok, float* losses, cudaStream_t st) override {
    const int b = cfg.chunk;
    // consecutive kernels on each stream overlap their launch and set-up
    // with the kernel before (each waits on it before touching memory)
    PdlScope pdl_scope(pdl_prefill && !prof_on);
    if (used) {
      err = "ttt_prefill needs a fresh or reset context";
      return TTT_ERR_STATE;
    }
    if (n_tok < 1 || n_tok > cfg.max_tokens) {
      err = "T must be in [1, max_tokens]";
      return TTT_ERR_SHAPE;
    }
    if (!tok || !losses) {
      err = "null tokens or losses";
      return TTT_ERR_INVALID;
    }
    const int nC = (int)((n_tok + b - 1) / b);
    const int32_t* tok_d = tok;
    if (!is_device_ptr(tok)) {
      CU_TRY(cudaMemcpyAsync(tok_stage, tok, sizeof(int32_t) * ns * n_tok, cudaMemcpyHostToDevice, st));
      tok_d = tok_stage;
    }
    const bool host_out = !is_device_ptr(losses);
    float* loss_d = host_out ? losses_stage : losses;
    int rc = clear_err(st);
    if (rc) return rc;
    used = true;
    const int d = cfg.d_model, hd = cfg.head_dim;
    // Two internal streams fork from `st`: s_bulk runs the bulk pass of the
    // frozen blocks one super-chunk ahead, s_loop the chunk loop.  Events order
    // the hand-offs: the chunk loop of super-chunk k waits for its bulk pass
    // (ev_a); the bulk pass of super-chunk k+2 reuses buffer k & 1 and waits
    // for the chunk loop of k (ev_b).  Both join back into `st`.  With
    // profiling on, both roles run on `st` itself, in the same order.
    cudaStream_t s_bulk = prof_on ? st : sa, s_loop = prof_on ? st : sb;
    CU_TRY(cudaEventRecord(ev_fork, st));
    CU_TRY(cudaStreamWaitEvent(s_bulk, ev_fork, 0));
    CU_TRY(cudaStreamWaitEvent(s_loop, ev_fork, 0));
    const int nS = (int)((n_tok + S_bulk - 1) / S_bulk);
    auto bulk = [&](int k) {
      const int64_t s0 = (int64_t)k * S_bulk;
      const int sn = (int)std::min<int64_t>(S_bulk, n_tok - s0);
      if (k >= 2) cudaStreamWaitEvent(s_bulk, ev_b[k & 1], 0);
      static_fwd(tok_d, n_tok, s0, sn, k & 1, s_bulk, &rc);
      cudaEventRecord(ev_a[k & 1], s_bulk);
    };
    bulk(0);
    for (int k = 0; k < nS && rc == TTT_OK; ++k) {
      if (k + 1 < nS) bulk(k + 1);
      const int64_t s0 = (int64_t)k * S_bulk;
      const int sn = (int)std::min<int64_t>(S_bulk, n_tok - s0);
      CU_TRY(cudaStreamWaitEvent(s_loop, ev_a[k & 1], 0));
      x_lo = x_lo_buf[k & 1];
      cs_bulk = cs_bulk_buf[k & 1];
      for (int64_t s = s0; s < s0 + sn && rc == TTT_OK; s += b) {
        const int c = (int)(s / b);
        const int n = (int)std::min<int64_t>(b, n_tok - s);
        const int n_tgt = (int)std::min<int64_t>(n, n_tok - 1 - s);
        const float* xin = x_lo + (s - s0) * d;
        if (ns > 1) {
          // the chunk's rows of every sequence (sn rows apart in the
          // super-chunk's output), stacked for the chunk loop
          CU_TRY(cudaMemcpy2DAsync(xs[0], sizeof(float) * (size_t)n * d, xin, sizeof(float) * (size_t)sn * d,
                                   sizeof(float) * (size_t)n * d, ns, cudaMemcpyDeviceToDevice, s_loop));
          xin = xs[0];
        }
        fast_fwd(xin, cs_bulk + (s - s0) * (hd / 2), s, n, s_loop, &rc, ns);
        if (n_tgt <= 0) {
          for (int q = 0; q < ns; ++q)
            CU_TRY(cudaMemsetAsync(loss_d + (int64_t)q * nC + c, 0, sizeof(float), s_loop));
          continue;
        }
        // without fast blocks the chunk loop only scores the chunk
        cross_entropy(tok_d, n_tok, s, n, n_tgt, loss_d, c, s_loop, &rc, cfg.n_ttt_layers > 0, ns, n_tok, nC);
        if (cfg.n_ttt_layers > 0) {
          sgd_side = sgd_side_ok;
          backward(s, n, s_loop, &rc, ns);
          sgd_side = false;
        }
        CU_TRY(cudaPeekAtLastError());
      }
      CU_TRY(cudaEventRecord(ev_b[k & 1], s_loop));
    }
    CU_TRY(cudaEventRecord(ev_join_a, s_bulk));
    CU_TRY(cudaEventRecord(ev_join_b, s_loop));
    CU_TRY(cudaStreamWaitEvent(st, ev_join_a, 0));
    CU_TRY(cudaStreamWaitEvent(st, ev_join_b, 0));
    if (rc) {
      cudaStreamSynchronize(st);
      return rc;
    }
    pos = n_tok;
    if (host_out)
      CU_TRY(cudaMemcpyAsync(losses, loss_d, sizeof(float) * ns * nC, cudaMemcpyDeviceToHost, st));
    return finish(st, "ttt_prefill");
  }

  // One decode step at the position held in dstate: every block over the
  // step's input token with the current weights (the one-query attention
  // splitting the window over the GPU), then, for kind 1, the greedy pick;
  // the tail kernel stores the first fast block's input row, the tokens and
  // the next input, and advances the state.  Nothing issued here depends on
  // the host's copy of the position, so the same launches serve every step.
  void decode_step(int kind, cudaStream_t st, int* rc) {
    const int b = cfg.chunk, d = cfg.d_model, V = cfg.vocab;
    const int lo = cfg.n_layers - cfg.n_ttt_layers;
    dec_part = dec_buf;
    dpos = &dstate->pos;
    // consecutive kernels of the step overlap their start-up (and the
    // one-row products their first weight loads) with the kernel before
    set_pdl(pdl_ok && !prof_on);
    forward_all(&dstate->tok, pos, 1, st, rc);
    dpos = nullptr;
    dec_part = nullptr;
    if (kind == 1) {
      // lm_head with the greedy pick fused: each block folds its columns'
      // keys and takes one atomic max on dec_pick (no logits are stored)
      Epi e = epi(EPI_ARGMAX);
      e.out = dec_pick;
      gemm_cls = P_GEMM_LMHEAD;
      gemm(1, V, d, hf, d, 0, Wlm, d, 0, e, st, rc);
      gemm_cls = -1;
    }
    row((double)d * 8, st, [&] { launch_decode_tail(dstate, xlow[lo & 1], xdec, d, dtok, dec_pick, b, st); });
    set_pdl(false);
  }
  // Record the launches of one decode step of the given kind into a graph
  // (on a stream of the engine's own: capture needs one that is not the
  // legacy default stream).  The step has run once directly before, so
  // every lazy set-up (kernel attributes, scratch) is done.  A failed
  // capture leaves the steps issued directly.
  void capture_decode_step(int kind) {
    if (!cap_st && cudaStreamCreateWithFlags(&cap_st, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      dec_graph_off = true;
      return;
    }
    cudaGraph_t g = nullptr;
    int rc = TTT_OK;
    if (cudaStreamBeginCapture(cap_st, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
      decode_step(kind, cap_st, &rc);
      if (cudaStreamEndCapture(cap_st, &g) != cudaSuccess) g = nullptr;
    }
    if (!g || rc != TTT_OK || cudaGraphInstantiate(&dec_graph[kind], g, 0) != cudaSuccess) {
      dec_graph[kind] = nullptr;
      dec_graph_off = true;
    }
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
  }

  // Decode-time test-time training: one token per step through every block
  // with the current weights, then the greedy next token; when a chunk of b
  // positions is complete, the same test-time step as the prefill's chunk
  // loop (fast blocks recomputed over the chunk, loss, backward, SGD).
  // The first step of each kind is issued directly and then captured; later
  // ones replay the graph (one launch from the host instead of one per
  // kernel).  The chunk's test-time step is issued directly.
  int decode(const int32_t* tokens, int64_t n_given, int64_t n_steps, int32_t* tokens_out, float* losses,
             cudaStream_t st) override {
    const int b = cfg.chunk, d = cfg.d_model, hd = cfg.head_dim, V = cfg.vocab;
    if (!tokens || !tokens_out || !losses) {
      err = "null tokens, tokens_out or chunk_losses";
      return TTT_ERR_INVALID;
    }
    if (ns > 1) {
      err = "ttt_decode takes a context of one sequence (n_seq <= 1)";
      return TTT_ERR_STATE;
    }
    if (n_steps < 1 || n_given < 1 || n_given > n_steps + 1) {
      err = "need 1 <= n_given <= n_steps + 1";
      return TTT_ERR_INVALID;
    }
    if (pos + n_steps > cfg.max_tokens || n_given > std::max<int64_t>(cfg.max_tokens, b)) {
      err = "decode past max_tokens";
      return TTT_ERR_SHAPE;
    }
    if (dec_fill == 0 && pos % b != 0) {
      err = "decode starts at a chunk boundary (a prefill of a multiple of the chunk length)";
      return TTT_ERR_STATE;
    }
    if (!xdec) {
      A_TRY(xdec, (size_t)b * d);
      A_TRY(dtok, (size_t)b + 1);
      A_TRY(dec_out, (size_t)cfg.max_tokens + 1);
      const int64_t part_elems = attn_decode_scratch_elems(cfg.n_heads, hd);
      A_TRY(dec_buf, (size_t)part_elems);
      // the one-query attention's per-KV-head counters start at zero
      CU_TRY(cudaMemsetAsync(dec_buf, 0, sizeof(float) * part_elems, st));
      A_TRY(dec_pick, 1);
      CU_TRY(mem.alloc((void**)&dstate, sizeof(DecodeState)));
    }
    const int32_t* given = tokens;
    if (!is_device_ptr(tokens)) {
      CU_TRY(cudaMemcpyAsync(tok_stage, tokens, sizeof(int32_t) * n_given, cudaMemcpyHostToDevice, st));
      given = tok_stage;
    }
    const bool host_tok = !is_device_ptr(tokens_out), host_loss = !is_device_ptr(losses);
    int32_t* tok_d = host_tok ? dec_out : tokens_out;
    float* loss_d = host_loss ? losses_stage : losses;
    int rc = clear_err(st);
    if (rc) return rc;
    used = true;
    row(0.0, st, [&] { launch_decode_begin(dstate, pos, dec_fill, given, (int)n_given, tok_d, dec_pick, st); });
    int done = 0;  // chunks completed by this call
    for (int64_t i = 0; i < n_steps && rc == TTT_OK; ++i) {
      const int kind = i + 1 < n_given ? 0 : 1;  // 0: next input given, 1: greedy
      if (dec_graph[kind] && !prof_on) {
        CU_TRY(cudaGraphLaunch(dec_graph[kind], st));
      } else {
        decode_step(kind, st, &rc);
        if (rc == TTT_OK && !prof_on && !dec_graph_off) capture_decode_step(kind);
      }
      pos += 1;
      dec_fill += 1;
      if (dec_fill == b) {
        // chunk [s, s + b) complete; its targets are dtok[1..b]
        const int64_t s = pos - b;
        row((double)b * hd * 4, st, [&] { launch_rope_table(s, b, hd, cfg.rope_theta, cs, st); });
        fast_fwd(xdec, cs, s, b, st, &rc);
        cross_entropy(dtok, b + 1, 0, b, b, loss_d, done, st, &rc, cfg.n_ttt_layers > 0);
        if (cfg.n_ttt_layers > 0) backward(s, b, st, &rc);
        CU_TRY(cudaMemcpyAsync(dtok, dtok + b, sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
        dec_fill = 0;
        ++done;
      }
      CU_TRY(cudaPeekAtLastError());
    }
    if (rc) {
      cudaStreamSynchronize(st);
      return rc;
    }
    // the prediction after the last step (the next input)
    CU_TRY(cudaMemcpyAsync(tok_d + n_steps, dtok + dec_fill, sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    if (host_tok)
      CU_TRY(cudaMemcpyAsync(tokens_out, tok_d, sizeof(int32_t) * (n_steps + 1), cudaMemcpyDeviceToHost, st));
    if (host_loss && done > 0)
      CU_TRY(cudaMemcpyAsync(losses, loss_d, sizeof(float) * done, cudaMemcpyDeviceToHost, st));
    return finish(st, "ttt_decode");
  }

  int logits(const int32_t* cont, int n, float* out, cudaStream_t st) override {
    if (n < 1 || n > cfg.chunk) {
      err = "n must be in [1, chunk]";
      return TTT_ERR_SHAPE;
    }
    if (!cont || !out) {
      err = "null continuation or logits";
      return TTT_ERR_INVALID;
    }
    if (ns > 1) {
      err = "ttt_logits takes a context of one sequence (n_seq <= 1)";
      return TTT_ERR_STATE;
    }
    const int32_t* c_d = cont;
    if (!is_device_ptr(cont)) {
      CU_TRY(cudaMemcpyAsync(tok_stage, cont, sizeof(int32_t) * n, cudaMemcpyHostToDevice, st));
      c_d = tok_stage;
    }
    const bool host_out = !is_device_ptr(out);
    float* o = out;
    if (host_out) {
      if (!logits_stage) A_TRY(logits_stage, (size_t)cfg.chunk * cfg.vocab);
      o = logits_stage;
    }
    int rc = clear_err(st);
    if (rc) return rc;
    forward_all(c_d, pos, n, st, &rc);
    Epi e = epi(EPI_STORE);
    e.out_f32 = 1;
    e.out = o;
    e.ldo = cfg.vocab;
    gemm(n, cfg.vocab, cfg.d_model, hf, cfg.d_model, 0, Wlm, cfg.d_model, 0, e, st, &rc);
    if (rc) return rc;
    if (host_out)
      CU_TRY(cudaMemcpyAsync(out, o, sizeof(float) * (size_t)n * cfg.vocab, cudaMemcpyDeviceToHost, st));
    return finish(st, "ttt_logits");
  }

  int get_fast(int block, int which, float* dst, cudaStream_t st) override {
    const int d = cfg.d_model, ff = cfg.d_ff;
    // with several sequences, block counts over them: sequence q's block i
    // is q * n_ttt_layers + i
    if (block < 0 || block >= ns * cfg.n_ttt_layers || which < 0 || which > 2 || !dst) {
      err = "bad block/which/dst";
      return TTT_ERR_INVALID;
    }
    const int q = block / cfg.n_ttt_layers, i = block % cfg.n_ttt_layers;
    Layer& y = layers[cfg.n_layers - cfg.n_ttt_layers + i];
    if (which == 2) {
      CU_TRY(cudaMemcpyAsync(dst, y.wd32 + q * y.d_elems, sizeof(float) * (size_t)d * ff, cudaMemcpyDefault, st));
    } else {
      CU_TRY(cudaMemcpy2DAsync(dst, sizeof(float) * d, y.wgu32 + q * y.gu_elems + (which == 1 ? d : 0),
                               sizeof(float) * 2 * d, sizeof(float) * d, ff, cudaMemcpyDefault, st));
    }
    CU_TRY(cudaStreamSynchronize(st));
    return TTT_OK;
  }

  int reset(cudaStream_t st) override {
    const int L = cfg.n_layers, d = cfg.d_model, ff = cfg.d_ff;
    for (int l = 0; l < L; ++l) {
      Layer& y = layers[l];
      CU_TRY(cudaMemsetAsync(y.kring, 0, sizeof(T) * (size_t)ns * y.ring_elems, st));
      CU_TRY(cudaMemsetAsync(y.vring, 0, sizeof(T) * (size_t)ns * y.ring_elems, st));
      if (l >= L - cfg.n_ttt_layers) {
        for (int q = 0; q < ns; ++q) {
          CU_TRY(cudaMemcpyAsync(y.wgu32 + q * y.gu_elems, y.wgu32_init, sizeof(float) * 2 * ff * (size_t)d,
                                 cudaMemcpyDeviceToDevice, st));
          CU_TRY(cudaMemcpyAsync(y.wd32 + q * y.d_elems, y.wd32_init, sizeof(float) * (size_t)d * ff,
                                 cudaMemcpyDeviceToDevice, st));
        }
        if (kBF16) {
          const double nb = 2.0 * ff * d * ns;
          row(nb * 8, st, [&] { launch_split_bf16(y.wgu32, ns * y.gu_elems, (bf16*)y.wgu, (bf16*)y.wgu_lo, st); });
          row(nb * 4, st, [&] { launch_split_bf16(y.wd32, ns * y.d_elems, (bf16*)y.wd, (bf16*)y.wd_lo, st); });
        }
      }
    }
    CU_TRY(cudaGetLastError());
    CU_TRY(cudaStreamSynchronize(st));
    if (prof_on) prof_collect();
    pos = 0;
    used = false;
    dec_fill = 0;
    return TTT_OK;
  }
};

}  // namespace ttt

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
struct ttt_ctx {
  std::unique_ptr<ttt::EngineBase> eng;
};

static int validate(const ttt_config* c, std::string& msg) {
  if (c->precision != TTT_BF16 && c->precision != TTT_FP32_CHECK) {
    msg = "precision must be TTT_BF16 or TTT_FP32_CHECK";
    return TTT_ERR_INVALID;
  }
  if (c->n_layers < 1 || c->d_model < 2 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 2 ||
      c->d_ff < 2 || c->vocab < 2 || c->window < 1 || c->chunk < 1 || c->n_ttt_layers < 0 ||
      c->max_tokens < 1) {
    msg = "every size must be positive (n_ttt_layers >= 0)";
    return TTT_ERR_INVALID;
  }
  if (c->n_ttt_layers > c->n_layers) {
    msg = "n_ttt_layers > n_layers";
    return TTT_ERR_INVALID;
  }
  if (c->dual_mlp != 0 && c->dual_mlp != 1) {
    msg = "dual_mlp must be 0 or 1";
    return TTT_ERR_INVALID;
  }
  if (c->bulk_tokens < 0) {
    msg = "bulk_tokens must be >= 0 (0: automatic)";
    return TTT_ERR_INVALID;
  }
  if (c->fast_bf16_single != 0 && c->fast_bf16_single != 1) {
    msg = "fast_bf16_single must be 0 or 1";
    return TTT_ERR_INVALID;
  }
  if (c->n_seq < 0 || c->n_seq > 64) {
    msg = "n_seq must be in [0, 64] (0 or 1: one sequence)";
    return TTT_ERR_INVALID;
  }
  if (c->n_heads % c->n_kv_heads) {
    msg = "n_heads must be a multiple of n_kv_heads";
    return TTT_ERR_SHAPE;
  }
  if ((c->head_dim & 1) || (c->d_model & 1) || (c->d_ff & 1) || (c->vocab & 1) || c->head_dim > 256) {
    msg = "head_dim, d_model, d_ff and vocab must be even; head_dim <= 256";
    return TTT_ERR_SHAPE;
  }
  if (!std::isfinite(c->lr)) {
    msg = "lr is not finite";
    return TTT_ERR_NONFINITE;
  }
  if (!(c->rope_theta > 0.f) || !std::isfinite(c->rope_theta) || !(c->norm_eps >= 0.f) ||
      !std::isfinite(c->norm_eps)) {
    msg = "rope_theta must be positive and norm_eps non-negative (both finite)";
    return TTT_ERR_INVALID;
  }
  return TTT_OK;
}

extern "C" int ttt_create(const ttt_config* cfg, const ttt_weights* w, void* stream, ttt_ctx** out) {
  ttt::g_create_error.clear();
  if (!out) {
    ttt::g_create_error = "out is null";
    return TTT_ERR_INVALID;
  }
  *out = nullptr;
  if (!cfg || !w) {
    ttt::g_create_error = "cfg or weights is null";
    return TTT_ERR_INVALID;
  }
  std::string msg;
  int rc = validate(cfg, msg);
  if (rc) {
    ttt::g_create_error = msg;
    return rc;
  }
  std::unique_ptr<ttt::EngineBase> eng;
  try {
    if (cfg->precision == TTT_BF16) eng.reset(new ttt::Engine<ttt::bf16>());
    else eng.reset(new ttt::Engine<float>());
  } catch (...) {
    ttt::g_create_error = "host allocation failed";
    return TTT_ERR_OOM;
  }
  eng->cfg = *cfg;
  eng->ns = cfg->n_seq > 1 ? cfg->n_seq : 1;
  eng->prof_clear();
  const int need = cfg->window + cfg->chunk - 1;
  eng->R = ((need + 127) / 128) * 128;
  // super-chunk of the bulk static pass: a multiple of b, about 16K tokens
  // unless the configuration names another length, never more than the
  // longest sequence needs
  {
    const int64_t b = cfg->chunk;
    const int64_t asked = cfg->bulk_tokens > 0 ? cfg->bulk_tokens : 16384;
    const int64_t want = std::max<int64_t>(b, (asked / b) * b);
    const int64_t cap = ((cfg->max_tokens + b - 1) / b) * b;
    eng->S_bulk = (int)std::min(want, cap);
    const int64_t need_s = (int64_t)cfg->window + eng->S_bulk - 1;
    eng->R_s = (int)(((need_s + 127) / 128) * 128);
  }
  eng->qkv_cols = (cfg->n_heads + 2 * cfg->n_kv_heads) * cfg->head_dim;
  eng->Vs = 0;  // set in init(), once the SM count is known
  const bool bf = cfg->precision == TTT_BF16;
  const char* g = getenv("TTT_GEMM_IMPL");
  const char* a = getenv("TTT_ATTN_IMPL");
  eng->use_tc_gemm = bf && !(g && strcmp(g, "simt") == 0);
  // attention runs on the tensor-core kernels for every shape they support;
  // TTT_ATTN_IMPL=simt keeps it on the SIMT kernels (a GPU-side cross-check)
  eng->use_tc_attn = bf && !(a && strcmp(a, "simt") == 0);
  eng->use_tc_attn_bwd = eng->use_tc_attn;
  // decode steps: TTT_DECODE_LAUNCH=graph keeps the captured graphs without
  // programmatic dependent launch, =direct issues every kernel from the
  // host (the same kernels and results; for measuring the launch modes)
  // TTT_PREFILL_UPDATES=inline: the prefill's weight updates on the chunk
  // loop's stream (for comparison)
  const char* pu = getenv("TTT_PREFILL_UPDATES");
  eng->sgd_side_ok = !(pu && strcmp(pu, "inline") == 0);
  // TTT_PREFILL_LAUNCH=pdl: programmatic dependent launch in the prefill's
  // chunk loop (for comparison; the default launches plainly)
  const char* pl = getenv("TTT_PREFILL_LAUNCH");
  eng->pdl_prefill = pl && strcmp(pl, "pdl") == 0;
  const char* dl = getenv("TTT_DECODE_LAUNCH");
  eng->pdl_ok = !(dl && (strcmp(dl, "graph") == 0 || strcmp(dl, "direct") == 0));
  eng->dec_graph_off = dl && strcmp(dl, "direct") == 0;
  if (eng->use_tc_gemm) {
    int r = ttt::gemm_tc_init();
    if (r) {
      ttt::g_create_error = "tensor-core GEMM initialisation failed";
      return TTT_ERR_CUDA;
    }
  }
  cudaStream_t st = (cudaStream_t)stream;
  try {
    rc = eng->init(w, st);
  } catch (...) {
    rc = TTT_ERR_INTERNAL;
    eng->err = "exception during initialisation";
  }
  if (rc) {
    ttt::g_create_error = eng->err;
    cudaStreamSynchronize(st);
    return rc;
  }
  ttt_ctx* c = new (std::nothrow) ttt_ctx();
  if (!c) {
    ttt::g_create_error = "host allocation failed";
    return TTT_ERR_OOM;
  }
  c->eng = std::move(eng);
  *out = c;
  return TTT_OK;
}

#define CTX_GUARD(ctx)                 \
  if (!(ctx) || !(ctx)->eng) return TTT_ERR_INVALID;

extern "C" int ttt_prefill(ttt_ctx* ctx, const int32_t* tokens, int64_t T, float* chunk_losses,
                           void* stream) {
  CTX_GUARD(ctx);
  ctx->eng->err.clear();
  try {
    return ctx->eng->prefill(tokens, T, chunk_losses, (cudaStream_t)stream);
  } catch (...) {
    ctx->eng->err = "exception in ttt_prefill";
    return TTT_ERR_INTERNAL;
  }
}

extern "C" int ttt_prefill_batch(ttt_ctx* const* ctxs, int32_t n_ctx, const int32_t* const* tokens,
                                 const int64_t* T, float* const* chunk_losses, void* const* streams) {
  if (!ctxs || !tokens || !T || !chunk_losses || n_ctx < 1) return TTT_ERR_INVALID;
  for (int i = 0; i < n_ctx; ++i) {
    if (!ctxs[i] || !ctxs[i]->eng) return TTT_ERR_INVALID;
    for (int j = 0; j < i; ++j)
      if (ctxs[j] == ctxs[i]) return TTT_ERR_INVALID;  // one sequence per context
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TTT_ERR_CUDA;
  std::vector<int> rc(n_ctx, TTT_OK);
  auto run = [&](int i) {
    ttt::EngineBase* e = ctxs[i]->eng.get();
    e->err.clear();
    try {
      rc[i] = e->prefill(tokens[i], T[i], chunk_losses[i], streams ? (cudaStream_t)streams[i] : nullptr);
    } catch (...) {
      e->err = "exception in ttt_prefill_batch";
      rc[i] = TTT_ERR_INTERNAL;
    }
  };
  // one host thread per further sequence, so that every context issues its
  // work while the others run; the calling thread takes the first
  std::vector<std::thread> th;
  try {
    for (int i = 1; i < n_ctx; ++i)
      th.emplace_back([&, i] {
        if (cudaSetDevice(dev) != cudaSuccess) {
          rc[i] = TTT_ERR_CUDA;
          return;
        }
        run(i);
      });
  } catch (...) {
    // no more threads: the remaining sequences run on this thread
    for (size_t i = th.size() + 1; i < (size_t)n_ctx; ++i) run((int)i);
  }
  run(0);
  for (std::thread& t : th) t.join();
  for (int i = 0; i < n_ctx; ++i)
    if (rc[i] != TTT_OK) return rc[i];
  return TTT_OK;
}

extern "C" int ttt_decode(ttt_ctx* ctx, const int32_t* tokens, int64_t n_given, int64_t n_steps, int32_t* tokens_out,
                          float* chunk_losses, void* stream) {
  CTX_GUARD(ctx);
  ctx->eng->err.clear();
  try {
    return ctx->eng->decode(tokens, n_given, n_steps, tokens_out, chunk_losses, (cudaStream_t)stream);
  } catch (...) {
    ctx->eng->err = "exception in ttt_decode";
    return TTT_ERR_INTERNAL;
  }
}

extern "C" int ttt_logits(ttt_ctx* ctx, const int32_t* cont, int32_t n, float* logits, void* stream) {
  CTX_GUARD(ctx);
  ctx->eng->err.clear();
  try {
    return ctx->eng->logits(cont, n, logits, (cudaStream_t)stream);
  } catch (...) {
    ctx->eng->err = "exception in ttt_logits";
    return TTT_ERR_INTERNAL;
  }
}

extern "C" int ttt_get_fast_weights(ttt_ctx* ctx, int32_t block, int32_t which, float* dst, void* stream) {
  CTX_GUARD(ctx);
  ctx->eng->err.clear();
  return ctx->eng->get_fast(block, which, dst, (cudaStream_t)stream);
}

extern "C" int ttt_profile(ttt_ctx* ctx, int32_t on) {
  CTX_GUARD(ctx);
  ctx->eng->err.clear();
  ctx->eng->prof_clear();
  ctx->eng->prof_on = on != 0;
  return TTT_OK;
}

extern "C" int ttt_profile_read(ttt_ctx* ctx, ttt_kernel_stat* out, int32_t cap, int32_t* n_out) {
  CTX_GUARD(ctx);
  if (!n_out || (cap > 0 && !out) || cap < 0) {
    ctx->eng->err = "bad output arguments";
    return TTT_ERR_INVALID;
  }
  const int n = std::min<int>(cap, ttt::EngineBase::P_N);
  for (int i = 0; i < n; ++i) out[i] = ctx->eng->prof_stat[i];
  *n_out = ttt::EngineBase::P_N;
  return TTT_OK;
}

extern "C" int ttt_reset(ttt_ctx* ctx) {
  CTX_GUARD(ctx);
  ctx->eng->err.clear();
  return ctx->eng->reset((cudaStream_t)0);
}

extern "C" void ttt_destroy(ttt_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  delete ctx;
}

extern "C" const char* ttt_last_error(const ttt_ctx* ctx) {
  if (!ctx || !ctx->eng) return ttt::g_create_error.c_str();
  return ctx->eng->err.c_str();
}

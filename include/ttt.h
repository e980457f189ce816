/*
 * ttt.h — C ABI of the TTT-E2E test-time inner loop on one B300 (sm_103a).
 *
 * The method ("End-to-End Test-Time Training for Long Context"): a
 * decoder-only Transformer with sliding-window attention reads a long
 * context in mini-batches ("chunks") of b tokens; on each chunk it runs the
 * forward pass, takes the next-token cross-entropy loss, back-propagates
 * into the MLPs of the last quarter of the blocks only, and takes one plain
 * gradient step on them, so the next chunk is read by the updated weights
 * (summary page, Method; podcast page, 6:36 and 7:08; NVIDIA blog, "Our
 * method: compressing context into weights").  Keys and values of earlier
 * chunks stay cached and are not differentiated.  The meta-learned outer
 * loop is not part of this library.
 *
 * Conventions for every call:
 *   - Return value: TTT_OK (0) or a negative TTT_ERR_* code.  Nothing aborts
 *     and no C++ exception crosses this boundary.  ttt_last_error() returns
 *     a NUL-terminated description of the last failure on that context
 *     (owned by the context, valid until the next call on it).
 *   - Matrices use the [out, in] row-major layout of a linear layer
 *     (y = x W^T): wq [H*hd, d], wk/wv [Hkv*hd, d], wo [d, H*hd],
 *     w_gate/w_up [d_ff, d], w_down [d, d_ff], tok_embed/lm_head [vocab, d].
 *     Embeddings are untied.  Norm gains are [d].
 *   - Pointers may be host memory or device memory of the current device;
 *     the library tells them apart with cudaPointerGetAttributes and copies
 *     host data itself.  The library never keeps a caller pointer after a
 *     call returns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  The device
 *     work of a call starts after the work already queued on `stream` and
 *     finishes before anything queued on it later (ttt_prefill forks two
 *     internal streams from `stream` and joins them back into it).
 */
#ifndef TTT_H_
#define TTT_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  TTT_OK = 0,
  TTT_ERR_INVALID = -1,   /* null pointer, bad enum, bad config value          */
  TTT_ERR_SHAPE = -2,     /* sizes the kernels do not support                  */
  TTT_ERR_OOM = -3,       /* device allocation failed                          */
  TTT_ERR_CUDA = -4,      /* a CUDA runtime/driver call failed                 */
  TTT_ERR_NONFINITE = -5, /* a chunk loss was NaN/Inf (chunk index in message) */
  TTT_ERR_STATE = -6,     /* call not allowed in the context's current state   */
  TTT_ERR_INTERNAL = -7   /* a device-side check or bounded wait failed        */
};

enum {
  TTT_BF16 = 0,       /* bf16 storage, fp32 accumulation, tensor cores          */
  TTT_FP32_CHECK = 1  /* fp32 everywhere, SIMT kernels (correctness mode)        */
};

/* Model and loop configuration.
 *   n_layers L, d_model d, n_heads H, n_kv_heads Hkv (H % Hkv == 0),
 *   head_dim hd (even), d_ff, vocab V, window W (query t sees keys j with
 *   t-W < j <= t), chunk b (test-time mini-batch), n_ttt_layers (the MLPs
 *   of blocks [L-n_ttt_layers, L) are the fast weights; 0: no test-time
 *   training, ttt_prefill only scores the chunks of a frozen model, e.g. a
 *   full-attention Transformer with window >= T), precision
 *   (TTT_BF16 | TTT_FP32_CHECK), lr (SGD step), rope_theta, norm_eps,
 *   max_tokens (longest sequence ttt_prefill will be given; sizes the
 *   device staging of host token arrays), dual_mlp (0 or 1: each fast block
 *   carries a second, static SwiGLU MLP after its fast one, with its own
 *   pre-norm and residual: y = h2 + MLP2(n(h2)), h2 = h + MLP_fast(n(h));
 *   podcast page, 7:08), bulk_tokens (>= 0: tokens per super-chunk of the
 *   frozen blocks' bulk pass in ttt_prefill, rounded down to a multiple of
 *   chunk and at least one chunk; 0 picks about 16K tokens.  It changes how
 *   the work is batched, never what is computed), fast_bf16_single (0 or
 *   1, TTT_BF16 only: how the forward reads a fast weight w, whose value is
 *   an fp32 master updated in place.  0: as the bf16 pair hi = rn(w),
 *   lo = rn(w - hi), read as hi + lo, which carries about 16 significant
 *   bits, so every update reaches the forward.  1: one bf16 copy rn(w),
 *   re-rounded after every update, at half the tensor work of the fast
 *   MLPs' forward products; an update smaller than half a bf16 step of w
 *   leaves that copy unchanged, so at small lr the forward does not see
 *   the test-time training until updates accumulate past that step),
 *   n_seq (0 or 1: the context holds one sequence; 2 .. 64: it holds n_seq
 *   independent sequences, each with its own fast weights and key/value
 *   cache, sharing the static weights.  ttt_prefill then reads all of them
 *   at once: the products with static weights take every sequence's rows in
 *   one launch, and the fast MLPs' products run as grouped GEMMs, one
 *   weight set per sequence.  ttt_decode and ttt_logits need n_seq <= 1.)  */
typedef struct ttt_config {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ff, vocab;
  int32_t window, chunk, n_ttt_layers, precision;
  float lr, rope_theta, norm_eps;
  int64_t max_tokens;
  int32_t dual_mlp;
  int32_t bulk_tokens;
  int32_t fast_bf16_single;
  int32_t n_seq;
} ttt_config;

/* Initial weights, fp32 values (host or device).  Per-layer fields are
 * arrays of n_layers pointers (the arrays themselves live in host memory). */
typedef struct ttt_weights {
  const float* tok_embed;  /* [V, d] */
  const float* final_norm; /* [d]    */
  const float* lm_head;    /* [V, d] */
  const float* const* attn_norm; /* [d]        */
  const float* const* wq;        /* [H*hd, d]  */
  const float* const* wk;        /* [Hkv*hd, d]*/
  const float* const* wv;        /* [Hkv*hd, d]*/
  const float* const* wo;        /* [d, H*hd]  */
  const float* const* mlp_norm;  /* [d]        */
  const float* const* w_gate;    /* [d_ff, d]  */
  const float* const* w_up;      /* [d_ff, d]  */
  const float* const* w_down;    /* [d, d_ff]  */
  /* dual_mlp only: the static second MLP of each fast block (entries of
   * other blocks are ignored and may be NULL; the arrays may be NULL when
   * dual_mlp is 0) */
  const float* const* mlp2_norm; /* [d]        */
  const float* const* w_gate2;   /* [d_ff, d]  */
  const float* const* w_up2;     /* [d_ff, d]  */
  const float* const* w_down2;   /* [d, d_ff]  */
} ttt_weights;

typedef struct ttt_ctx ttt_ctx;

/* Validate `cfg`, allocate all device state (weights in the working
 * precision, fp32 masters of the fast weights, the key/value ring of
 * W+b-1 positions per layer, per-chunk activations), copy and convert the
 * weights (bf16 by round-to-nearest-even in TTT_BF16 mode), and return the
 * context in *out.  The context is fresh: position 0, initial fast weights.
 * Errors: INVALID (null args, bad enum), SHAPE (unsupported sizes), OOM,
 * CUDA.  On error *out is NULL and nothing is leaked.
 * Environment, read here, for cross-checks and measurement only (results
 * are those of the method in every setting): TTT_GEMM_IMPL=simt and
 * TTT_ATTN_IMPL=simt keep the products / the attention on SIMT kernels;
 * TTT_PREFILL_LAUNCH=pdl launches ttt_prefill's chunk loop with
 * programmatic dependent launch; TTT_PREFILL_UPDATES=inline keeps its
 * weight updates on the chunk loop's stream; TTT_DECODE_LAUNCH as under
 * ttt_decode. */
int ttt_create(const ttt_config* cfg, const ttt_weights* w, void* stream, ttt_ctx** out);

/* The test-time inner loop over tokens[0..T) (int32 ids in [0, V)).
 * Chunk c covers positions [c*b, min(T,(c+1)*b)); the target of position t
 * is tokens[t+1] when t+1 < T.  For each chunk: forward with the current
 * weights, loss = mean over the chunk's targets of (logsumexp(z_t) -
 * z_t[target]), backward into w_gate/w_up/w_down of the fast blocks with
 * earlier keys/values held constant, then W <- W - lr * dW (fp32 master;
 * its bf16 pair, or the single bf16 copy, is re-rounded).  A chunk without targets reports loss 0 and
 * makes no update.
 *   chunk_losses: [ceil(T/b)] fp32, host or device.
 * With n_seq > 1 the context reads n_seq sequences of the same length T:
 * tokens is [n_seq][T] and chunk_losses [n_seq][ceil(T/b)], row q for
 * sequence q; each sequence is trained on exactly as if it were alone.
 * Requires a fresh (or reset) context and 1 <= T <= cfg.max_tokens;
 * otherwise STATE / SHAPE.  Returns after the work has completed on
 * `stream`.  A NaN/Inf chunk loss returns NONFINITE with the first such
 * chunk index in ttt_last_error(); the context is then left as is.  After
 * success the context holds the final fast weights and the ring at
 * position T.  Internally the call forks streams from `stream`: one runs
 * the frozen blocks' bulk pass a super-chunk ahead, one the chunk loop, and
 * one the chunk loop's weight updates beside the backward of the layers
 * below; all join back into `stream` before the call returns. */
int ttt_prefill(ttt_ctx* ctx, const int32_t* tokens, int64_t T, float* chunk_losses,
                void* stream);

/* Several sequences in one call: ttt_prefill on each of n_ctx distinct
 * contexts, every context with its own fast weights and ring (scope row
 * "batched sequences").  The contexts run concurrently: the calling thread
 * drives the first and one host thread each of the others, each on
 * streams[i] (streams may be NULL: every context then uses the legacy
 * default stream, which orders them one after another).  Arguments are
 * arrays of n_ctx entries with the meaning of ttt_prefill's.  Each
 * context's result and ttt_last_error are as if ttt_prefill had been called
 * on it alone; the return value is the first non-OK code in index order.
 * Two entries naming the same context are INVALID. */
int ttt_prefill_batch(ttt_ctx* const* ctxs, int32_t n_ctx, const int32_t* const* tokens, const int64_t* T,
                      float* const* chunk_losses, void* const* streams);

/* Decode-time test-time training: generation one token per step, with the
 * same test-time step as ttt_prefill's chunk loop once every b positions
 * (the latency per token stays constant in the context length: summary
 * page, Key claims; podcast 5:55).  Step i (position pos + i, where pos is
 * the context's position) runs the token through every block with the
 * current weights, writing its keys and values to the ring, and forms the
 * next input: tokens[i + 1] while given, else the greedy prediction (the
 * index of the largest logit, the smallest index on ties).  When position
 * p completes a chunk [p + 1 - b, p + 1), the chunk is trained on as in
 * ttt_prefill: its fast blocks are recomputed over the chunk, the loss is
 * the mean over its b positions of (logsumexp(z_t) - z_t[token t+1]), where
 * the target of the chunk's last position is that step's next input, and
 * one SGD step updates the fast weights.  Teacher-forced decode of
 * tokens[0..n_steps] therefore trains exactly like ttt_prefill over those
 * n_steps + 1 tokens, chunk for chunk.
 *   tokens:       [n_given] int32 (host or device), 1 <= n_given <= n_steps + 1;
 *                 tokens[0] is the input at position pos.
 *   tokens_out:   [n_steps + 1] int32 (host or device): the input token of
 *                 every step, then the next input after the last step.
 *   chunk_losses: losses of the chunks completed by this call, in order
 *                 (at most (n_steps + b - 1) / b + 1 of them).
 * A chunk left incomplete carries over to the next ttt_decode call.  The
 * first decode on a context must start at a chunk boundary (pos a multiple
 * of b: a fresh or reset context, or after ttt_prefill of a multiple of b
 * tokens), else STATE; pos + n_steps <= max_tokens, else SHAPE.  A non-finite
 * chunk loss returns NONFINITE with its index within this call.  Returns
 * after the work has completed on `stream`; pos advances by n_steps.
 * The steps' position and tokens live in device memory, so the first step
 * of each kind (next input given, or greedy) is issued kernel by kernel and
 * recorded into a CUDA graph on a stream the context owns; later steps, in
 * this and later calls, replay that graph on `stream`.  The chunk's
 * test-time step is always issued kernel by kernel.  Do not call ttt_decode
 * while a stream capture is active on the calling thread.  Environment
 * TTT_DECODE_LAUNCH (read at ttt_create): "graph" replays graphs without
 * programmatic dependent launch between their kernels, "direct" issues every
 * step kernel by kernel; results are the same in every mode. */
int ttt_decode(ttt_ctx* ctx, const int32_t* tokens, int64_t n_given, int64_t n_steps, int32_t* tokens_out,
               float* chunk_losses, void* stream);

/* Forward only: logits of a continuation cont[0..n) placed at positions
 * P..P+n-1, where P is the number of positions consumed so far, using the
 * current fast weights and the cached keys/values.  1 <= n <= cfg.chunk.
 *   logits: [n, V] fp32 row-major, host or device.
 * The context's weights, position and visible cache are unchanged (ring
 * slots beyond position P may be overwritten; they are outside every later
 * query's window). */
int ttt_logits(ttt_ctx* ctx, const int32_t* cont, int32_t n, float* logits, void* stream);

/* Copy the current fp32 value of one fast weight:
 *   block in [0, n_ttt_layers) (0 = layer L-n_ttt_layers); with n_seq > 1,
 *   block in [0, n_seq * n_ttt_layers): block q * n_ttt_layers + i is
 *   block i of sequence q,
 *   which 0 = w_gate [d_ff, d], 1 = w_up [d_ff, d], 2 = w_down [d, d_ff],
 *   dst host or device, in the [out, in] layout above. */
int ttt_get_fast_weights(ttt_ctx* ctx, int32_t block, int32_t which, float* dst, void* stream);

/* Restore the initial fast weights, empty the ring, set position 0.
 * Synchronous. */
int ttt_reset(ttt_ctx* ctx);

/* Per-launch timing of the kernels of the loop, by kernel class.  With
 * profiling on, every kernel launch of ttt_prefill / ttt_logits is
 * bracketed by two CUDA events on the call's stream; the pairs are resolved
 * when the call synchronises and summed per class:
 *   "gemm_fwd"      projections of the chunk loop's forward (q/k/v + RoPE + ring write,
 *                   output + residual, gate/up + SwiGLU, down + residual)
 *   "gemm_lm_head"  the streamed lm_head products of the cross-entropy
 *   "gemm_bwd_dx"   input-gradient products of the backward
 *   "gemm_dw_sgd"   weight-gradient products with the fused SGD step
 *   "attn_fwd"      sliding-window attention forward
 *   "attn_bwd"      chunk-local attention backward
 *   "rowwise"       embedding, norms, softmax statistics, RoPE backward
 *   "gemm_fwd_bulk" forward projections of the frozen blocks, run over
 *                   spans longer than a chunk (ttt_prefill)
 *   "attn_fwd_bulk" their sliding-window attention forward
 * `flops` counts 2 per multiply-add of the operation as defined (attention:
 * unmasked query/key pairs only; no recomputation, no padding), `bytes`
 * the operands read once and results written once.  While profiling is
 * on, ttt_prefill runs its bulk pass and chunk loop on the call's stream
 * alone (no overlap), so that each event pair times one kernel by itself.
 * The events add a few microseconds per launch on the host; device time is
 * unaffected apart from the gaps they leave between kernels. */
typedef struct ttt_kernel_stat {
  char name[24];
  int64_t launches;
  double ms;    /* summed event-to-event device time */
  double flops; /* algorithmic FLOPs of those launches */
  double bytes; /* algorithmic bytes of those launches */
} ttt_kernel_stat;

/* Switch per-launch timing on (on != 0) or off; clears the counters. */
int ttt_profile(ttt_ctx* ctx, int32_t on);

/* Copy up to `cap` class records (in the order listed above) into out and
 * set *n_out to the number of classes.  Counters accumulate over calls
 * until ttt_profile() is called again. */
int ttt_profile_read(ttt_ctx* ctx, ttt_kernel_stat* out, int32_t cap, int32_t* n_out);

/* Free everything owned by ctx (NULL is ignored). */
void ttt_destroy(ttt_ctx* ctx);

/* Description of the last error on ctx ("" if none).  With ctx == NULL:
 * the last error of a failed ttt_create on this thread. */
const char* ttt_last_error(const ttt_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* TTT_H_ */

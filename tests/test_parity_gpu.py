"""Parity of the CUDA inner loop (through the C ABI) with the CPU oracle.

Tolerances: fp32 check mode <= 1e-4, bf16 mode <= 2e-2, on the per-chunk
loss (relative) and on the final fast weights (relative Frobenius norm);
chunk count and target bookkeeping are exact.

Because W_final is dominated by W_0 at these step sizes, and every chunk
loss of a randomly initialised model sits near ln V, two further checks make
a wrong hidden state fail in bf16 as well as in fp32:
  * the update itself, dW = W_final - W_0, to the same relative Frobenius
    tolerance;
  * the losses' departure from the uniform predictor: the vector
    (loss_c - ln V) over the chunks, compared in relative 2-norm.
"""
import math

import numpy as np
import pytest

from long_context_lm_ttt_b300 import inputs
from oracle import ttt_ref as O

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_lm_ttt_b300 import ttt as T
    T.load()
    return T


def run_gpu(s, w, tok, precision, lr=None, bulk_tokens=0, fast_bf16_single=False, profile=False):
    T = _lib()
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    m = T.TTT(s, w, prec, max_tokens=len(tok), lr=lr, bulk_tokens=bulk_tokens, fast_bf16_single=fast_bf16_single)
    try:
        if profile:
            m.profile(True)
        losses = m.prefill(np.ascontiguousarray(tok, np.int32)).astype(np.float64)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    return losses, fast


def run_oracle(s, w, tok, lr=None, n_chunks=None, return_state=False):
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    return O.prefill(cfg, w, tok, lr=lr, n_chunks=n_chunks, return_state=return_state)


def rel_fro(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


def check_against(s, w, g_loss, g_fast, r, precision, check_delta=None):
    """Losses, fast weights, their updates and the losses' departure from
    ln V against the oracle's run r."""
    tol = TOL[precision]
    n_tok = s.seq_len
    assert len(g_loss) == len(r["losses"])
    rel = np.abs(g_loss - r["losses"]) / np.maximum(np.abs(r["losses"]), 1e-12)
    assert rel.max() <= tol, (rel.max(), g_loss[:4], r["losses"][:4])
    # departure from the uniform predictor; chunks without targets report 0
    has_tgt = np.array([min(e, n_tok - 1) > st for st, e in O.chunk_bounds(n_tok, s.chunk)])
    dev_ref = r["losses"][has_tgt] - math.log(s.vocab)
    dev_err = float(np.linalg.norm(g_loss[has_tgt] - r["losses"][has_tgt]) / max(np.linalg.norm(dev_ref), 1e-30))
    assert dev_err <= tol, ("loss - ln V", dev_err)
    L, Lt = s.n_layers, s.n_ttt_layers
    worst_delta = 0.0
    for i in range(Lt):
        for k in O.FAST:
            assert rel_fro(g_fast[i][k], r["fast"][i][k]) <= tol
            w0 = np.asarray(w["layers"][L - Lt + i][k], np.float64)
            if np.any(r["fast"][i][k] != w0):
                worst_delta = max(worst_delta, rel_fro(g_fast[i][k] - w0, r["fast"][i][k] - w0))
    if check_delta is None:
        check_delta = tol
    assert worst_delta <= check_delta, ("dW", worst_delta)
    return rel.max(), worst_delta, dev_err


def compare(s, w, tok, precision, lr=None, check_delta=None, bulk_tokens=0, fast_bf16_single=False):
    assert len(tok) == s.seq_len
    g_loss, g_fast = run_gpu(s, w, tok, precision, lr, bulk_tokens=bulk_tokens, fast_bf16_single=fast_bf16_single)
    r = run_oracle(s, w, tok, lr)
    assert len(g_loss) == -(-len(tok) // s.chunk)
    return check_against(s, w, g_loss, g_fast, r, precision, check_delta)


# ---------------------------------------------------------------------------
# fp32 check mode: tight parity on the tiny shapes and their edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "tiny-ttt2", "tiny-gqa"])
def test_fp32_parity(name):
    s = inputs.shape(name)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "fp32", check_delta=1e-4)


@pytest.mark.parametrize("T_len", [1, 2, 31, 33, 100, 257])
def test_fp32_ragged_lengths(T_len):
    """T not a multiple of b; a last chunk with a single position has no target."""
    s = inputs.shape("tiny-ttt2", seq_len=T_len)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s, T_len), "fp32")


# ---------------------------------------------------------------------------
# several super-chunks of the frozen blocks' bulk pass: the two-stream
# hand-off (bulk pass of super-chunk k+1 overlapping the chunk loop of k),
# the double-buffered hand-off buffers and the static blocks' ring wrapping
# across super-chunks, at sizes the oracle runs in seconds
# ---------------------------------------------------------------------------
SUPER = [
    # name, overrides, bulk tokens: 4 super-chunks of 2 chunks each
    ("tiny-ttt2", dict(n_layers=3), 64),
    ("tiny-gqa", dict(), 64),
]


@pytest.mark.parametrize("name,kw,bulk", SUPER)
def test_fp32_super_chunks(name, kw, bulk):
    s = inputs.shape(name, **kw)
    assert -(-s.seq_len // bulk) >= 3
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "fp32", check_delta=1e-4, bulk_tokens=bulk)


@pytest.mark.parametrize("name,kw,bulk", SUPER)
def test_bf16_super_chunks(name, kw, bulk):
    s = inputs.shape(name, bf16=True, **kw)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "bf16", bulk_tokens=bulk)


# tensor-core attention and GEMM shapes (head dim 64, chunks of 128, a
# ragged last chunk) over 3 super-chunks of 2 chunks, 2 static blocks
TC_SUPER = dict(n_layers=4, n_heads=4, n_kv_heads=2, head_dim=64, d_model=256, d_ff=512, chunk=128, window=200,
                seq_len=700)


def test_bf16_super_chunks_tensor_cores():
    s = inputs.shape("tiny-gqa", bf16=True, **TC_SUPER)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s, s.seq_len), "bf16", bulk_tokens=256)


def test_super_chunks_overlap_is_bitwise_serial():
    """The two-stream prefill (bulk pass one super-chunk ahead) gives bitwise
    the result of the same work on one stream (profiling on), so the event
    hand-offs order every read after its write."""
    s = inputs.shape("tiny-gqa", bf16=True, **TC_SUPER)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s, s.seq_len)
    a, fa = run_gpu(s, w, tok, "bf16", bulk_tokens=256)
    b, fb = run_gpu(s, w, tok, "bf16", bulk_tokens=256, profile=True)
    c, fc = run_gpu(s, w, tok, "bf16", bulk_tokens=0)
    assert np.array_equal(a, b) and np.array_equal(a, c)
    for x, y, z in zip(fa, fb, fc):
        for k in O.FAST:
            assert np.array_equal(x[k], y[k]) and np.array_equal(x[k], z[k])


def test_fp32_window_smaller_than_chunk():
    s = inputs.shape("tiny-gqa", window=13, chunk=32)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "fp32")


def test_fp32_window_covers_everything():
    s = inputs.shape("tiny-ttt2", window=4096)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "fp32")


def test_fp32_head_dim_64_gqa_group_3():
    s = inputs.shape("tiny-gqa", n_heads=6, n_kv_heads=2, head_dim=64, d_model=192, seq_len=160)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s, 160), "fp32")


def test_fp32_lr0_is_plain_swa_transformer():
    s = inputs.shape("tiny-ttt2")
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s)
    g, fast = run_gpu(s, w, tok, "fp32", lr=0.0)
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    full = O.full_forward_losses(cfg, w, tok)
    b, T = s.chunk, len(tok)
    ref = np.array([full[c * b:min(T - 1, (c + 1) * b)].mean() for c in range(-(-T // b))])
    np.testing.assert_allclose(g, ref, rtol=1e-4)
    L, Lt = s.n_layers, s.n_ttt_layers
    for i in range(Lt):
        for k in O.FAST:
            assert np.array_equal(fast[i][k], w["layers"][L - Lt + i][k])


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_causality_and_determinism(precision):
    """Bit-exact indexing: chunks whose last target precedes p are bitwise
    unchanged when token p changes; two identical runs are bitwise equal."""
    s = inputs.shape("tiny-ttt2")
    w = inputs.make_weights(s, bf16=precision == "bf16")
    tok = inputs.make_tokens(s)
    p = 150
    tok2 = tok.copy()
    tok2[p] = (tok2[p] + 7) % s.vocab
    a, _ = run_gpu(s, w, tok, precision)
    a2, _ = run_gpu(s, w, tok, precision)
    b_, _ = run_gpu(s, w, tok2, precision)
    assert np.array_equal(a, a2)
    for c, (s0, e0) in enumerate(O.chunk_bounds(len(tok), s.chunk)):
        if e0 <= p:
            assert a[c] == b_[c]


# ---------------------------------------------------------------------------
# bf16 mode
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "tiny-ttt2", "tiny-gqa"])
def test_bf16_parity_tiny(name):
    s = inputs.shape(name, bf16=True)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "bf16")


def test_bf16_parity_125m_shape_4_layers():
    """125M tile shapes (d=768, 12x64 heads, ff 2048, V=32000, b=512, W=2048)
    with 4 blocks, 2 of them fast, over 6 chunks (window wraps the ring)."""
    s = inputs.shape("125m", n_layers=4, n_ttt_layers=2, seq_len=3000)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s, 3000)
    compare(s, w, tok, "bf16")


def test_bf16_parity_760m_shape_2_layers():
    """760M head layout: hd=96, 16 q heads over 4 KV heads."""
    s = inputs.shape("760m", n_layers=2, n_ttt_layers=2, seq_len=2500, window=1024, chunk=512)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s, 2500)
    compare(s, w, tok, "bf16")


def test_bf16_parity_tc_attention_small():
    """Head dim 64 and chunks of 128 put the attention forward and backward
    on the tensor-core kernels at a size the oracle runs in seconds; a
    ragged last chunk and a window shorter than the sequence."""
    s = inputs.shape("tiny-gqa", n_heads=4, n_kv_heads=2, head_dim=64, d_model=256, d_ff=512, chunk=128,
                     window=200, seq_len=700, bf16=True)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s, 700), "bf16")


@pytest.mark.parametrize("name,kw", [
    ("tiny-ttt2", dict()),
    ("tiny-gqa", dict(n_heads=4, n_kv_heads=2, head_dim=64, d_model=256, d_ff=512, chunk=128, window=200,
                      seq_len=700)),
])
def test_bf16_fast_weights_as_one_copy(name, kw):
    """The optional forward read of the fast weights as one bf16 copy
    (fast_bf16_single = 1) against the oracle, updates included, at the
    tiny shapes' step size (lr 1e-2), where a chunk's update is not far
    below half a bf16 step of the weights.  At the 125M-3B step sizes it is
    (lr 5e-4 to 1e-3): there the copy keeps its initial value for many
    chunks and the option is not held to the oracle."""
    s = inputs.shape(name, bf16=True, **kw)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s, s.seq_len), "bf16", fast_bf16_single=True)


def test_bf16_3b_shapes_four_blocks():
    """The 3B tile shapes end to end: d 3072, 24 query / 8 KV heads x 128,
    d_ff 8192, V 128256 (the streamed cross-entropy's vocabulary slabs),
    chunks of 1024 with the CTA-pair, split-K and wide-tile GEMM plans the
    3B model runs, over two blocks of each kind.  The window is shortened to
    1024 so the fast blocks' ring wraps within 4 chunks, and the frozen
    blocks' bulk pass runs as 2 super-chunks."""
    s = inputs.shape("3b-4layer", window=1024, seq_len=4096)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s, s.seq_len)
    compare(s, w, tok, "bf16", bulk_tokens=2048)


# ---------------------------------------------------------------------------
# ttt_logits: predictions after reading a context
# ---------------------------------------------------------------------------
LOGITS_CASES = [
    ("fp32", "tiny-gqa", dict(seq_len=96), 20),
    ("bf16", "tiny-gqa", dict(seq_len=96), 20),
    ("bf16", "tiny-gqa", dict(n_heads=4, n_kv_heads=2, head_dim=64, d_model=256, d_ff=512, chunk=128,
                              window=200, seq_len=384), 128),
]


@pytest.mark.parametrize("precision,name,kw,n", LOGITS_CASES)
def test_logits_after_prefill(precision, name, kw, n):
    """ttt_logits after a prefill of several chunks against the oracle's
    forward with the trained weights and the cache (logits_after), element
    by element relative to each row's largest logit.  The call changes
    nothing: a second call gives bitwise the same logits, the fast weights
    are unchanged, and a decode that follows matches one without it."""
    T = _lib()
    s = inputs.shape(name, bf16=precision == "bf16", **kw)
    w = inputs.make_weights(s)
    full = inputs.make_tokens(s.replace(seq_len=s.seq_len + n + 1), s.seq_len + n + 1)
    tok, cont = full[:s.seq_len], full[s.seq_len:s.seq_len + n]
    r = run_oracle(s, w, tok, return_state=True)
    ref = O.logits_after(r["state"], cont)
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    outs = []
    for with_logits in (True, False):
        m = T.TTT(s, w, prec, max_tokens=len(full))
        try:
            m.prefill(np.ascontiguousarray(tok, np.int32))
            if with_logits:
                z = m.logits(np.ascontiguousarray(cont, np.int32)).astype(np.float64)
                z2 = m.logits(np.ascontiguousarray(cont, np.int32)).astype(np.float64)
                fast_before = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
            toks_out, dl = m.decode(np.ascontiguousarray(full[s.seq_len:], np.int32), n)
            outs.append((toks_out.copy(), dl.copy()))
        finally:
            m.close()
    assert z.shape == ref.shape == (n, s.vocab)
    err = np.abs(z - ref).max(axis=1) / np.abs(ref).max(axis=1)
    assert err.max() <= TOL[precision], err.max()
    assert np.array_equal(z, z2)
    L, Lt = s.n_layers, s.n_ttt_layers
    for i in range(Lt):
        for k in O.FAST:
            w0 = np.asarray(w["layers"][L - Lt + i][k], np.float64)
            assert rel_fro(fast_before[i][k] - w0, r["fast"][i][k] - w0) <= TOL[precision]
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])



@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_full_attention_without_test_time_training(precision):
    """n_ttt_layers = 0 with a window covering the whole sequence: a plain
    full-attention Transformer scoring its chunks (the baseline the pages
    compare against), against the un-chunked oracle forward."""
    s = inputs.shape("tiny-gqa", n_ttt_layers=0, window=4096, seq_len=200, bf16=precision == "bf16")
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s)
    g, fast = run_gpu(s, w, tok, precision)
    assert fast == []
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    full = O.full_forward_losses(cfg, w, tok)
    b, T = s.chunk, len(tok)
    ref = np.array([full[c * b:min(T - 1, (c + 1) * b)].mean() for c in range(-(-T // b))])
    np.testing.assert_allclose(g, ref, rtol=TOL[precision])


# ---------------------------------------------------------------------------
# fast blocks with a static second MLP (dual_mlp)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny-ttt2", "tiny-gqa"])
def test_fp32_parity_dual_mlp(name):
    s = inputs.shape(name, dual_mlp=True)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "fp32", check_delta=1e-4)


@pytest.mark.parametrize("name", ["tiny-ttt2", "tiny-gqa"])
def test_bf16_parity_dual_mlp(name):
    s = inputs.shape(name, dual_mlp=True, bf16=True)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s), "bf16")


def test_bf16_parity_dual_mlp_tc_attention():
    """Tensor-core attention shapes (head dim 64, chunks of 128) with the
    static second MLP in both fast blocks."""
    s = inputs.shape("tiny-gqa", n_heads=4, n_kv_heads=2, head_dim=64, d_model=256, d_ff=512, chunk=128,
                     window=200, seq_len=520, bf16=True, dual_mlp=True)
    compare(s, inputs.make_weights(s), inputs.make_tokens(s, 520), "bf16")


def test_fp32_dual_mlp_lr0_is_plain_forward():
    """lr = 0: the dual-MLP model scores its chunks like one un-chunked
    forward of the same model."""
    s = inputs.shape("tiny-ttt2", dual_mlp=True)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s)
    g, _ = run_gpu(s, w, tok, "fp32", lr=0.0)
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    full = O.full_forward_losses(cfg, w, tok)
    b, T = s.chunk, len(tok)
    ref = np.array([full[c * b:min(T - 1, (c + 1) * b)].mean() for c in range(-(-T // b))])
    np.testing.assert_allclose(g, ref, rtol=1e-4)

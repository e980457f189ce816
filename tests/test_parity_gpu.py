"""Parity of the CUDA inner loop (through the C ABI) with the CPU oracle.

Tolerances: fp32 check mode <= 1e-4, bf16 mode <= 2e-2, both on the
per-chunk loss (relative) and on the final fast weights (relative Frobenius
norm); chunk count and target bookkeeping are exact.
"""
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


def run_gpu(s, w, tok, precision, lr=None, host=True):
    T = _lib()
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    m = T.TTT(s, w, prec, max_tokens=len(tok), lr=lr)
    try:
        losses = m.prefill(np.ascontiguousarray(tok, np.int32)).astype(np.float64)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    return losses, fast


def run_oracle(s, w, tok, lr=None, n_chunks=None):
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    return O.prefill(cfg, w, tok, lr=lr, n_chunks=n_chunks)


def rel_fro(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


def compare(s, w, tok, precision, lr=None, check_delta=None):
    g_loss, g_fast = run_gpu(s, w, tok, precision, lr)
    r = run_oracle(s, w, tok, lr)
    tol = TOL[precision]
    assert len(g_loss) == len(r["losses"]) == -(-len(tok) // s.chunk)
    rel = np.abs(g_loss - r["losses"]) / np.maximum(np.abs(r["losses"]), 1e-12)
    assert rel.max() <= tol, (rel.max(), g_loss[:4], r["losses"][:4])
    L, Lt = s.n_layers, s.n_ttt_layers
    worst_delta = 0.0
    for i in range(Lt):
        for k in O.FAST:
            assert rel_fro(g_fast[i][k], r["fast"][i][k]) <= tol
            w0 = np.asarray(w["layers"][L - Lt + i][k], np.float64)
            worst_delta = max(worst_delta, rel_fro(g_fast[i][k] - w0, r["fast"][i][k] - w0))
    if check_delta is not None:
        assert worst_delta <= check_delta, worst_delta
    return rel.max(), worst_delta


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

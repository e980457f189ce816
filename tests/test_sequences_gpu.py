"""Several sequences in one context (ttt_config.n_seq > 1): one ttt_prefill
reads them all, the products with static weights take every sequence's rows
in one launch, and the fast MLPs' products run as grouped GEMMs with one
weight set per sequence.  Every sequence must come out as the oracle's run
of that sequence alone: its chunk losses, its final fast weights and their
update, at the precision's tolerance (fp32 check mode 1e-4, bf16 2e-2)."""
import numpy as np
import pytest

from long_context_lm_ttt_b300 import inputs
from oracle import ttt_ref as O

from test_parity_gpu import TOL, check_against

pytestmark = pytest.mark.gpu


def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_lm_ttt_b300 import ttt as T
    T.load()
    return T


def run_sequences(s, w, toks, precision, bulk_tokens=0):
    T = _lib()
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    ns = len(toks)
    m = T.TTT(s, w, prec, max_tokens=s.seq_len, bulk_tokens=bulk_tokens, n_seq=ns)
    try:
        losses = m.prefill(np.ascontiguousarray(np.stack(toks), np.int32)).astype(np.float64)
        fast = [[m.fast_weights(i, seq=q) for i in range(s.n_ttt_layers)] for q in range(ns)]
        # a reset context gives the same again
        m.reset()
        again = m.prefill(np.ascontiguousarray(np.stack(toks), np.int32)).astype(np.float64)
    finally:
        m.close()
    assert np.array_equal(losses, again)
    return losses, fast


def compare_sequences(s, w, toks, precision, bulk_tokens=0, check_delta=None):
    losses, fast = run_sequences(s, w, toks, precision, bulk_tokens)
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    assert losses.shape == (len(toks), -(-s.seq_len // s.chunk))
    for q, tk in enumerate(toks):
        r = O.prefill(cfg, w, tk)
        check_against(s, w, losses[q], fast[q], r, precision, check_delta)


SEQ_CASES = [
    # name, overrides, sequences, bulk tokens (several super-chunks)
    ("tiny-ttt2", dict(n_layers=3), 3, 64),
    ("tiny-gqa", dict(), 2, 0),
]


@pytest.mark.parametrize("name,kw,ns,bulk", SEQ_CASES)
def test_fp32_sequences(name, kw, ns, bulk):
    s = inputs.shape(name, **kw)
    w = inputs.make_weights(s)
    toks = [inputs.make_tokens(s, seed=1 + q) for q in range(ns)]
    compare_sequences(s, w, toks, "fp32", bulk, check_delta=1e-4)


@pytest.mark.parametrize("name,kw,ns,bulk", SEQ_CASES)
def test_bf16_sequences(name, kw, ns, bulk):
    s = inputs.shape(name, bf16=True, **kw)
    w = inputs.make_weights(s)
    toks = [inputs.make_tokens(s, seed=1 + q) for q in range(ns)]
    compare_sequences(s, w, toks, "bf16", bulk)


def test_bf16_sequences_tensor_cores():
    """Head dim 64, chunks of 128: tensor-core attention per sequence and
    grouped GEMMs over 128-row groups (single-CTA tiles), 3 sequences over
    3 super-chunks with a ragged last chunk."""
    s = inputs.shape("tiny-gqa", bf16=True, n_layers=4, n_heads=4, n_kv_heads=2, head_dim=64, d_model=256,
                     d_ff=512, chunk=128, window=200, seq_len=700)
    w = inputs.make_weights(s)
    toks = [inputs.make_tokens(s, s.seq_len, seed=1 + q) for q in range(3)]
    compare_sequences(s, w, toks, "bf16", bulk_tokens=256)


def test_bf16_sequences_3b_shapes():
    """The 3B tile shapes with two sequences: grouped GEMMs over 1024-row
    groups on CTA pairs, the stacked static products at M = 2048, two
    super-chunks, the window (1024) wrapping the ring."""
    s = inputs.shape("3b-4layer", window=1024, seq_len=2048)
    w = inputs.make_weights(s)
    toks = [inputs.make_tokens(s, s.seq_len, seed=1 + q) for q in range(2)]
    compare_sequences(s, w, toks, "bf16", bulk_tokens=1024)


def test_sequences_match_separate_contexts():
    """The same sequences through one context each agree with the
    multi-sequence context to the bf16 tolerance (the grouped and stacked
    products change only the order of fp32 sums)."""
    T = _lib()
    s = inputs.shape("tiny-gqa", bf16=True, n_layers=4, n_heads=4, n_kv_heads=2, head_dim=64, d_model=256,
                     d_ff=512, chunk=128, window=200, seq_len=512)
    w = inputs.make_weights(s)
    toks = [inputs.make_tokens(s, s.seq_len, seed=5 + q) for q in range(2)]
    losses, fast = run_sequences(s, w, toks, "bf16", bulk_tokens=256)
    for q, tk in enumerate(toks):
        m = T.TTT(s, w, T.TTT_BF16, max_tokens=s.seq_len, bulk_tokens=256)
        try:
            one = m.prefill(np.ascontiguousarray(tk, np.int32)).astype(np.float64)
            f1 = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
        finally:
            m.close()
        assert np.abs(one - losses[q]).max() / np.abs(one).max() <= TOL["bf16"] / 10
        for i in range(s.n_ttt_layers):
            for k in O.FAST:
                a, b = fast[q][i][k].astype(np.float64), f1[i][k].astype(np.float64)
                assert np.linalg.norm(a - b) / np.linalg.norm(b) <= TOL["bf16"] / 10


def test_sequences_reject_decode_and_logits():
    T = _lib()
    s = inputs.shape("tiny-gqa")
    w = inputs.make_weights(s)
    m = T.TTT(s, w, T.TTT_FP32_CHECK, max_tokens=s.seq_len, n_seq=2)
    try:
        with pytest.raises(T.TTTError) as e:
            m.logits(np.zeros(4, np.int32))
        assert e.value.code == T.TTT_ERR_STATE
        with pytest.raises(T.TTTError) as e:
            m.decode(np.zeros(1, np.int32), 4)
        assert e.value.code == T.TTT_ERR_STATE
    finally:
        m.close()

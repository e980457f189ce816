"""Decode-time test-time training through the C ABI (ttt_decode) against the
CPU oracle's decode.

Tolerances as for the prefill parity: fp32 check mode <= 1e-4, bf16 mode
<= 2e-2 on the chunk losses (relative) and the final fast weights (relative
Frobenius norm).  Greedy tokens are an integer decision taken on the GPU's
own fp32 logits: a generated token must be the oracle's largest logit or
within the precision's margin of it, given the same preceding tokens.
"""
import numpy as np
import pytest

from long_context_lm_ttt_b300 import inputs
from oracle import ttt_ref as O

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}
# a greedy pick may differ from the oracle's argmax only between logits this
# close (relative to the largest logit magnitude of the step)
MARGIN = {"fp32": 1e-4, "bf16": 3e-2}


def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_lm_ttt_b300 import ttt as T
    T.load()
    return T


def _model(s, w, precision, max_tokens):
    T = _lib()
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    return T, T.TTT(s, w, prec, max_tokens=max_tokens)


def rel_fro(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


def _check_losses_weights(g_loss, g_fast, r, tol):
    assert len(g_loss) == len(r["losses"])
    rel = np.abs(np.asarray(g_loss, np.float64) - r["losses"]) / np.maximum(np.abs(r["losses"]), 1e-12)
    assert rel.max() <= tol, (rel.max(), g_loss, r["losses"])
    for gb, rb in zip(g_fast, r["fast"]):
        for k in O.FAST:
            assert rel_fro(gb[k], rb[k]) <= tol


def _shape(name, precision, **kw):
    return inputs.shape(name, bf16=precision == "bf16", **kw)


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
@pytest.mark.parametrize("name", ["tiny-ttt2", "tiny-gqa"])
def test_teacher_forced_decode_parity(name, precision):
    s = _shape(name, precision)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    N = 3 * s.chunk
    T, m = _model(s, w, precision, N + 1)
    try:
        out, losses = m.decode(np.ascontiguousarray(tok[:N + 1], np.int32), N)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    assert np.array_equal(out, tok[:N + 1])
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    r = O.decode(cfg, w, tok[:N + 1], N)
    _check_losses_weights(losses[:3], fast, r, TOL[precision])


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_decode_equals_gpu_prefill(precision):
    """Teacher-forced decode of tokens[0..N] and ttt_prefill of the same
    N + 1 tokens train alike (the prefill's last chunk has no target)."""
    s = _shape("tiny-ttt2", precision)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    N = 2 * s.chunk
    T, m = _model(s, w, precision, N + 1)
    try:
        _, dl = m.decode(np.ascontiguousarray(tok[:N + 1], np.int32), N)
        df = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
        m.reset()
        pl = m.prefill(np.ascontiguousarray(tok[:N + 1], np.int32))
        pf = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    tol = 1e-5 if precision == "fp32" else 1e-2
    np.testing.assert_allclose(dl[:2], pl[:2], rtol=tol)
    for a, b in zip(df, pf):
        for k in O.FAST:
            assert rel_fro(a[k], b[k]) <= tol


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_greedy_decode_parity(precision):
    """Greedy generation from a 5-token prompt over two chunks and a bit:
    every pick is the oracle's argmax up to the margin, and the oracle fed
    the GPU's tokens trains to the same losses and weights."""
    s = _shape("tiny-ttt2", precision)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    N = 2 * s.chunk + 7
    T, m = _model(s, w, precision, N + 1)
    try:
        out, losses = m.decode(np.ascontiguousarray(tok[:5], np.int32), N)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    assert np.array_equal(out[:5], tok[:5])
    assert out.min() >= 0 and out.max() < s.vocab
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    r = O.decode(cfg, w, out, N)  # the GPU's sequence, teacher-forced
    assert np.array_equal(r["tokens"], out)
    for i in range(4, N):
        z = r["logits"][i]
        assert z[out[i + 1]] >= z.max() - MARGIN[precision] * np.abs(z).max(), (i, out[i + 1], z.argmax())
    _check_losses_weights(losses[:2], fast, r, TOL[precision])


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_decode_after_prefill(precision):
    """A prefill of two chunks, then decode continues at the boundary: the
    oracle's decode from the oracle prefill's state."""
    s = _shape("tiny-gqa", precision)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    b = s.chunk
    P, N = 2 * b, 2 * b + 3
    T, m = _model(s, w, precision, P + N + 1)
    try:
        pl = m.prefill(np.ascontiguousarray(tok[:P], np.int32))
        out, dl = m.decode(np.ascontiguousarray(tok[P:P + N + 1], np.int32), N)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    rp = O.prefill(cfg, w, tok[:P], return_state=True)
    r = O.decode(cfg, w, tok[P:P + N + 1], N, state=rp["state"])
    np.testing.assert_allclose(pl, rp["losses"], rtol=TOL[precision])
    assert np.array_equal(out, tok[P:P + N + 1])
    _check_losses_weights(dl[:2], fast, r, TOL[precision])


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_decode_split_over_calls_is_bitwise_one_call(precision):
    """A chunk left incomplete carries over to the next call."""
    s = _shape("tiny-ttt2", precision)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    b = s.chunk
    N1, N2 = b + 5, b + 11
    T, m = _model(s, w, precision, N1 + N2 + 1)
    try:
        o1, l1 = m.decode(np.ascontiguousarray(tok[:N1], np.int32), N1)
        o2, l2 = m.decode(np.ascontiguousarray(tok[N1:N1 + 3], np.int32), N2)
        f_split = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
        m.reset()
        given = np.concatenate([tok[:N1], tok[N1:N1 + 3]]).astype(np.int32)
        o, l = m.decode(given, N1 + N2)
        f_one = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    # the first call's last prediction was replaced by the second call's
    # first given token, as the single call's given tokens do
    assert np.array_equal(np.concatenate([o1[:N1], o2]), o)
    assert np.array_equal(np.concatenate([l1[:1], l2[:1]]), l[:2])
    for a, c in zip(f_split, f_one):
        for k in O.FAST:
            assert np.array_equal(a[k], c[k])


def test_decode_tensor_core_attention_bf16():
    """Head dim 64 puts the one-query attention on the tensor-core kernel."""
    s = inputs.shape("tiny-gqa", n_heads=4, n_kv_heads=2, head_dim=64, d_model=256, d_ff=512, chunk=128,
                     window=200, seq_len=700, bf16=True)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s, 700)
    N = 2 * s.chunk + 3
    T, m = _model(s, w, "bf16", N + 1)
    try:
        out, losses = m.decode(np.ascontiguousarray(tok[:N + 1], np.int32), N)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    r = O.decode(cfg, w, tok[:N + 1], N)
    _check_losses_weights(losses[:2], fast, r, TOL["bf16"])


def test_decode_errors():
    s = inputs.shape("tiny-ttt2")
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    T, m = _model(s, w, "fp32", 100)
    try:
        t32 = np.ascontiguousarray(tok[:40], np.int32)
        out = np.zeros(101, np.int32)
        loss = np.zeros(8, np.float32)
        with pytest.raises(T.TTTError) as e:
            T.ttt_decode(m.ctx, t32, 0, 5, out, loss)
        assert e.value.code == -1  # INVALID: nothing given
        with pytest.raises(T.TTTError) as e:
            T.ttt_decode(m.ctx, t32, 7, 5, out, loss)
        assert e.value.code == -1  # INVALID: more given than steps + 1
        with pytest.raises(T.TTTError) as e:
            T.ttt_decode(m.ctx, t32, 1, 101, out, loss)
        assert e.value.code == -2  # SHAPE: past max_tokens
        m.prefill(np.ascontiguousarray(tok[:40], np.int32))  # 40 is not a multiple of 32
        with pytest.raises(T.TTTError) as e:
            T.ttt_decode(m.ctx, t32, 1, 5, out, loss)
        assert e.value.code == -6  # STATE: not at a chunk boundary
        m.reset()
        bad = t32.copy()
        bad[3] = s.vocab
        with pytest.raises(T.TTTError) as e:
            T.ttt_decode(m.ctx, bad, 10, 10, out, loss)
        assert e.value.code == -1  # INVALID: token id out of range
    finally:
        m.close()


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_teacher_forced_decode_dual_mlp(precision):
    """Decode-time test-time training with the static second MLP."""
    s = inputs.shape("tiny-ttt2", dual_mlp=True, bf16=precision == "bf16")
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    N = 2 * s.chunk
    T, m = _model(s, w, precision, N + 1)
    try:
        out, losses = m.decode(np.ascontiguousarray(tok[:N + 1], np.int32), N)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    r = O.decode(cfg, w, tok[:N + 1], N)
    _check_losses_weights(losses[:2], fast, r, TOL[precision])


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_decode_graph_replay_is_bitwise_direct_issue(precision):
    """Decode steps replayed from the captured graphs give bit for bit what
    the same steps give when every kernel is issued directly (per-launch
    profiling keeps the engine on direct issue).  Mixes given and greedy
    steps across two calls and a completed chunk."""
    s = _shape("tiny-gqa", precision)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    N = 2 * s.chunk + 5
    given = np.ascontiguousarray(tok[:s.chunk // 2], np.int32)
    runs = []
    for profiled in (False, True):
        T, m = _model(s, w, precision, N + 1)
        try:
            if profiled:
                m.profile(True)
            o1, l1 = m.decode(given, s.chunk + 3)
            o2, l2 = m.decode(o1[-1:], N - (s.chunk + 3))
            fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
        finally:
            m.close()
        runs.append((o1, l1, o2, l2, fast))
    (a1, al1, a2, al2, af), (b1, bl1, b2, bl2, bf) = runs
    assert np.array_equal(a1, b1) and np.array_equal(a2, b2)
    assert np.array_equal(np.asarray(al1), np.asarray(bl1)) and np.array_equal(np.asarray(al2), np.asarray(bl2))
    for fa, fb in zip(af, bf):
        for k in O.FAST:
            assert np.array_equal(fa[k], fb[k])


def test_decode_3b_widths_after_prefill():
    """Decode at the 3B widths (d 3072, 24 query / 8 KV heads x 128, d_ff
    8192, V 128256) after a two-chunk prefill, through a completed chunk and
    into greedy picks: the one-row products at these widths (the lm_head
    with the fused greedy pick among them), the bulk-copy one-query
    attention with three query heads per KV head, the graph replay and the
    chunk's test-time step.  Two blocks, one fast; chunks of 128 and a
    window of 300 keep the oracle's run short."""
    s = inputs.shape("3b-4layer", n_layers=2, n_ttt_layers=1, chunk=128, window=300, seq_len=512)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    b = s.chunk
    P, N, n_given = 2 * b, b + 6, b - 10  # greedy from step n_given - 1 on
    T, m = _model(s, w, "bf16", P + N + 1)
    try:
        pl = m.prefill(np.ascontiguousarray(tok[:P], np.int32))
        out, dl = m.decode(np.ascontiguousarray(tok[P:P + n_given], np.int32), N)
        fast = [m.fast_weights(i) for i in range(s.n_ttt_layers)]
    finally:
        m.close()
    assert np.array_equal(out[:n_given], tok[P:P + n_given])
    assert out.min() >= 0 and out.max() < s.vocab
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    rp = O.prefill(cfg, w, tok[:P], return_state=True)
    r = O.decode(cfg, w, out, N, state=rp["state"])  # the GPU's tokens, teacher-forced
    np.testing.assert_allclose(pl, rp["losses"], rtol=TOL["bf16"])
    for i in range(n_given - 1, N):
        z = r["logits"][i]
        assert z[out[i + 1]] >= z.max() - MARGIN["bf16"] * np.abs(z).max(), (i, out[i + 1], z.argmax())
    _check_losses_weights(dl[:1], fast, r, TOL["bf16"])
    # the updates themselves (prefill and decode chunks), not only the
    # weights they were added to
    L = s.n_layers
    for k in O.FAST:
        w0 = np.asarray(w["layers"][L - 1][k], np.float64)
        assert rel_fro(fast[0][k] - w0, r["fast"][0][k] - w0) <= TOL["bf16"], k

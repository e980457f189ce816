"""Plant plausible mistakes in the oracle (CPU only) and check that the pins
catch each of them.  Every plant is undone by monkeypatch after its test."""
import numpy as np
import pytest

from oracle import ttt_ref as O
import test_oracle_pins as P


def _fails(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except AssertionError:
        return True
    return False


def test_wrong_rope_backward_sign_is_caught(monkeypatch):
    monkeypatch.setattr(O, "rope_bwd", O.rope)
    assert P.fd_check("tiny-ttt2", 0) > 1e-3


def test_dropped_rmsnorm_backward_term_is_caught(monkeypatch):
    monkeypatch.setattr(O, "rmsnorm_bwd", lambda x, g, r, dy: r * (g * dy))
    assert P.fd_check("tiny", 0) > 1e-3


def test_stale_stash_in_backward_is_caught(monkeypatch):
    """The backward reads an up-projection that differs from the forward's."""
    orig = O.backward_chunk

    def bad_backward(st, z, acts, valid, tgt, n_tgt):
        for l in acts:
            if l != "final":
                acts[l] = dict(acts[l], up=acts[l]["up"] * 1.0001 + 1e-3)
        return orig(st, z, acts, valid, tgt, n_tgt)

    monkeypatch.setattr(O, "backward_chunk", bad_backward)
    assert P.fd_check("tiny", 0) > 1e-4


def test_wrong_kv_head_grouping_is_caught(monkeypatch):
    """Query head i paired with KV head i % Hkv instead of i // (H/Hkv)."""
    import math

    def bad_attention(q, kw, vw, qpos, kpos, window, group):
        head_kv = np.arange(q.shape[1]) % kw.shape[1]
        kh, vh = kw[:, head_kv, :], vw[:, head_kv, :]
        S = np.einsum("nhd,mhd->hnm", q, kh) / math.sqrt(q.shape[-1])
        rel = qpos[:, None] - kpos[None, :]
        S = np.where(((rel >= 0) & (rel < window))[None], S, -np.inf)
        E = np.exp(S - S.max(-1, keepdims=True))
        Pm = E / E.sum(-1, keepdims=True)
        return np.einsum("hnm,mhd->nhd", Pm, vh), Pm

    monkeypatch.setattr(O, "attention", bad_attention)
    assert _fails(P.test_forward_matches_torch_library_restatement, "tiny-gqa", False)


def test_window_off_by_one_is_caught(monkeypatch):
    orig = O.attention
    monkeypatch.setattr(O, "attention",
                        lambda q, kw, vw, qp, kp, window, group: orig(q, kw, vw, qp, kp, window + 1, group))
    assert _fails(P.test_attention_band_matches_sdpa_with_mask)


def test_target_shift_is_caught(monkeypatch):
    def bad_targets(tokens, s, e):
        T = len(tokens)
        t = np.arange(s, e)
        valid = (t + 1) < T
        return valid, np.where(valid, np.asarray(tokens)[t], 0)

    monkeypatch.setattr(O, "chunk_targets", bad_targets)
    assert _fails(P.test_lr0_chunked_equals_unchunked, "tiny", False)


def test_update_sign_is_caught(monkeypatch):
    orig = O.step_chunk

    def bad_step(st, tokens, s, e, lr, update=True, want_grads=False):
        return orig(st, tokens, s, e, -lr, update, want_grads)

    monkeypatch.setattr(O, "step_chunk", bad_step)
    assert _fails(P.test_loss_falls_on_repeated_context)


def test_skipped_static_mlp_backward_is_caught(monkeypatch):
    """With a static second MLP, the backward treats it as the identity
    (passes dy straight to the fast MLP)."""
    orig = O.backward_chunk

    def bad_backward(st, z, acts, valid, tgt, n_tgt):
        import copy
        st2 = copy.copy(st)
        st2.cfg = O.dataclasses.replace(st.cfg, dual_mlp=False)
        return orig(st2, z, acts, valid, tgt, n_tgt)

    monkeypatch.setattr(O, "backward_chunk", bad_backward)
    assert P.fd_check("tiny-ttt2", 0, dual_mlp=True) > 1e-3


def test_logits_after_at_a_shifted_position_is_caught(monkeypatch):
    """The continuation rotated as if it started one position early."""
    def bad_logits_after(st, cont):
        z, _ = O.forward_span(st, np.asarray(cont), st.pos - 1, write_cache=False)
        return z

    monkeypatch.setattr(O, "logits_after", bad_logits_after)
    assert _fails(P.test_logits_after_prefill_match_torch_forward, 0.0)
    assert _fails(P.test_logits_after_prefill_match_torch_forward, None)


def test_logits_after_with_the_initial_weights_is_caught(monkeypatch):
    """The continuation scored by the fast weights before the context's
    updates (those of the pin's configuration, tiny)."""
    from long_context_lm_ttt_b300 import inputs
    w0 = inputs.make_weights(inputs.shape("tiny"))

    def bad_logits_after(st, cont):
        L = st.cfg.n_layers
        saved = {k: st.layers[L - 1][k] for k in O.FAST}
        try:
            for k in O.FAST:
                st.layers[L - 1][k] = np.asarray(w0["layers"][L - 1][k], st.dtype)
            z, _ = O.forward_span(st, np.asarray(cont), st.pos, write_cache=False)
        finally:
            st.layers[L - 1].update(saved)
        return z

    monkeypatch.setattr(O, "logits_after", bad_logits_after)
    assert _fails(P.test_logits_after_prefill_match_torch_forward, None)

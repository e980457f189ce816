"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one part of the oracle to what the pages or mathematics fix:
library routines for the special cases they cover, central finite
differences for the gradients, closed forms for the update, invariants
(chunking, causality, repetition) for the loop.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from long_context_lm_ttt_b300 import inputs
from oracle import ttt_ref as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _setup(name, **kw):
    s = inputs.shape(name, **kw)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s)
    return s, O.OracleConfig.from_mapping(s.as_dict()), w, tok


# ---------------------------------------------------------------------------
# building blocks against library routines / closed forms
# ---------------------------------------------------------------------------
def test_rmsnorm_matches_torch_library():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 48))
    g = rng.standard_normal(48)
    y, r = O.rmsnorm(x, g, 1e-6)
    ref = F.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_rmsnorm_bwd_finite_differences():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 16))
    g = rng.standard_normal(16)
    dy = rng.standard_normal((3, 16))
    _, r = O.rmsnorm(x, g, 1e-6)
    dx = O.rmsnorm_bwd(x, g, r, dy)
    eps = 1e-6
    num = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += eps
            xm[i, j] -= eps
            num[i, j] = (np.sum(O.rmsnorm(xp, g, 1e-6)[0] * dy) -
                         np.sum(O.rmsnorm(xm, g, 1e-6)[0] * dy)) / (2 * eps)
    np.testing.assert_allclose(dx, num, rtol=1e-7, atol=1e-8)


def test_rope_is_complex_rotation():
    """Rotate-half RoPE == multiplying (x_i + i x_{i+h}) by exp(i t theta^(-2i/hd))."""
    rng = np.random.default_rng(7)
    n, nh, hd = 9, 3, 16
    x = rng.standard_normal((n, nh, hd))
    pos = np.arange(100, 100 + n)
    ang = O.rope_angles(pos, hd, 10000.0)
    y = O.rope(x, ang)
    h = hd // 2
    zc = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos[:, None, None] *
                                                  (10000.0 ** (-np.arange(h) * 2.0 / hd)))
    np.testing.assert_allclose(y[..., :h], zc.real, atol=1e-12)
    np.testing.assert_allclose(y[..., h:], zc.imag, atol=1e-12)
    # the backward is the inverse rotation, and rotations keep inner products
    np.testing.assert_allclose(O.rope_bwd(y, ang), x, atol=1e-12)
    k = rng.standard_normal((n, nh, hd))
    np.testing.assert_allclose(np.einsum("nhd,nhd->nh", y, O.rope(k, ang)),
                               np.einsum("nhd,nhd->nh", x, k), atol=1e-10)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (6, 2)])
def test_attention_full_window_is_sdpa_causal(H, Hkv):
    """window >= T: banded attention is plain causal attention (library)."""
    rng = np.random.default_rng(8)
    n, hd = 13, 8
    q = rng.standard_normal((n, H, hd))
    k = rng.standard_normal((n, Hkv, hd))
    v = rng.standard_normal((n, Hkv, hd))
    pos = np.arange(n)
    o, _ = O.attention(q, k, v, pos, pos, window=10 ** 6, group=H // Hkv)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(H // Hkv, 0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(H // Hkv, 0)[None]
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_attention_band_matches_sdpa_with_mask():
    rng = np.random.default_rng(9)
    n, H, hd, W = 20, 2, 8, 5
    q = rng.standard_normal((n, H, hd))
    k = rng.standard_normal((n, H, hd))
    v = rng.standard_normal((n, H, hd))
    pos = np.arange(n)
    o, _ = O.attention(q, k, v, pos, pos, window=W, group=1)
    i = torch.arange(n)
    mask = (i[:, None] >= i[None, :]) & (i[:, None] - i[None, :] < W)
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask)[0].permute(1, 0, 2)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# whole forward against a restatement made of torch library routines
# ---------------------------------------------------------------------------
def _torch_forward_logits(s, w, tok, fast=None):
    """Un-chunked SWA forward from library pieces (rms_norm, sdpa with a band
    mask, silu; RoPE as complex rotation).  fp64 logits [T, V].  ``fast``
    maps a block index to weights that replace that block's own."""
    T = len(tok)
    H, Hkv, hd = s.n_heads, s.n_kv_heads, s.head_dim
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.float64)
    pos = torch.arange(T, dtype=torch.float64)
    half = hd // 2
    inv = s.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / hd)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64), pos[:, None] * inv[None])

    def rope(x):                                     # x [T, nh, hd]
        zc = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([zc.real, zc.imag], dim=-1)

    i = torch.arange(T)
    band = (i[:, None] >= i[None, :]) & (i[:, None] - i[None, :] < s.window)
    x = t(w["tok_embed"])[torch.as_tensor(tok, dtype=torch.long)]
    for l, lw in enumerate(w["layers"]):
        lwt = {k: t(v) for k, v in lw.items()}
        if fast is not None and l in fast:
            lwt.update(fast[l])
        xn = F.rms_norm(x, (s.d_model,), lwt["attn_norm"], eps=s.norm_eps)
        q = rope(F.linear(xn, lwt["wq"]).view(T, H, hd))
        k = rope(F.linear(xn, lwt["wk"]).view(T, Hkv, hd))
        v = F.linear(xn, lwt["wv"]).view(T, Hkv, hd)
        rep = H // Hkv
        o = F.scaled_dot_product_attention(
            q.permute(1, 0, 2)[None], k.permute(1, 0, 2).repeat_interleave(rep, 0)[None],
            v.permute(1, 0, 2).repeat_interleave(rep, 0)[None], attn_mask=band)
        o = o[0].permute(1, 0, 2).reshape(T, H * hd)
        h = x + F.linear(o, lwt["wo"])
        hn = F.rms_norm(h, (s.d_model,), lwt["mlp_norm"], eps=s.norm_eps)
        x = h + F.linear(F.silu(F.linear(hn, lwt["w_gate"])) * F.linear(hn, lwt["w_up"]),
                         lwt["w_down"])
        if s.dual_mlp and l >= s.n_layers - s.n_ttt_layers:
            hn2 = F.rms_norm(x, (s.d_model,), lwt["mlp2_norm"], eps=s.norm_eps)
            x = x + F.linear(F.silu(F.linear(hn2, lwt["w_gate2"])) * F.linear(hn2, lwt["w_up2"]),
                             lwt["w_down2"])
    return F.linear(F.rms_norm(x, (s.d_model,), t(w["final_norm"]), eps=s.norm_eps), t(w["lm_head"]))


def _torch_forward_losses(s, w, tok, fast=None):
    """Per-position next-token losses of that forward (cross_entropy)."""
    z = _torch_forward_logits(s, w, tok, fast)
    return F.cross_entropy(z[:-1], torch.as_tensor(tok[1:], dtype=torch.long), reduction="none")


@pytest.mark.parametrize("name,dual", [("tiny", False), ("tiny-gqa", False), ("tiny-gqa", True)])
def test_forward_matches_torch_library_restatement(name, dual):
    s, cfg, w, tok = _setup(name, dual_mlp=dual)
    ours = O.full_forward_losses(cfg, w, tok)
    ref = _torch_forward_losses(s, w, tok).numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("lr", [0.0, None])
def test_logits_after_prefill_match_torch_forward(lr):
    """logits_after (what ttt_logits returns): the logits of a continuation
    after reading a context.  With one fast block, the last, the cached keys
    and values of earlier positions do not depend on the fast weights (each
    block's MLP follows its attention, and no fast block lies below another
    block), so the continuation's logits equal one plain forward over context
    and continuation with the final fast weights (the initial ones at lr = 0).
    The call leaves the state as it was."""
    s, cfg, w, tok = _setup("tiny")
    assert s.n_ttt_layers == 1
    P, n = 3 * s.chunk + 5, 9  # a ragged context, then n more tokens
    cont = tok[P:P + n]
    r = O.prefill(cfg, w, tok[:P], lr=lr, return_state=True)
    st = r["state"]
    pos0 = st.pos
    z = O.logits_after(st, cont)
    assert st.pos == pos0
    np.testing.assert_array_equal(O.logits_after(st, cont), z)
    L = s.n_layers
    fast = {L - 1: {k: torch.as_tensor(np.asarray(v), dtype=torch.float64) for k, v in r["fast"][-1].items()}}
    if lr is None:  # the context did move the fast weights
        assert max(np.abs(r["fast"][-1][k] - w["layers"][L - 1][k]).max() for k in O.FAST) > 0
    ref = _torch_forward_logits(s, w, np.concatenate([tok[:P], cont]), fast=fast)[P:P + n].numpy()
    np.testing.assert_allclose(z, ref, rtol=0, atol=1e-10 * np.abs(ref).max())


@pytest.mark.parametrize("name,dual", [("tiny", False), ("tiny-ttt2", False), ("tiny-gqa", False),
                                       ("tiny-ttt2", True)])
def test_lr0_chunked_equals_unchunked(name, dual):
    """With lr=0 the chunk losses are those of one plain SWA forward."""
    s, cfg, w, tok = _setup(name, dual_mlp=dual)
    r0 = O.prefill(cfg, w, tok, lr=0.0)
    full = O.full_forward_losses(cfg, w, tok)
    T, b = len(tok), s.chunk
    ref = np.array([full[c * b:min(T - 1, (c + 1) * b)].mean() for c in range(-(-T // b))])
    np.testing.assert_allclose(r0["losses"], ref, rtol=1e-12, atol=1e-12)


def test_window_at_least_T_is_full_causal_attention():
    s, cfg, w, tok = _setup("tiny", window=10 ** 6)
    r0 = O.prefill(cfg, w, tok, lr=0.0)
    # brute force: full causal attention via the library restatement
    ref = _torch_forward_losses(s.replace(window=len(tok) + 1), w, tok).numpy()
    T, b = len(tok), s.chunk
    ref_c = np.array([ref[c * b:min(T - 1, (c + 1) * b)].mean() for c in range(-(-T // b))])
    np.testing.assert_allclose(r0["losses"], ref_c, rtol=1e-11)


# ---------------------------------------------------------------------------
# gradients
# ---------------------------------------------------------------------------
def _snapshot_before_chunk(cfg, w, tok, c, lr):
    """Oracle state right before chunk c (earlier chunks applied)."""
    st = O.OracleState(cfg, w, max_positions=len(tok))
    for s0, e0 in O.chunk_bounds(len(tok), cfg.chunk)[:c]:
        O.step_chunk(st, tok, s0, e0, lr)
    return st


def _loss_with_cache_fixed(st, tok, s, e):
    z, _ = O.forward_span(st, np.asarray(tok)[s:e], s, write_cache=False)
    valid, tgt = O.chunk_targets(tok, s, e)
    return O.chunk_loss_from_logits(z, valid, tgt)[0]


def fd_check(name, c, n_dirs=3, eps=1e-5, **kw):
    """Directional central differences of loss_c along random directions of
    every fast matrix vs <grad, direction>; returns worst relative error."""
    s, cfg, w, tok = _setup(name, **kw)
    st = _snapshot_before_chunk(cfg, w, tok, c, s.lr)
    s0, e0 = O.chunk_bounds(len(tok), cfg.chunk)[c]
    import copy
    st_g = copy.deepcopy(st)
    _, grads = O.step_chunk(st_g, tok, s0, e0, lr=0.0, update=False, want_grads=True)
    rng = np.random.default_rng(11)
    worst = 0.0
    for l, gl in grads.items():
        for key in O.FAST:
            for _ in range(n_dirs):
                D = rng.standard_normal(gl[key].shape)
                st_p, st_m = copy.deepcopy(st), copy.deepcopy(st)
                st_p.layers[l][key] += eps * D
                st_m.layers[l][key] -= eps * D
                num = (_loss_with_cache_fixed(st_p, tok, s0, e0) -
                       _loss_with_cache_fixed(st_m, tok, s0, e0)) / (2 * eps)
                ana = float(np.sum(gl[key] * D))
                worst = max(worst, abs(num - ana) / max(abs(ana), 1e-12))
    return worst


@pytest.mark.parametrize("name,c", [("tiny", 0), ("tiny", 5), ("tiny-ttt2", 0), ("tiny-ttt2", 4),
                                    ("tiny-gqa", 3)])
def test_gradients_central_differences(name, c):
    assert fd_check(name, c) < 1e-6


@pytest.mark.parametrize("name,c", [("tiny-ttt2", 0), ("tiny-gqa", 2)])
def test_gradients_central_differences_dual_mlp(name, c):
    """Fast blocks with a static second MLP after the fast one: the fast
    weights' gradients pass through the static MLP's input gradient."""
    assert fd_check(name, c, dual_mlp=True) < 1e-6


@pytest.mark.parametrize("dual", [False, True])
def test_gradients_match_torch_autograd(dual):
    """One chunk's fast-weight gradients against torch.autograd (fp64) on the
    library restatement (first chunk: no cache involved)."""
    s, cfg, w, tok = _setup("tiny-gqa", dual_mlp=dual)
    b = s.chunk
    tok1 = tok[:b + 1]                      # chunk 0 plus its last target
    st = O.OracleState(cfg, w, max_positions=b + 1)
    _, grads = O.step_chunk(st, tok1, 0, b, lr=0.0, update=False, want_grads=True)
    L, Lt = s.n_layers, s.n_ttt_layers
    fast = {l: {k: torch.tensor(w["layers"][l][k], dtype=torch.float64, requires_grad=True)
                for k in O.FAST} for l in range(L - Lt, L)}
    losses = _torch_forward_losses(s, w, tok1, fast=fast)
    losses[:b].mean().backward()
    for l in fast:
        for k in O.FAST:
            np.testing.assert_allclose(grads[l][k], fast[l][k].grad.numpy(), rtol=1e-8, atol=1e-13)


# ---------------------------------------------------------------------------
# the update and the loop
# ---------------------------------------------------------------------------
def test_update_is_one_sgd_step():
    s, cfg, w, tok = _setup("tiny-ttt2")
    b = s.chunk
    st = O.OracleState(cfg, w, max_positions=len(tok))
    _, grads = O.step_chunk(st, tok, 0, b, lr=s.lr)
    for l, gl in grads.items():
        for k in O.FAST:
            np.testing.assert_allclose(st.layers[l][k] - np.asarray(w["layers"][l][k], np.float64),
                                       -s.lr * gl[k], rtol=1e-9, atol=1e-16)
    # static weights untouched
    L, Lt = s.n_layers, s.n_ttt_layers
    for l in range(L):
        for k in inputs.LAYER_TENSORS:
            if l >= L - Lt and k in O.FAST:
                continue
            assert np.array_equal(st.layers[l][k], w["layers"][l][k])


def test_first_order_closed_form():
    """loss_1(lr) - loss_1(0) = -lr <g0, g1> + O(lr^2)."""
    s, cfg, w, tok = _setup("tiny-ttt2")
    b = s.chunk
    st = O.OracleState(cfg, w, max_positions=len(tok))
    _, g0 = O.step_chunk(st, tok, 0, b, lr=0.0, update=False, want_grads=True)
    _, g1 = O.step_chunk(st, tok, b, 2 * b, lr=0.0, update=False, want_grads=True)
    dot = sum(float(np.sum(g0[l][k] * g1[l][k])) for l in g0 for k in O.FAST)
    base = O.prefill(cfg, w, tok, lr=0.0, n_chunks=2)["losses"][1]
    errs = []
    for lr in (1e-3, 5e-4):
        l1 = O.prefill(cfg, w, tok, lr=lr, n_chunks=2)["losses"][1]
        errs.append(abs((l1 - base) - (-lr * dot)))
        assert abs((l1 - base) / (-lr * dot) - 1) < 0.05
    assert errs[1] < errs[0] * 0.4           # second-order remainder shrinks ~4x


def test_loss_falls_on_repeated_context():
    """Learning the context compresses it: on a repeated block the loss falls
    chunk after chunk, and stays below the no-update run."""
    s = inputs.shape("tiny")
    w = inputs.make_weights(s)
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    T = 16 * s.chunk
    tok = inputs.make_repeated_tokens(s, T, s.chunk)
    l0 = O.prefill(cfg, w, tok, lr=0.0)["losses"]
    l1 = O.prefill(cfg, w, tok, lr=s.lr)["losses"]
    # the receptive field grows by window-1 positions per block, so without
    # updates the loss is periodic once L*(W-1) positions precede the chunk
    first = -(-(s.n_layers * (s.window - 1)) // s.chunk)
    np.testing.assert_allclose(l0[first:-1], l0[first], rtol=1e-12)
    assert np.all(np.diff(l1[first:]) < 0)
    assert np.all(l1[first:] < l0[first:])


def test_initial_loss_near_log_vocab():
    s, cfg, w, tok = _setup("tiny")
    r = O.prefill(cfg, w, tok, lr=0.0, n_chunks=1)
    assert abs(r["losses"][0] - math.log(s.vocab)) < 0.1


# ---------------------------------------------------------------------------
# indexing
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,b", [(256, 32), (257, 32), (33, 32), (1, 32), (100, 7)])
def test_chunks_and_targets(T, b):
    bounds = O.chunk_bounds(T, b)
    assert len(bounds) == -(-T // b)
    assert bounds[0][0] == 0 and bounds[-1][1] == T
    assert all(bounds[i][1] == bounds[i + 1][0] for i in range(len(bounds) - 1))
    tok = np.arange(T)
    n_tgt = [int(O.chunk_targets(tok, s0, e0)[0].sum()) for s0, e0 in bounds]
    assert sum(n_tgt) == T - 1
    assert n_tgt[-1] == bounds[-1][1] - bounds[-1][0] - 1
    for s0, e0 in bounds:
        valid, tgt = O.chunk_targets(tok, s0, e0)
        assert np.array_equal(tgt[valid], np.arange(s0, e0)[valid] + 1)


def test_chunk_without_targets_reports_zero_and_keeps_weights():
    s, cfg, w, tok = _setup("tiny")
    tok = tok[:s.chunk + 1]                 # last chunk holds one position, no target
    r = O.prefill(cfg, w, tok)
    assert len(r["losses"]) == 2 and r["losses"][1] == 0.0
    r1 = O.prefill(cfg, w, tok, n_chunks=1)
    for a, b_ in zip(r["fast"], r1["fast"]):
        for k in O.FAST:
            assert np.array_equal(a[k], b_[k])


@pytest.mark.parametrize("lr", [0.0, 1e-2])
def test_causality(lr):
    """Changing token p leaves every chunk that ends before p-1 bit-identical."""
    s, cfg, w, tok = _setup("tiny")
    p = 150
    tok2 = tok.copy()
    tok2[p] = (tok2[p] + 1) % s.vocab
    a = O.prefill(cfg, w, tok, lr=lr)["losses"]
    b_ = O.prefill(cfg, w, tok2, lr=lr)["losses"]
    for c, (s0, e0) in enumerate(O.chunk_bounds(len(tok), s.chunk)):
        if e0 <= p:                          # last target tok[e0] lies before p
            assert a[c] == b_[c]
        if s0 <= p - 1 < e0:
            assert a[c] != b_[c]


# ---------------------------------------------------------------------------
# the pages' own numbers, and the regression lock
# ---------------------------------------------------------------------------
def test_shapes_follow_the_pages():
    with open(os.path.join(GOLDEN, "pages_hparams.json")) as f:
        g = json.load(f)
    s = inputs.shape("3b")
    assert s.window == g["window_tokens"]
    assert s.chunk == g["ttt_minibatch_tokens"]
    for name in ("125m", "760m", "3b"):
        sh = inputs.shape(name)
        assert sh.n_ttt_layers * g["updated_fraction_of_blocks_denominator"] == sh.n_layers
    assert abs(inputs.n_params(s) / 1e9 - g["params_billion"]) < 0.7


def test_oracle_regression_lock():
    """Chunk losses of the tiny shapes as written by tests/golden/make_golden.py
    (which calls only the oracle); guards the oracle against silent edits."""
    with open(os.path.join(GOLDEN, "oracle_tiny_losses.json")) as f:
        g = json.load(f)
    for name, ref in g["losses"].items():
        s, cfg, w, tok = _setup(name)
        np.testing.assert_allclose(O.prefill(cfg, w, tok)["losses"], ref, rtol=1e-12)


def test_no_fast_blocks_is_a_frozen_model():
    """n_ttt_layers = 0: nothing is trained at test time, so the chunk losses
    are the chunk means of one un-chunked forward, for any lr."""
    s = inputs.shape("tiny-ttt2", n_ttt_layers=0, lr=0.5)
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s)
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    r = O.prefill(cfg, w, tok)
    full = O.full_forward_losses(cfg, w, tok)
    b, T = s.chunk, len(tok)
    ref = np.array([full[c * b:min(T - 1, (c + 1) * b)].mean() for c in range(-(-T // b))])
    np.testing.assert_allclose(r["losses"], ref, rtol=1e-12, atol=1e-12)
    assert r["fast"] == []


# ---------------------------------------------------------------------------
# decode-time test-time training
# ---------------------------------------------------------------------------
def test_teacher_forced_decode_trains_like_prefill():
    """Reading tokens one position at a time and training on each completed
    chunk gives the prefill's chunk losses and final fast weights over the
    same tokens (the prefill's extra last chunk has no target)."""
    s, cfg, w, tok = _setup("tiny-ttt2")
    b = s.chunk
    N = 3 * b
    d = O.decode(cfg, w, tok[:N + 1], N)
    r = O.prefill(cfg, w, tok[:N + 1])
    assert len(d["losses"]) == 3 and len(r["losses"]) == 4 and r["losses"][3] == 0.0
    np.testing.assert_allclose(d["losses"], r["losses"][:3], rtol=1e-11, atol=0)
    for a, c in zip(d["fast"], r["fast"]):
        for k in O.FAST:
            np.testing.assert_allclose(a[k], c[k], rtol=0, atol=1e-11 * np.abs(c[k]).max())
    assert np.array_equal(d["tokens"], tok[:N + 1])


def test_decode_step_logits_equal_one_unchunked_forward_at_lr0():
    """With lr = 0 nothing changes the weights, so the logits of every step
    equal the logits of one forward over the whole sequence."""
    s, cfg, w, tok = _setup("tiny-gqa", lr=0.0)
    N = 2 * s.chunk + 9
    d = O.decode(cfg, w, tok[:N + 1], N)
    st = O.OracleState(cfg, w, max_positions=N)
    z, _ = O.forward_span(st, tok[:N], 0)
    np.testing.assert_allclose(d["logits"], z, rtol=0, atol=1e-10 * np.abs(z).max())


def test_greedy_decode_picks_argmax_and_replays():
    """Greedy steps take the largest logit; feeding the generated tokens back
    as given inputs reproduces the run exactly."""
    s, cfg, w, tok = _setup("tiny-ttt2")
    N = 2 * s.chunk + 10
    g = O.decode(cfg, w, tok[:5], N)
    for i in range(4, N):
        assert g["tokens"][i + 1] == int(np.argmax(g["logits"][i]))
    assert np.array_equal(g["tokens"][:5], tok[:5])
    t = O.decode(cfg, w, g["tokens"], N)
    assert np.array_equal(t["tokens"], g["tokens"])
    np.testing.assert_array_equal(t["losses"], g["losses"])


def test_teacher_forced_decode_trains_like_prefill_dual_mlp():
    s, cfg, w, tok = _setup("tiny-gqa", dual_mlp=True)
    N = 2 * s.chunk
    d = O.decode(cfg, w, tok[:N + 1], N)
    r = O.prefill(cfg, w, tok[:N + 1])
    np.testing.assert_allclose(d["losses"], r["losses"][:2], rtol=1e-11, atol=0)
    for a, c in zip(d["fast"], r["fast"]):
        for k in O.FAST:
            np.testing.assert_allclose(a[k], c[k], rtol=0, atol=1e-11 * np.abs(c[k]).max())


def test_decode_without_fast_blocks_scores_a_frozen_model():
    """n_ttt_layers = 0: decoding only scores; its chunk losses are the
    chunk means of one un-chunked forward."""
    s, cfg, w, tok = _setup("tiny-ttt2", n_ttt_layers=0)
    b = s.chunk
    N = 3 * b
    d = O.decode(cfg, w, tok[:N + 1], N)
    full = O.full_forward_losses(cfg, w, tok[:N + 1])
    ref = np.array([full[c * b:(c + 1) * b].mean() for c in range(3)])
    np.testing.assert_allclose(d["losses"], ref, rtol=1e-12, atol=1e-12)
    assert d["fast"] == []

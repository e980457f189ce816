"""CPU oracle for the TTT-E2E test-time inner loop (prefill and decode).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, links or runs
this module; only the tests, the smoke check and the CPU-baseline leg of the
benchmark do.  It shares no code with the CUDA path: the two meet only in the
seeded inputs handed to both.

What it computes ("End-to-End Test-Time Training for Long Context"):
  * the model is a standard decoder-only Transformer whose self-attention is
    sliding-window attention (summary page, Method; podcast page 4:41);
  * at test time the model keeps training on the context it reads, by
    next-token prediction (summary page, Method; NVIDIA blog, "Our method");
  * the context is consumed in mini-batches of about 1K tokens under an 8K
    window, and only the MLP layers are updated; attention, embeddings and the
    rest stay fixed (podcast page, 6:36);
  * only the MLPs of the last quarter of the blocks are updated (podcast page,
    7:08); the configurations name that count ``n_ttt_layers``;
  * the update is plain gradient descent on the context ("mini-gradient
    descent", digitado repost, TL;DR).

Readings taken where the pages are silent (each is listed in the design
notes):
  * block: pre-norm RMSNorm (no bias, gain g, eps), RoPE rotate-half with
    theta at absolute positions, grouped KV heads (q head i uses KV head
    i // (H/Hkv)), SwiGLU MLP  Wd (silu(Wg u) * (Wu u)), final RMSNorm and an
    untied lm_head;
  * window: query t sees keys j with t - W < j <= t (W keys, itself included);
  * the target of position t is token t+1 for t+1 < T, so a chunk's last
    position predicts the first token of the next chunk; the chunk loss is the
    mean over the chunk's targets; a chunk without targets reports 0 and does
    not update;
  * the chunk is scored by the weights before its own update (the same
    forward yields the reported loss and the gradient);
  * one SGD step per chunk, W <- W - lr * dL/dW, applied after all gradients
    of the chunk are formed; keys and values of earlier chunks are constants
    (cached, detached), so gradients reach only the current chunk's own
    queries, keys and values;
  * optionally (``dual_mlp``) each updated block keeps a static second MLP
    (podcast page, 7:08), placed after its fast MLP with its own pre-norm
    and residual; it is never updated, and gradients pass through it;
  * decoding (``decode``) keeps the same loop, one chunk step per b
    positions read, as stated in its docstring.

Everything runs in float64 (``dtype`` may be lowered for timing only).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

FAST = ("w_gate", "w_up", "w_down")


@dataclasses.dataclass
class OracleConfig:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    window: int
    chunk: int
    n_ttt_layers: int
    lr: float
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6
    dual_mlp: bool = False

    @classmethod
    def from_mapping(cls, m) -> "OracleConfig":
        names = {f.name for f in dataclasses.fields(cls)}
        return cls(**{k: v for k, v in dict(m).items() if k in names})


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------
def rmsnorm(x, g, eps):
    """n(x) = g * x / sqrt(mean(x^2) + eps), row-wise.  Returns (n(x), r)
    with r = 1/sqrt(mean(x^2)+eps) of shape [rows, 1]."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return g * x * r, r


def rmsnorm_bwd(x, g, r, dy):
    """Gradient of n(x) w.r.t. x:  r*(g*dy) - r^3 * x * mean(x*g*dy)."""
    d = x.shape[-1]
    s = np.sum(x * g * dy, axis=-1, keepdims=True) / d
    return r * (g * dy) - (r ** 3) * x * s


def rope_angles(pos, head_dim, theta):
    """angle[t, i] = pos[t] * theta^(-2i/hd), i in [0, hd/2)."""
    half = head_dim // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]


def rope(x, ang):
    """Rotate-half RoPE: pairs (i, i+hd/2) rotated by ang.  x: [n, heads, hd]."""
    half = x.shape[-1] // 2
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_bwd(dy, ang):
    """Transpose of ``rope`` (rotation by -ang)."""
    half = dy.shape[-1] // 2
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = dy[..., :half], dy[..., half:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def logsumexp(z):
    m = np.max(z, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True)))[..., 0]


# ---------------------------------------------------------------------------
# state
# ---------------------------------------------------------------------------
class OracleState:
    """Weights (fast ones are updated in place), the per-layer key/value cache
    indexed by absolute position, and the number of positions consumed."""

    def __init__(self, cfg: OracleConfig, weights: dict, max_positions: int, dtype=np.float64):
        self.cfg = cfg
        self.dtype = dtype
        cv = lambda a: np.array(a, dtype=dtype, copy=True)
        self.tok_embed = cv(weights["tok_embed"])
        self.final_norm = cv(weights["final_norm"])
        self.lm_head = cv(weights["lm_head"])
        self.layers = [{k: cv(v) for k, v in lw.items()} for lw in weights["layers"]]
        H, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        self.kcache = [np.zeros((max_positions, Hkv, hd), dtype) for _ in range(cfg.n_layers)]
        self.vcache = [np.zeros((max_positions, Hkv, hd), dtype) for _ in range(cfg.n_layers)]
        self.pos = 0

    def fast_weights(self) -> List[Dict[str, np.ndarray]]:
        L, Lt = self.cfg.n_layers, self.cfg.n_ttt_layers
        return [{k: self.layers[l][k].copy() for k in FAST} for l in range(L - Lt, L)]


# ---------------------------------------------------------------------------
# forward of one span of positions [s, e) with the current weights
# ---------------------------------------------------------------------------
def attention(q, kw, vw, qpos, kpos, window, group):
    """Banded causal attention with grouped heads.

    q: [n, H, hd] (roped), kw/vw: [m, Hkv, hd] for key positions kpos.
    Query at position t sees keys j with t - window < j <= t.
    Returns o [n, H, hd] and the probabilities P [H, n, m].
    """
    hd = q.shape[-1]
    head_kv = np.arange(q.shape[1]) // group
    kh = kw[:, head_kv, :]                     # [m, H, hd]
    vh = vw[:, head_kv, :]
    # per head: S_h = q_h k_h^T / sqrt(hd), as batched matrix products
    S = np.matmul(q.transpose(1, 0, 2), kh.transpose(1, 2, 0)) / math.sqrt(hd)   # [H, n, m]
    rel = qpos[:, None] - kpos[None, :]
    allowed = (rel >= 0) & (rel < window)
    S = np.where(allowed[None], S, -np.inf)
    m = np.max(S, axis=-1, keepdims=True)
    E = np.exp(S - m)
    P = E / np.sum(E, axis=-1, keepdims=True)
    o = np.matmul(P, vh.transpose(1, 0, 2)).transpose(1, 0, 2)                    # [n, H, hd]
    return o, P


def forward_span(st: OracleState, tok_span, s, write_cache=True, keep=None):
    """Run positions [s, s+n) through all blocks; returns (z, acts).

    ``keep`` is the set of layers whose intermediates are kept for backward.
    Keys and values of these positions are written to the cache.
    """
    cfg = st.cfg
    n = len(tok_span)
    e = s + n
    H, Hkv, hd, W = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.window
    group = H // Hkv
    pos = np.arange(s, e)
    ang = rope_angles(pos, hd, cfg.rope_theta)
    lo = max(0, s - W + 1)
    kpos = np.arange(lo, e)
    x = st.tok_embed[np.asarray(tok_span)]
    acts = {}
    keep = set() if keep is None else keep
    for l, lw in enumerate(st.layers):
        xn, r1 = rmsnorm(x, lw["attn_norm"], cfg.norm_eps)
        q = (xn @ lw["wq"].T).reshape(n, H, hd)
        k = (xn @ lw["wk"].T).reshape(n, Hkv, hd)
        v = (xn @ lw["wv"].T).reshape(n, Hkv, hd)
        qr, kr = rope(q, ang), rope(k, ang)
        kc, vc = st.kcache[l], st.vcache[l]
        if write_cache:
            kc[s:e] = kr
            vc[s:e] = v
            kw, vw = kc[lo:e], vc[lo:e]
        else:
            kw = np.concatenate([kc[lo:s], kr], axis=0)
            vw = np.concatenate([vc[lo:s], v], axis=0)
        o, P = attention(qr, kw, vw, pos, kpos, W, group)
        of = o.reshape(n, H * hd)
        h = x + of @ lw["wo"].T
        hn, r2 = rmsnorm(h, lw["mlp_norm"], cfg.norm_eps)
        gp = hn @ lw["w_gate"].T
        up = hn @ lw["w_up"].T
        a = silu(gp) * up
        y = h + a @ lw["w_down"].T
        if l in keep:
            acts[l] = dict(x=x, xn=xn, r1=r1, qr=qr, kw=kw, vw=vw, P=P, o=of, h=h, hn=hn,
                           r2=r2, gp=gp, up=up, a=a, v=v)
        if cfg.dual_mlp and l >= cfg.n_layers - cfg.n_ttt_layers:
            # the fast block's static second MLP, after the fast one, with
            # its own pre-norm and residual
            h2 = y
            hn2, r3 = rmsnorm(h2, lw["mlp2_norm"], cfg.norm_eps)
            gp2 = hn2 @ lw["w_gate2"].T
            up2 = hn2 @ lw["w_up2"].T
            y = h2 + (silu(gp2) * up2) @ lw["w_down2"].T
            if l in keep:
                acts[l].update(h2=h2, r3=r3, gp2=gp2, up2=up2)
        x = y
    hf, rf = rmsnorm(x, st.final_norm, cfg.norm_eps)
    z = hf @ st.lm_head.T
    acts["final"] = dict(x=x, rf=rf, hf=hf, ang=ang, lo=lo, s=s, n=n)
    return z, acts


def chunk_targets(tokens, s, e):
    """Targets of positions [s, e): token t+1 where t+1 < T.  Returns
    (valid mask [n], target ids [n] with 0 where invalid)."""
    T = len(tokens)
    t = np.arange(s, e)
    valid = (t + 1) < T
    tgt = np.where(valid, np.asarray(tokens)[np.minimum(t + 1, T - 1)], 0)
    return valid, tgt


def chunk_loss_from_logits(z, valid, tgt):
    """mean over valid rows of logsumexp(z_t) - z_t[y_t]; 0 without targets."""
    n_tgt = int(valid.sum())
    if n_tgt == 0:
        return 0.0, n_tgt
    lse = logsumexp(z)
    zy = z[np.arange(z.shape[0]), tgt]
    return float(np.sum((lse - zy)[valid]) / n_tgt), n_tgt


# ---------------------------------------------------------------------------
# backward of one chunk's loss into the fast weights
# ---------------------------------------------------------------------------
def backward_chunk(st: OracleState, z, acts, valid, tgt, n_tgt):
    """Manual backward of the chunk loss w.r.t. w_gate, w_up, w_down of the
    fast blocks.  Cached keys/values of earlier chunks are constants."""
    cfg = st.cfg
    L, Lt = cfg.n_layers, cfg.n_ttt_layers
    H, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    group = H // Hkv
    fin = acts["final"]
    n, s, lo, ang = fin["n"], fin["s"], fin["lo"], fin["ang"]
    # d loss / d z = (softmax(z) - onehot(y)) / n_tgt on rows with a target
    lse = logsumexp(z)
    dz = np.exp(z - lse[:, None])
    dz[np.arange(n), tgt] -= 1.0
    dz *= (valid[:, None] / n_tgt)
    dhf = dz @ st.lm_head
    dy = rmsnorm_bwd(fin["x"], st.final_norm, fin["rf"], dhf)
    grads = {}
    n_cached = s - lo                       # keys before the chunk: constants
    for l in range(L - 1, L - Lt - 1, -1):
        lw, A = st.layers[l], acts[l]
        if cfg.dual_mlp:
            # y = h2 + a2 Wd2^T with a2 = silu(n(h2) Wg2^T) * (n(h2) Wu2^T):
            # the static MLP's input gradient, then dy is the one at h2
            da2 = dy @ lw["w_down2"]
            sg2 = sigmoid(A["gp2"])
            dgp2 = da2 * A["up2"] * (sg2 * (1.0 + A["gp2"] * (1.0 - sg2)))
            dup2 = da2 * A["gp2"] * sg2
            dhn2 = dgp2 @ lw["w_gate2"] + dup2 @ lw["w_up2"]
            dy = dy + rmsnorm_bwd(A["h2"], lw["mlp2_norm"], A["r3"], dhn2)
        # y = h + a Wd^T
        da = dy @ lw["w_down"]
        g_down = dy.T @ A["a"]
        sg = sigmoid(A["gp"])
        dgp = da * A["up"] * (sg * (1.0 + A["gp"] * (1.0 - sg)))
        dup = da * A["gp"] * sg
        g_gate = dgp.T @ A["hn"]
        g_up = dup.T @ A["hn"]
        grads[l] = {"w_gate": g_gate, "w_up": g_up, "w_down": g_down}
        if l == L - Lt:
            break                            # nothing below holds fast weights
        dhn = dgp @ lw["w_gate"] + dup @ lw["w_up"]
        dh = dy + rmsnorm_bwd(A["h"], lw["mlp_norm"], A["r2"], dhn)
        # h = x + o Wo^T
        do = (dh @ lw["wo"]).reshape(n, H, hd)
        P = A["P"]                                            # [H, n, m]
        head_kv = np.arange(H) // group
        kh = A["kw"][:, head_kv, :]
        vh = A["vw"][:, head_kv, :]
        # per head h (batched matrix products over the head axis):
        # dP_h = do_h v_h^T, dq_h = dS_h k_h, and for the chunk's own keys
        # dk_h = dS_h^T q_h, dv_h = P_h^T do_h
        dP = np.matmul(do.transpose(1, 0, 2), vh.transpose(1, 2, 0))               # [H, n, m]
        o = A["o"].reshape(n, H, hd)
        Dt = np.sum(do * o, axis=-1).T[..., None]                                  # [H, n, 1]
        dS = P * (dP - Dt) / math.sqrt(hd)
        dq = np.matmul(dS, kh.transpose(1, 0, 2)).transpose(1, 0, 2)               # [n, H, hd]
        # keys / values of the chunk itself: the last n columns of the window
        dk_h = np.matmul(dS[:, :, n_cached:].transpose(0, 2, 1), A["qr"].transpose(1, 0, 2)).transpose(1, 0, 2)
        dv_h = np.matmul(P[:, :, n_cached:].transpose(0, 2, 1), do.transpose(1, 0, 2)).transpose(1, 0, 2)
        dk = dk_h.reshape(n, Hkv, group, hd).sum(axis=2)
        dv = dv_h.reshape(n, Hkv, group, hd).sum(axis=2)
        dq = rope_bwd(dq, ang).reshape(n, H * hd)
        dk = rope_bwd(dk, ang).reshape(n, Hkv * hd)
        dv = dv.reshape(n, Hkv * hd)
        dxn = dq @ lw["wq"] + dk @ lw["wk"] + dv @ lw["wv"]
        dy = dh + rmsnorm_bwd(A["x"], lw["attn_norm"], A["r1"], dxn)
    return grads


# ---------------------------------------------------------------------------
# the inner loop
# ---------------------------------------------------------------------------
def chunk_bounds(T: int, b: int):
    """Chunk c covers positions [c*b, min(T, (c+1)*b))."""
    return [(c * b, min(T, (c + 1) * b)) for c in range(-(-T // b))]


def step_chunk(st: OracleState, tokens, s, e, lr, update=True, want_grads=False):
    """Forward chunk [s, e) with the current weights, its loss, its gradient,
    then (if update) one SGD step on the fast weights."""
    cfg = st.cfg
    L, Lt = cfg.n_layers, cfg.n_ttt_layers
    keep = set(range(L - Lt, L))
    z, acts = forward_span(st, np.asarray(tokens)[s:e], s, write_cache=True, keep=keep)
    valid, tgt = chunk_targets(tokens, s, e)
    loss, n_tgt = chunk_loss_from_logits(z, valid, tgt)
    grads = None
    if n_tgt > 0 and (update or want_grads):
        grads = backward_chunk(st, z, acts, valid, tgt, n_tgt)
        if update:
            for l, gl in grads.items():
                for k in FAST:
                    st.layers[l][k] -= lr * gl[k]
    st.pos = e
    return loss, grads


def prefill(cfg: OracleConfig, weights: dict, tokens, lr: Optional[float] = None,
            n_chunks: Optional[int] = None, dtype=np.float64, return_state=False):
    """The test-time inner loop over ``tokens``.

    Returns dict(losses=[nC] float64, fast=[{w_gate,w_up,w_down}] for blocks
    L-Lt..L-1, state=OracleState if requested).  ``n_chunks`` stops after a
    prefix of chunks (their losses are exactly those of the full run, since
    chunk c only sees tokens up to its last target).
    """
    lr = cfg.lr if lr is None else lr
    tokens = np.asarray(tokens)
    T = len(tokens)
    bounds = chunk_bounds(T, cfg.chunk)
    if n_chunks is not None:
        bounds = bounds[:n_chunks]
    st = OracleState(cfg, weights, max_positions=max(1, bounds[-1][1] if bounds else 1), dtype=dtype)
    losses = []
    for s, e in bounds:
        loss, _ = step_chunk(st, tokens, s, e, lr)
        losses.append(loss)
    out = {"losses": np.array(losses, dtype=np.float64), "fast": st.fast_weights()}
    if return_state:
        out["state"] = st
    return out


def decode(cfg: OracleConfig, weights: dict, tokens, n_steps: int, lr: Optional[float] = None,
           dtype=np.float64, state: Optional[OracleState] = None):
    """Decode-time test-time training: generation one position at a time,
    training on every completed chunk.  It starts at position 0, or at
    ``state.pos`` (a chunk boundary) of a state left by ``prefill``.

    The pages state that the method's latency per token stays constant in
    the context length, like a recurrent model (summary page, Key claims;
    podcast page, 5:55): generation keeps the same inner loop, one gradient
    step per chunk of the tokens read.  Readings taken here:
      * step i reads input token x_i at position i with the current weights
        (its keys and values enter the cache) and gives the logits z_i;
      * the next input is tokens[i + 1] while given, else the greedy choice
        argmax z_i (the first index on ties);
      * when position p completes a chunk [p + 1 - b, p + 1), that chunk is
        trained on exactly as in the prefill (``step_chunk``): its targets
        are the inputs that followed each position, the last one being the
        input chosen at step p.
    So teacher-forced decoding of tokens[0..n_steps] trains like ``prefill``
    over those n_steps + 1 tokens, chunk for chunk.

    Returns dict(tokens=[n_steps + 1] (the inputs, then the next input after
    the last step), logits=[n_steps, V] (z_i before any update of the chunk
    holding i), losses=[completed chunks], fast=final fast weights).
    """
    lr = cfg.lr if lr is None else lr
    tokens = np.asarray(tokens)
    n_given = len(tokens)
    assert 1 <= n_given <= n_steps + 1
    b = cfg.chunk
    if state is None:
        st = OracleState(cfg, weights, max_positions=n_steps + 1, dtype=dtype)
    else:
        st = state
        assert st.pos % b == 0
        grow = st.pos + n_steps + 1 - st.kcache[0].shape[0]
        if grow > 0:
            for l in range(cfg.n_layers):
                st.kcache[l] = np.concatenate([st.kcache[l], np.zeros((grow,) + st.kcache[l].shape[1:], st.dtype)])
                st.vcache[l] = np.concatenate([st.vcache[l], np.zeros((grow,) + st.vcache[l].shape[1:], st.dtype)])
    p0 = st.pos
    seq = np.zeros(p0 + n_steps + 1, np.int64)  # inputs by absolute position
    seq[p0] = tokens[0]
    logits, losses = [], []
    for i in range(n_steps):
        p = p0 + i
        z, _ = forward_span(st, seq[p:p + 1], p, write_cache=True)
        logits.append(z[0])
        seq[p + 1] = tokens[i + 1] if i + 1 < n_given else int(np.argmax(z[0]))
        st.pos = p + 1
        if (p + 1) % b == 0:
            loss, _ = step_chunk(st, seq[:p + 2], p + 1 - b, p + 1, lr)
            losses.append(loss)
    return {"tokens": seq[p0:], "logits": np.array(logits), "losses": np.array(losses, dtype=np.float64),
            "fast": st.fast_weights()}


def logits_after(st: OracleState, cont) -> np.ndarray:
    """Logits of a continuation at positions pos..pos+n-1 with the current
    weights and cache; the state is left unchanged."""
    z, _ = forward_span(st, np.asarray(cont), st.pos, write_cache=False)
    return z


def full_forward_losses(cfg: OracleConfig, weights: dict, tokens, dtype=np.float64):
    """Per-position next-token losses of ONE un-chunked sliding-window forward
    over all tokens with fixed weights (no test-time training).  Returns the
    vector loss_t for t in [0, T-1)."""
    tokens = np.asarray(tokens)
    T = len(tokens)
    st = OracleState(cfg, weights, max_positions=T, dtype=dtype)
    z, _ = forward_span(st, tokens, 0, write_cache=True)
    lse = logsumexp(z[:-1])
    return lse - z[np.arange(T - 1), tokens[1:]]

"""Seeded synthetic workloads: model shapes, weights and token streams.

This module holds no arithmetic of the method itself. It only names the model
shapes that are run, and draws the inputs (initial weights, token ids) that
both the CUDA path and the CPU oracle receive. Everything is deterministic in
the seeds below.

Shapes follow the end-to-end test-time-training pages ("End-to-End Test-Time
Training for Long Context"): a decoder-only Transformer with sliding-window
attention (window 8K at 3B), test-time mini-batches of 1K tokens, and fast
weights in the MLPs of the last quarter of the blocks (the podcast page, the
6:36 and 7:08 segments).

Recipe:
  * weights: tensor number k in the fixed order
      tok_embed, then per block (attn_norm, wq, wk, wv, wo, mlp_norm,
      w_gate, w_up, w_down), then final_norm, lm_head, then (dual-MLP
      shapes only) per fast block (mlp2_norm, w_gate2, w_up2, w_down2)
    is default_rng([seed, k]).standard_normal(shape, float32) * 0.02;
    norm gains are ones (they still take their index k).  With
    ``bf16=True`` every value is rounded to the nearest bfloat16
    (ties to even), so both sides start from identical weights.
  * tokens: seed 1.  ``uniform`` draws ids uniformly in [0, V);
    ``zipf`` draws a truncated Zipf(1.1) law p(i) ~ (i+1)^-1.1 over
    [0, V) by inverse CDF, the id being the rank.
  * repeated blocks: seed 2, one block of ``block`` ids repeated.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Sizes of one workload (plain data; no behaviour)."""

    name: str
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
    seq_len: int
    bf16: bool
    tokens: str = "zipf"          # "uniform" | "zipf"
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6
    # fast blocks carry a second, static MLP after the fast one (podcast
    # page, 7:08)
    dual_mlp: bool = False

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)

    @property
    def n_chunks(self) -> int:
        return -(-self.seq_len // self.chunk)

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)


# The workloads.  ``tiny`` is small enough for the oracle to run in seconds;
# the others are the 125M / 760M / 3B classes.  ``tiny-ttt2`` and
# ``tiny-gqa`` exercise the attention backward (two fast blocks) and grouped
# KV heads; ``3b-4layer`` keeps the 3B tile shapes with four blocks.
SHAPES: Dict[str, ModelShape] = {
    "tiny": ModelShape("tiny", 2, 128, 4, 4, 32, 512, 512, 64, 32, 1, 1e-2, 256,
                       bf16=False, tokens="uniform"),
    "tiny-ttt2": ModelShape("tiny-ttt2", 2, 128, 4, 4, 32, 512, 512, 64, 32, 2, 1e-2, 256,
                            bf16=False, tokens="uniform"),
    "tiny-gqa": ModelShape("tiny-gqa", 3, 128, 4, 2, 32, 384, 512, 48, 32, 2, 1e-2, 200,
                           bf16=False, tokens="uniform"),
    "125m": ModelShape("125m", 12, 768, 12, 12, 64, 2048, 32000, 2048, 512, 3, 1e-3, 32768,
                       bf16=True),
    "760m": ModelShape("760m", 24, 1536, 16, 4, 96, 4096, 32000, 4096, 1024, 6, 1e-3, 131072,
                       bf16=True),
    "3b": ModelShape("3b", 28, 3072, 24, 8, 128, 8192, 128256, 8192, 1024, 7, 5e-4, 131072,
                     bf16=True),
    "3b-4layer": ModelShape("3b-4layer", 4, 3072, 24, 8, 128, 8192, 128256, 8192, 1024, 2,
                            5e-4, 4096, bf16=True),
}


def shape(name: str, **overrides) -> ModelShape:
    s = SHAPES[name]
    return s.replace(**overrides) if overrides else s


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")
# the static second MLP of a fast block (dual-MLP shapes)
LAYER2_TENSORS = ("mlp2_norm", "w_gate2", "w_up2", "w_down2")


def _layer_shapes(s: ModelShape) -> Dict[str, tuple]:
    q = s.n_heads * s.head_dim
    kv = s.n_kv_heads * s.head_dim
    return {
        "attn_norm": (s.d_model,),
        "wq": (q, s.d_model),
        "wk": (kv, s.d_model),
        "wv": (kv, s.d_model),
        "wo": (s.d_model, q),
        "mlp_norm": (s.d_model,),
        "w_gate": (s.d_ff, s.d_model),
        "w_up": (s.d_ff, s.d_model),
        "w_down": (s.d_model, s.d_ff),
    }


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 value (ties to even),
    returned as float32.  Input preparation only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _draw(seed: int, k: int, shp: tuple, bf16: bool) -> np.ndarray:
    rng = np.random.default_rng([seed, k])
    w = rng.standard_normal(shp, dtype=np.float32)
    w *= np.float32(0.02)
    return round_bf16(w) if bf16 else w


def weight_plan(s: ModelShape) -> List[tuple]:
    """(k, path, shape, is_gain) for every tensor, in drawing order."""
    plan = [(0, ("tok_embed",), (s.vocab, s.d_model), False)]
    k = 1
    ls = _layer_shapes(s)
    for l in range(s.n_layers):
        for name in LAYER_TENSORS:
            plan.append((k, ("layers", l, name), ls[name], name.endswith("norm")))
            k += 1
    plan.append((k, ("final_norm",), (s.d_model,), True))
    plan.append((k + 1, ("lm_head",), (s.vocab, s.d_model), False))
    k += 2
    if s.dual_mlp:
        for l in range(s.n_layers - s.n_ttt_layers, s.n_layers):
            for name in LAYER2_TENSORS:
                plan.append((k, ("layers", l, name), ls[name[:-1] if name != "mlp2_norm" else "mlp_norm"],
                             name.endswith("norm")))
                k += 1
    return plan


def make_weights(s: ModelShape, seed: int = 0, threads: Optional[int] = None,
                 bf16: Optional[bool] = None) -> dict:
    """Initial weights as float32 numpy arrays (bf16-representable when the
    shape is a bf16 one), in the ``nn.Linear`` layout [out, in]."""
    bf16 = s.bf16 if bf16 is None else bf16
    out: dict = {"layers": [dict() for _ in range(s.n_layers)]}
    plan = weight_plan(s)

    def one(item):
        k, path, shp, is_gain = item
        arr = np.ones(shp, np.float32) if is_gain else _draw(seed, k, shp, bf16)
        return path, arr

    nthreads = threads or min(16, max(1, len(__import__("os").sched_getaffinity(0))))
    with ThreadPoolExecutor(nthreads) as ex:
        for path, arr in ex.map(one, plan):
            if path[0] == "layers":
                out["layers"][path[1]][path[2]] = arr
            else:
                out[path[0]] = arr
    return out


def n_params(s: ModelShape) -> int:
    return sum(int(np.prod(shp)) for _, _, shp, _ in weight_plan(s))


# --------------------------------------------------------------------------
# tokens
# --------------------------------------------------------------------------
def make_tokens(s: ModelShape, T: Optional[int] = None, seed: int = 1,
                kind: Optional[str] = None) -> np.ndarray:
    """int32 token ids of length T (default: the shape's sequence length)."""
    T = s.seq_len if T is None else T
    kind = s.tokens if kind is None else kind
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return rng.integers(0, s.vocab, size=T, dtype=np.int64).astype(np.int32)
    if kind == "zipf":
        p = (np.arange(s.vocab, dtype=np.float64) + 1.0) ** -1.1
        cdf = np.cumsum(p)
        cdf /= cdf[-1]
        ids = np.searchsorted(cdf, rng.random(T), side="left")
        return np.minimum(ids, s.vocab - 1).astype(np.int32)
    raise ValueError(kind)


def make_repeated_tokens(s: ModelShape, T: int, block: int, seed: int = 2) -> np.ndarray:
    """One random block of ``block`` ids (uniform), repeated to length T."""
    rng = np.random.default_rng(seed)
    blk = rng.integers(0, s.vocab, size=block, dtype=np.int64).astype(np.int32)
    reps = -(-T // block)
    return np.tile(blk, reps)[:T].copy()


def flops_per_sequence(s: ModelShape, T: Optional[int] = None) -> Dict[str, float]:
    """Algorithmic FLOPs of one prefill pass (2 per multiply-add).

    Attention counts only the unmasked (query, key) pairs; nothing recomputed
    or wasted on masked tiles is counted.  Returns forward, backward, total.
    """
    T = s.seq_len if T is None else T
    d, H, Hkv, hd, ff, V, W, b = (s.d_model, s.n_heads, s.n_kv_heads, s.head_dim,
                                  s.d_ff, s.vocab, s.window, s.chunk)
    L, Lt = s.n_layers, s.n_ttt_layers
    n_attn = d * H * hd + 2 * d * Hkv * hd + H * hd * d       # q,k,v,o weights
    n_mlp = 3 * d * ff
    # unmasked pairs over the whole sequence: sum_t min(t+1, W)
    t = np.arange(T, dtype=np.float64)
    P = float(np.minimum(t + 1, W).sum())
    # in-chunk pairs (query and key in the same chunk, inside the window)
    P_local = 0.0
    for c0 in range(0, T, b):
        n = min(b, T - c0)
        tt = np.arange(n, dtype=np.float64)
        P_local += float(np.minimum(tt + 1, W).sum())
    fwd = 2.0 * (n_attn + n_mlp) * L * T + 2.0 * d * V * T + 4.0 * L * H * hd * P
    if s.dual_mlp:
        fwd += 2.0 * n_mlp * Lt * T
    if Lt == 0:  # no fast blocks: the chunks are only scored
        return {"fwd": fwd, "bwd": 0.0, "total": fwd}
    bwd = (2.0 * d * V * T                                    # d hidden from lm_head
           + 2.0 * Lt * n_mlp * T                             # MLP weight grads
           + 2.0 * (Lt - 1) * (n_mlp + n_attn) * T            # dX through upper fast blocks
           + (Lt - 1) * (6.0 * H * hd * P + 4.0 * H * hd * P_local))
    # the lowest fast block still needs dX of its down projection (da = dy Wd)
    bwd += 2.0 * d * ff * T
    if s.dual_mlp:  # dX through every static second MLP
        bwd += 2.0 * Lt * n_mlp * T
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}

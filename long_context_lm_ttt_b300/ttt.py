"""Python binding of the C ABI in include/ttt.h (argument marshalling only).

The functions below carry the C names and forward to libttt.so; every step
of the inner loop runs in the library's CUDA kernels.  Arrays may be numpy
arrays (host memory) or torch CUDA tensors (device memory); the library
tells the two apart.  If libttt.so is missing the import fails loudly:
there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_void_p
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# TTT_LIBRARY=debug selects libttt_debug.so, the same library built with the
# range checks (python -m long_context_lm_ttt_b300.build --debug-bounds)
LIB_PATH = os.path.join(_HERE, "libttt_debug.so" if os.environ.get("TTT_LIBRARY") == "debug" else "libttt.so")

TTT_OK = 0
TTT_ERR_INVALID = -1
TTT_ERR_SHAPE = -2
TTT_ERR_OOM = -3
TTT_ERR_CUDA = -4
TTT_ERR_NONFINITE = -5
TTT_ERR_STATE = -6
TTT_ERR_INTERNAL = -7
ERR_NAMES = {0: "OK", -1: "INVALID", -2: "SHAPE", -3: "OOM", -4: "CUDA", -5: "NONFINITE",
             -6: "STATE", -7: "INTERNAL"}

TTT_BF16 = 0
TTT_FP32_CHECK = 1

EXPORTS = ("ttt_create", "ttt_prefill", "ttt_prefill_batch", "ttt_decode", "ttt_logits", "ttt_get_fast_weights",
           "ttt_reset", "ttt_destroy", "ttt_last_error", "ttt_profile", "ttt_profile_read")


class ttt_config(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("d_model", c_int32), ("n_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("d_ff", c_int32),
                ("vocab", c_int32), ("window", c_int32), ("chunk", c_int32),
                ("n_ttt_layers", c_int32), ("precision", c_int32), ("lr", c_float),
                ("rope_theta", c_float), ("norm_eps", c_float), ("max_tokens", c_int64),
                ("dual_mlp", c_int32), ("bulk_tokens", c_int32), ("fast_bf16_single", c_int32),
                ("n_seq", c_int32)]


class ttt_weights(ctypes.Structure):
    _fields_ = [("tok_embed", c_void_p), ("final_norm", c_void_p), ("lm_head", c_void_p)] + [
        (name, POINTER(c_void_p)) for name in
        ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down",
         "mlp2_norm", "w_gate2", "w_up2", "w_down2")]


class ttt_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", c_int64), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libttt.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it with `python -m long_context_lm_ttt_b300.build`")
    lib = ctypes.CDLL(path)
    lib.ttt_create.argtypes = [POINTER(ttt_config), POINTER(ttt_weights), c_void_p, POINTER(c_void_p)]
    lib.ttt_create.restype = c_int32
    lib.ttt_prefill.argtypes = [c_void_p, c_void_p, c_int64, c_void_p, c_void_p]
    lib.ttt_prefill.restype = c_int32
    lib.ttt_prefill_batch.argtypes = [POINTER(c_void_p), c_int32, POINTER(c_void_p), POINTER(c_int64),
                                      POINTER(c_void_p), POINTER(c_void_p)]
    lib.ttt_prefill_batch.restype = c_int32
    lib.ttt_decode.argtypes = [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_void_p]
    lib.ttt_decode.restype = c_int32
    lib.ttt_logits.argtypes = [c_void_p, c_void_p, c_int32, c_void_p, c_void_p]
    lib.ttt_logits.restype = c_int32
    lib.ttt_get_fast_weights.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    lib.ttt_get_fast_weights.restype = c_int32
    lib.ttt_reset.argtypes = [c_void_p]
    lib.ttt_reset.restype = c_int32
    lib.ttt_destroy.argtypes = [c_void_p]
    lib.ttt_destroy.restype = None
    lib.ttt_last_error.argtypes = [c_void_p]
    lib.ttt_last_error.restype = c_char_p
    lib.ttt_profile.argtypes = [c_void_p, c_int32]
    lib.ttt_profile.restype = c_int32
    lib.ttt_profile_read.argtypes = [c_void_p, POINTER(ttt_kernel_stat), c_int32, POINTER(c_int32)]
    lib.ttt_profile_read.restype = c_int32
    lib.ttt_kernel_gemm.argtypes = [c_int32, c_int32, c_int32, c_void_p, c_int64, c_int32, c_void_p,
                                    c_int64, c_int32, c_void_p, c_void_p, c_int64, c_int32, c_void_p]
    lib.ttt_kernel_gemm.restype = c_int32
    i32 = c_int32
    lib.ttt_kernel_gemm_sgd.argtypes = [i32, i32, i32, c_void_p, c_int64, i32, c_void_p, c_int64, i32, c_void_p,
                                        c_void_p, c_void_p, c_int64, c_float, i32, c_void_p]
    lib.ttt_kernel_gemm_sgd.restype = c_int32
    lib.ttt_kernel_gemm_grouped.argtypes = [i32, i32, i32, i32, c_void_p, c_int64, c_void_p, c_int64, i32, c_int64,
                                            c_void_p, c_void_p, c_int64, i32, c_void_p]
    lib.ttt_kernel_gemm_grouped.restype = c_int32
    lib.ttt_kernel_attn_fwd.argtypes = [i32, i32, i32, i32, i32, i32, i32, c_int64, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, i32, c_void_p]
    lib.ttt_kernel_attn_fwd.restype = c_int32
    lib.ttt_kernel_attn_bwd.argtypes = [i32, i32, i32, i32, i32, i32, i32, c_int64, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, i32, c_void_p, c_void_p, c_void_p,
                                        c_void_p]
    lib.ttt_kernel_attn_bwd.restype = c_int32
    lib.ttt_kernel_wait_selftest.argtypes = [c_int64, c_void_p]
    lib.ttt_kernel_wait_selftest.restype = c_int32
    lib.ttt_kernel_error.argtypes = []
    lib.ttt_kernel_error.restype = c_int32
    lib.ttt_kernel_bounds_checked.argtypes = []
    lib.ttt_kernel_bounds_checked.restype = c_int32
    lib.ttt_kernel_bounds.argtypes = [POINTER(c_int32), POINTER(c_int64), POINTER(c_int64)]
    lib.ttt_kernel_bounds.restype = c_int32
    lib.ttt_kernel_bounds_selftest.argtypes = [c_int64, c_int64, c_void_p]
    lib.ttt_kernel_bounds_selftest.restype = c_int32
    _lib = lib
    return lib


class TTTError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


def _ptr(a) -> int:
    """Address of a numpy array (host) or torch tensor (device or host)."""
    if a is None:
        return 0
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return a.data_ptr()
    raise TypeError(type(a))


def _stream(stream) -> int:
    if stream is None:
        return 0
    return int(getattr(stream, "cuda_stream", stream))


# ---------------------------------------------------------------------------
# the C calls, same names
# ---------------------------------------------------------------------------
def ttt_last_error(ctx=None) -> str:
    m = load().ttt_last_error(ctx)
    return m.decode() if m else ""


def _check(rc: int, ctx=None):
    if rc != TTT_OK:
        raise TTTError(rc, ttt_last_error(ctx))


def make_config(shape, precision: int = TTT_BF16, max_tokens: Optional[int] = None,
                lr: Optional[float] = None, bulk_tokens: int = 0, fast_bf16_single: bool = False,
                n_seq: int = 1) -> ttt_config:
    """ttt_config from any object with the ModelShape field names."""
    return ttt_config(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                      shape.d_ff, shape.vocab, shape.window, shape.chunk, shape.n_ttt_layers, precision,
                      shape.lr if lr is None else lr, shape.rope_theta, shape.norm_eps,
                      max_tokens if max_tokens is not None else shape.seq_len,
                      1 if getattr(shape, "dual_mlp", False) else 0, int(bulk_tokens),
                      1 if fast_bf16_single else 0, int(n_seq))


def make_weights(w: dict):
    """ttt_weights from a dict of fp32 arrays (numpy host or torch device);
    returns (struct, keepalive)."""
    keep = []
    layers = w["layers"]

    def arr(name):
        a = (c_void_p * len(layers))(*[_ptr(lw.get(name)) for lw in layers])
        keep.append(a)
        return ctypes.cast(a, POINTER(c_void_p))

    for lw in layers:
        for v in lw.values():
            if isinstance(v, np.ndarray) and v.dtype != np.float32:
                raise TypeError("weights must be float32")
    s = ttt_weights(_ptr(w["tok_embed"]), _ptr(w["final_norm"]), _ptr(w["lm_head"]),
                    arr("attn_norm"), arr("wq"), arr("wk"), arr("wv"), arr("wo"), arr("mlp_norm"),
                    arr("w_gate"), arr("w_up"), arr("w_down"),
                    arr("mlp2_norm"), arr("w_gate2"), arr("w_up2"), arr("w_down2"))
    return s, keep


def ttt_create(cfg: ttt_config, weights: ttt_weights, stream=None) -> c_void_p:
    ctx = c_void_p()
    _check(load().ttt_create(ctypes.byref(cfg), ctypes.byref(weights), _stream(stream), ctypes.byref(ctx)))
    return ctx


def ttt_prefill(ctx, tokens, T: int, chunk_losses, stream=None) -> int:
    rc = load().ttt_prefill(ctx, _ptr(tokens), int(T), _ptr(chunk_losses), _stream(stream))
    _check(rc, ctx)
    return rc


def ttt_prefill_batch(ctxs, tokens, T, chunk_losses, streams=None) -> int:
    """ttt_prefill on several contexts at once (lists of equal length)."""
    n = len(ctxs)
    arr = lambda vals: (c_void_p * n)(*vals)
    c_ctx = arr([c.value if isinstance(c, c_void_p) else c for c in ctxs])
    c_tok = arr([_ptr(t) for t in tokens])
    c_T = (c_int64 * n)(*[int(t) for t in T])
    c_loss = arr([_ptr(l) for l in chunk_losses])
    c_st = arr([_stream(s) for s in streams]) if streams is not None else None
    rc = load().ttt_prefill_batch(c_ctx, n, c_tok, c_T, c_loss, c_st)
    if rc != 0:
        bad = next((c for c in ctxs if load().ttt_last_error(c)), ctxs[0])
        _check(rc, bad)
    return rc


def ttt_decode(ctx, tokens, n_given: int, n_steps: int, tokens_out, chunk_losses, stream=None) -> int:
    rc = load().ttt_decode(ctx, _ptr(tokens), int(n_given), int(n_steps), _ptr(tokens_out), _ptr(chunk_losses),
                           _stream(stream))
    _check(rc, ctx)
    return rc


def ttt_logits(ctx, cont, n: int, logits, stream=None) -> int:
    rc = load().ttt_logits(ctx, _ptr(cont), int(n), _ptr(logits), _stream(stream))
    _check(rc, ctx)
    return rc


def ttt_get_fast_weights(ctx, block: int, which: int, dst, stream=None) -> int:
    rc = load().ttt_get_fast_weights(ctx, int(block), int(which), _ptr(dst), _stream(stream))
    _check(rc, ctx)
    return rc


def ttt_reset(ctx) -> int:
    rc = load().ttt_reset(ctx)
    _check(rc, ctx)
    return rc


def ttt_profile(ctx, on: bool) -> int:
    rc = load().ttt_profile(ctx, 1 if on else 0)
    _check(rc, ctx)
    return rc


def ttt_profile_read(ctx) -> dict:
    """{class name: dict(launches, ms, flops, bytes)} of the profiled launches."""
    buf = (ttt_kernel_stat * 16)()
    n = c_int32()
    _check(load().ttt_profile_read(ctx, buf, 16, ctypes.byref(n)), ctx)
    return {buf[i].name.decode(): dict(launches=int(buf[i].launches), ms=float(buf[i].ms),
                                       flops=float(buf[i].flops), bytes=float(buf[i].bytes))
            for i in range(min(n.value, 16))}


def ttt_destroy(ctx) -> None:
    if ctx:
        load().ttt_destroy(ctx)


# kernel-level entry points (include/ttt_kernels.h)
GEMM_TC, GEMM_SIMT_BF16, GEMM_SIMT_F32 = 0, 1, 2


def ttt_kernel_gemm(M, N, K, A, lda, a_mn, B, ldb, b_mn, B2, C, ldc, impl, stream=None) -> int:
    rc = load().ttt_kernel_gemm(int(M), int(N), int(K), _ptr(A), int(lda), int(a_mn), _ptr(B), int(ldb),
                                int(b_mn), _ptr(B2), _ptr(C), int(ldc), int(impl), _stream(stream))
    _check(rc)
    return rc


def ttt_kernel_gemm_sgd(M, N, K, A, lda, a_mn, B, ldb, b_mn, w32, w16, w16lo, ldw, lr, impl, stream=None) -> int:
    rc = load().ttt_kernel_gemm_sgd(int(M), int(N), int(K), _ptr(A), int(lda), int(a_mn), _ptr(B), int(ldb),
                                    int(b_mn), _ptr(w32), _ptr(w16), _ptr(w16lo), int(ldw), float(lr), int(impl),
                                    _stream(stream))
    _check(rc)
    return rc


def ttt_kernel_gemm_grouped(groups, group_rows, N, K, A, lda, B, ldb, b_mn, group_stride, B2, C, ldc, impl,
                            stream=None) -> int:
    rc = load().ttt_kernel_gemm_grouped(int(groups), int(group_rows), int(N), int(K), _ptr(A), int(lda), _ptr(B),
                                        int(ldb), int(b_mn), int(group_stride), _ptr(B2), _ptr(C), int(ldc), int(impl),
                                        _stream(stream))
    _check(rc)
    return rc


def ttt_kernel_error() -> int:
    return int(load().ttt_kernel_error())


def ttt_kernel_bounds_checked() -> bool:
    return bool(load().ttt_kernel_bounds_checked())


def ttt_kernel_bounds():
    """(count, kernel id, index, limit) of the failed range checks since the
    last call on the current device; count 0 means none."""
    k, i, n = c_int32(0), c_int64(0), c_int64(0)
    rc = int(load().ttt_kernel_bounds(ctypes.byref(k), ctypes.byref(i), ctypes.byref(n)))
    if rc < 0:
        raise RuntimeError(f"ttt_kernel_bounds: {ERR_NAMES.get(rc, rc)}")
    return rc, int(k.value), int(i.value), int(n.value)


# ---------------------------------------------------------------------------
# a small object wrapper around one context
# ---------------------------------------------------------------------------
class TTT:
    """One test-time-training context on the current CUDA device."""

    def __init__(self, shape, weights: dict, precision: int = TTT_BF16,
                 max_tokens: Optional[int] = None, lr: Optional[float] = None, stream=None,
                 bulk_tokens: int = 0, fast_bf16_single: bool = False, n_seq: int = 1):
        self.shape = shape
        self.n_seq = max(1, int(n_seq))
        self.cfg = make_config(shape, precision, max_tokens, lr, bulk_tokens, fast_bf16_single, n_seq)
        ws, keep = make_weights(weights)
        self.ctx = ttt_create(self.cfg, ws, stream)
        del keep

    def n_chunks(self, T: int) -> int:
        return -(-T // self.cfg.chunk)

    def prefill(self, tokens, chunk_losses=None, stream=None):
        """Run the inner loop; returns the chunk losses (numpy for host
        tokens, else the given / a new float32 CUDA tensor).  With n_seq > 1,
        tokens is [n_seq, T] and the losses [n_seq, ceil(T / b)]."""
        T = tokens.shape[-1] if self.n_seq > 1 else len(tokens)
        shape = (self.n_seq, self.n_chunks(T)) if self.n_seq > 1 else (self.n_chunks(T),)
        if chunk_losses is None:
            if isinstance(tokens, np.ndarray):
                chunk_losses = np.zeros(shape, np.float32)
            else:
                import torch
                chunk_losses = torch.zeros(shape, dtype=torch.float32, device=tokens.device)
        ttt_prefill(self.ctx, tokens, T, chunk_losses, stream)
        return chunk_losses

    def decode(self, tokens, n_steps: int, tokens_out=None, chunk_losses=None, stream=None):
        """Decode-time test-time training for n_steps positions, inputs
        given by ``tokens`` while they last, then greedy.  Returns
        (tokens_out [n_steps + 1], chunk losses of the chunks completed);
        numpy for host tokens, else CUDA tensors on the tokens' device."""
        n_given = len(tokens)
        n_loss = n_steps // self.cfg.chunk + 1
        if tokens_out is None or chunk_losses is None:
            if isinstance(tokens, np.ndarray):
                tokens_out = np.zeros(n_steps + 1, np.int32) if tokens_out is None else tokens_out
                chunk_losses = np.zeros(n_loss, np.float32) if chunk_losses is None else chunk_losses
            else:
                import torch
                dev = tokens.device
                if tokens_out is None:
                    tokens_out = torch.zeros(n_steps + 1, dtype=torch.int32, device=dev)
                if chunk_losses is None:
                    chunk_losses = torch.zeros(n_loss, dtype=torch.float32, device=dev)
        ttt_decode(self.ctx, tokens, n_given, n_steps, tokens_out, chunk_losses, stream)
        return tokens_out, chunk_losses

    def logits(self, cont, out=None, stream=None):
        n = len(cont)
        if out is None:
            out = np.zeros((n, self.cfg.vocab), np.float32)
        ttt_logits(self.ctx, cont, n, out, stream)
        return out

    def fast_weights(self, block: int, seq: int = 0) -> dict:
        d, ff = self.cfg.d_model, self.cfg.d_ff
        out = {}
        for which, name, shp in ((0, "w_gate", (ff, d)), (1, "w_up", (ff, d)), (2, "w_down", (d, ff))):
            a = np.zeros(shp, np.float32)
            ttt_get_fast_weights(self.ctx, seq * self.cfg.n_ttt_layers + block, which, a)
            out[name] = a
        return out

    def reset(self):
        ttt_reset(self.ctx)

    def profile(self, on: bool = True):
        ttt_profile(self.ctx, on)

    def profile_read(self) -> dict:
        return ttt_profile_read(self.ctx)

    def close(self):
        if self.ctx:
            ttt_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

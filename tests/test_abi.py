"""The C-ABI library without a GPU: it loads, exports every call that
include/ttt.h declares, the ctypes mirrors match the C structs, and argument
checks that run before any device work return their error codes."""
import ctypes
import os
import re

import numpy as np
import pytest

from long_context_lm_ttt_b300 import inputs
from long_context_lm_ttt_b300 import ttt as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:int|void|const char\*)\s+(ttt_\w+)\s*\(", src, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(T.LIB_PATH):
        from long_context_lm_ttt_b300 import build
        build.build()
    return T.load()


def test_exports_every_declared_call(lib):
    declared = _declared()
    assert set(T.EXPORTS) <= declared
    for name in declared:
        assert hasattr(lib, name), name


def test_struct_layout():
    # 11 int32, 3 float, int64 max_tokens, int32 dual_mlp, bulk_tokens,
    # fast_bf16_single and n_seq, as the C declaration lays them out
    assert ctypes.sizeof(T.ttt_config) == 11 * 4 + 3 * 4 + 8 + 4 * 4
    assert T.ttt_config.max_tokens.offset == 56
    assert T.ttt_config.dual_mlp.offset == 64
    assert T.ttt_config.bulk_tokens.offset == 68
    assert T.ttt_config.fast_bf16_single.offset == 72
    assert T.ttt_config.n_seq.offset == 76
    assert ctypes.sizeof(T.ttt_weights) == 16 * ctypes.sizeof(ctypes.c_void_p)


def _cfg(**kw):
    c = T.make_config(inputs.shape("tiny"), T.TTT_FP32_CHECK)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,code", [
    (dict(precision=7), T.TTT_ERR_INVALID),
    (dict(n_layers=0), T.TTT_ERR_INVALID),
    (dict(n_ttt_layers=3), T.TTT_ERR_INVALID),
    (dict(n_ttt_layers=-1), T.TTT_ERR_INVALID),
    (dict(dual_mlp=2), T.TTT_ERR_INVALID),
    (dict(bulk_tokens=-1), T.TTT_ERR_INVALID),
    (dict(fast_bf16_single=2), T.TTT_ERR_INVALID),
    (dict(n_seq=-1), T.TTT_ERR_INVALID),
    (dict(n_seq=65), T.TTT_ERR_INVALID),
    (dict(n_kv_heads=3), T.TTT_ERR_SHAPE),
    (dict(head_dim=31), T.TTT_ERR_SHAPE),
    (dict(lr=float("nan")), T.TTT_ERR_NONFINITE),
    (dict(lr=float("inf")), T.TTT_ERR_NONFINITE),
    (dict(max_tokens=0), T.TTT_ERR_INVALID),
])
def test_create_rejects_bad_config(lib, kw, code):
    ws = T.ttt_weights()
    ctx = ctypes.c_void_p()
    rc = lib.ttt_create(ctypes.byref(_cfg(**kw)), ctypes.byref(ws), None, ctypes.byref(ctx))
    assert rc == code
    assert not ctx.value
    assert T.ttt_last_error(None) != ""


def test_null_arguments(lib):
    ctx = ctypes.c_void_p()
    assert lib.ttt_create(None, None, None, ctypes.byref(ctx)) == T.TTT_ERR_INVALID
    assert lib.ttt_create(ctypes.byref(_cfg()), None, None, None) == T.TTT_ERR_INVALID
    assert lib.ttt_prefill(None, None, 0, None, None) == T.TTT_ERR_INVALID
    assert lib.ttt_logits(None, None, 1, None, None) == T.TTT_ERR_INVALID
    assert lib.ttt_decode(None, None, 1, 1, None, None, None) == T.TTT_ERR_INVALID
    assert lib.ttt_get_fast_weights(None, 0, 0, None, None) == T.TTT_ERR_INVALID
    assert lib.ttt_reset(None) == T.TTT_ERR_INVALID
    lib.ttt_destroy(None)


def test_prefill_batch_rejects_null_contexts(lib):
    """The batch entry checks every context before any device work."""
    toks = [np.zeros(8, np.int32), np.zeros(8, np.int32)]
    losses = [np.zeros(1, np.float32), np.zeros(1, np.float32)]
    with pytest.raises(T.TTTError) as e:
        T.ttt_prefill_batch([ctypes.c_void_p(), ctypes.c_void_p()], toks, [8, 8], losses)
    assert e.value.code == T.TTT_ERR_INVALID
    assert lib.ttt_prefill_batch(None, 2, None, None, None, None) == T.TTT_ERR_INVALID


@pytest.mark.parametrize("offset", [0, 2, 8])
def test_decode_attention_rejects_misaligned_rows(lib, offset):
    """The one-query attention kernel (impl 4) reads rows with 16-byte loads:
    a key, value, query or output pointer off a 16-byte boundary returns
    TTT_ERR_SHAPE before any device work.  The addresses are never
    dereferenced (an aligned set is rejected for its head count instead)."""
    base = 0x10000
    H, Hkv, hd, W = 4, 2, 64, 64
    R = 128
    args = [base, base + 0x1000, base + 0x2000, base + 0x3000]
    for i in range(4):
        a = list(args)
        a[i] += offset
        # 9 query heads per KV head exceed the kernel's limit: even the
        # aligned case stops at the shape check, so nothing reaches a GPU
        Hq = Hkv * 9 if offset == 0 else H
        rc = lib.ttt_kernel_attn_fwd(4, 1, Hq, Hkv, hd, W, R, 5, a[0], a[1], a[2], a[3], base + 0x4000, 1, None)
        assert rc == T.TTT_ERR_SHAPE, (i, offset, rc)


def test_debug_library_exports_every_declared_call():
    """libttt_debug.so, the same sources built with the range checks, exports
    the same calls and says that it carries the checks (no device work);
    libttt.so says that it does not."""
    path = os.path.join(ROOT, "long_context_lm_ttt_b300", "libttt_debug.so")
    if not os.path.exists(path):
        from long_context_lm_ttt_b300 import build
        build.build(debug_bounds=True)
    dbg = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(dbg, name), name
    dbg.ttt_kernel_bounds_checked.restype = ctypes.c_int32
    assert dbg.ttt_kernel_bounds_checked() == 1
    assert T.load().ttt_kernel_bounds_checked() == 0

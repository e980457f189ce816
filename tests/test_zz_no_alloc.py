"""The attention backward entry point that allocates nothing
(ttt_kernel_attn_bwd_noalloc), for callers that must not call cudaMalloc:
code inside a global-mode CUDA graph capture, code whose device memory
belongs to a caching allocator or a fixed budget.  Its scratch is a fixed
device array inside the library.  Two calls in a row, with different
inputs, must each agree with the allocating entry point
ttt_kernel_attn_bwd (tensor cores) on the same inputs: the second call
also shows that what the first one left in the shared scratch does not
leak into its result.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_lm_ttt_b300 import ttt as T
    lib = T.load()
    i32, vp = ctypes.c_int32, ctypes.c_void_p
    lib.ttt_kernel_attn_bwd_noalloc.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_int64, vp, vp, vp, vp, vp,
                                                i32, vp, vp, vp, vp]
    lib.ttt_kernel_attn_bwd_noalloc.restype = i32
    return torch, T, lib


def _inputs(torch, n, H, Hkv, hd, R, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((n, H * hd), device="cuda", generator=g).to(torch.bfloat16)
    kr = torch.randn((Hkv, R, hd), device="cuda", generator=g).to(torch.bfloat16)
    vr = torch.randn((Hkv, R, hd), device="cuda", generator=g).to(torch.bfloat16)
    dout = torch.randn((n, H * hd), device="cuda", generator=g).to(torch.bfloat16)
    return q, kr, vr, dout


@pytest.mark.parametrize("shape", [
    # n, H, Hkv, hd, W, pos0: a 3B-class chunk deep in the sequence, a small
    # ragged one with head dim 96
    (1024, 24, 8, 128, 8192, 40960),
    (200, 6, 2, 96, 300, 1024),
])
def test_noalloc_matches_allocating_entry_point(shape):
    torch, T, lib = _env()
    n, H, Hkv, hd, W, pos0 = shape
    R = ((W + n - 1 + 127) // 128) * 128
    for call in range(2):
        q, kr, vr, dout = _inputs(torch, n, H, Hkv, hd, R, seed=10 * call + n)
        o = torch.empty((n, H * hd), device="cuda", dtype=torch.bfloat16)
        lse = torch.empty((H, n), device="cuda", dtype=torch.float32)
        assert lib.ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, pos0, q.data_ptr(), kr.data_ptr(), vr.data_ptr(),
                                       o.data_ptr(), lse.data_ptr(), n, None) == 0
        outs = []
        for fn in ("ref", "noalloc"):
            dsum = torch.empty((H, n), device="cuda", dtype=torch.float32)
            g = torch.full((n, (H + 2 * Hkv) * hd), float("nan"), device="cuda", dtype=torch.bfloat16)
            args = (n, H, Hkv, hd, W, R, pos0, q.data_ptr(), kr.data_ptr(), vr.data_ptr(), o.data_ptr(),
                    lse.data_ptr(), n, dout.data_ptr(), dsum.data_ptr(), g.data_ptr(), None)
            rc = lib.ttt_kernel_attn_bwd(0, *args) if fn == "ref" else lib.ttt_kernel_attn_bwd_noalloc(*args)
            assert rc == 0, (fn, rc)
            torch.cuda.synchronize()
            outs.append(g.float().cpu().numpy())
        assert T.ttt_kernel_error() == 0
        ref, got = outs
        assert np.isfinite(got).all()
        err = np.abs(got - ref).max() / np.abs(ref).max()
        assert err <= TOL, (call, err)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    torch, T, lib = _env()
    # 2 * n * H * hd floats must fit in 8 Mi floats
    n, H, Hkv, hd, W = 8192, 32, 8, 128, 64
    R = ((W + n - 1 + 127) // 128) * 128
    z = torch.zeros(16, device="cuda", dtype=torch.float32)
    p = z.data_ptr()
    rc = lib.ttt_kernel_attn_bwd_noalloc(n, H, Hkv, hd, W, R, 0, p, p, p, p, p, n, p, p, p, None)
    assert rc == T.TTT_ERR_SHAPE


def test_noalloc_against_fp64_restatement():
    """The no-alloc backward's dq, dk, dv against the fp64 restatement of
    the attention backward (the same check as the allocating entry point's
    in test_attn_gpu.py), on a ragged chunk with head dim 96 whose window
    wraps the ring."""
    torch, T, lib = _env()
    from test_attn_gpu import make_case, ref_backward
    from long_context_lm_ttt_b300 import inputs
    n, H, Hkv, hd, W, pos0, R = 256, 6, 2, 96, 300, 1024, 640
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=2 * n + hd)
    rng = np.random.default_rng(n)
    dout = inputs.round_bf16(rng.standard_normal((n, H * hd)).astype(np.float32))
    cu = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    dq_, dk_, dv_, do_ = cu(q), cu(kr), cu(vr), cu(dout)
    o = torch.zeros((n, H * hd), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    assert lib.ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), n, None) == 0
    dsum = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    g = torch.full((n, (H + 2 * Hkv) * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.ttt_kernel_attn_bwd_noalloc(n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                         o.data_ptr(), lse.data_ptr(), n, do_.data_ptr(), dsum.data_ptr(),
                                         g.data_ptr(), None)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    got = g.float().cpu().numpy().astype(np.float64)
    rq, rk, rv = ref_backward(q, kr, vr, dout, n, H, Hkv, hd, W, pos0)
    for name, a, b in (("dq", got[:, :H * hd], rq), ("dk", got[:, H * hd:(H + Hkv) * hd], rk),
                       ("dv", got[:, (H + Hkv) * hd:], rv)):
        err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-6)
        assert err < 2e-2, (name, err)

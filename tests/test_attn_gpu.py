"""Unit tests of the sliding-window attention kernels through the kernel-level
C entry points (include/ttt_kernels.h): the tensor-core kernels (impl 0) and
the SIMT ones (impl 1) against a float64 restatement of banded causal
attention on the CPU, on bf16 inputs.

The restatement: query t sees keys j with t - W < j <= t, key j read from
ring slot j mod R of KV head h // (H / Hkv); o = softmax(q k^T / sqrt(hd)) v,
lse = log-sum-exp of the scaled scores.  Backward: dq over the whole window,
dk / dv for the chunk's own keys only (earlier keys are constants), summed
over the query heads that share a KV head.
"""
import math

import numpy as np
import pytest

from long_context_lm_ttt_b300 import inputs

pytestmark = pytest.mark.gpu


def _env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_lm_ttt_b300 import ttt as T
    T.load()
    return torch, T


def make_case(n, H, Hkv, hd, W, pos0, R, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    bf = lambda a: inputs.round_bf16(a.astype(np.float32))
    q = bf(rng.standard_normal((n, H * hd)) * scale)
    kr = bf(rng.standard_normal((Hkv, R, hd)) * scale)
    vr = bf(rng.standard_normal((Hkv, R, hd)))
    return q, kr, vr


def ref_forward(q, kr, vr, n, H, Hkv, hd, W, pos0, rows=None):
    R = kr.shape[1]
    g = H // Hkv
    rows = range(n) if rows is None else rows
    o = {}
    lse = {}
    for r in rows:
        t = pos0 + r
        js = np.arange(max(0, t - W + 1), t + 1)
        slots = js % R
        for h in range(H):
            qv = q[r, h * hd:(h + 1) * hd].astype(np.float64)
            K = kr[h // g, slots].astype(np.float64)
            V = vr[h // g, slots].astype(np.float64)
            s = K @ qv / math.sqrt(hd)
            m = s.max()
            e = np.exp(s - m)
            o[(r, h)] = (e / e.sum()) @ V
            lse[(r, h)] = m + math.log(e.sum())
    return o, lse


def run_fwd(T, torch, impl, q, kr, vr, n, H, Hkv, hd, W, pos0):
    R = kr.shape[1]
    cu = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    dq, dk, dv = cu(q), cu(kr), cu(vr)
    o = torch.full((n, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, n), float("nan"), dtype=torch.float32, device="cuda")
    rc = T.load().ttt_kernel_attn_fwd(impl, n, H, Hkv, hd, W, R, pos0, dq.data_ptr(), dk.data_ptr(),
                                      dv.data_ptr(), o.data_ptr(), lse.data_ptr(), n, None)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


FWD_CASES = [
    # n, H, Hkv, hd, W, pos0, R
    (128, 2, 1, 64, 64, 0, 256),          # first chunk, W < tile
    (200, 4, 2, 64, 1000, 0, 1280),       # ragged tile, window covers all
    (256, 6, 2, 96, 300, 1024, 640),      # hd 96, GQA 3, ring wraps
    (130, 3, 3, 128, 77, 4096 + 64, 256), # odd window, tile of 2 rows
    (512, 4, 1, 128, 2048, 5000, 2560),   # unaligned pos0
]


@pytest.mark.parametrize("case", FWD_CASES)
@pytest.mark.parametrize("impl", [0, 1, 2, 3])
def test_attn_fwd(case, impl):
    """impl 0: tensor cores (variant by size), 1: SIMT, 2: tensor cores with
    one query tile per CTA, 3: two tiles per CTA with P in tensor memory."""
    torch, T = _env()
    n, H, Hkv, hd, W, pos0, R = case
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=n + hd)
    o, lse = run_fwd(T, torch, impl, q, kr, vr, n, H, Hkv, hd, W, pos0)
    ro, rl = ref_forward(q, kr, vr, n, H, Hkv, hd, W, pos0)
    err_o = max(np.abs(o[r, h * hd:(h + 1) * hd] - v).max() for (r, h), v in ro.items())
    err_l = max(abs(lse[h, r] - v) for (r, h), v in rl.items())
    assert err_o < 2e-2, err_o
    assert err_l < 2e-3, err_l


DECODE_CASES = [
    # H, Hkv, hd, W, pos0, R: one query position
    (24, 8, 128, 8192, 40 * 1024 + 17, 9216),  # 3B heads deep in the sequence, ring wraps
    (24, 8, 128, 8192, 5, 9216),               # fewer keys than one slice
    (4, 4, 32, 64, 300, 128),                  # hd 32, one query head per KV head
    (6, 2, 96, 300, 1024, 640),                # hd 96, GQA 3
    (16, 2, 64, 1000, 999, 1024),              # GQA 8, window covers everything
    (10, 2, 160, 500, 2000, 512),              # hd 160 (odd dims per lane), ring wraps
    (8, 2, 256, 4096, 5000, 4608),             # hd 256, GQA 4
]


@pytest.mark.parametrize("case", DECODE_CASES)
def test_attn_fwd_one_query(case):
    """impl 4: the decode step's one-query kernel (key range split over
    CTAs, slices folded) against the restatement."""
    torch, T = _env()
    H, Hkv, hd, W, pos0, R = case
    q, kr, vr = make_case(1, H, Hkv, hd, W, pos0, R, seed=hd + H)
    o, lse = run_fwd(T, torch, 4, q, kr, vr, 1, H, Hkv, hd, W, pos0)
    ro, rl = ref_forward(q, kr, vr, 1, H, Hkv, hd, W, pos0)
    err_o = max(np.abs(o[r, h * hd:(h + 1) * hd] - v).max() for (r, h), v in ro.items())
    err_l = max(abs(lse[h, r] - v) for (r, h), v in rl.items())
    assert err_o < 2e-2, err_o
    assert err_l < 2e-3, err_l


def test_attn_fwd_one_query_repeated_calls():
    """The one-query kernel's last CTA per KV head folds the slices and
    resets that head's counter: back-to-back calls at other positions stay
    right, and a repeated call gives the same bits."""
    torch, T = _env()
    H, Hkv, hd, W, R = 24, 8, 128, 2048, 4096
    outs = []
    for pos0 in (3000, 3001, 100, 3000):
        q, kr, vr = make_case(1, H, Hkv, hd, W, pos0, R, seed=11)
        o, lse = run_fwd(T, torch, 4, q, kr, vr, 1, H, Hkv, hd, W, pos0)
        ro, rl = ref_forward(q, kr, vr, 1, H, Hkv, hd, W, pos0)
        err_o = max(np.abs(o[r, h * hd:(h + 1) * hd] - v).max() for (r, h), v in ro.items())
        assert err_o < 2e-2, (pos0, err_o)
        outs.append((o.copy(), lse.copy()))
    assert np.array_equal(outs[0][0], outs[3][0]) and np.array_equal(outs[0][1], outs[3][1])


@pytest.mark.parametrize("impl", [0, 2, 3])
def test_attn_fwd_3b_shape_sampled(impl):
    """3B head layout (24 q / 8 KV heads x 128) over a full 1024-row chunk
    deep in the sequence (window 8192 of a 9216-slot ring); sampled rows.
    impl 0 splits each tile pair's key range into parts there."""
    torch, T = _env()
    n, H, Hkv, hd, W, R = 1024, 24, 8, 128, 8192, 9216
    pos0 = 40 * 1024
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=7)
    o, lse = run_fwd(T, torch, impl, q, kr, vr, n, H, Hkv, hd, W, pos0)
    rows = [0, 1, 127, 128, 500, 777, 1023]
    ro, rl = ref_forward(q, kr, vr, n, H, Hkv, hd, W, pos0, rows=rows)
    err_o = max(np.abs(o[r, h * hd:(h + 1) * hd] - v).max() for (r, h), v in ro.items())
    err_l = max(abs(lse[h, r] - v) for (r, h), v in rl.items())
    assert err_o < 2e-2, err_o
    assert err_l < 2e-3, err_l
    assert np.isfinite(o).all()


@pytest.mark.parametrize("impl", [0, 3])
def test_attn_fwd_long_span_sampled(impl):
    """A 4096-row span of the 3B head layout one super-chunk into the
    sequence (window 8192), the shape of the frozen blocks' pass: sixteen
    tile pairs per head, 66 key blocks of 128 per pair, the ring wrapping
    inside the span; sampled rows."""
    torch, T = _env()
    n, H, Hkv, hd, W = 4096, 24, 8, 128, 8192
    R = 12288
    pos0 = 16384 + 512
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=17)
    o, lse = run_fwd(T, torch, impl, q, kr, vr, n, H, Hkv, hd, W, pos0)
    rows = [0, 63, 64, 255, 256, 2047, 3000, 4095]
    ro, rl = ref_forward(q, kr, vr, n, H, Hkv, hd, W, pos0, rows=rows)
    err_o = max(np.abs(o[r, h * hd:(h + 1) * hd] - v).max() for (r, h), v in ro.items())
    err_l = max(abs(lse[h, r] - v) for (r, h), v in rl.items())
    assert err_o < 2e-2, err_o
    assert err_l < 2e-3, err_l
    assert np.isfinite(o).all()


@pytest.mark.parametrize("impl", [0, 2, 3])
def test_attn_fwd_large_scores(impl):
    """Scores spread over a wide range exercise the lazy rescaling of the
    output accumulator (the running max grows by more than 2^8)."""
    torch, T = _env()
    n, H, Hkv, hd, W, pos0, R = 256, 2, 2, 64, 512, 256, 768
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=3, scale=3.0)
    # make later keys dominate so that the max keeps growing along the row
    ramp = np.linspace(0.2, 3.0, R, dtype=np.float32)[None, :, None]
    kr = inputs.round_bf16(kr * ramp)
    o, lse = run_fwd(T, torch, impl, q, kr, vr, n, H, Hkv, hd, W, pos0)
    ro, rl = ref_forward(q, kr, vr, n, H, Hkv, hd, W, pos0)
    err_o = max(np.abs(o[r, h * hd:(h + 1) * hd] - v).max() for (r, h), v in ro.items())
    err_l = max(abs(lse[h, r] - v) / max(1.0, abs(v)) for (r, h), v in rl.items())
    assert err_o < 3e-2, err_o
    assert err_l < 2e-3, err_l


def test_attn_tc_rejects_unsupported_head_dim():
    torch, T = _env()
    n, H, Hkv, hd, W, R = 32, 2, 2, 32, 32, 128
    z = torch.zeros((n * H * hd + Hkv * R * hd,), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    rc = T.load().ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, 0, z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                      z.data_ptr(), lse.data_ptr(), n, None)
    assert rc == T.TTT_ERR_SHAPE


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------
def ref_backward(q, kr, vr, dout, n, H, Hkv, hd, W, pos0):
    """dq over the window; dk, dv of keys pos0 .. pos0+n-1 (the chunk's own),
    summed over the query heads of each KV head."""
    R = kr.shape[1]
    g = H // Hkv
    dq = np.zeros((n, H * hd))
    dk = np.zeros((n, Hkv * hd))
    dv = np.zeros((n, Hkv * hd))
    for r in range(n):
        t = pos0 + r
        js = np.arange(max(0, t - W + 1), t + 1)
        slots = js % R
        own = js >= pos0
        for h in range(H):
            kv = h // g
            qv = q[r, h * hd:(h + 1) * hd].astype(np.float64)
            go = dout[r, h * hd:(h + 1) * hd].astype(np.float64)
            K = kr[kv, slots].astype(np.float64)
            V = vr[kv, slots].astype(np.float64)
            s = K @ qv / math.sqrt(hd)
            P = np.exp(s - s.max())
            P /= P.sum()
            o = P @ V
            dP = V @ go
            dS = P * (dP - go @ o) / math.sqrt(hd)
            dq[r, h * hd:(h + 1) * hd] = dS @ K
            jl = js[own] - pos0
            dk[jl, kv * hd:(kv + 1) * hd] += dS[own, None] * qv[None, :]
            dv[jl, kv * hd:(kv + 1) * hd] += P[own, None] * go[None, :]
    return dq, dk, dv


BWD_CASES = [
    # n, H, Hkv, hd, W, pos0, R
    (128, 2, 1, 64, 64, 0, 256),
    (200, 4, 2, 64, 1000, 0, 1280),
    (256, 6, 2, 96, 300, 1024, 640),
    (192, 3, 3, 128, 77, 4096, 384),
    (256, 4, 1, 128, 1024, 2048, 1280),
]


@pytest.mark.parametrize("case", BWD_CASES)
@pytest.mark.parametrize("impl", [0, 1])
def test_attn_bwd(case, impl):
    torch, T = _env()
    n, H, Hkv, hd, W, pos0, R = case
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=2 * n + hd)
    rng = np.random.default_rng(n)
    dout = inputs.round_bf16(rng.standard_normal((n, H * hd)).astype(np.float32))
    cu = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    dq_, dk_, dv_, do_ = cu(q), cu(kr), cu(vr), cu(dout)
    o = torch.zeros((n, H * hd), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    lib = T.load()
    assert lib.ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), n, None) == 0
    dsum = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    g = torch.full((n, (H + 2 * Hkv) * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.ttt_kernel_attn_bwd(impl, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), n, do_.data_ptr(), dsum.data_ptr(), g.data_ptr(), None)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    got = g.float().cpu().numpy().astype(np.float64)
    rq, rk, rv = ref_backward(q, kr, vr, dout, n, H, Hkv, hd, W, pos0)
    for name, a, b in (("dq", got[:, :H * hd], rq), ("dk", got[:, H * hd:(H + Hkv) * hd], rk),
                       ("dv", got[:, (H + Hkv) * hd:], rv)):
        err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-6)
        assert err < 2e-2, (name, err)


def test_attn_bwd_deterministic():
    """Split key ranges are summed in a fixed order: identical runs agree
    bitwise."""
    torch, T = _env()
    n, H, Hkv, hd, W, pos0, R = 1024, 24, 8, 128, 8192, 16384, 9216
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=11)
    rng = np.random.default_rng(12)
    dout = inputs.round_bf16(rng.standard_normal((n, H * hd)).astype(np.float32))
    cu = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    dq_, dk_, dv_, do_ = cu(q), cu(kr), cu(vr), cu(dout)
    lib = T.load()
    o = torch.zeros((n, H * hd), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    assert lib.ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), n, None) == 0
    outs = []
    for _ in range(2):
        dsum = torch.zeros((H, n), dtype=torch.float32, device="cuda")
        g = torch.zeros((n, (H + 2 * Hkv) * hd), dtype=torch.bfloat16, device="cuda")
        assert lib.ttt_kernel_attn_bwd(0, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(),
                                       dv_.data_ptr(), o.data_ptr(), lse.data_ptr(), n, do_.data_ptr(),
                                       dsum.data_ptr(), g.data_ptr(), None) == 0
        torch.cuda.synchronize()
        outs.append(g.cpu())
    assert T.ttt_kernel_error() == 0
    assert torch.equal(outs[0], outs[1])
    assert torch.isfinite(outs[0].float()).all()


def ref_backward_heads(q, kr, vr, dout, n, H, Hkv, hd, W, pos0, kv_heads):
    """The backward restated with whole-chunk matrix products for the query
    heads of the given KV heads: {('dq', h): [n, hd], ('dk', kv): [n, hd],
    ('dv', kv): [n, hd]} (dk, dv of the chunk's own keys, summed over the
    KV head's query heads)."""
    R = kr.shape[1]
    g = H // Hkv
    js = np.arange(max(0, pos0 - W + 1), pos0 + n)
    slots = js % R
    t = pos0 + np.arange(n)
    rel = t[:, None] - js[None, :]
    allowed = (rel >= 0) & (rel < W)
    own = js >= pos0
    out = {}
    for kv in kv_heads:
        K = kr[kv, slots].astype(np.float64)
        V = vr[kv, slots].astype(np.float64)
        dk = np.zeros((n, hd))
        dv = np.zeros((n, hd))
        for h in range(kv * g, (kv + 1) * g):
            Q = q[:, h * hd:(h + 1) * hd].astype(np.float64)
            dO = dout[:, h * hd:(h + 1) * hd].astype(np.float64)
            S = np.where(allowed, Q @ K.T / math.sqrt(hd), -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            O = P @ V
            dS = P * (dO @ V.T - (dO * O).sum(axis=1, keepdims=True)) / math.sqrt(hd)
            out[("dq", h)] = dS @ K
            dk += dS[:, own].T @ Q
            dv += P[:, own].T @ dO
        out[("dk", kv)] = dk
        out[("dv", kv)] = dv
    return out


@pytest.mark.parametrize("pos0", [40 * 1024, 1024])
def test_attn_bwd_3b_shape_heads(pos0):
    """The backward at the 3B chunk shape (1024 rows, 24 q / 8 KV heads x
    128, window 8192 in a 9216-slot ring) as the inner loop runs it: deep in
    the sequence the dq kernel splits the window's key blocks into parts
    summed in a fixed order; near the start the window is still short.
    Every row of two KV groups (KV heads 0 and 7 with their 6 query heads)
    against the restatement in float64."""
    torch, T = _env()
    n, H, Hkv, hd, W, R = 1024, 24, 8, 128, 8192, 9216
    q, kr, vr = make_case(n, H, Hkv, hd, W, pos0, R, seed=5 + pos0 % 7)
    rng = np.random.default_rng(pos0)
    dout = inputs.round_bf16(rng.standard_normal((n, H * hd)).astype(np.float32))
    cu = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    dq_, dk_, dv_, do_ = cu(q), cu(kr), cu(vr), cu(dout)
    lib = T.load()
    o = torch.zeros((n, H * hd), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    assert lib.ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), n, None) == 0
    dsum = torch.zeros((H, n), dtype=torch.float32, device="cuda")
    g = torch.full((n, (H + 2 * Hkv) * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert lib.ttt_kernel_attn_bwd(0, n, H, Hkv, hd, W, R, pos0, dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), n, do_.data_ptr(), dsum.data_ptr(), g.data_ptr(),
                                   None) == 0
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    got = g.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    ref = ref_backward_heads(q, kr, vr, dout, n, H, Hkv, hd, W, pos0, kv_heads=(0, Hkv - 1))
    for (name, h), b in ref.items():
        if name == "dq":
            a = got[:, h * hd:(h + 1) * hd]
        elif name == "dk":
            a = got[:, (H + h) * hd:(H + h + 1) * hd]
        else:
            a = got[:, (H + Hkv + h) * hd:(H + Hkv + h + 1) * hd]
        err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-6)
        assert err < 2e-2, (name, h, err)

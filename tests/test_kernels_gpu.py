"""Unit tests of single CUDA kernels through the kernel-level C entry points
(include/ttt_kernels.h), against float64 products computed on the CPU."""
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


def _operand(rng, rows, cols, mn, bf16=True):
    """Logical [rows (M or N), cols (K)] operand and its storage."""
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    if bf16:
        x = inputs.round_bf16(x)
    store = np.ascontiguousarray(x.T) if mn else x      # mn: stored [K, rows]
    return x.astype(np.float64), store


SHAPES = [(128, 128, 64), (256, 384, 192), (100, 200, 96), (32, 128, 32), (130, 258, 70),
          (1024, 3072, 1024), (512, 512, 4096), (520, 640, 200), (300, 136, 1000),
          (1, 256, 200), (1, 3072, 3072),
          # one-row products: several K ranges per column pair (a ragged last
          # one), many pairs per SM, and a single pair
          (1, 16384, 3072), (1, 3072, 8192), (1, 258, 5000), (1, 2, 64),
          # 192-wide tiles with ragged edges (planner: pairs for a K-major B,
          # single CTAs otherwise)
          (1000, 3000, 200)]

# impl 0: tensor cores, planner's choice; 3: 128-row tiles on one CTA;
# 4: 256-row tiles on a CTA pair (also for M < 256: the second CTA's rows
# are all out of range); 1: SIMT


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("impl", [0, 1, 3, 4])
def test_gemm_bf16(M, N, K, a_mn, b_mn, impl):
    torch, T = _env()
    if impl == 1 and M * N * K > 2 ** 28:
        pytest.skip("SIMT reference only on the small shapes")
    rng = np.random.default_rng(M * 7 + N * 3 + K + 11 * a_mn + 5 * b_mn)
    a, a_st = _operand(rng, M, K, a_mn)
    b, b_st = _operand(rng, N, K, b_mn)
    ref = a @ b.T
    dA = torch.from_numpy(a_st).to(torch.bfloat16).cuda()
    dB = torch.from_numpy(b_st).to(torch.bfloat16).cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lda = M if a_mn else K
    ldb = N if b_mn else K
    if impl != 1 and (lda % 8 or ldb % 8):
        pytest.skip("TMA needs 16-byte row pitch")
    T.ttt_kernel_gemm(M, N, K, dA, lda, a_mn, dB, ldb, b_mn, None, C, N, impl)
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    got = C.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref).max() / np.abs(ref).max()
    # fp32 accumulation of exact bf16 products: the rounding error of a sum
    # grows with its number of terms (at most linearly, Higham's n u bound),
    # so the bound grows with K beyond 4096
    assert err < 1e-5 * max(1.0, K / 4096), err


@pytest.mark.parametrize("impl", [0, 1, 3, 4])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("M,K", [(200, 320), (1, 320), (1, 5000)])
def test_gemm_dual_b(impl, b_mn, M, K):
    """C = A B^T + A B2^T (the hi + lo fast-weight pair); M = 1 is the
    one-row product of a decode step (K 5000: several K ranges per pair)."""
    torch, T = _env()
    N = 384
    rng = np.random.default_rng(3)
    a, a_st = _operand(rng, M, K, 0)
    b, b_st = _operand(rng, N, K, b_mn)
    b2, b2_st = _operand(rng, N, K, b_mn)
    ref = a @ b.T + a @ b2.T
    cu = lambda x: torch.from_numpy(x).to(torch.bfloat16).cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    T.ttt_kernel_gemm(M, N, K, cu(a_st), K, 0, cu(b_st), N if b_mn else K, b_mn, cu(b2_st), C, N, impl)
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    err = np.abs(C.cpu().numpy() - ref).max() / np.abs(ref).max()
    # 2 K products per output: the fp32 summation bound grows with them
    assert err < 1e-5 * max(1.0, 2 * K / 4096), err


def test_gemm_fp32_simt():
    torch, T = _env()
    M, N, K = 70, 130, 50
    rng = np.random.default_rng(4)
    a = rng.standard_normal((M, K)).astype(np.float32)
    b = rng.standard_normal((K, N)).astype(np.float32)      # MN-major B
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    T.ttt_kernel_gemm(M, N, K, torch.from_numpy(a).cuda(), K, 0, torch.from_numpy(b).cuda(), N, 1, None,
                      C, N, 2)
    torch.cuda.synchronize()
    ref = a.astype(np.float64) @ b.astype(np.float64)
    assert np.abs(C.cpu().numpy() - ref).max() / np.abs(ref).max() < 1e-5


@pytest.mark.parametrize("M,N,K", [(3072, 8192, 1024), (16384, 3072, 1024), (200, 96, 40), (256, 384, 512),
                                   (392, 160, 72)])
@pytest.mark.parametrize("impl", [0, 1, 2, 3])
def test_gemm_sgd(M, N, K, impl):
    """Weight gradient + fused SGD step: w32 -= lr A^T B (both operands stored
    [K, M] / [K, N], as the chunk's activations are), then the bf16 pair
    hi = rn(w32), lo = rn(w32 - hi).  impl 0 tensor cores (planner), 2 one
    CTA per tile, 3 CTA pairs, 1 SIMT."""
    torch, T = _env()
    if impl == 1 and M * N * K > 2 ** 30:
        pytest.skip("SIMT reference only on the small shapes")
    rng = np.random.default_rng(M + N + K + impl)
    a, a_st = _operand(rng, M, K, 1)
    b, b_st = _operand(rng, N, K, 1)
    w0 = (rng.standard_normal((M, N)) * 0.02).astype(np.float32)
    lr = 1e-3
    cu = lambda x: torch.from_numpy(x).to(torch.bfloat16).cuda()
    w32 = torch.from_numpy(w0).cuda()
    hi = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    lo = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    T.ttt_kernel_gemm_sgd(M, N, K, cu(a_st), M, 1, cu(b_st), N, 1, w32, hi, lo, N, lr, impl)
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    ref = w0.astype(np.float64) - lr * (a @ b.T)
    got = w32.cpu().numpy().astype(np.float64)
    upd = np.abs(lr * (a @ b.T)).max()
    assert np.abs(got - ref).max() <= 1e-5 * upd + 2e-9, np.abs(got - ref).max()
    g32 = w32.cpu()
    assert torch.equal(hi.cpu(), g32.to(torch.bfloat16))
    assert torch.equal(lo.cpu(), (g32 - g32.to(torch.bfloat16).float()).to(torch.bfloat16))


@pytest.mark.parametrize("impl", [0, 2, 3])
def test_gemm_sgd_without_low_half(impl):
    """The SGD step with one bf16 copy (no low half), the forward read the
    inner loop uses by default: w32 as above, w16 = rn(w32) exactly."""
    torch, T = _env()
    M, N, K = 3072, 8192, 1024
    rng = np.random.default_rng(17 + impl)
    a, a_st = _operand(rng, M, K, 1)
    b, b_st = _operand(rng, N, K, 1)
    w0 = (rng.standard_normal((M, N)) * 0.02).astype(np.float32)
    lr = 1e-3
    cu = lambda x: torch.from_numpy(x).to(torch.bfloat16).cuda()
    w32 = torch.from_numpy(w0).cuda()
    hi = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    T.ttt_kernel_gemm_sgd(M, N, K, cu(a_st), M, 1, cu(b_st), N, 1, w32, hi, None, N, lr, impl)
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    ref = w0.astype(np.float64) - lr * (a @ b.T)
    got = w32.cpu().numpy().astype(np.float64)
    upd = np.abs(lr * (a @ b.T)).max()
    assert np.abs(got - ref).max() <= 1e-5 * upd + 2e-9, np.abs(got - ref).max()
    assert torch.equal(hi.cpu(), w32.cpu().to(torch.bfloat16))



@pytest.mark.parametrize("groups,R,N,K", [(3, 1024, 3072, 512), (2, 128, 640, 256), (3, 96, 384, 128)])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("dual", [False, True])
@pytest.mark.parametrize("impl", [0, 3, 4, 1])
def test_gemm_grouped(groups, R, N, K, b_mn, dual, impl):
    """Grouped product: group g's rows against its own B (and B2).  R =
    1024 runs every group in one launch on CTA pairs, R = 128 in one launch
    on single CTAs (a pair tile would straddle two groups), R = 96 one
    launch per group."""
    torch, T = _env()
    if impl == 1 and groups * R * N * K > 2 ** 30:
        pytest.skip("SIMT reference only on the small shapes")
    rng = np.random.default_rng(groups * 1000 + R + N + K + 7 * b_mn + 3 * dual + impl)
    a, a_st = _operand(rng, groups * R, K, 0)
    bs = [_operand(rng, N, K, b_mn) for _ in range(groups)]
    b2s = [_operand(rng, N, K, b_mn) for _ in range(groups)] if dual else None
    stride = N * K
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).cuda()
    B = cu(np.stack([st for _, st in bs]))
    B2 = cu(np.stack([st for _, st in b2s])) if dual else None
    C = torch.full((groups * R, N), float("nan"), dtype=torch.float32, device="cuda")
    ldb = N if b_mn else K
    T.ttt_kernel_gemm_grouped(groups, R, N, K, cu(a_st), K, B, ldb, b_mn, stride, B2, C, N, impl)
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0
    got = C.cpu().numpy().astype(np.float64)
    for g in range(groups):
        ref = a[g * R:(g + 1) * R] @ bs[g][0].T
        if dual:
            ref = ref + a[g * R:(g + 1) * R] @ b2s[g][0].T
        err = np.abs(got[g * R:(g + 1) * R] - ref).max() / np.abs(ref).max()
        assert err < 1e-5, (g, err)

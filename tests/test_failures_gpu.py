"""Failure handling of the C ABI on the GPU, with no fault, trap or hang:
non-finite values, bad token ids, bad sizes and call order are reported as
error codes, and a device-side wait that can never complete gives up after
its budget and reports instead of hanging.  The context stays usable."""
import numpy as np
import pytest

from long_context_lm_ttt_b300 import inputs

pytestmark = pytest.mark.gpu


def _T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_lm_ttt_b300 import ttt as T
    T.load()
    return torch, T


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_nonfinite_weight_reports_chunk(precision):
    torch, T = _T()
    s = inputs.shape("tiny-ttt2", bf16=precision == "bf16")
    w = inputs.make_weights(s)
    w["lm_head"][5, 3] = np.nan
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    m = T.TTT(s, w, prec, max_tokens=s.seq_len)
    try:
        with pytest.raises(T.TTTError) as ei:
            m.prefill(inputs.make_tokens(s))
        assert ei.value.code == T.TTT_ERR_NONFINITE
        assert "chunk 0" in str(ei.value)
        # the context is still usable after a reset
        m.reset()
    finally:
        m.close()


def test_bad_token_size_and_order():
    torch, T = _T()
    s = inputs.shape("tiny-ttt2", bf16=True)
    w = inputs.make_weights(s)
    m = T.TTT(s, w, T.TTT_BF16, max_tokens=64)
    try:
        bad = np.zeros(64, np.int32)
        bad[10] = s.vocab + 3
        with pytest.raises(T.TTTError) as ei:
            m.prefill(bad)
        assert ei.value.code == T.TTT_ERR_INVALID
        m.reset()
        with pytest.raises(T.TTTError) as ei:
            m.prefill(np.zeros(65, np.int32))          # longer than max_tokens
        assert ei.value.code == T.TTT_ERR_SHAPE
        tok = inputs.make_tokens(s, 64)
        m.prefill(tok)
        with pytest.raises(T.TTTError) as ei:           # prefill twice without reset
            m.prefill(tok)
        assert ei.value.code == T.TTT_ERR_STATE
        m.reset()
        losses = m.prefill(tok)                         # usable again
        assert np.isfinite(losses).all()
    finally:
        m.close()


def test_bounded_wait_gives_up_and_reports():
    """A wait on an mbarrier nothing completes: ~5 ms of clocks, then the
    kernel records code 199 and returns; the device keeps working."""
    torch, T = _T()
    lib = T.load()
    assert T.ttt_kernel_error() == 0
    assert lib.ttt_kernel_wait_selftest(10_000_000, None) == 0
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 199
    assert T.ttt_kernel_error() == 0                   # read clears it
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0

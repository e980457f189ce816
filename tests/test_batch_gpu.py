"""Several sequences in one call (ttt_prefill_batch): every context keeps its
own fast weights and ring, the contexts run concurrently on their own
streams, and each result is bitwise the one ttt_prefill gives alone."""
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


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_batch_equals_one_at_a_time(precision):
    torch, T = _env()
    s = inputs.shape("tiny-ttt2", bf16=precision == "bf16")
    w = inputs.make_weights(s)
    prec = T.TTT_FP32_CHECK if precision == "fp32" else T.TTT_BF16
    lens = [256, 200, 97]
    toks = [np.ascontiguousarray(inputs.make_tokens(s, L, seed=1 + i), np.int32) for i, L in enumerate(lens)]
    models = [T.TTT(s, w, prec, max_tokens=256) for _ in lens]
    try:
        streams = [torch.cuda.Stream() for _ in lens]
        losses = [np.zeros(m.n_chunks(L), np.float32) for m, L in zip(models, lens)]
        T.ttt_prefill_batch([m.ctx for m in models], toks, lens, losses, streams)
        fast = [[m.fast_weights(i) for i in range(s.n_ttt_layers)] for m in models]
        for m, tk, lb, fb in zip(models, toks, losses, fast):
            m.reset()
            la = m.prefill(tk)
            assert np.array_equal(la, lb)
            for i in range(s.n_ttt_layers):
                for k, v in m.fast_weights(i).items():
                    assert np.array_equal(v, fb[i][k])
    finally:
        for m in models:
            m.close()


def test_batch_reports_a_bad_sequence_and_finishes_the_others():
    torch, T = _env()
    s = inputs.shape("tiny-ttt2")
    w = inputs.make_weights(s)
    good = np.ascontiguousarray(inputs.make_tokens(s, 256, seed=3), np.int32)
    bad = good.copy()
    bad[17] = s.vocab  # out of range
    models = [T.TTT(s, w, T.TTT_FP32_CHECK, max_tokens=256) for _ in range(2)]
    try:
        losses = [np.zeros(8, np.float32), np.zeros(8, np.float32)]
        with pytest.raises(T.TTTError) as e:
            T.ttt_prefill_batch([m.ctx for m in models], [good, bad], [256, 256], losses,
                                [torch.cuda.Stream(), torch.cuda.Stream()])
        assert e.value.code == T.TTT_ERR_INVALID
        ref = T.TTT(s, w, T.TTT_FP32_CHECK, max_tokens=256)
        try:
            assert np.array_equal(ref.prefill(good), losses[0])
        finally:
            ref.close()
        # the same context twice is refused before anything runs
        with pytest.raises(T.TTTError):
            T.ttt_prefill_batch([models[0].ctx, models[0].ctx], [good, good], [256, 256], losses)
    finally:
        for m in models:
            m.close()

"""The seeded input recipe (CPU): the dual-MLP tensors are drawn after every
other tensor, so turning the option on leaves the shared weights unchanged;
the FLOP model counts the static second MLP once forward and once through
its input gradient."""
import numpy as np

from long_context_lm_ttt_b300 import inputs


def test_dual_mlp_adds_tensors_without_changing_others():
    s = inputs.shape("tiny-gqa")
    sd = s.replace(dual_mlp=True)
    w, wd = inputs.make_weights(s), inputs.make_weights(sd)
    for k in ("tok_embed", "final_norm", "lm_head"):
        assert np.array_equal(w[k], wd[k])
    L, Lt = s.n_layers, s.n_ttt_layers
    for l in range(L):
        for k, v in w["layers"][l].items():
            assert np.array_equal(v, wd["layers"][l][k])
        extra = set(wd["layers"][l]) - set(w["layers"][l])
        assert extra == (set(inputs.LAYER2_TENSORS) if l >= L - Lt else set())
    lw = wd["layers"][L - 1]
    assert lw["w_gate2"].shape == (s.d_ff, s.d_model) and lw["w_down2"].shape == (s.d_model, s.d_ff)
    assert np.all(lw["mlp2_norm"] == 1.0)
    assert not np.array_equal(lw["w_gate2"], lw["w_gate"])


def test_dual_mlp_flop_model():
    s = inputs.shape("3b")
    a = inputs.flops_per_sequence(s)
    b = inputs.flops_per_sequence(s.replace(dual_mlp=True))
    extra = 2.0 * 3 * s.d_model * s.d_ff * s.n_ttt_layers * s.seq_len
    assert np.isclose(b["fwd"] - a["fwd"], extra)
    assert np.isclose(b["bwd"] - a["bwd"], extra)

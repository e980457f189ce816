"""Writes oracle_tiny_losses.json: chunk losses of the tiny shapes, computed
by the CPU oracle alone.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from long_context_lm_ttt_b300 import inputs  # noqa: E402  (seeded inputs only)
from oracle import ttt_ref as O  # noqa: E402


def main():
    out = {"_note": "oracle chunk losses (float64) on the seeded tiny shapes", "losses": {}}
    for name in ("tiny", "tiny-ttt2", "tiny-gqa"):
        s = inputs.shape(name)
        cfg = O.OracleConfig.from_mapping(s.as_dict())
        r = O.prefill(cfg, inputs.make_weights(s), inputs.make_tokens(s))
        out["losses"][name] = [float(v) for v in r["losses"]]
    with open(os.path.join(HERE, "oracle_tiny_losses.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()

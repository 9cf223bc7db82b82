"""Writes conv_adversarial.txt: conv weight rows (four fp32 taps, hex floats)
for a conv fed with inputs of 1.0, chosen where a conv + SiLU code is hard to
decide.  Inputs only: the expected codes come from the oracle, which the CPU
pins check against an arbitrary-precision evaluation of the same rows.

  near   SiLU of the tap sum placed 2^-45 .. 2^-30 (relative) from a bf16
         rounding boundary, the sum split into four fp32 pieces;
  tie    a single tap 3 v 2^k (65 .. 16 000) exactly on a bf16 midpoint,
         where double precision cannot tell SiLU(y) from y;
  large  four random taps summing to |y| beyond 87 (where e^-|y| leaves the
         fp32 range), either sign.

Run from the repository root: python tests/golden/make_conv_adversarial.py
(needs mpmath)."""
from __future__ import annotations

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
from test_oracle_pins import _large_midpoint_sums, _near_boundary_inputs  # noqa: E402


def main() -> None:
    rows = []
    w, x, _, _ = _near_boundary_inputs(400, seed=41)
    rows += [("near", r) for r in w * x]
    w, x, _, _ = _large_midpoint_sums(seed=43)
    rows += [("tie", r) for r in w * x]
    rng = np.random.default_rng(47)
    for _ in range(120):
        y = rng.uniform(87.5, 400.0) * rng.choice([-1.0, 1.0])
        parts = rng.dirichlet(np.ones(4)) * y
        rows += [("large", parts.astype(np.float32).astype(np.float64))]
    with open(os.path.join(HERE, "conv_adversarial.txt"), "w") as f:
        f.write("# Conv weight rows for inputs of 1.0 (tap sum = row sum), written by\n"
                "# make_conv_adversarial.py; the code of each row is SiLU of the exact sum,\n"
                "# correctly rounded to bf16 ([state] \"vllm.models.kimi_k3.nvidia.specialized_decode.\n"
                "# recoverssm.state\", deferred_recoverssm_verify: causal_conv1d_update(..., activation=\"silu\")).\n"
                "# kind  w0 w1 w2 w3 (fp32 values as hex floats)\n")
        for kind, r in rows:
            f.write(kind + " " + " ".join(float(np.float32(v)).hex() for v in r) + "\n")


if __name__ == "__main__":
    main()

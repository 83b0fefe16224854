"""Writes s80_layer_seed.json: the first seed whose 80B-shaped router logits (oracle, double) have a
top-10 margin (10th minus 11th largest logit) above 1e-2, as the single-layer 80B workload asks.
Calls only the oracle and the input generator."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402
from int4_routed_expert_05_b300 import synth  # noqa: E402

sh = synth.S80
for seed in range(1000):
    lg, _ = oracle.router_logits(synth.router_bits(sh, seed, 0), synth.activation_bits(sh, seed, 0)[0])
    s = np.sort(lg)[::-1]
    margin = float(s[sh.top_k - 1] - s[sh.top_k])
    if margin > 1e-2:
        break
out = {"source": "seed search over synth seeds 0.. with the oracle's double router logits; accept the first "
                  "seed whose top-10 margin exceeds 1e-2 (80B-shaped single layer workload)",
       "seed": seed, "margin": margin}
json.dump(out, open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "s80_layer_seed.json"), "w"), indent=1)
print(out)

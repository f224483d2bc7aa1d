"""Writes tests/golden/oracle_small_case.json from the oracle alone (no GPU code involved).

The fixture freezes the oracle's output on one small seeded case so that any later change to
the oracle's arithmetic shows up as a failing test and has to be justified.  Run from the
repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_ssm_gb300.synth import Geometry, prefill_inputs  # noqa: E402

GEO = Geometry(num_k_heads=2, num_v_heads=6, head_k_dim=8, head_v_dim=4, conv_width=4)
LENGTHS = [3, 70]
SEED = 42


def compute():
    inp = prefill_inputs(LENGTHS, seed=SEED, geo=GEO, random_conv_state=True)
    r = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                       inp["norm_w"], GEO.num_k_heads, GEO.num_v_heads, GEO.head_k_dim,
                       GEO.head_v_dim, GEO.q_scale, 1e-6, 1e-6, state_in=inp["state0"],
                       conv_state_in=inp["conv_state0"])
    return {
        "geometry": [GEO.num_k_heads, GEO.num_v_heads, GEO.head_k_dim, GEO.head_v_dim, GEO.conv_width],
        "lengths": LENGTHS, "seed": SEED, "q_scale": GEO.q_scale, "l2_eps": 1e-6, "rms_eps": 1e-6,
        "out_rows": {f"{t},{h}": r["out"][t, h].tolist() for t, h in [(0, 0), (2, 5), (3, 1), (66, 2), (72, 4)]},
        "o_rows": {f"{t},{h}": r["o"][t, h].tolist() for t, h in [(1, 3), (67, 0)]},
        "state_seq1_head5": r["state"][1, 5].reshape(-1).tolist(),
        "conv_state_seq0_ch0": r["conv_state"][0, 0].float().tolist(),
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_case.json")
    with open(out, "w") as f:
        json.dump(compute(), f, indent=1)
    print("wrote", out)

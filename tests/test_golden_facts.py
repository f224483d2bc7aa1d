"""The geometry, chunking and tolerance facts the pages print (tests/golden/pages_facts.txt),
checked against the synthetic workload definition and the oracle (CPU only)."""
import json
import os

import torch

import oracle
from linear_attention_ssm_gb300.synth import QWEN_GDN, Geometry, prefill_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def facts():
    out = {}
    with open(os.path.join(HERE, "golden", "pages_facts.txt")) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = v
    return out


def test_workload_geometry_matches_pages():
    F = facts()
    assert QWEN_GDN.num_k_heads == int(F["num_k_heads"])
    assert QWEN_GDN.num_v_heads == int(F["num_v_heads"])
    assert QWEN_GDN.head_k_dim == QWEN_GDN.head_v_dim == int(F["head_dim"])
    assert QWEN_GDN.num_v_heads // QWEN_GDN.num_k_heads == int(F["v_per_k_head"])
    assert QWEN_GDN.conv_width == int(F["conv_width"])
    assert F["output_gate"] == "sigmoid"
    assert float(F["rms_norm_eps"]) == 1e-6
    assert F["state_layout"] == "value,key"


def test_chunk_counts_match_pages():
    F = facts()
    chunk = 64
    for S in (16, 64, 80, 128):
        assert (S + chunk - 1) // chunk == int(F[f"chunks_S{S}"])


def test_oracle_reproduces_frozen_small_case():
    with open(os.path.join(HERE, "golden", "oracle_small_case.json")) as f:
        gold = json.load(f)
    hk, hv, dk, dv, W = gold["geometry"]
    geo = Geometry(hk, hv, dk, dv, W)
    inp = prefill_inputs(gold["lengths"], seed=gold["seed"], geo=geo, random_conv_state=True)
    r = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                       inp["norm_w"], hk, hv, dk, dv, gold["q_scale"], gold["l2_eps"], gold["rms_eps"],
                       state_in=inp["state0"], conv_state_in=inp["conv_state0"])
    for key, row in gold["out_rows"].items():
        t, h = map(int, key.split(","))
        assert torch.allclose(r["out"][t, h], torch.tensor(row, dtype=torch.float64), rtol=1e-12, atol=1e-14)
    for key, row in gold["o_rows"].items():
        t, h = map(int, key.split(","))
        assert torch.allclose(r["o"][t, h], torch.tensor(row, dtype=torch.float64), rtol=1e-12, atol=1e-14)
    st = torch.tensor(gold["state_seq1_head5"], dtype=torch.float64)
    assert torch.allclose(r["state"][1, 5].reshape(-1), st, rtol=1e-12, atol=1e-14)
    assert r["conv_state"][0, 0].float().tolist() == gold["conv_state_seq0_ch0"]

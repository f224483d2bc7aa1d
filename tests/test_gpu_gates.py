"""GPU parity of the gate derivation (g, beta from the a / b projections, A_log, dt_bias) against
the oracle's (parity unpinned against the pages, which give no formula), alone and feeding the
chunk prefill."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import gate_inputs, prefill_inputs
from tests.gpu_common import DEV, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu
A = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128)


@pytest.mark.parametrize("rows", [1, 257, 4096])
def test_gates_match_oracle(rows):
    g = lib()
    gi = gate_inputs(rows, seed=80 + rows)
    gg, bb = g.gdn_gates(gi["a"].to(DEV), gi["b"].to(DEV), gi["A_log"].to(DEV), gi["dt_bias"].to(DEV))
    g.gdn_check_device_errors()
    want_g, want_b = oracle.gates(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"])
    # fp32 evaluation of exp, log1p and the division: a few ulps
    assert torch.allclose(gg.cpu().double(), want_g, rtol=2e-6, atol=1e-30)
    assert torch.allclose(bb.cpu().double(), want_b, rtol=2e-6, atol=1e-30)
    assert (gg <= 0).all()


def test_prefill_from_gate_projections():
    """gdn_gates feeding the whole prefill equals the oracle prefill fed the oracle's gates."""
    g = lib()
    lengths = [150, 70]
    inp = prefill_inputs(lengths, seed=81)
    T = sum(lengths)
    gi = gate_inputs(T, seed=82)
    gg, bb = g.gdn_gates(gi["a"].to(DEV), gi["b"].to(DEV), gi["A_log"].to(DEV), gi["dt_bias"].to(DEV))
    st = inp["state0"].to(DEV).clone()
    out = g.gdn_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), inp["cu_seqlens"].to(DEV), gg, bb,
                        inp["z"].to(DEV), inp["norm_w"].to(DEV), inp["q_scale"], state_in=st, state_out=st)
    g.gdn_check_device_errors()
    og, ob = oracle.gates(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"])
    ref = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], og.float(), ob.float(), inp["z"],
                         inp["norm_w"], q_scale=inp["q_scale"], state_in=inp["state0"], **A)
    assert_out_close(out.cpu(), ref["out"])
    for n in range(len(lengths)):
        assert_state_close(st[n].cpu(), ref["state"][n], f"state of sequence {n}")


def test_gates_head_count_not_a_multiple_of_eight():
    """6 V heads: the element-at-a-time path."""
    from linear_attention_ssm_gb300.synth import Geometry
    g = lib()
    geo = Geometry(num_k_heads=2, num_v_heads=6)
    gi = gate_inputs(333, seed=83, geo=geo)
    gg, bb = g.gdn_gates(gi["a"].to(DEV), gi["b"].to(DEV), gi["A_log"].to(DEV), gi["dt_bias"].to(DEV), geometry=geo)
    g.gdn_check_device_errors()
    want_g, want_b = oracle.gates(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"])
    assert torch.allclose(gg.cpu().double(), want_g, rtol=2e-6, atol=1e-30)
    assert torch.allclose(bb.cpu().double(), want_b, rtol=2e-6, atol=1e-30)

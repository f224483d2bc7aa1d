"""GPU parity of the fused gate derivation: gdn_chunk_prefill_fused_gates and
gdn_decode_step_fused_gates derive g and beta inside the prefill's prep kernel (or the fused
kernel) and the decode kernel from the projections a, b and A_log, dt_bias.  Their results equal
gdn_gates followed by the plain call bit for bit (one device definition of the gate arithmetic),
and match the oracle fed the oracle's gates within the usual tolerances.  The gate formula itself
is parity unpinned against the pages (they name the inputs but give no formula)."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import Geometry, decode_inputs, gate_inputs, prefill_inputs
from tests.gpu_common import (DEV, assert_out_close, assert_state_close, chunk_mode,  # noqa: F401
                              lib)
from tests.test_gpu_chunk import run_oracle

pytestmark = pytest.mark.gpu
A = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128)


def _gates_dev(gi):
    return [gi[k].to(DEV) for k in ("a", "b", "A_log", "dt_bias")]


@pytest.mark.parametrize("lengths,geo", [([150, 64, 7], Geometry()), ([3000, 1, 1351], Geometry(2, 6))],
                         ids=["small", "segmented"])
def test_prefill_fused_gates(lengths, geo, mode):
    g = lib()
    inp = prefill_inputs(lengths, seed=90, geo=geo)
    T = sum(lengths)
    gi = gate_inputs(T, seed=91, geo=geo)
    og, ob = oracle.gates(gi["a"], gi["b"], gi["A_log"], gi["dt_bias"])
    inp_o = dict(inp, g=og.float(), beta=ob.float())
    heads = None if geo.num_v_heads <= 6 else [0, 17, 47]
    ref = run_oracle(inp_o, geo=geo, heads=heads)
    y = ref["y"].to(DEV)
    d = {k: inp[k].to(DEV) for k in ("cu_seqlens", "state0", "z", "norm_w")}
    a, b, A_log, dt_bias = _gates_dev(gi)
    st = torch.empty_like(d["state0"])
    out = g.gdn_chunk_prefill_fused_gates(y, a, b, A_log, dt_bias, d["cu_seqlens"], inp["q_scale"], 1e-6,
                                          d["state0"], st, d["z"], d["norm_w"], 1e-6, geometry=geo)
    g.gdn_check_device_errors()
    # the unfused route: the gates kernel, then the plain call
    gg, bb = g.gdn_gates(a, b, A_log, dt_bias, geometry=geo)
    st2 = torch.empty_like(d["state0"])
    out2 = g.gdn_chunk_prefill(y, gg, bb, d["cu_seqlens"], inp["q_scale"], 1e-6, d["state0"], st2, d["z"],
                               d["norm_w"], 1e-6, geometry=geo)
    g.gdn_check_device_errors()
    assert torch.equal(out, out2) and torch.equal(st, st2)
    for h in (heads or range(geo.num_v_heads)):
        assert_out_close(out[:, h], ref["out"][:, h], f"out, head {h}")
        for n in range(len(lengths)):
            assert_state_close(st[n, h], ref["state"][n, h], f"state of sequence {n}, head {h}")


def test_decode_fused_gates():
    g = lib()
    B, steps = 6, 4
    d = decode_inputs(B, steps, seed=92)
    gis = [gate_inputs(B, seed=93 + s) for s in range(steps)]
    dw, dnw = d["conv_w"].to(DEV), d["norm_w"].to(DEV)
    cs, st = d["conv_state0"].to(DEV).clone(), d["state0"].to(DEV).clone()
    cs2, st2 = cs.clone(), st.clone()
    cs_ref, st_ref = d["conv_state0"], d["state0"].double()
    for s in range(steps):
        a, b, A_log, dt_bias = _gates_dev(gis[s])
        out = g.gdn_decode_step_fused_gates(d["x"][s].to(DEV), dw, cs, a, b, A_log, dt_bias, st, d["z"][s].to(DEV),
                                            dnw, d["q_scale"])
        gg, bb = g.gdn_gates(a, b, A_log, dt_bias)
        out2 = g.gdn_decode_step(d["x"][s].to(DEV), dw, cs2, gg, bb, st2, d["z"][s].to(DEV), dnw, d["q_scale"])
        g.gdn_check_device_errors()
        assert torch.equal(out, out2) and torch.equal(st, st2) and torch.equal(cs, cs2)
        og, ob = oracle.gates(gis[s]["a"], gis[s]["b"], gis[s]["A_log"], gis[s]["dt_bias"])
        ref, _, cs_ref, st_ref = oracle.decode_step(d["x"][s], d["conv_w"], cs_ref, og.float(), ob.float(), st_ref,
                                                    d["z"][s], d["norm_w"], q_scale=d["q_scale"], **A)
        assert_out_close(out, ref, f"out of step {s}")
        assert_state_close(st, st_ref, f"state after step {s}")

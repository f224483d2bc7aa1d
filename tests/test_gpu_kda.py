"""GPU parity of the KDA decode step (per-channel decay) against the oracle: consecutive steps at
the 64-head geometry, the decay clamp, and agreement with the GDN step for a decay that is the
same on every key channel."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import KDA_GEO, QWEN_GDN, decode_inputs, kda_decode_inputs
from tests.gpu_common import DEV, Guarded, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu


def _a(geo):
    return dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
                head_v_dim=geo.head_v_dim)


@pytest.mark.parametrize("g_min", [float("-inf"), -0.5], ids=["no_clamp", "clamp"])
def test_kda_decode_steps_match_oracle(g_min):
    g = lib()
    geo = KDA_GEO
    B, steps = 3, 3
    d = kda_decode_inputs(B, steps, seed=90)
    cs, st = d["conv_state0"].to(DEV).clone(), d["state0"].to(DEV).clone()
    cs_ref, st_ref = d["conv_state0"], d["state0"].double()
    for s in range(steps):
        out = Guarded((B, geo.num_v_heads, 128), torch.bfloat16)
        g.gdn_kda_decode_step(d["x"][s].to(DEV), d["conv_w"].to(DEV), cs, d["g"][s].to(DEV), d["beta"][s].to(DEV),
                              st, d["z"][s].to(DEV), d["norm_w"].to(DEV), d["q_scale"], g_min, 1e-6, 1e-6, out.t,
                              geometry=geo)
        g.gdn_check_device_errors()
        out.check("out")
        ref, _, cs_ref, st_ref = oracle.kda_decode_step(d["x"][s], d["conv_w"], cs_ref, d["g"][s], d["beta"][s],
                                                        st_ref, d["z"][s], d["norm_w"], q_scale=d["q_scale"],
                                                        g_min=g_min, **_a(geo))
        assert_out_close(out.t, ref, f"out of step {s}")
        for b in range(B):
            assert_state_close(st[b], st_ref[b], f"state of sequence {b} after step {s}")
        assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_kda_with_a_channel_constant_decay_matches_the_gdn_step():
    """The per-channel kernel with every channel's decay equal to the head's agrees with the
    scalar-decay decode kernel (the delta rule's projection is summed in another order)."""
    g = lib()
    geo = QWEN_GDN
    B = 4
    d = decode_inputs(B, 1, seed=91)
    g_vec = d["g"][0][:, :, None].expand(B, geo.num_v_heads, geo.head_k_dim).contiguous()
    cs1, st1 = d["conv_state0"].to(DEV).clone(), d["state0"].to(DEV).clone()
    cs2, st2 = d["conv_state0"].to(DEV).clone(), d["state0"].to(DEV).clone()
    o1 = g.gdn_kda_decode_step(d["x"][0].to(DEV), d["conv_w"].to(DEV), cs1, g_vec.to(DEV), d["beta"][0].to(DEV),
                               st1, d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"])
    o2 = g.gdn_decode_step(d["x"][0].to(DEV), d["conv_w"].to(DEV), cs2, d["g"][0].to(DEV), d["beta"][0].to(DEV),
                           st2, d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"])
    g.gdn_check_device_errors()
    assert torch.equal(cs1, cs2)
    for b in range(B):
        assert_state_close(st1[b], st2[b].double(), f"state of sequence {b}", tol=1e-5)
    assert_out_close(o1, o2.double())

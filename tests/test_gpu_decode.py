"""GPU parity of the fused decode step against the oracle: consecutive steps, the one-token
prefill equivalence, in-place state updates, and the negative controls."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import QWEN_GDN, decode_inputs, cu_seqlens_of
from tests.gpu_common import (DEV, Guarded, NEG_CONTROL_RATIO, STATE_TOL_F16, assert_out_close, assert_state_close,
                              lib, out_error_ratio)

pytestmark = pytest.mark.gpu
GEO = QWEN_GDN
A = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128)


def test_decode_steps_match_oracle():
    g = lib()
    B, steps = 5, 6
    d = decode_inputs(B, steps, seed=21)
    cs = d["conv_state0"].to(DEV).clone()
    st = d["state0"].to(DEV).clone()
    cs_ref, st_ref = d["conv_state0"], d["state0"].double()
    for s in range(steps):
        out = Guarded((B, 48, 128), torch.bfloat16)
        g.gdn_decode_step(d["x"][s].to(DEV), d["conv_w"].to(DEV), cs, d["g"][s].to(DEV), d["beta"][s].to(DEV), st,
                          d["z"][s].to(DEV), d["norm_w"].to(DEV), d["q_scale"], 1e-6, 1e-6, out.t)
        g.gdn_check_device_errors()
        out.check("out")
        ref, _, cs_ref, st_ref = oracle.decode_step(d["x"][s], d["conv_w"], cs_ref, d["g"][s], d["beta"][s], st_ref,
                                                    d["z"][s], d["norm_w"], q_scale=d["q_scale"], **A)
        assert_out_close(out.t, ref, f"out of step {s}")
        assert_state_close(st, st_ref, f"state after step {s}")
        assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_decode_equals_one_token_prefill():
    """A decode step and a one-token prefill (conv with the same conv state, chunk prefill with
    the same recurrent state, fused gate) agree."""
    g = lib()
    B = 3
    d = decode_inputs(B, 1, seed=22)
    st_dec = d["state0"].to(DEV).clone()
    cs_dec = d["conv_state0"].to(DEV).clone()
    out_dec = g.gdn_decode_step(d["x"][0].to(DEV), d["conv_w"].to(DEV), cs_dec, d["g"][0].to(DEV),
                                d["beta"][0].to(DEV), st_dec, d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"])
    st_pre = d["state0"].to(DEV).clone()
    cs_pre = d["conv_state0"].to(DEV).clone()
    out_pre = g.gdn_prefill(d["x"][0].to(DEV), d["conv_w"].to(DEV), cu_seqlens_of([1] * B).to(DEV),
                            d["g"][0].to(DEV), d["beta"][0].to(DEV), d["z"][0].to(DEV), d["norm_w"].to(DEV),
                            d["q_scale"], state_in=st_pre, state_out=st_pre, conv_state_in=cs_pre,
                            conv_state_out=cs_pre)
    g.gdn_check_device_errors()
    assert_out_close(out_dec, out_pre.double())
    assert_state_close(st_dec, st_pre.double())
    assert torch.equal(cs_dec.cpu(), cs_pre.cpu())


@pytest.mark.parametrize("mutation", [oracle.MUT_SILU_GATE, oracle.MUT_CONV_SHIFT, oracle.MUT_TRANSPOSE,
                                      oracle.MUT_TILED_HEADS],
                         ids=["silu_gate", "conv_shift", "transposed_state", "tiled_heads"])
def test_decode_negative_controls(mutation):
    g = lib()
    B = 4
    d = decode_inputs(B, 1, seed=23)
    st = d["state0"].to(DEV).clone()
    cs = d["conv_state0"].to(DEV).clone()
    out = g.gdn_decode_step(d["x"][0].to(DEV), d["conv_w"].to(DEV), cs, d["g"][0].to(DEV), d["beta"][0].to(DEV),
                            st, d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"])
    args = (d["x"][0], d["conv_w"], d["conv_state0"], d["g"][0], d["beta"][0], d["state0"].double(), d["z"][0],
            d["norm_w"])
    ref = oracle.decode_step(*args, q_scale=d["q_scale"], **A)[0]
    bad = oracle.decode_step(*args, q_scale=d["q_scale"], mutation=mutation, **A)[0]
    assert out_error_ratio(out, ref) <= 1.0
    assert out_error_ratio(out, bad) > NEG_CONTROL_RATIO


# ------------------------------------------------------------------ fp16 (binary16) recurrent state

def _f16_quantum(v):
    """Spacing of binary16 values at |v| (2^-24 in the subnormal range)."""
    _, ex = torch.frexp(v.abs().double())
    return torch.exp2(torch.clamp(ex - 11, min=-24).double())


def test_fp16_state_one_step_is_within_one_rounding_of_the_oracle():
    """From the same binary16 state, one step stores every element either as the oracle's rounding
    of the exact value or as its neighbour (the fp32 arithmetic put the value on the other side of
    a rounding midpoint); such neighbours are rare."""
    g = lib()
    B = 6
    d = decode_inputs(B, 1, seed=24)
    h0 = d["state0"].to(torch.float16)
    st = h0.to(DEV).clone()
    cs = d["conv_state0"].to(DEV).clone()
    out = Guarded((B, 48, 128), torch.bfloat16)
    g.gdn_decode_step_fp16_state(d["x"][0].to(DEV), d["conv_w"].to(DEV), cs, d["g"][0].to(DEV),
                                 d["beta"][0].to(DEV), st, d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"],
                                 1e-6, 1e-6, out.t)
    g.gdn_check_device_errors()
    out.check("out")
    ref, _, cs_ref, st_ref = oracle.decode_step_h16(d["x"][0], d["conv_w"], d["conv_state0"], d["g"][0],
                                                    d["beta"][0], h0, d["z"][0], d["norm_w"], q_scale=d["q_scale"],
                                                    **A)
    assert_out_close(out.t, ref)
    got, want = st.cpu().double(), st_ref.double()
    assert torch.isfinite(got).all()
    diff = (got - want).abs()
    # one rounding, plus the fp32 error of the step's terms (2^-20 of the state's scale bounds it)
    # where cancellation leaves a value whose quantum is smaller than that error
    bound = _f16_quantum(want) + 2.0 ** -20 * want.abs().max()
    assert (diff <= bound).all(), "an element is more than one rounding away"
    assert (diff > 0).double().mean().item() < 1e-2
    assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_fp16_state_decode_steps_match_oracle():
    """Consecutive fp16-state steps: GPU chain against the oracle's binary16 chain."""
    g = lib()
    B, steps = 5, 6
    d = decode_inputs(B, steps, seed=25)
    st = d["state0"].to(torch.float16).to(DEV)
    cs = d["conv_state0"].to(DEV).clone()
    cs_ref, st_ref = d["conv_state0"], d["state0"].to(torch.float16)
    for s in range(steps):
        out = g.gdn_decode_step_fp16_state(d["x"][s].to(DEV), d["conv_w"].to(DEV), cs, d["g"][s].to(DEV),
                                           d["beta"][s].to(DEV), st, d["z"][s].to(DEV), d["norm_w"].to(DEV),
                                           d["q_scale"])
        g.gdn_check_device_errors()
        ref, _, cs_ref, st_ref = oracle.decode_step_h16(d["x"][s], d["conv_w"], cs_ref, d["g"][s], d["beta"][s],
                                                        st_ref, d["z"][s], d["norm_w"], q_scale=d["q_scale"], **A)
        assert_out_close(out, ref, f"out of step {s}")
        assert_state_close(st.double(), st_ref.double(), f"state after step {s}", tol=STATE_TOL_F16)
        assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_fp16_state_zero_gate_and_beta_keep_the_state_bits():
    """g = 0 and beta = 0: the step leaves every (nonzero) binary16 state pattern unchanged."""
    g = lib()
    B = 2
    d = decode_inputs(B, 1, seed=26)
    h0 = d["state0"].to(torch.float16)
    h0 = torch.where(h0 == 0, torch.full_like(h0, 0.25), h0)
    st = h0.to(DEV).clone()
    g.gdn_decode_step_fp16_state(d["x"][0].to(DEV), d["conv_w"].to(DEV), d["conv_state0"].to(DEV).clone(),
                                 torch.zeros_like(d["g"][0]).to(DEV), torch.zeros_like(d["beta"][0]).to(DEV), st,
                                 d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"])
    g.gdn_check_device_errors()
    assert torch.equal(st.cpu().view(torch.int16), h0.view(torch.int16))


def test_fp16_state_rejects_an_fp32_state():
    g = lib()
    d = decode_inputs(1, 1, seed=27)
    with pytest.raises(TypeError):
        g.gdn_decode_step_fp16_state(d["x"][0].to(DEV), d["conv_w"].to(DEV), d["conv_state0"].to(DEV),
                                     d["g"][0].to(DEV), d["beta"][0].to(DEV), d["state0"].to(DEV), d["z"][0].to(DEV),
                                     d["norm_w"].to(DEV), d["q_scale"])

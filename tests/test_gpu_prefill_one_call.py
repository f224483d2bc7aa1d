"""GPU tests of gdn_prefill, the one-call prefill sublayer (conv1d+SiLU, then the chunk-wise gated
delta rule with the gated norm): every result has the same bits as the two calls
gdn_conv1d_prefill and gdn_chunk_prefill in sequence, and matches the oracle."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import BATCHED_LENGTHS, Geometry, prefill_inputs
from tests.gpu_common import DEV, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu


def _both(g, inp, geo, in_place=False):
    d = {k: v.to(DEV) for k, v in inp.items() if torch.is_tensor(v)}
    # the two calls
    cs1 = torch.empty_like(d["conv_state0"])
    qkv1 = g.gdn_conv1d_prefill(d["x"], d["conv_w"], d["cu_seqlens"], d["conv_state0"], cs1, geometry=geo)
    st1 = torch.empty_like(d["state0"])
    out1 = g.gdn_chunk_prefill(qkv1, d["g"], d["beta"], d["cu_seqlens"], inp["q_scale"], 1e-6, d["state0"], st1,
                               d["z"], d["norm_w"], 1e-6, geometry=geo)
    # one call
    if in_place:
        st2, cs2 = d["state0"].clone(), d["conv_state0"].clone()
        s_in, c_in = st2, cs2
    else:
        st2, cs2 = torch.empty_like(d["state0"]), torch.empty_like(d["conv_state0"])
        s_in, c_in = d["state0"], d["conv_state0"]
    qkv2 = torch.full_like(qkv1, float("nan"))
    out2 = g.gdn_prefill(d["x"], d["conv_w"], d["cu_seqlens"], d["g"], d["beta"], d["z"], d["norm_w"], inp["q_scale"],
                         state_in=s_in, state_out=st2, conv_state_in=c_in, conv_state_out=cs2, qkv_buf=qkv2,
                         geometry=geo)
    g.gdn_check_device_errors()
    assert torch.equal(qkv1.view(torch.int16), qkv2.view(torch.int16)), "conv output"
    assert torch.equal(out1, out2), "out"
    assert torch.equal(st1, st2), "states"
    assert torch.equal(cs1.view(torch.int16), cs2.view(torch.int16)), "conv states"
    return out2, st2, cs2


@pytest.mark.parametrize("in_place", [False, True], ids=["out_of_place", "in_place"])
def test_one_call_prefill_equals_two_calls(in_place):
    """4,484 tokens on the small geometry (three chunk segments on the fast path): ragged lengths,
    an empty sequence and a nonzero conv state, states updated out of place and in place."""
    g = lib()
    geo = Geometry(num_k_heads=2, num_v_heads=6)
    lengths = [3000, 0, 1351, 70, 63]
    inp = prefill_inputs(lengths, seed=95, geo=geo, random_conv_state=True)
    out, st, cs = _both(g, inp, geo, in_place)
    ref = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"], inp["norm_w"],
                         2, 6, 128, 128, inp["q_scale"], state_in=inp["state0"], conv_state_in=inp["conv_state0"])
    assert_out_close(out, ref["out"])
    for n in range(len(lengths)):
        assert_state_close(st[n], ref["state"][n], f"state of sequence {n}")
    assert torch.equal(cs.cpu().view(torch.int16), ref["conv_state"].view(torch.int16))


def test_short_prefill_one_segment():
    """97 tokens: one chunk segment, everything on the caller's stream."""
    g = lib()
    geo = Geometry()
    inp = prefill_inputs([80, 17], seed=96, random_conv_state=True)
    _both(g, inp, geo)


def test_full_size_prefill_equals_two_calls():
    """The 4 x 4096-token workload: the one call and the two calls agree bit for bit."""
    g = lib()
    inp = prefill_inputs(BATCHED_LENGTHS, seed=97)
    _both(g, inp, Geometry())

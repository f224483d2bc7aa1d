"""GPU parity of the memory-bound legs: conv1d+SiLU prefill and the gated RMSNorm."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import QWEN_GDN, prefill_inputs, cu_seqlens_of
from tests.gpu_common import (DEV, Guarded, assert_bf16_within_one_ulp, assert_out_close, conv_accumulation_floor,
                              lib, out_error_ratio, NEG_CONTROL_RATIO)

pytestmark = pytest.mark.gpu
GEO = QWEN_GDN
C = GEO.conv_dim


@pytest.mark.parametrize("lengths,with_state", [
    ([16], False),
    ([1, 2, 3, 5, 17, 64, 65], True),
    ([0, 7, 0, 40, 1], True),
    ([63, 64, 65, 80, 128], False),
])
def test_conv1d_prefill_matches_oracle(lengths, with_state):
    g = lib()
    inp = prefill_inputs(lengths, seed=sum(lengths), random_conv_state=with_state)
    cs_in = inp["conv_state0"] if with_state else None
    y_ref, _, cs_ref = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], cs_in)
    T, N = sum(lengths), len(lengths)
    y = Guarded((T, C), torch.bfloat16)
    cs_out = Guarded((N, C, 3), torch.bfloat16)
    g.gdn_conv1d_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), inp["cu_seqlens"].to(DEV),
                         None if cs_in is None else cs_in.to(DEV), cs_out.t, y.t)
    g.gdn_check_device_errors()
    y.check("y")
    cs_out.check("conv_state_out")
    floor = conv_accumulation_floor(inp["x"], inp["conv_w"], inp["cu_seqlens"], cs_in)
    exact = assert_bf16_within_one_ulp(y.t, y_ref, floor, "conv output")
    assert exact > 0.99, f"only {exact:.4f} of the conv outputs are bit-exact"
    assert torch.equal(cs_out.t.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_conv1d_state_in_place_and_split_call():
    """conv_state_out may be conv_state_in; two calls with the state carried equal one call."""
    g = lib()
    inp = prefill_inputs([37], seed=5, random_conv_state=True)
    x, w = inp["x"].to(DEV), inp["conv_w"].to(DEV)
    y_all = g.gdn_conv1d_prefill(x, w, cu_seqlens_of([37]).to(DEV), inp["conv_state0"].to(DEV))
    st = inp["conv_state0"].to(DEV).clone()
    y1 = g.gdn_conv1d_prefill(x[:20].contiguous(), w, cu_seqlens_of([20]).to(DEV), st, st)
    y2 = g.gdn_conv1d_prefill(x[20:].contiguous(), w, cu_seqlens_of([17]).to(DEV), st, st)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([y1, y2]).view(torch.int16), y_all.view(torch.int16))
    _, _, cs_ref = oracle.conv1d_prefill(inp["x"], inp["conv_w"], [0, 37], inp["conv_state0"])
    assert torch.equal(st.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_conv1d_rejects_bad_cu_seqlens_on_device():
    g = lib()
    inp = prefill_inputs([8, 8], seed=6)
    bad = torch.tensor([0, 12, 5], dtype=torch.int32, device=DEV)   # not monotonic
    y = Guarded((16, C), torch.bfloat16)
    g.gdn_conv1d_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), bad, None, None, y.t)
    with pytest.raises(g.GdnError) as e:
        g.gdn_check_device_errors()
    assert e.value.name == "GDN_ERR_DEVICE_ARGUMENT"
    y.check("y")
    g.gdn_check_device_errors()   # the word was cleared


@pytest.mark.parametrize("T", [1, 33, 200])
def test_gated_rmsnorm_matches_oracle(T):
    g = lib()
    gen = torch.Generator().manual_seed(T)
    o = torch.randn(T, GEO.num_v_heads, 128, generator=gen).to(torch.bfloat16)
    z = torch.randn(T, GEO.num_v_heads, 128, generator=gen).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    ref = oracle.gated_rmsnorm(o.double(), z, w, 1e-6)
    out = Guarded((T, GEO.num_v_heads, 128), torch.bfloat16)
    g.gdn_gated_rmsnorm(o.to(DEV), z.to(DEV), w.to(DEV), 1e-6, out.t)
    g.gdn_check_device_errors()
    out.check("out")
    assert_out_close(out.t, ref)
    # the gate is sigmoid, not SiLU: the silu-gated oracle misses by far more than the bound
    silu = oracle.gated_rmsnorm(o.double(), z, w, 1e-6, mutation=oracle.MUT_SILU_GATE)
    assert out_error_ratio(out.t, silu) > NEG_CONTROL_RATIO

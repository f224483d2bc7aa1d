"""GPU parity of the KDA paths (per-key-channel decay) at the method's degenerate cases, against
the fp64 oracle of the KDA recurrence (GLM-5.3-Flash kernel TDD ledger, slices I2 and I4):

  beta = 0            the delta correction vanishes: pure per-channel decay,
                      S_T = S_0 diag(exp(sum_t g_t)) on the key dimension
  beta = 1, g = 0     no decay and a full projection per token: the memory spans every chunk, the
                      chunk form takes its tensor-core way for A and P in every chunk, and
                      (I + A)^-1 is at its worst for the split-bf16 operands
  g = -30 per token   every channel's decay underflows fp32 within a few tokens (the chunk form
                      takes its CUDA-core way)
  z = +-40            the sigmoid output gate saturates at 0 and 1

Each runs through the chunk-wise prefill, the sequential prefill and the decode step."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import KDA_GEO, kda_decode_inputs, kda_prefill_inputs
from tests.gpu_common import DEV, assert_out_close, assert_state_close, lib
from tests.test_gpu_kda_chunk import GEO2, _a, _conv, _oracle, _run

pytestmark = pytest.mark.gpu
CASES = ["beta0", "beta1_nodecay", "strong_decay", "gate_saturated"]


def _edge(inp, case):
    """Rewrite g, beta or z of a KDA prefill / decode input dict for one degenerate case."""
    if case == "beta0":
        inp["beta"] = torch.zeros_like(inp["beta"])
        inp["g"] = inp["g"] * 0.02  # weak decay, so that the decayed state stays far above fp32's range floor
    elif case == "beta1_nodecay":
        inp["beta"] = torch.ones_like(inp["beta"])
        inp["g"] = torch.zeros_like(inp["g"])
    elif case == "strong_decay":
        inp["g"] = torch.full_like(inp["g"], -30.0)
    elif case == "gate_saturated":
        z = inp["z"].float()
        inp["z"] = torch.where(z >= 0, 40.0, -40.0).to(torch.bfloat16)
    else:
        raise ValueError(case)
    return inp


def _sequential(g, y, inp, geo, state_out):
    return g.gdn_kda_recurrence(y.to(DEV), inp["g"].to(DEV), inp["beta"].to(DEV), inp["cu_seqlens"].to(DEV),
                                inp["q_scale"], state_in=inp["state0"].to(DEV), state_out=state_out,
                                z=inp["z"].to(DEV), norm_w=inp["norm_w"].to(DEV), geometry=geo)


@pytest.mark.parametrize("form", ["chunked", "sequential"])
@pytest.mark.parametrize("case", CASES)
def test_kda_prefill_edge_case(case, form):
    g = lib()
    geo = GEO2
    lengths = [1100] if case == "beta1_nodecay" else [130, 64, 5]
    N = len(lengths)
    inp = _edge(kda_prefill_inputs(lengths, seed=360 + CASES.index(case), geo=geo), case)
    y = _conv(inp)
    st = torch.empty((N, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    if form == "chunked":
        out = _run(g, y, inp, geo, state_in=inp["state0"].to(DEV), state_out=st)
    else:
        out = _sequential(g, y, inp, geo, st)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, state_in=inp["state0"])
    assert_out_close(out, want_o)
    for n in range(N):
        assert_state_close(st[n], want_s[n], f"state of sequence {n}")
    if case == "beta0":  # the closed form itself: every token only decays the state, channel by channel
        start = 0
        for n, L in enumerate(lengths):
            decay = torch.exp(inp["g"][start:start + L].double().sum(0))  # [Hv, Dk]
            want = inp["state0"][n].double() * decay[:, None, :]
            assert_state_close(st[n], want, f"closed form, sequence {n}")
            start += L
    if case == "gate_saturated":  # elements whose gate is closed (z = -40) come out as zeros
        closed = (inp["z"].float() < 0).to(DEV)
        assert out[closed].abs().max().item() <= 1e-6 * out.abs().max().item()


@pytest.mark.parametrize("case", CASES)
def test_kda_decode_edge_case(case):
    g = lib()
    geo = KDA_GEO
    B, steps = 3, 4
    d = _edge(kda_decode_inputs(B, steps, seed=380 + CASES.index(case)), case)
    cs, st = d["conv_state0"].to(DEV).clone(), d["state0"].to(DEV).clone()
    cs_ref, st_ref = d["conv_state0"], d["state0"].double()
    for s in range(steps):
        out = g.gdn_kda_decode_step(d["x"][s].to(DEV), d["conv_w"].to(DEV), cs, d["g"][s].to(DEV),
                                    d["beta"][s].to(DEV), st, d["z"][s].to(DEV), d["norm_w"].to(DEV), d["q_scale"],
                                    geometry=geo)
        g.gdn_check_device_errors()
        ref, _, cs_ref, st_ref = oracle.kda_decode_step(d["x"][s], d["conv_w"], cs_ref, d["g"][s], d["beta"][s],
                                                        st_ref, d["z"][s], d["norm_w"], q_scale=d["q_scale"],
                                                        **_a(geo))
        assert_out_close(out, ref, f"out of step {s}")
        for b in range(B):
            assert_state_close(st[b], st_ref[b], f"state of sequence {b} after step {s}")
    if case == "beta0":
        want = d["state0"].double() * torch.exp(d["g"].double().sum(0))[:, :, None, :]
        for b in range(B):
            assert_state_close(st[b], want[b], f"closed form, sequence {b}")

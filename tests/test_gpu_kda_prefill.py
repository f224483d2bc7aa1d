"""GPU parity of the KDA prefill (conv1d, then the KDA recurrence with the gated RMSNorm fused, in
its sequential and its chunk-wise form) against the oracle: ragged lengths around the 16-token
staging blocks and the 63/64/65 chunk boundary, an empty sequence, the decay clamp, o without the
norm, in-place states, one-token sequences against the KDA decode kernel, bad cu_seqlens on the
device, and the 64-head 4 x 4096 workload on sampled heads."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import KDA_GEO, Geometry, cu_seqlens_of, kda_decode_inputs, kda_prefill_inputs
from tests.gpu_common import DEV, Guarded, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu

GEO2 = Geometry(num_k_heads=2, num_v_heads=4, head_k_dim=128, head_v_dim=128, conv_width=4)  # 2 V heads per K head
LENGTHS = [0, 1, 15, 16, 17, 63, 64, 65, 130]


def _a(geo):
    return dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
                head_v_dim=geo.head_v_dim)


@pytest.mark.parametrize("chunked", [False, True], ids=["sequential", "chunked"])
@pytest.mark.parametrize("g_min", [float("-inf"), -1.0], ids=["no_clamp", "clamp"])
def test_kda_prefill_matches_oracle(g_min, chunked):
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs(LENGTHS, seed=300, geo=geo, random_conv_state=True)
    T, N = sum(LENGTHS), len(LENGTHS)
    out = Guarded((T, geo.num_v_heads, 128), torch.bfloat16)
    st = Guarded((N, geo.num_v_heads, 128, 128), torch.float32)
    cs = torch.empty((N, geo.conv_dim, geo.conv_width - 1), dtype=torch.bfloat16, device=DEV)
    g.gdn_kda_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), inp["cu_seqlens"].to(DEV), inp["g"].to(DEV),
                      inp["beta"].to(DEV), inp["z"].to(DEV), inp["norm_w"].to(DEV), inp["q_scale"], g_min,
                      state_in=inp["state0"].to(DEV), state_out=st.t, conv_state_in=inp["conv_state0"].to(DEV),
                      conv_state_out=cs, out=out.t, chunked=chunked, geometry=geo)
    g.gdn_check_device_errors()
    out.check("out")
    st.check("state_out")
    ref = oracle.kda_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                             inp["norm_w"], q_scale=inp["q_scale"], g_min=g_min, state_in=inp["state0"],
                             conv_state_in=inp["conv_state0"], **_a(geo))
    assert_out_close(out.t, ref["out"])
    for n, L in enumerate(LENGTHS):
        if L == 0:   # an empty sequence passes its state through unchanged
            assert torch.equal(st.t[n].cpu(), inp["state0"][n])
        else:
            assert_state_close(st.t[n], ref["state"][n], f"state of sequence {n} ({L} tokens)")
    assert torch.equal(cs.cpu().view(torch.int16), ref["conv_state"].view(torch.int16))


def test_kda_recurrence_without_z_returns_o_and_updates_the_state_in_place():
    """From the oracle's own conv output: out is o = q_scale S q (bf16), and state_out may be
    state_in."""
    g = lib()
    geo = GEO2
    lengths = [20, 47, 33]
    inp = kda_prefill_inputs(lengths, seed=301, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    st = inp["state0"].to(DEV).clone()
    out = g.gdn_kda_recurrence(y.to(DEV), inp["g"].to(DEV), inp["beta"].to(DEV), inp["cu_seqlens"].to(DEV),
                               inp["q_scale"], state_in=st, state_out=st, geometry=geo)
    g.gdn_check_device_errors()
    o, st_ref = oracle.kda_recurrence(y, inp["g"], inp["beta"], inp["cu_seqlens"], q_scale=inp["q_scale"],
                                      state_in=inp["state0"], **_a(geo))
    assert_out_close(out, o)
    for n in range(len(lengths)):
        assert_state_close(st[n], st_ref[n], f"state of sequence {n}")


def test_kda_recurrence_from_zero_state():
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs([70, 9], seed=302, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    st = torch.empty((2, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = g.gdn_kda_recurrence(y.to(DEV), inp["g"].to(DEV), inp["beta"].to(DEV), inp["cu_seqlens"].to(DEV),
                               inp["q_scale"], state_out=st, z=inp["z"].to(DEV), norm_w=inp["norm_w"].to(DEV),
                               geometry=geo)
    g.gdn_check_device_errors()
    o, st_ref = oracle.kda_recurrence(y, inp["g"], inp["beta"], inp["cu_seqlens"], q_scale=inp["q_scale"], **_a(geo))
    assert_out_close(out, oracle.gated_rmsnorm(o, inp["z"], inp["norm_w"]))
    for n in range(2):
        assert_state_close(st[n], st_ref[n], f"state of sequence {n}")


def test_one_token_sequences_match_the_kda_decode_kernel():
    """B sequences of one token each: the prefill and the decode kernel (its own conv step) give
    the same outputs and states."""
    g = lib()
    geo = GEO2
    B = 6
    d = kda_decode_inputs(B, 1, seed=303, geo=geo)
    args = dict(geometry=geo)
    st_dec, cs_dec = d["state0"].to(DEV).clone(), d["conv_state0"].to(DEV).clone()
    out_dec = g.gdn_kda_decode_step(d["x"][0].to(DEV), d["conv_w"].to(DEV), cs_dec, d["g"][0].to(DEV),
                                    d["beta"][0].to(DEV), st_dec, d["z"][0].to(DEV), d["norm_w"].to(DEV),
                                    d["q_scale"], -2.0, **args)
    st_pre = d["state0"].to(DEV).clone()
    cs_pre = torch.empty_like(cs_dec)
    out_pre = g.gdn_kda_prefill(d["x"][0].to(DEV), d["conv_w"].to(DEV), cu_seqlens_of([1] * B).to(DEV),
                                d["g"][0].to(DEV), d["beta"][0].to(DEV), d["z"][0].to(DEV), d["norm_w"].to(DEV),
                                d["q_scale"], -2.0, state_in=st_pre, state_out=st_pre,
                                conv_state_in=d["conv_state0"].to(DEV), conv_state_out=cs_pre, chunked=False, **args)
    g.gdn_check_device_errors()
    assert torch.equal(cs_pre, cs_dec)
    assert_out_close(out_pre, out_dec.double())
    for b in range(B):
        assert_state_close(st_pre[b], st_dec[b].double(), f"state of sequence {b}", tol=1e-5)


def test_kda_recurrence_rejects_bad_cu_seqlens_on_device():
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs([8, 8], seed=304, geo=geo)
    bad = torch.tensor([0, 12, 5], dtype=torch.int32, device=DEV)   # not monotonic
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    out = Guarded((16, geo.num_v_heads, 128), torch.bfloat16)
    st = Guarded((2, geo.num_v_heads, 128, 128), torch.float32)
    g.gdn_kda_recurrence(y.to(DEV), inp["g"].to(DEV), inp["beta"].to(DEV), bad, inp["q_scale"], state_out=st.t,
                         out=out.t, geometry=geo)
    with pytest.raises(g.GdnError) as e:
        g.gdn_check_device_errors()
    assert e.value.name == "GDN_ERR_DEVICE_ARGUMENT"
    out.check("out")
    st.check("state_out")
    g.gdn_check_device_errors()   # the word was cleared


def _one_head(inp, geo, h):
    """The inputs of V head h (and its K head) alone, as a one-head problem: the conv is
    depthwise and the heads' recurrences are independent, so its results are those of head h."""
    hk, dk, dv, j = geo.num_k_heads, geo.head_k_dim, geo.head_v_dim, h // (geo.num_v_heads // geo.num_k_heads)
    ch = torch.cat([torch.arange(j * dk, (j + 1) * dk), torch.arange((hk + j) * dk, (hk + j + 1) * dk),
                    torch.arange(2 * hk * dk + h * dv, 2 * hk * dk + (h + 1) * dv)])
    return dict(x=inp["x"][:, ch].contiguous(), conv_w=inp["conv_w"][ch].contiguous(),
                g=inp["g"][:, h:h + 1].contiguous(), beta=inp["beta"][:, h:h + 1].contiguous(),
                z=inp["z"][:, h:h + 1].contiguous(), state_in=inp["state0"][:, h:h + 1].contiguous())


@pytest.mark.parametrize("chunked", [False, True], ids=["sequential", "chunked"])
def test_kda_prefill_full_size_sampled_heads(chunked):
    """The 64-head workload, 4 sequences x 4096 tokens, in the launch configurations the benchmark
    times; the oracle computes three of the 64 V heads, each from its own channels."""
    g = lib()
    geo = KDA_GEO
    lengths = [4096] * 4
    inp = kda_prefill_inputs(lengths, seed=305, geo=geo)
    T = sum(lengths)
    st = torch.empty((4, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = g.gdn_kda_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), inp["cu_seqlens"].to(DEV), inp["g"].to(DEV),
                            inp["beta"].to(DEV), inp["z"].to(DEV), inp["norm_w"].to(DEV), inp["q_scale"],
                            state_in=inp["state0"].to(DEV), state_out=st, chunked=chunked, geometry=geo)
    g.gdn_check_device_errors()
    assert out.shape == (T, geo.num_v_heads, 128)
    for h in (0, 37, 63):
        one = _one_head(inp, geo, h)
        ref = oracle.kda_prefill(one["x"], one["conv_w"], inp["cu_seqlens"], one["g"], one["beta"], one["z"],
                                 inp["norm_w"], 1, 1, 128, 128, inp["q_scale"], state_in=one["state_in"])
        assert_out_close(out[:, h], ref["out"][:, 0], f"out of head {h}")
        for n in range(4):
            assert_state_close(st[n, h], ref["state"][n, 0], f"state of sequence {n}, head {h}")


def test_kda_weak_decay_long_memory():
    """Per-channel decays fifty times weaker than the workload's: the state carries across many
    16-token blocks and the fp32 chain is checked at the state tolerance."""
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs([1024, 300], seed=306, geo=geo)
    inp["g"] = inp["g"] * 0.02
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    st = torch.empty((2, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = g.gdn_kda_recurrence(y.to(DEV), inp["g"].to(DEV), inp["beta"].to(DEV), inp["cu_seqlens"].to(DEV),
                               inp["q_scale"], state_in=inp["state0"].to(DEV), state_out=st, z=inp["z"].to(DEV),
                               norm_w=inp["norm_w"].to(DEV), geometry=geo)
    g.gdn_check_device_errors()
    o, st_ref = oracle.kda_recurrence(y, inp["g"], inp["beta"], inp["cu_seqlens"], q_scale=inp["q_scale"],
                                      state_in=inp["state0"], **_a(geo))
    assert_out_close(out, oracle.gated_rmsnorm(o, inp["z"], inp["norm_w"]))
    for n in range(2):
        assert_state_close(st[n], st_ref[n], f"state of sequence {n}")

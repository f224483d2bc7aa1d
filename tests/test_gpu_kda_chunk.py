"""GPU parity of the chunk-wise KDA prefill (gdn_kda_chunk_prefill: a prep kernel per (chunk, V
head), then the state chain on the tensor cores) against the sequential fp64 oracle of the KDA
recurrence (GLM-5.3-Flash kernel TDD ledger, slices I2, I2a and I4): ragged lengths around the
16-token blocks and the 63 / 64 / 65 chunk boundary, an empty sequence, the decay clamp, decays
strong enough to underflow inside a chunk, weak decays over long sequences, o without the norm,
in-place and zero states, bad cu_seqlens on the device, many short sequences, and the 64-head
4 x 4096 workload on sampled heads in the launch configuration the benchmark times."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import KDA_GEO, Geometry, cu_seqlens_of, kda_prefill_inputs
from tests.gpu_common import DEV, Guarded, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu

GEO2 = Geometry(num_k_heads=2, num_v_heads=4, head_k_dim=128, head_v_dim=128, conv_width=4)  # 2 V heads per K head
LENGTHS = [0, 1, 15, 16, 17, 63, 64, 65, 130]


def _a(geo):
    return dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
                head_v_dim=geo.head_v_dim)


def _conv(inp):
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    return y


def _run(g, y, inp, geo, g_min=float("-inf"), state_in=None, state_out=None, gated=True, out=None, gate=None):
    gg = inp["g"] if gate is None else gate
    return g.gdn_kda_chunk_prefill(y.to(DEV), gg.to(DEV), inp["beta"].to(DEV), inp["cu_seqlens"].to(DEV),
                                   inp["q_scale"], g_min, state_in=state_in, state_out=state_out,
                                   z=inp["z"].to(DEV) if gated else None,
                                   norm_w=inp["norm_w"].to(DEV) if gated else None, out=out, geometry=geo)


def _oracle(y, inp, geo, g_min=float("-inf"), state_in=None, gated=True, gate=None):
    gg = inp["g"] if gate is None else gate
    o, st = oracle.kda_recurrence(y, gg, inp["beta"], inp["cu_seqlens"], q_scale=inp["q_scale"], g_min=g_min,
                                  state_in=state_in, **_a(geo))
    return (oracle.gated_rmsnorm(o, inp["z"], inp["norm_w"]) if gated else o), st


@pytest.mark.parametrize("g_min", [float("-inf"), -1.0], ids=["no_clamp", "clamp"])
def test_kda_chunk_matches_oracle(g_min):
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs(LENGTHS, seed=320, geo=geo)
    y = _conv(inp)
    T, N = sum(LENGTHS), len(LENGTHS)
    out = Guarded((T, geo.num_v_heads, 128), torch.bfloat16)
    st = Guarded((N, geo.num_v_heads, 128, 128), torch.float32)
    _run(g, y, inp, geo, g_min, state_in=inp["state0"].to(DEV), state_out=st.t, out=out.t)
    g.gdn_check_device_errors()
    out.check("out")
    st.check("state_out")
    want_o, want_s = _oracle(y, inp, geo, g_min, state_in=inp["state0"])
    assert_out_close(out.t, want_o)
    for n, L in enumerate(LENGTHS):
        if L == 0:   # an empty sequence passes its state through unchanged
            assert torch.equal(st.t[n].cpu(), inp["state0"][n])
        else:
            assert_state_close(st.t[n], want_s[n], f"state of sequence {n} ({L} tokens)")


def test_kda_chunk_without_z_in_place():
    """out is o = q_scale S q (bf16) itself, and state_out may be state_in."""
    g = lib()
    geo = GEO2
    lengths = [20, 47, 200, 33]
    inp = kda_prefill_inputs(lengths, seed=321, geo=geo)
    y = _conv(inp)
    st = inp["state0"].to(DEV).clone()
    out = _run(g, y, inp, geo, state_in=st, state_out=st, gated=False)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, state_in=inp["state0"], gated=False)
    assert_out_close(out, want_o)
    for n in range(len(lengths)):
        assert_state_close(st[n], want_s[n], f"state of sequence {n}")


def test_kda_chunk_from_zero_state():
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs([70, 9, 128], seed=322, geo=geo)
    y = _conv(inp)
    st = torch.empty((3, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = _run(g, y, inp, geo, state_out=st)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo)
    assert_out_close(out, want_o)
    for n in range(3):
        assert_state_close(st[n], want_s[n], f"state of sequence {n}")


def test_kda_chunk_decay_underflow_and_clamp():
    """Log decays down to -30 per token, clamped at -20: inside a chunk e^gamma underflows to zero
    for many channels, and the chunk form must still give the sequential results (the factors
    between tokens are formed as differences of running sums, never as quotients)."""
    g = lib()
    geo = GEO2
    lengths = [64, 130, 77]
    inp = kda_prefill_inputs(lengths, seed=323, geo=geo)
    gen = torch.Generator().manual_seed(3230)
    strong = -30.0 * torch.rand(inp["g"].shape, generator=gen)
    weak = inp["g"] * 0.01
    pick = torch.rand(inp["g"].shape, generator=gen) < 0.5   # half of the channels nearly keep their memory
    gate = torch.where(pick, weak, strong)
    y = _conv(inp)
    st = torch.empty((3, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = _run(g, y, inp, geo, -20.0, state_in=inp["state0"].to(DEV), state_out=st, gate=gate)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, -20.0, state_in=inp["state0"], gate=gate)
    assert_out_close(out, want_o)
    for n in range(3):
        assert_state_close(st[n], want_s[n], f"state of sequence {n}")


def test_kda_chunk_mixed_decay_spans():
    """Chunks whose decays span more than the tensor-core way takes (about 60 nats between a token
    and the chunk's middle) next to chunks that span less, in one sequence: each chunk's A and P
    come from its own way, and the state carries across both."""
    g = lib()
    geo = GEO2
    lengths = [300, 64]
    inp = kda_prefill_inputs(lengths, seed=329, geo=geo)
    gate = inp["g"] * 0.05
    strong = torch.zeros(sum(lengths), dtype=torch.bool)
    strong[64:128] = True          # the second chunk of the first sequence
    strong[256:300] = True         # its ragged last chunk
    gate[strong] = -3.0 - torch.rand(gate[strong].shape, generator=torch.Generator().manual_seed(3290))
    y = _conv(inp)
    st = torch.empty((2, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = _run(g, y, inp, geo, state_in=inp["state0"].to(DEV), state_out=st, gate=gate)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, state_in=inp["state0"], gate=gate)
    assert_out_close(out, want_o)
    for n in range(2):
        assert_state_close(st[n], want_s[n], f"state of sequence {n}")


def test_kda_chunk_weak_decay_long_memory():
    """Decays fifty times weaker than the workload's: the state carries across many chunks and
    the fp32 chain is checked at the state tolerance."""
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs([1024, 300], seed=324, geo=geo)
    gate = inp["g"] * 0.02
    y = _conv(inp)
    st = torch.empty((2, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = _run(g, y, inp, geo, state_in=inp["state0"].to(DEV), state_out=st, gate=gate)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, state_in=inp["state0"], gate=gate)
    assert_out_close(out, want_o)
    for n in range(2):
        assert_state_close(st[n], want_s[n], f"state of sequence {n}")


def test_kda_chunk_many_short_sequences():
    """More (sequence, V head) items than CTAs, with lengths 0..150: the persistent state kernel's
    work queue and the prep kernel's chunk-to-sequence search."""
    g = lib()
    geo = Geometry(num_k_heads=4, num_v_heads=8, head_k_dim=128, head_v_dim=128, conv_width=4)
    gen = torch.Generator().manual_seed(3250)
    lengths = torch.randint(0, 151, (60,), generator=gen).tolist()
    inp = kda_prefill_inputs(lengths, seed=325, geo=geo)
    y = _conv(inp)
    N = len(lengths)
    st = torch.empty((N, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = _run(g, y, inp, geo, -5.0, state_in=inp["state0"].to(DEV), state_out=st)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, -5.0, state_in=inp["state0"])
    assert_out_close(out, want_o)
    for n, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(st[n].cpu(), inp["state0"][n])
        else:
            assert_state_close(st[n], want_s[n], f"state of sequence {n} ({L} tokens)")


def test_kda_chunk_rejects_bad_cu_seqlens_on_device():
    g = lib()
    geo = GEO2
    inp = kda_prefill_inputs([8, 8], seed=326, geo=geo)
    y = _conv(inp)
    bad = torch.tensor([0, 12, 5], dtype=torch.int32, device=DEV)   # not monotonic
    out = Guarded((16, geo.num_v_heads, 128), torch.bfloat16)
    st = Guarded((2, geo.num_v_heads, 128, 128), torch.float32)
    g.gdn_kda_chunk_prefill(y.to(DEV), inp["g"].to(DEV), inp["beta"].to(DEV), bad, inp["q_scale"], state_out=st.t,
                            out=out.t, geometry=geo)
    with pytest.raises(g.GdnError) as e:
        g.gdn_check_device_errors()
    assert e.value.name == "GDN_ERR_DEVICE_ARGUMENT"
    out.check("out")
    st.check("state_out")
    g.gdn_check_device_errors()   # the word was cleared


def test_kda_chunk_empty_call_copies_states():
    """total_tokens = 0 with sequences: every state passes through unchanged."""
    g = lib()
    geo = GEO2
    s0 = torch.randn((3, geo.num_v_heads, 128, 128), generator=torch.Generator().manual_seed(327))
    st = torch.full_like(s0, float("nan")).to(DEV)
    qkv = torch.empty((0, geo.conv_dim), dtype=torch.bfloat16, device=DEV)
    g.gdn_kda_chunk_prefill(qkv, torch.empty((0, geo.num_v_heads, 128), device=DEV),
                            torch.empty((0, geo.num_v_heads), device=DEV), cu_seqlens_of([0, 0, 0]).to(DEV), 0.088,
                            state_in=s0.to(DEV), state_out=st, geometry=geo)
    g.gdn_check_device_errors()
    assert torch.equal(st.cpu(), s0)


def _one_head(inp, geo, h):
    """The inputs of V head h (and its K head) alone, as a one-head problem: the conv is
    depthwise and the heads' recurrences are independent, so its results are those of head h."""
    hk, dk, dv, j = geo.num_k_heads, geo.head_k_dim, geo.head_v_dim, h // (geo.num_v_heads // geo.num_k_heads)
    ch = torch.cat([torch.arange(j * dk, (j + 1) * dk), torch.arange((hk + j) * dk, (hk + j + 1) * dk),
                    torch.arange(2 * hk * dk + h * dv, 2 * hk * dk + (h + 1) * dv)])
    return dict(x=inp["x"][:, ch].contiguous(), conv_w=inp["conv_w"][ch].contiguous(),
                g=inp["g"][:, h:h + 1].contiguous(), beta=inp["beta"][:, h:h + 1].contiguous(),
                z=inp["z"][:, h:h + 1].contiguous(), state_in=inp["state0"][:, h:h + 1].contiguous())


def test_kda_chunk_full_size_sampled_heads():
    """The 64-head workload, 4 sequences x 4096 tokens, through the same calls the benchmark
    times (the conv kernel, then the chunk prefill); the oracle computes three of the 64 V heads,
    each from its own channels."""
    g = lib()
    geo = KDA_GEO
    lengths = [4096] * 4
    inp = kda_prefill_inputs(lengths, seed=328, geo=geo)
    T = sum(lengths)
    st = torch.empty((4, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    cu = inp["cu_seqlens"].to(DEV)
    y = g.gdn_conv1d_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), cu, geometry=geo)
    out = g.gdn_kda_chunk_prefill(y, inp["g"].to(DEV), inp["beta"].to(DEV), cu, inp["q_scale"],
                                  state_in=inp["state0"].to(DEV), state_out=st, z=inp["z"].to(DEV),
                                  norm_w=inp["norm_w"].to(DEV), geometry=geo)
    g.gdn_check_device_errors()
    assert out.shape == (T, geo.num_v_heads, 128)
    for h in (0, 37, 63):
        one = _one_head(inp, geo, h)
        ref = oracle.kda_prefill(one["x"], one["conv_w"], inp["cu_seqlens"], one["g"], one["beta"], one["z"],
                                 inp["norm_w"], 1, 1, 128, 128, inp["q_scale"], state_in=one["state_in"])
        assert_out_close(out[:, h], ref["out"][:, 0], f"out of head {h}")
        for n in range(4):
            assert_state_close(st[n, h], ref["state"][n, 0], f"state of sequence {n}, head {h}")


def test_kda_chunk_inside_a_captured_graph():
    """The chunk-wise KDA call launches on the caller's stream only (no side streams, no host
    synchronisation), so it can be captured in a CUDA graph; replays give the oracle's results."""
    g = lib()
    geo = GEO2
    lengths = [130, 64, 7]
    inp = kda_prefill_inputs(lengths, seed=330, geo=geo)
    y = _conv(inp).to(DEV)
    N, T = len(lengths), sum(lengths)
    d = {k: inp[k].to(DEV) for k in ("g", "beta", "cu_seqlens", "z", "norm_w", "state0")}
    ws = torch.empty(g.gdn_kda_chunk_prefill_workspace_size(N, T, geometry=geo), dtype=torch.uint8, device=DEV)
    st = torch.empty_like(d["state0"])
    out = torch.empty((T, geo.num_v_heads, 128), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.gdn_kda_chunk_prefill(y, d["g"], d["beta"], d["cu_seqlens"], inp["q_scale"], -4.0, state_in=d["state0"],
                                    state_out=st, z=d["z"], norm_w=d["norm_w"], out=out, workspace=ws, geometry=geo,
                                    stream=s)
    want_o, want_s = _oracle(_conv(inp), inp, geo, -4.0, state_in=inp["state0"])
    for _ in range(2):
        st.fill_(float("nan"))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        g.gdn_check_device_errors()
        assert_out_close(out, want_o)
        for n in range(N):
            assert_state_close(st[n], want_s[n], f"state of sequence {n}")


def test_kda_chunk_thousands_of_short_sequences():
    """5,000 sequences of 0..12 tokens: more than the schedule sorts (its unsorted order is taken),
    one chunk each, so consecutive prep units lie in different sequences and their sequence is
    searched for each time."""
    g = lib()
    geo = GEO2
    gen = torch.Generator().manual_seed(3310)
    lengths = torch.randint(0, 13, (5000,), generator=gen).tolist()
    inp = kda_prefill_inputs(lengths, seed=331, geo=geo)
    y = _conv(inp)
    N = len(lengths)
    st = torch.empty((N, geo.num_v_heads, 128, 128), dtype=torch.float32, device=DEV)
    out = _run(g, y, inp, geo, -6.0, state_in=inp["state0"].to(DEV), state_out=st)
    g.gdn_check_device_errors()
    want_o, want_s = _oracle(y, inp, geo, -6.0, state_in=inp["state0"])
    assert_out_close(out, want_o)
    for n in range(0, N, 97):  # a sample of the states, every length represented
        if lengths[n] == 0:
            assert torch.equal(st[n].cpu(), inp["state0"][n])
        else:
            assert_state_close(st[n], want_s[n], f"state of sequence {n} ({lengths[n]} tokens)")


def test_kda_one_call_prefill_equals_the_two_calls():
    """gdn_kda_prefill (conv, then the chunk-wise recurrence, in one call) gives the bits of
    gdn_conv1d_prefill followed by gdn_kda_chunk_prefill: conv output, output, states, conv states."""
    g = lib()
    geo = GEO2
    lengths = [150, 0, 64, 33]
    inp = kda_prefill_inputs(lengths, seed=332, geo=geo, random_conv_state=True)
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
    N = len(lengths)
    st1, st2 = torch.empty_like(d["state0"]), torch.empty_like(d["state0"])
    cs1, cs2 = torch.empty_like(d["conv_state0"]), torch.empty_like(d["conv_state0"])
    qkv1 = torch.empty_like(d["x"])
    out1 = g.gdn_kda_prefill(d["x"], d["conv_w"], d["cu_seqlens"], d["g"], d["beta"], d["z"], d["norm_w"],
                             inp["q_scale"], -3.0, state_in=d["state0"], state_out=st1, conv_state_in=d["conv_state0"],
                             conv_state_out=cs1, qkv_buf=qkv1, geometry=geo)
    qkv2 = g.gdn_conv1d_prefill(d["x"], d["conv_w"], d["cu_seqlens"], d["conv_state0"], cs2, geometry=geo)
    out2 = g.gdn_kda_chunk_prefill(qkv2, d["g"], d["beta"], d["cu_seqlens"], inp["q_scale"], -3.0,
                                   state_in=d["state0"], state_out=st2, z=d["z"], norm_w=d["norm_w"], geometry=geo)
    g.gdn_check_device_errors()
    assert torch.equal(qkv1, qkv2)
    assert torch.equal(out1, out2)
    assert torch.equal(st1, st2)
    assert torch.equal(cs1, cs2)
    ref = oracle.kda_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                             inp["norm_w"], q_scale=inp["q_scale"], g_min=-3.0, state_in=inp["state0"],
                             conv_state_in=inp["conv_state0"], **_a(geo))
    assert_out_close(out1, ref["out"])
    for n, L in enumerate(lengths):
        if L:
            assert_state_close(st1[n], ref["state"][n], f"state of sequence {n}")

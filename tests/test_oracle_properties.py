"""Randomised pins of the oracle (CPU only): the invariants of the pin tests, drawn over random
small geometries (head ratios 1..3, Dk != Dv), ragged lengths (empty sequences included) and
decays, so that no pin holds only at the hand-picked sizes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from linear_attention_ssm_gb300.synth import Geometry, kda_prefill_inputs, prefill_inputs  # noqa: E402
from tests.chunked_numpy import chunked_chain, chunked_chain_kda, l2n  # noqa: E402

geometries = st.builds(
    lambda hk, ratio, dk, dv: Geometry(num_k_heads=hk, num_v_heads=hk * ratio, head_k_dim=dk, head_v_dim=dv,
                                       conv_width=4),
    st.integers(1, 2), st.integers(1, 3), st.sampled_from([4, 8, 16]), st.sampled_from([4, 6, 8]))
length_lists = st.lists(st.integers(0, 40), min_size=1, max_size=4)
SETTINGS = settings(max_examples=25, deadline=None, derandomize=True)


def _args(geo, q_scale=0.5):
    return (geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim, q_scale)


@SETTINGS
@given(geo=geometries, lengths=length_lists, seed=st.integers(0, 10_000), kda=st.booleans())
def test_packed_call_equals_separate_calls(geo, lengths, seed, kda):
    inp = (kda_prefill_inputs if kda else prefill_inputs)(lengths, seed=seed, geo=geo, random_conv_state=True)
    run = oracle.kda_prefill if kda else oracle.prefill
    packed = run(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"], inp["norm_w"],
                 *_args(geo), state_in=inp["state0"], conv_state_in=inp["conv_state0"], nthreads=1)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        one = run(inp["x"][s:e], inp["conv_w"], [0, e - s], inp["g"][s:e], inp["beta"][s:e], inp["z"][s:e],
                  inp["norm_w"], *_args(geo), state_in=inp["state0"][n:n + 1],
                  conv_state_in=inp["conv_state0"][n:n + 1], nthreads=1)
        assert torch.equal(one["out"], packed["out"][s:e])
        assert torch.equal(one["state"][0], packed["state"][n])


@SETTINGS
@given(geo=geometries, L=st.integers(1, 140), seed=st.integers(0, 10_000), kda=st.booleans(),
       chunk=st.sampled_from([16, 64]))
def test_sequential_chain_equals_the_chunked_form(geo, L, seed, kda, chunk):
    inp = (kda_prefill_inputs if kda else prefill_inputs)([L], seed=seed, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    rec = oracle.kda_recurrence if kda else oracle.gdn_recurrence
    o, s = rec(y, inp["g"], inp["beta"], [0, L], *_args(geo), state_in=inp["state0"], nthreads=1)
    hk, hv, dk, dv = geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim
    a = y.double().numpy()
    for h in range(hv):
        j = h // (hv // hk)
        q = l2n(a[:, j * dk:(j + 1) * dk], 1e-6)
        k = l2n(a[:, (hk + j) * dk:(hk + j + 1) * dk], 1e-6)
        v = a[:, 2 * hk * dk + h * dv:2 * hk * dk + (h + 1) * dv]
        form = chunked_chain_kda if kda else chunked_chain
        O, S = form(q, k, v, inp["g"][:, h].double().numpy(), inp["beta"][:, h].double().numpy(),
                    inp["state0"][0, h].double().numpy(), 0.5, chunk=chunk)
        np.testing.assert_allclose(o[:, h].numpy(), O, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(s[0, h].numpy(), S, rtol=1e-9, atol=1e-11)


@SETTINGS
@given(geo=geometries, L=st.integers(1, 12), seed=st.integers(0, 10_000))
def test_decode_steps_equal_a_prefill(geo, L, seed):
    inp = prefill_inputs([L], seed=seed, geo=geo, random_conv_state=True)
    pre = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"], inp["norm_w"],
                         *_args(geo), state_in=inp["state0"], conv_state_in=inp["conv_state0"], nthreads=1)
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.5, nthreads=1)
    cs, stt = inp["conv_state0"], inp["state0"].double()
    for t in range(L):
        out, _, cs, stt = oracle.decode_step(inp["x"][t:t + 1], inp["conv_w"], cs, inp["g"][t:t + 1],
                                             inp["beta"][t:t + 1], stt, inp["z"][t:t + 1], inp["norm_w"], **a)
        np.testing.assert_allclose(out[0].numpy(), pre["out"][t].numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(stt[0].numpy(), pre["state"][0].numpy(), rtol=1e-10, atol=1e-13)
    assert torch.equal(cs[0].view(torch.int16), pre["conv_state"][0].view(torch.int16))

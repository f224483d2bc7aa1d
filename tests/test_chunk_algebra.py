"""The chunk-wise KDA form in the precision and factorisation a tensor-core kernel can use (CPU
only): fp32 throughout, intra-chunk decay weights formed by 16-token sub-blocks around references
that keep every factor a decay in (0, 1].  Checked against the fp64 sequential oracle, including
decays far stronger than any workload's, where the plain factorisation exp(Gamma_t) * exp(-Gamma_j)
leaves the range of fp32.  Then the tensor-core precision plan: with every contraction a bf16
product (fp32 accumulation), which operands must be bf16 hi + lo pairs for the state to hold its
1e-4 tolerance when it carries across many chunks.  GLM-5.3-Flash kernel TDD ledger, slice I4 (the
chunk path matches the sequential state and output at 63/64/65 tokens)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from linear_attention_ssm_gb300.synth import Geometry, kda_prefill_inputs
from tests.chunked_numpy import (TC_SPLIT_ALL, chunked_chain_kda_fp32, chunked_chain_kda_tc, chunked_chain_kda_tc_middle,
                                 kda_gram_middle_reference, kda_intra_chunk_weights,
                                 l2n)

GEO = Geometry(num_k_heads=1, num_v_heads=1, head_k_dim=128, head_v_dim=128, conv_width=4)


def _case(L, seed, g_scale=1.0):
    inp = kda_prefill_inputs([L], seed=seed, geo=GEO)
    inp["g"] = inp["g"] * g_scale
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    o, st = oracle.kda_recurrence(y, inp["g"], inp["beta"], [0, L], 1, 1, 128, 128, GEO.q_scale,
                                  state_in=inp["state0"])
    a = y.double().numpy()
    q, k, v = l2n(a[:, :128], 1e-6), l2n(a[:, 128:256], 1e-6), a[:, 256:]
    return inp, q, k, v, o[:, 0].numpy(), st[0, 0].numpy()


def _rel(got, want):
    return float(np.linalg.norm(got.astype(np.float64) - want) / np.linalg.norm(want))


@pytest.mark.parametrize("L", [63, 64, 65, 130])
def test_fp32_subblock_chunk_form_matches_the_oracle(L):
    inp, q, k, v, o, st = _case(L, 400 + L)
    O, S = chunked_chain_kda_fp32(q, k, v, inp["g"][:, 0].double().numpy(), inp["beta"][:, 0].double().numpy(),
                                  inp["state0"][0, 0].double().numpy(), GEO.q_scale)
    assert np.isfinite(O).all() and np.isfinite(S).all()
    assert np.abs(O - o).max() <= 2e-2 * np.abs(o).max() / 100   # well inside the output tolerance
    assert _rel(S, st) <= 1e-5                                   # and the state's


def test_fp32_subblock_weights_survive_decays_that_overflow_the_plain_factorisation():
    """g = -U(0.001, 2) x 10 per token and channel (total log decays near -640 over a chunk): the
    sub-block weights stay finite and match fp64; exp(-Gamma) alone already overflows fp32."""
    inp, q, k, v, o, st = _case(64, 410, g_scale=10.0)
    g = inp["g"][:, 0].double().numpy()
    gam = np.cumsum(g, axis=0)
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.exp(-gam.astype(np.float32))).all()
    M = kda_intra_chunk_weights(k, k, gam)
    exact = np.einsum("ti,ji,tji->tj", k, k, np.exp(np.where(np.tril(np.ones((64, 64)))[:, :, None] > 0,
                                                             gam[:, None, :] - gam[None, :, :], -np.inf)))
    assert np.isfinite(M).all()
    np.testing.assert_allclose(M, exact, rtol=0, atol=1e-6)
    O, S = chunked_chain_kda_fp32(q, k, v, g, inp["beta"][:, 0].double().numpy(), inp["state0"][0, 0].double().numpy(),
                                  GEO.q_scale)
    assert np.isfinite(O).all() and np.isfinite(S).all()
    assert np.abs(O - o).max() <= 2e-2 * np.abs(o).max() / 100
    assert _rel(S, st) <= 1e-5


def test_the_plain_factorisation_fails_where_the_subblocks_do_not():
    """Negative control: the same weights formed as one product (K * exp(Gamma)) (K * exp(-Gamma))^T
    about the chunk's start, in fp32, are not finite under the strong decay (an inf times a zero
    factor), so the sub-blocks are needed, not a refinement."""
    inp, q, k, v, o, st = _case(64, 412, g_scale=10.0)
    gam = np.cumsum(inp["g"][:, 0].double().numpy(), axis=0).astype(np.float32)
    kf = k.astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        plain = (kf * np.exp(gam)) @ (kf * np.exp(-gam)).T
    assert not np.isfinite(np.tril(plain)).all()
    assert np.isfinite(kda_intra_chunk_weights(k, k, gam)).all()


# ------------------------------------------------------------------ the tensor-core precision plan

def _weak(L, seed):
    """A sequence whose per-channel decays are fifty times weaker than the workload's, so the state
    carries across many chunks (under the workload's decay a chunk forgets its start, which hides
    errors of the state path)."""
    inp = kda_prefill_inputs([L], seed=seed, geo=GEO)
    inp["g"] = inp["g"] * 0.02
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    o, st = oracle.kda_recurrence(y, inp["g"], inp["beta"], [0, L], 1, 1, 128, 128, GEO.q_scale,
                                  state_in=inp["state0"])
    a = y.double().numpy()
    args = (l2n(a[:, :128], 1e-6), l2n(a[:, 128:256], 1e-6), a[:, 256:], inp["g"][:, 0].double().numpy(),
            inp["beta"][:, 0].double().numpy(), inp["state0"][0, 0].double().numpy(), GEO.q_scale)
    return args, o[:, 0].numpy(), st[0, 0].numpy()


def _errors(args, o, st, split):
    O, S = chunked_chain_kda_tc(*args, split=split)
    return np.abs(O - o).max() / (2e-2 * np.abs(o).max()), _rel(S, st)


def test_tensor_core_plan_split_state_path_plain_output_path():
    """bf16 hi + lo on every state-path operand and plain bf16 on the output-only products: the
    state stays far inside 1e-4 relative L2 over 512 tokens of long memory, the output inside its
    bound."""
    args, o, st = _weak(512, 420)
    plan = dict(TC_SPLIT_ALL, Qg=False, S_o=False, P=False, E_o=False)
    out_ratio, state_rel = _errors(args, o, st, plan)
    assert out_ratio <= 0.5
    assert state_rel <= 1e-5


@pytest.mark.parametrize("operand", ["Kd", "E", "R", "T", "Kg", "S"])
def test_each_state_path_operand_needs_its_split(operand):
    """Negative controls: any one state-path operand left plain bf16 puts the state beyond its
    1e-4 tolerance under long memory."""
    args, o, st = _weak(512, 420)
    plan = dict(TC_SPLIT_ALL, Qg=False, S_o=False, P=False, E_o=False)
    plan[operand] = False
    _, state_rel = _errors(args, o, st, plan)
    assert state_rel > 1e-4, (operand, state_rel)


def test_tensor_core_gram_around_the_middle_token():
    """A and P of a chunk as one bf16 hi / lo tensor-core product around token 31 (the KDA prep
    kernel's way when the chunk's decay span allows it): against the 16-token sub-block form the
    lower triangle agrees to the split's precision, and the whole chain keeps the state within
    1e-5 relative L2 of the fp64 oracle over 512 tokens of long memory and under the workload's
    decay, the output within half its bound."""
    args, o, st = _weak(512, 420)
    q, k, gam = args[0][:64], args[1][:64], np.cumsum(args[3][:64].astype(np.float32), axis=0).astype(np.float32)
    exact = kda_intra_chunk_weights(k, k, gam).astype(np.float64)
    got = kda_gram_middle_reference(k, k, gam)
    low = np.tril(np.ones((64, 64), dtype=bool))
    assert np.abs(got - exact)[low].max() <= 1e-4 * np.abs(exact[low]).max()
    O, S = chunked_chain_kda_tc_middle(*args)
    assert np.abs(O - o).max() <= 0.5 * 2e-2 * np.abs(o).max()
    assert _rel(S, st) <= 1e-5
    inp = kda_prefill_inputs([256], seed=421, geo=GEO)   # the workload's decay, -U(0.001, 2)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    o2, st2 = oracle.kda_recurrence(y, inp["g"], inp["beta"], [0, 256], 1, 1, 128, 128, GEO.q_scale,
                                    state_in=inp["state0"])
    a = y.double().numpy()
    O2, S2 = chunked_chain_kda_tc_middle(l2n(a[:, :128], 1e-6), l2n(a[:, 128:256], 1e-6), a[:, 256:],
                                         inp["g"][:, 0].double().numpy(), inp["beta"][:, 0].double().numpy(),
                                         inp["state0"][0, 0].double().numpy(), GEO.q_scale)
    assert np.abs(O2 - o2[:, 0].numpy()).max() <= 0.5 * 2e-2 * np.abs(o2[:, 0].numpy()).max()
    assert _rel(S2, st2[0, 0].numpy()) <= 1e-5

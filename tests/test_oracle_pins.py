"""Pins of the CPU oracle against facts other than itself (CPU only).

Each test checks the oracle against a library routine, a closed form, an invariant the pages
state, exact rational arithmetic, or an independently structured algorithm, chosen so that a
dropped term, a wrong sign, a wrong index or a transposed operand in the oracle fails one of
them.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from linear_attention_ssm_gb300.synth import (Geometry, prefill_inputs, decode_inputs, cu_seqlens_of,
                                              kda_prefill_inputs)
from tests.chunked_numpy import chunked_chain, chunked_chain_kda, l2n

SMALL = Geometry(num_k_heads=2, num_v_heads=6, head_k_dim=8, head_v_dim=4, conv_width=4)


def bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


# ------------------------------------------------------------------ bf16 rounding

def _nearest_bf16_bruteforce(x: float) -> int:
    """Nearest bf16 to x among the three neighbours of a candidate, ties to the even pattern."""
    cand = int(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)[0]) & 0xFFFF
    best = None
    for b in (cand - 1, cand, cand + 1):
        b &= 0xFFFF
        val = float(torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)[0].float())
        if math.isnan(val) or math.isinf(val):
            continue
        d = abs(Fraction(x) - Fraction(val))
        key = (d, b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def test_round_bf16_matches_bruteforce_and_ties_to_even():
    rng = np.random.default_rng(0)
    xs = list(rng.standard_normal(300) * np.exp(rng.uniform(-20, 20, 300)))
    # exact midpoints between consecutive bf16 values must go to the even pattern
    for b in (0x3F80, 0x3F81, 0x4049, 0xC2F7, 0x0081):
        lo = float(torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)[0].float())
        hi = float(torch.tensor([b + 1], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)[0].float())
        xs.append((lo + hi) / 2)
    got = oracle.round_bf16(torch.tensor(xs, dtype=torch.float64)).view(torch.int16)
    for x, gbits in zip(xs, got.tolist()):
        assert (gbits & 0xFFFF) == _nearest_bf16_bruteforce(x), x


# ------------------------------------------------------------------ conv1d + SiLU

def _torch_conv_silu(x, w, cu, state_in):
    """Depthwise causal conv1d via torch.nn.functional.conv1d (fp64), then F.silu."""
    C, W = w.shape
    outs, states = [], []
    for n in range(cu.numel() - 1):
        s, e = int(cu[n]), int(cu[n + 1])
        hist = state_in[n].double().T if state_in is not None else torch.zeros(W - 1, C, dtype=torch.float64)
        seq = torch.cat([hist, x[s:e].double()], 0)  # [W-1+L, C]
        y = F.conv1d(seq.T[None], w.double()[:, None, :], groups=C)[0].T  # [L, C]
        outs.append(F.silu(y))
        states.append(seq[-(W - 1):].T)
    return torch.cat(outs, 0), torch.stack(states, 0)


@pytest.mark.parametrize("with_state", [False, True])
def test_conv_matches_torch_conv1d(with_state):
    gen = torch.Generator().manual_seed(1)
    lengths = [1, 2, 3, 5, 9]
    cu = cu_seqlens_of(lengths)
    T, C, W = sum(lengths), 24, 4
    x = torch.randn(T, C, generator=gen).to(torch.bfloat16)
    w = (0.5 * torch.randn(C, W, generator=gen)).to(torch.bfloat16)
    st = torch.randn(len(lengths), C, W - 1, generator=gen).to(torch.bfloat16) if with_state else None
    y, y_exact, st_out = oracle.conv1d_prefill(x, w, cu, st)
    ref, ref_state = _torch_conv_silu(x, w, cu, st)
    assert torch.allclose(y_exact, ref, rtol=1e-12, atol=1e-14)
    # the stored conv output is the exact value rounded once to bf16
    assert torch.equal(y.view(torch.int16), oracle.round_bf16(y_exact).view(torch.int16))
    # torch's own bf16 rounding of the fp64 value agrees to within one ulp everywhere
    ulp_gap = (y.view(torch.int16).int() - ref.to(torch.bfloat16).view(torch.int16).int()).abs()
    assert int(ulp_gap.max()) <= 1
    assert torch.equal(st_out.double(), ref_state)


def test_conv_split_call_equals_one_call():
    gen = torch.Generator().manual_seed(2)
    C, W, T = 16, 4, 11
    x = torch.randn(T, C, generator=gen).to(torch.bfloat16)
    w = torch.randn(C, W, generator=gen).to(torch.bfloat16)
    st0 = torch.randn(1, C, W - 1, generator=gen).to(torch.bfloat16)
    y_all, _, st_all = oracle.conv1d_prefill(x, w, [0, T], st0)
    for cut in (1, 2, 3, 7):
        y1, _, st1 = oracle.conv1d_prefill(x[:cut], w, [0, cut], st0)
        y2, _, st2 = oracle.conv1d_prefill(x[cut:], w, [0, T - cut], st1)
        assert torch.equal(torch.cat([y1, y2]).view(torch.int16), y_all.view(torch.int16))
        assert torch.equal(st2.view(torch.int16), st_all.view(torch.int16))


# ------------------------------------------------------------------ the recurrence

def _expand_qkv(qkv, geo):
    hk, hv, dk, dv = geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim
    T = qkv.shape[0]
    a = qkv.double().numpy()
    q = a[:, : hk * dk].reshape(T, hk, dk)
    k = a[:, hk * dk: 2 * hk * dk].reshape(T, hk, dk)
    v = a[:, 2 * hk * dk:].reshape(T, hv, dv)
    return q, k, v


def _product_form(qkv, g, beta, cu, geo, q_scale, eps, state0):
    """S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with explicit matrices;
    q/k heads expanded with np.repeat (repeat_interleave)."""
    hk, hv, dk = geo.num_k_heads, geo.num_v_heads, geo.head_k_dim
    q, k, v = _expand_qkv(qkv, geo)
    q = np.repeat(q, hv // hk, axis=1)
    k = np.repeat(k, hv // hk, axis=1)
    T = qkv.shape[0]
    o = np.zeros((T, hv, geo.head_v_dim))
    S_fin = np.zeros((len(cu) - 1, hv, geo.head_v_dim, dk))
    for n in range(len(cu) - 1):
        for h in range(hv):
            S = state0[n, h].double().numpy().copy()
            for t in range(int(cu[n]), int(cu[n + 1])):
                kn = l2n(k[t, h], eps)
                qn = l2n(q[t, h], eps)
                b = float(beta[t, h])
                S = math.exp(float(g[t, h])) * S @ (np.eye(dk) - b * np.outer(kn, kn)) + b * np.outer(v[t, h], kn)
                o[t, h] = q_scale * S @ qn
            S_fin[n, h] = S
    return o, S_fin


def test_recurrence_matches_product_form():
    geo = SMALL
    inp = prefill_inputs([5, 1, 9], seed=3, geo=geo, random_conv_state=True)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["conv_state0"])
    o, st = oracle.gdn_recurrence(y, inp["g"], inp["beta"], inp["cu_seqlens"], geo.num_k_heads,
                                  geo.num_v_heads, geo.head_k_dim, geo.head_v_dim, 0.37, 1e-6,
                                  inp["state0"])
    o_ref, st_ref = _product_form(y, inp["g"], inp["beta"], inp["cu_seqlens"], geo, 0.37, 1e-6, inp["state0"])
    np.testing.assert_allclose(o.numpy(), o_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(st.numpy(), st_ref, rtol=1e-11, atol=1e-13)


def test_recurrence_exact_rational_case():
    """Two tokens, Dk = Dv = 2, one head, eps = 0, g = 0: checked in exact rational arithmetic.
    k's are (3,4)/5 and (0,1); with g = 0 the product form has rational entries only."""
    geo = Geometry(num_k_heads=1, num_v_heads=1, head_k_dim=2, head_v_dim=2, conv_width=4)
    qraw = [[1.0, 0.0], [0.0, 2.0]]
    kraw = [[3.0, 4.0], [0.0, 1.0]]
    vraw = [[1.0, -2.0], [0.5, 3.0]]
    betas = [0.5, 0.25]
    qkv = bf([qraw[t] + kraw[t] + vraw[t] for t in range(2)])
    g = torch.zeros(2, 1)
    beta = torch.tensor([[b] for b in betas])
    S0 = torch.tensor([[[[0.5, -1.0], [2.0, 0.25]]]])
    o, st = oracle.gdn_recurrence(qkv, g, beta, [0, 2], 1, 1, 2, 2, 1.0, 0.0, S0)

    def nrm(x):
        n2 = sum(Fraction(a) ** 2 for a in x)
        r = Fraction(math.isqrt(n2.numerator), math.isqrt(n2.denominator))
        assert r * r == n2
        return [Fraction(a) / r for a in x]

    S = [[Fraction(0.5), Fraction(-1)], [Fraction(2), Fraction(0.25)]]
    outs = []
    for t in range(2):
        kn, qn, b = nrm(kraw[t]), nrm(qraw[t]), Fraction(betas[t])
        M = [[(1 if i == j else 0) - b * kn[i] * kn[j] for j in range(2)] for i in range(2)]
        S = [[sum(S[r][i] * M[i][c] for i in range(2)) + b * Fraction(vraw[t][r]) * kn[c]
              for c in range(2)] for r in range(2)]
        outs.append([sum(S[r][i] * qn[i] for i in range(2)) for r in range(2)])
    for t in range(2):
        for r in range(2):
            assert abs(float(o[t, 0, r]) - float(outs[t][r])) < 1e-14
    for r in range(2):
        for c in range(2):
            assert abs(float(st[0, 0, r, c]) - float(S[r][c])) < 1e-14


def test_beta_zero_is_pure_decay_closed_form():
    geo = SMALL
    inp = prefill_inputs([7, 3], seed=4, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    beta0 = torch.zeros_like(inp["beta"])
    o, st = oracle.gdn_recurrence(y, inp["g"], beta0, inp["cu_seqlens"], geo.num_k_heads, geo.num_v_heads,
                                  geo.head_k_dim, geo.head_v_dim, 0.5, 1e-6, inp["state0"])
    q, _, _ = _expand_qkv(y, geo)
    cu = inp["cu_seqlens"].tolist()
    for n in range(2):
        s, e = cu[n], cu[n + 1]
        for h in range(geo.num_v_heads):
            S0 = inp["state0"][n, h].double().numpy()
            gam = np.cumsum(inp["g"][s:e, h].double().numpy())
            np.testing.assert_allclose(st[n, h].numpy(), math.exp(gam[-1]) * S0, rtol=1e-12)
            for i, t in enumerate(range(s, e)):
                qn = l2n(q[t, h // 3], 1e-6)
                np.testing.assert_allclose(o[t, h].numpy(), 0.5 * math.exp(gam[i]) * S0 @ qn, rtol=1e-11, atol=1e-14)


def test_beta_one_projects_key_onto_value():
    """beta = 1, g = 0: after each token the state maps that token's (normalised) key to its value."""
    geo = SMALL
    inp = prefill_inputs([6], seed=5, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    _, k, v = _expand_qkv(y, geo)
    for L in range(1, 7):
        o, st = oracle.gdn_recurrence(y[:L], torch.zeros(L, geo.num_v_heads), torch.ones(L, geo.num_v_heads),
                                      [0, L], geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim,
                                      1.0, 1e-6, inp["state0"])
        for h in range(geo.num_v_heads):
            kn = l2n(k[L - 1, h // 3], 1e-6)
            # S k_hat = v exactly when ||k_hat|| = 1; with eps the norm is 1 - O(eps)
            Sk = st[0, h].numpy() @ kn
            resid = v[L - 1, h] - Sk
            assert np.abs(resid).max() < 1e-5 * max(1.0, np.abs(v[L - 1, h]).max())
    # with eps = 0 the property is exact to rounding
    o, st = oracle.gdn_recurrence(y[:3], torch.zeros(3, geo.num_v_heads), torch.ones(3, geo.num_v_heads),
                                  [0, 3], geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim,
                                  1.0, 0.0, inp["state0"])
    for h in range(geo.num_v_heads):
        kn = l2n(k[2, h // 3], 0.0)
        np.testing.assert_allclose(st[0, h].numpy() @ kn, v[2, h], rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_closed_form():
    """g = 0, beta = 1, orthonormal keys: S = S0 (I - sum k k^T) + sum v k^T."""
    dk, dv = 4, 3
    geo = Geometry(num_k_heads=1, num_v_heads=1, head_k_dim=dk, head_v_dim=dv, conv_width=4)
    gen = torch.Generator().manual_seed(6)
    T = 3
    keys = torch.zeros(T, dk)
    keys[0, 2], keys[1, 0], keys[2, 3] = 2.0, -1.0, 0.5   # orthogonal; normalised by the oracle
    qs = torch.randn(T, dk, generator=gen)
    vs = torch.randn(T, dv, generator=gen)
    qkv = torch.cat([qs, keys, vs], 1).to(torch.bfloat16)
    S0 = torch.randn(1, 1, dv, dk, generator=gen)
    o, st = oracle.gdn_recurrence(qkv, torch.zeros(T, 1), torch.ones(T, 1), [0, T], 1, 1, dk, dv, 1.0, 0.0, S0)
    kn = l2n(keys.double().numpy(), 0.0)
    vb = qkv[:, 2 * dk:].double().numpy()
    ref = S0[0, 0].double().numpy() @ (np.eye(dk) - kn.T @ kn) + vb.T @ kn
    np.testing.assert_allclose(st[0, 0].numpy(), ref, rtol=1e-12, atol=1e-12)


def test_state_layout_is_value_by_key():
    """With beta = 0 and g = 0 the output is q_scale * S0 q_hat: rows of S0 index the value dim."""
    dk, dv = 8, 4
    gen = torch.Generator().manual_seed(7)
    qkv = torch.randn(1, 2 * dk + dv, generator=gen).to(torch.bfloat16)
    S0 = torch.randn(1, 1, dv, dk, generator=gen)
    o, _ = oracle.gdn_recurrence(qkv, torch.zeros(1, 1), torch.zeros(1, 1), [0, 1], 1, 1, dk, dv, 1.0, 0.0, S0)
    qn = F.normalize(qkv[0, :dk].double(), dim=0)       # library normalisation (eps = 0 case)
    np.testing.assert_allclose(o[0, 0].numpy(), (S0[0, 0].double() @ qn).numpy(), rtol=1e-12)


def test_l2_norm_form_is_sqrt_sum_plus_eps():
    """A tiny q (norm 1e-4, eps 1e-6): x/sqrt(sum x^2 + eps), not x/max(||x||, eps)."""
    dk, dv = 2, 1
    qkv = torch.tensor([[1e-4, 0.0, 1.0, 0.0, 1.0]]).to(torch.bfloat16)
    q0 = float(qkv[0, 0].float())
    S0 = torch.tensor([[[[1.0, 0.0]]]])
    o, _ = oracle.gdn_recurrence(qkv, torch.zeros(1, 1), torch.zeros(1, 1), [0, 1], 1, 1, dk, dv, 1.0, 1e-6, S0)
    assert abs(float(o[0, 0, 0]) - q0 / math.sqrt(q0 * q0 + 1e-6)) < 1e-15
    assert abs(float(o[0, 0, 0]) - 1.0) > 0.5   # the max(norm, eps) form would give 1


def test_head_expansion_is_repeat_interleave():
    geo = SMALL
    ratio = geo.num_v_heads // geo.num_k_heads
    inp = prefill_inputs([9], seed=8, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    hk, dk = geo.num_k_heads, geo.head_k_dim
    T = y.shape[0]
    q = y[:, : hk * dk].reshape(T, hk, dk).repeat_interleave(ratio, dim=1).reshape(T, -1)
    k = y[:, hk * dk: 2 * hk * dk].reshape(T, hk, dk).repeat_interleave(ratio, dim=1).reshape(T, -1)
    expanded = torch.cat([q, k, y[:, 2 * hk * dk:]], 1)
    args = (inp["g"], inp["beta"], [0, T])
    o1, s1 = oracle.gdn_recurrence(y, *args, hk, geo.num_v_heads, dk, geo.head_v_dim, 0.3, 1e-6, inp["state0"])
    o2, s2 = oracle.gdn_recurrence(expanded, *args, geo.num_v_heads, geo.num_v_heads, dk, geo.head_v_dim,
                                   0.3, 1e-6, inp["state0"])
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    o3, _ = oracle.gdn_recurrence(y, *args, hk, geo.num_v_heads, dk, geo.head_v_dim, 0.3, 1e-6,
                                  inp["state0"], mutation=oracle.MUT_TILED_HEADS)
    assert not torch.allclose(o1, o3)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 80, 128, 130])
def test_sequential_oracle_equals_chunked_wy_form(L):
    geo = Geometry(num_k_heads=1, num_v_heads=3, head_k_dim=128, head_v_dim=128, conv_width=4)
    inp = prefill_inputs([L], seed=100 + L, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    qs = geo.q_scale
    o, st = oracle.gdn_recurrence(y, inp["g"], inp["beta"], [0, L], 1, 3, 128, 128, qs, 1e-6, inp["state0"])
    q, k, v = _expand_qkv(y, geo)
    for h in range(3):
        O, S = chunked_chain(l2n(q[:, 0], 1e-6), l2n(k[:, 0], 1e-6), v[:, h], inp["g"][:, h].double().numpy(),
                             inp["beta"][:, h].double().numpy(), inp["state0"][0, h].double().numpy(), qs)
        np.testing.assert_allclose(o[:, h].numpy(), O, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(st[0, h].numpy(), S, rtol=1e-9, atol=1e-11)


def test_split_sequence_with_carried_state_equals_one_call():
    geo = SMALL
    inp = prefill_inputs([20], seed=9, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    a = (geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim, 0.25, 1e-6)
    o, st = oracle.gdn_recurrence(y, inp["g"], inp["beta"], [0, 20], *a, inp["state0"])
    o1, st1 = oracle.gdn_recurrence(y[:13], inp["g"][:13], inp["beta"][:13], [0, 13], *a, inp["state0"])
    o2, st2 = oracle.gdn_recurrence(y[13:], inp["g"][13:], inp["beta"][13:], [0, 7], *a, st1)
    assert torch.equal(torch.cat([o1, o2]), o) and torch.equal(st2, st)


# ------------------------------------------------------------------ gated RMSNorm

def test_gated_rmsnorm_matches_torch_rms_norm_times_sigmoid():
    gen = torch.Generator().manual_seed(10)
    o = torch.randn(5, 3, 16, generator=gen, dtype=torch.float64)
    z = torch.randn(5, 3, 16, generator=gen).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(16, generator=gen)).to(torch.bfloat16)
    out = oracle.gated_rmsnorm(o, z, w, 1e-6)
    ref = F.rms_norm(o, (16,), weight=w.double(), eps=1e-6) * torch.sigmoid(z.double())
    assert torch.allclose(out, ref, rtol=1e-13, atol=1e-15)
    # sigma(0) = 1/2
    half = oracle.gated_rmsnorm(o, torch.zeros_like(z), w, 1e-6)
    assert torch.allclose(half, 0.5 * F.rms_norm(o, (16,), weight=w.double(), eps=1e-6), rtol=1e-14)
    # a constant row normalises to sign(o) * |o| / sqrt(o^2 + eps)
    c = torch.full((1, 16), -3.0, dtype=torch.float64)
    big = torch.full((1, 16), 40.0).to(torch.bfloat16)   # sigmoid(40) = 1 - 4e-18
    one = torch.ones(16).to(torch.bfloat16)
    out_c = oracle.gated_rmsnorm(c, big, one, 1e-6)
    assert torch.allclose(out_c, torch.full_like(c, -3.0 / math.sqrt(9.0 + 1e-6)), rtol=1e-14)
    silu = oracle.gated_rmsnorm(o, z, w, 1e-6, mutation=oracle.MUT_SILU_GATE)
    assert not torch.allclose(silu, out, rtol=1e-3)


# ------------------------------------------------------------------ decode

def test_decode_steps_equal_prefill():
    """T decode steps equal one T-token prefill of every sequence (conv step = full conv)."""
    geo = SMALL
    B, T = 3, 5
    d = decode_inputs(B, T, seed=11, geo=geo)
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    cs, st = d["conv_state0"], d["state0"].double()
    outs = []
    for s in range(T):
        out, _, cs, st = oracle.decode_step(d["x"][s], d["conv_w"], cs, d["g"][s], d["beta"][s], st,
                                            d["z"][s], d["norm_w"], **a)
        outs.append(out)
    dec = torch.stack(outs, 1)  # [B, T, Hv, Dv]
    # the same tokens as B packed sequences of length T
    x = d["x"].transpose(0, 1).reshape(B * T, -1)
    g = d["g"].transpose(0, 1).reshape(B * T, -1)
    beta = d["beta"].transpose(0, 1).reshape(B * T, -1)
    z = d["z"].transpose(0, 1).reshape(B * T, geo.num_v_heads, geo.head_v_dim)
    ref = oracle.prefill(x, d["conv_w"], cu_seqlens_of([T] * B), g, beta, z, d["norm_w"],
                         state_in=d["state0"], conv_state_in=d["conv_state0"], **a)
    assert torch.allclose(dec.reshape(B * T, geo.num_v_heads, -1), ref["out"], rtol=1e-12, atol=1e-14)
    assert torch.allclose(st, ref["state"], rtol=1e-12, atol=1e-14)
    assert torch.equal(cs.view(torch.int16), ref["conv_state"].view(torch.int16))


# ------------------------------------------------------------------ mutations are live

@pytest.mark.parametrize("mut", [oracle.MUT_NO_CONV, oracle.MUT_DROP_CARRY, oracle.MUT_TRANSPOSE,
                                 oracle.MUT_TILED_HEADS, oracle.MUT_CONV_SHIFT, oracle.MUT_DECAY_SIGN,
                                 oracle.MUT_NO_BETA, oracle.MUT_SILU_GATE, oracle.MUT_NO_QNORM])
def test_each_planted_mutation_changes_the_output(mut):
    geo = SMALL
    inp = prefill_inputs([130], seed=12, geo=geo)
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=geo.q_scale, state_in=inp["state0"])
    base = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                          inp["norm_w"], **a)
    mutd = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                          inp["norm_w"], mutation=mut, **a)
    assert (base["out"] - mutd["out"]).abs().max() > 1e-3


# ------------------------------------------------------------------ decode with an fp16 state

def _f16_bits_numpy(xs):
    """numpy's double -> binary16 conversion (round to nearest, ties to even), as bit patterns."""
    with np.errstate(over="ignore"):
        return np.asarray(xs, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_f16_widening_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_double(torch.from_numpy(bits.view(np.int16)).view(torch.float16)).numpy()
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))  # -0 stays -0


def test_round_f16_matches_numpy_and_ties_to_even():
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(2000) * np.exp2(rng.uniform(-30, 17, 2000)))
    # exact midpoints between neighbours (normal, subnormal, across a binade) go to the even pattern
    for b in (0x3C00, 0x3C01, 0x0001, 0x0002, 0x03FF, 0x0400, 0x7BFE, 0xBC00, 0x8001):
        lo = float(np.uint16(b).view(np.float16))
        hi = float(np.uint16(b + 1).view(np.float16))
        xs.append((lo + hi) / 2)
        xs.append(np.nextafter((lo + hi) / 2, np.inf))
        xs.append(np.nextafter((lo + hi) / 2, -np.inf))
    # overflow boundary: 65504 is the largest finite value; from the midpoint 65520 up -> inf
    xs += [65504.0, 65519.99, 65520.0, 65536.0, -65520.0, 1e6, 2.0 ** -25, 2.0 ** -26, -0.0, 0.0]
    got = oracle.round_f16(torch.tensor(xs, dtype=torch.float64)).view(torch.int16).numpy().view(np.uint16)
    want = _f16_bits_numpy(xs)
    bad = [(x, hex(a), hex(b)) for x, a, b in zip(xs, got, want) if a != b]
    assert not bad, bad[:5]
    # the midpoint between 1 and its successor goes down to the even 1.0, the next one up to 0x3C02
    assert int(got[2000]) == 0x3C00 and int(got[2003]) == 0x3C02


def _h16_decode_args(d, s=0):
    return (d["x"][s], d["conv_w"], d["conv_state0"], d["g"][s], d["beta"][s])


def test_decode_h16_beta_zero_is_rounded_decay():
    """beta = 0: the new fp16 state is exp(g) * S rounded once to binary16 (numpy's rounding of the
    double product), and g = 0 as well leaves every state pattern unchanged."""
    geo = SMALL
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    d = decode_inputs(3, 1, seed=31, geo=geo)
    h = d["state0"].to(torch.float16)
    beta0 = torch.zeros_like(d["beta"][0])
    x, cw, cs, g, _ = _h16_decode_args(d)
    _, _, _, st = oracle.decode_step_h16(x, cw, cs, g, beta0, h, d["z"][0], d["norm_w"], **a)
    alpha = np.exp(g.double().numpy())[:, :, None, None]
    want = _f16_bits_numpy(alpha * h.numpy().astype(np.float64))
    assert np.array_equal(st.view(torch.int16).numpy().view(np.uint16), want)
    h_nz = torch.where(h == 0, torch.full_like(h, 0.5), h)  # no zeros: -0 + 0 would give +0
    _, _, _, st0 = oracle.decode_step_h16(x, cw, cs, torch.zeros_like(g), beta0, h_nz, d["z"][0], d["norm_w"], **a)
    assert torch.equal(st0.view(torch.int16), h_nz.view(torch.int16))


def test_decode_h16_output_uses_the_state_before_rounding():
    """The output of an fp16-state step equals the fp64 step's output from the widened state (the
    rounding applies to the stored state only), and the stored state is within half a binary16
    quantum of the fp64 step's state."""
    geo = SMALL
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    d = decode_inputs(4, 1, seed=32, geo=geo)
    h = d["state0"].to(torch.float16)
    args = _h16_decode_args(d)
    out16, o16, cs16, st16 = oracle.decode_step_h16(*args, h, d["z"][0], d["norm_w"], **a)
    out64, o64, cs64, st64 = oracle.decode_step(*args, h.double(), d["z"][0], d["norm_w"], **a)
    assert torch.equal(out16, out64) and torch.equal(o16, o64)
    assert torch.equal(cs16.view(torch.int16), cs64.view(torch.int16))
    exact = st64.numpy()
    got = st16.numpy().astype(np.float64)
    _, ex = np.frexp(np.abs(exact))
    quantum = np.exp2(np.maximum(ex - 11, -24))
    assert np.all(np.abs(got - exact) <= quantum / 2)
    assert np.any(got != exact)  # the rounding is live


def test_decode_h16_drift_stays_at_rounding_level():
    """Eight fp16-state steps stay within a few binary16 half-quanta of the fp64-state chain."""
    geo = SMALL
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    d = decode_inputs(2, 8, seed=33, geo=geo)
    h, s64 = d["state0"].to(torch.float16), d["state0"].to(torch.float16).double()
    cs16 = cs64 = d["conv_state0"]
    for s in range(8):
        o16, _, cs16, h = oracle.decode_step_h16(d["x"][s], d["conv_w"], cs16, d["g"][s], d["beta"][s], h,
                                                 d["z"][s], d["norm_w"], **a)
        o64, _, cs64, s64 = oracle.decode_step(d["x"][s], d["conv_w"], cs64, d["g"][s], d["beta"][s], s64,
                                               d["z"][s], d["norm_w"], **a)
        rel = ((h.double() - s64).norm() / s64.norm()).item()
        assert rel < 2.0 ** -10, (s, rel)
        assert (o16 - o64).abs().max().item() <= 2e-2 * o64.abs().max().item()


# ------------------------------------------------------------------ multi-token verify + commit

def _verify_inputs(B, K, seed, geo):
    d = decode_inputs(B, K, seed=seed, geo=geo)
    # [steps, B, ...] -> [B, K, ...]
    return {k: (v.transpose(0, 1).contiguous() if k in ("x", "g", "beta", "z") else v) for k, v in d.items()}


def test_verify_rows_equal_a_prefill_and_commit_selects_the_prefix_state():
    """Verify outputs equal a K-token prefill of each sequence from the same states; the committed
    states equal an m-token prefill's final states (m = 0: the prior states, bit for bit), and the
    committed conv state is the last W-1 raw inputs of [prior conv state, the m rows]."""
    geo = SMALL
    B, K = 5, 6
    v = _verify_inputs(B, K, seed=41, geo=geo)
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    m = [0, 1, 3, 6, 2]
    out, cs, st = oracle.verify(v["x"], v["conv_w"], v["conv_state0"], v["g"], v["beta"], v["state0"], v["z"],
                                v["norm_w"], m, **a)
    C = v["x"].shape[-1]
    for b in range(B):
        ref = oracle.prefill(v["x"][b], v["conv_w"], cu_seqlens_of([K]), v["g"][b], v["beta"][b], v["z"][b],
                             v["norm_w"], state_in=v["state0"][b:b + 1], conv_state_in=v["conv_state0"][b:b + 1], **a)
        assert torch.allclose(out[b], ref["out"], rtol=1e-12, atol=1e-14)
        if m[b] == 0:
            assert torch.equal(st[b], v["state0"][b].double())
            assert torch.equal(cs[b].view(torch.int16), v["conv_state0"][b].view(torch.int16))
            continue
        pre = oracle.prefill(v["x"][b, :m[b]], v["conv_w"], cu_seqlens_of([m[b]]), v["g"][b, :m[b]],
                             v["beta"][b, :m[b]], v["z"][b, :m[b]], v["norm_w"], state_in=v["state0"][b:b + 1],
                             conv_state_in=v["conv_state0"][b:b + 1], **a)
        assert torch.allclose(st[b], pre["state"][0], rtol=1e-12, atol=1e-14)
        window = torch.cat([v["conv_state0"][b].T, v["x"][b, :m[b]]], 0)  # [3 + m, C], oldest first
        assert torch.equal(cs[b].view(torch.int16), window[-3:].T.contiguous().view(torch.int16))
        assert cs[b].shape == (C, 3)


def test_verify_refuses_committed_rows_out_of_range():
    geo = SMALL
    v = _verify_inputs(2, 3, seed=42, geo=geo)
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    for bad in ([0, 4], [-1, 0], [1]):
        with pytest.raises(ValueError):
            oracle.verify(v["x"], v["conv_w"], v["conv_state0"], v["g"], v["beta"], v["state0"], v["z"],
                          v["norm_w"], bad, **a)


def test_verify_h16_rounds_only_the_committed_state():
    """The binary16-state verify: outputs equal the fp64 verify's from the widened state; a
    committed state is numpy's binary16 rounding of the fp64 committed state; an abort keeps the
    bits."""
    geo = SMALL
    B, K = 3, 4
    v = _verify_inputs(B, K, seed=43, geo=geo)
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=0.3)
    h = v["state0"].to(torch.float16)
    m = [0, 2, 4]
    out16, cs16, st16 = oracle.verify_h16(v["x"], v["conv_w"], v["conv_state0"], v["g"], v["beta"], h, v["z"],
                                          v["norm_w"], m, **a)
    out64, cs64, st64 = oracle.verify(v["x"], v["conv_w"], v["conv_state0"], v["g"], v["beta"], h.double(), v["z"],
                                      v["norm_w"], m, **a)
    assert torch.equal(out16, out64) and torch.equal(cs16.view(torch.int16), cs64.view(torch.int16))
    assert torch.equal(st16[0].view(torch.int16), h[0].view(torch.int16))
    for b in (1, 2):
        want = _f16_bits_numpy(st64[b].numpy())
        assert np.array_equal(st16[b].view(torch.int16).numpy().view(np.uint16), want)


# ------------------------------------------------------------------ gate derivation (parity unpinned)

def test_gates_match_torch_softplus_and_sigmoid():
    """The gates against torch's own softplus and sigmoid in fp64 (library routines)."""
    gen = torch.Generator().manual_seed(44)
    T, hv = 37, 6
    a = (3 * torch.randn((T, hv), generator=gen)).to(torch.bfloat16)
    b = (3 * torch.randn((T, hv), generator=gen)).to(torch.bfloat16)
    A_log = torch.rand(hv, generator=gen) * 3 - 1
    dt_bias = torch.randn(hv, generator=gen)
    g, beta = oracle.gates(a, b, A_log, dt_bias)
    want_g = -torch.exp(A_log.double()) * F.softplus(a.double() + dt_bias.double(), threshold=1e9)
    assert torch.allclose(g, want_g, rtol=1e-13, atol=0)
    assert torch.allclose(beta, torch.sigmoid(b.double()), rtol=1e-14, atol=0)


def test_gates_closed_forms():
    """a = -dt_bias gives g = -exp(A_log) ln 2; b = 0 gives beta = 1/2; beta(-b) = 1 - beta(b);
    g < 0 and g -> 0 as a -> -inf; large arguments do not overflow."""
    hv = 3
    A_log = torch.tensor([0.0, 1.0, -2.0])
    dt_bias = torch.tensor([0.5, -1.0, 2.0])
    a = (-dt_bias).to(torch.bfloat16).reshape(1, hv)   # exact in bf16
    b = torch.zeros((1, hv), dtype=torch.bfloat16)
    g, beta = oracle.gates(a, b, A_log, dt_bias)
    assert torch.allclose(g[0], -torch.exp(A_log.double()) * math.log(2.0), rtol=1e-15, atol=0)
    assert torch.equal(beta, torch.full((1, hv), 0.5, dtype=torch.float64))
    bb = torch.tensor([[1.5, -1.5, 7.0]]).to(torch.bfloat16)
    _, b1 = oracle.gates(a, bb, A_log, dt_bias)
    _, b2 = oracle.gates(a, (-bb.float()).to(torch.bfloat16), A_log, dt_bias)
    assert torch.allclose(b1 + b2, torch.ones_like(b1), rtol=0, atol=1e-15)
    far = torch.tensor([[-80.0, 80.0, 800.0]]).to(torch.bfloat16)
    g2, _ = oracle.gates(far, b, A_log, torch.zeros(hv))
    assert torch.isfinite(g2).all() and (g2 < 0).all()
    assert abs(g2[0, 0].item()) < 1e-30                       # softplus(-80) ~ e^-80
    assert abs(g2[0, 2].item() + math.exp(-2.0) * 800.0) < 1e-9  # softplus(x) -> x


# ------------------------------------------------------------------ KDA decode (per-channel decay)

KDA_GEO = Geometry(num_k_heads=3, num_v_heads=3, head_k_dim=8, head_v_dim=4, conv_width=4)


def _kda_args(geo):
    return dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
                head_v_dim=geo.head_v_dim, q_scale=0.35)


def test_kda_with_a_channel_constant_decay_is_the_gdn_step():
    """A per-channel decay equal on every key channel is the scalar decay of the GDN step (an
    independent code path), for every output and state element."""
    geo = KDA_GEO
    d = decode_inputs(4, 1, seed=45, geo=geo)
    a = _kda_args(geo)
    g_vec = d["g"][0][:, :, None].expand(4, geo.num_v_heads, geo.head_k_dim).contiguous()
    args = (d["x"][0], d["conv_w"], d["conv_state0"])
    kda = oracle.kda_decode_step(*args, g_vec, d["beta"][0], d["state0"], d["z"][0], d["norm_w"], **a)
    gdn = oracle.decode_step(*args, d["g"][0], d["beta"][0], d["state0"], d["z"][0], d["norm_w"], **a)
    for got, want in zip((kda[0], kda[1], kda[3]), (gdn[0], gdn[1], gdn[3])):
        assert torch.allclose(got, want, rtol=1e-12, atol=1e-14)
    assert torch.equal(kda[2].view(torch.int16), gdn[2].view(torch.int16))


def test_kda_beta_zero_decays_each_key_column():
    """beta = 0: the new state is S with key column i scaled by exp(g_i) (numpy), and the clamp
    limits the decay to exp(g_min)."""
    geo = KDA_GEO
    d = decode_inputs(2, 1, seed=46, geo=geo)
    a = _kda_args(geo)
    gen = torch.Generator().manual_seed(46)
    g_vec = -4 * torch.rand((2, geo.num_v_heads, geo.head_k_dim), generator=gen)
    beta0 = torch.zeros_like(d["beta"][0])
    args = (d["x"][0], d["conv_w"], d["conv_state0"])
    _, _, _, st = oracle.kda_decode_step(*args, g_vec, beta0, d["state0"], d["z"][0], d["norm_w"], **a)
    want = d["state0"].double().numpy() * np.exp(g_vec.double().numpy())[:, :, None, :]
    np.testing.assert_allclose(st.numpy(), want, rtol=1e-14, atol=0)
    _, _, _, stc = oracle.kda_decode_step(*args, g_vec, beta0, d["state0"], d["z"][0], d["norm_w"],
                                          g_min=-1.0, **a)
    wantc = d["state0"].double().numpy() * np.exp(np.maximum(g_vec.double().numpy(), -1.0))[:, :, None, :]
    np.testing.assert_allclose(stc.numpy(), wantc, rtol=1e-14, atol=0)


@pytest.mark.parametrize("mut", [oracle.MUT_DECAY_SIGN, oracle.MUT_NO_BETA, oracle.MUT_TRANSPOSE,
                                 oracle.MUT_NO_QNORM])
def test_kda_planted_mutations_change_the_result(mut):
    """The ledger's RED list for the KDA decode (wrong decay sign, missing beta or q scaling,
    transposed state) is live in the oracle."""
    geo = KDA_GEO
    d = decode_inputs(3, 1, seed=47, geo=geo)
    a = _kda_args(geo)
    gen = torch.Generator().manual_seed(47)
    g_vec = -2 * torch.rand((3, geo.num_v_heads, geo.head_k_dim), generator=gen)
    args = (d["x"][0], d["conv_w"], d["conv_state0"], g_vec, d["beta"][0], d["state0"], d["z"][0], d["norm_w"])
    base = oracle.kda_decode_step(*args, **a)
    bad = oracle.kda_decode_step(*args, mutation=mut, **a)
    assert (base[0] - bad[0]).abs().max() > 1e-3 or (base[3] - bad[3]).abs().max() > 1e-3


# ------------------------------------------------------------------ KDA prefill (sequential form)

def _geo_args(geo):
    return (geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim)


def test_kda_recurrence_with_a_channel_constant_decay_is_the_gdn_recurrence():
    """Ragged sequences, 3 V heads per K head: a decay equal on every key channel reproduces the
    scalar-decay recurrence exactly."""
    geo = SMALL
    inp = prefill_inputs([7, 1, 12], seed=60, geo=geo, random_conv_state=True)
    T = sum(inp["lengths"])
    g_vec = inp["g"][:, :, None].expand(T, geo.num_v_heads, geo.head_k_dim).contiguous()
    common = (inp["x"], inp["conv_w"], inp["cu_seqlens"])
    tail = (inp["beta"], inp["z"], inp["norm_w"], *_geo_args(geo), 0.3)
    kda = oracle.kda_prefill(*common, g_vec, *tail, state_in=inp["state0"], conv_state_in=inp["conv_state0"])
    gdn = oracle.prefill(*common, inp["g"], *tail, state_in=inp["state0"], conv_state_in=inp["conv_state0"])
    for key in ("o", "out", "state"):
        assert torch.equal(kda[key], gdn[key]), key


@pytest.mark.parametrize("g_min", [float("-inf"), -1.0])
def test_kda_prefill_equals_consecutive_kda_decode_steps(g_min):
    """Per sequence, the prefill (conv over the packed rows, token chain) and one KDA decode step
    per token (conv shift register, the decode oracle's own step) give the same outputs and final
    states; the clamp enters both."""
    geo = Geometry(num_k_heads=2, num_v_heads=4, head_k_dim=8, head_v_dim=6, conv_width=4)
    lengths = [5, 1, 3]
    inp = kda_prefill_inputs(lengths, seed=61, geo=geo, random_conv_state=True)
    qs = 0.4
    pre = oracle.kda_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                             inp["norm_w"], *_geo_args(geo), qs, g_min=g_min, state_in=inp["state0"],
                             conv_state_in=inp["conv_state0"])
    a = dict(num_k_heads=geo.num_k_heads, num_v_heads=geo.num_v_heads, head_k_dim=geo.head_k_dim,
             head_v_dim=geo.head_v_dim, q_scale=qs, g_min=g_min)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        cs, st = inp["conv_state0"][n:n + 1], inp["state0"][n:n + 1].double()
        for t in range(cu[n], cu[n + 1]):
            out, _, cs, st = oracle.kda_decode_step(inp["x"][t:t + 1], inp["conv_w"], cs, inp["g"][t:t + 1],
                                                    inp["beta"][t:t + 1], st, inp["z"][t:t + 1], inp["norm_w"], **a)
            np.testing.assert_allclose(out[0].numpy(), pre["out"][t].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(st[0].numpy(), pre["state"][n].numpy(), rtol=1e-10, atol=1e-13)
        assert torch.equal(cs[0].view(torch.int16), pre["conv_state"][n].view(torch.int16))


def test_kda_recurrence_matches_the_matrix_product_form():
    """numpy, token by token, in the product form S_t = S_{t-1} diag(alpha_t) (I - beta k k^T) +
    beta v k^T with alpha_t = exp(max(g_t, g_min)) over the key channels; o_t = q_scale S_t q_t.
    Dk != Dv, so a decay on the value rows instead of the key columns cannot pass."""
    dk, dv, L, g_min, qs = 8, 5, 9, -1.5, 0.7
    gen = torch.Generator().manual_seed(62)
    qkv = torch.randn(L, 2 * dk + dv, generator=gen).to(torch.bfloat16)
    g = -4 * torch.rand(L, 1, dk, generator=gen)
    beta = torch.rand(L, 1, generator=gen)
    S0 = torch.randn(1, 1, dv, dk, generator=gen)
    o, st = oracle.kda_recurrence(qkv, g, beta, [0, L], 1, 1, dk, dv, qs, g_min, 1e-6, S0)
    y = qkv.double().numpy()
    S = S0[0, 0].double().numpy()
    for t in range(L):
        q, k, v = l2n(y[t, :dk], 1e-6), l2n(y[t, dk:2 * dk], 1e-6), y[t, 2 * dk:]
        alpha = np.exp(np.maximum(g[t, 0].double().numpy(), g_min))
        b = float(beta[t, 0])
        S = S @ np.diag(alpha) @ (np.eye(dk) - b * np.outer(k, k)) + b * np.outer(v, k)
        np.testing.assert_allclose(o[t, 0].numpy(), qs * S @ q, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(st[0, 0].numpy(), S, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 130])
def test_kda_sequential_oracle_equals_chunked_wy_form(L):
    """The ledger's KDA prefill boundary (63/64/65 tokens around a 64-token chunk): the token
    chain and the per-channel chunk-wise form agree in output and final state."""
    geo = Geometry(num_k_heads=1, num_v_heads=2, head_k_dim=128, head_v_dim=64, conv_width=4)
    inp = kda_prefill_inputs([L], seed=200 + L, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    qs = geo.q_scale
    o, st = oracle.kda_recurrence(y, inp["g"], inp["beta"], [0, L], *_geo_args(geo), qs, state_in=inp["state0"])
    q, k, v = _expand_qkv(y, geo)
    for h in range(2):
        O, S = chunked_chain_kda(l2n(q[:, 0], 1e-6), l2n(k[:, 0], 1e-6), v[:, h], inp["g"][:, h].double().numpy(),
                                 inp["beta"][:, h].double().numpy(), inp["state0"][0, h].double().numpy(), qs)
        np.testing.assert_allclose(o[:, h].numpy(), O, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(st[0, h].numpy(), S, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("mut", [oracle.MUT_DECAY_SIGN, oracle.MUT_NO_BETA, oracle.MUT_TRANSPOSE,
                                 oracle.MUT_DROP_CARRY])
def test_kda_recurrence_planted_mutations_fail_the_chunked_form(mut):
    """A wrong decay sign, a missing beta, a transposed state or a dropped carry in the oracle's
    KDA chain is caught by the chunked form."""
    geo = Geometry(num_k_heads=1, num_v_heads=1, head_k_dim=16, head_v_dim=16, conv_width=4)
    L = 70
    inp = kda_prefill_inputs([L], seed=63, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    o, st = oracle.kda_recurrence(y, inp["g"], inp["beta"], [0, L], *_geo_args(geo), 0.5,
                                  state_in=inp["state0"], mutation=mut)
    q, k, v = _expand_qkv(y, geo)
    O, S = chunked_chain_kda(l2n(q[:, 0], 1e-6), l2n(k[:, 0], 1e-6), v[:, 0], inp["g"][:, 0].double().numpy(),
                             inp["beta"][:, 0].double().numpy(), inp["state0"][0, 0].double().numpy(), 0.5)
    assert np.abs(o[:, 0].numpy() - O).max() > 1e-3 or np.abs(st[0, 0].numpy() - S).max() > 1e-3



# ------------------------------------------------------------------ normalisation and packing invariants

def test_l2_normalisation_makes_q_and_k_scale_free():
    """With eps = 0, doubling every q and k channel (exact in bf16) leaves outputs and states
    unchanged: the recurrence sees only q/||q|| and k/||k||.  The planted no-q-norm mistake is not
    scale free."""
    geo = SMALL
    inp = prefill_inputs([11, 6], seed=64, geo=geo)
    y, _, _ = oracle.conv1d_prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"])
    y2 = y.clone()
    nqk = 2 * geo.num_k_heads * geo.head_k_dim
    y2[:, :nqk] = y[:, :nqk] * 2
    a = (inp["g"], inp["beta"], inp["cu_seqlens"], geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim,
         0.3, 0.0, inp["state0"])
    o1, s1 = oracle.gdn_recurrence(y, *a)
    o2, s2 = oracle.gdn_recurrence(y2, *a)
    np.testing.assert_allclose(o2.numpy(), o1.numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(s2.numpy(), s1.numpy(), rtol=1e-13, atol=1e-15)
    b1, _ = oracle.gdn_recurrence(y, *a, mutation=oracle.MUT_NO_QNORM)
    b2, _ = oracle.gdn_recurrence(y2, *a, mutation=oracle.MUT_NO_QNORM)
    assert (b2 - b1).abs().max() > 1e-3


@pytest.mark.parametrize("kda", [False, True], ids=["gdn", "kda"])
def test_packed_sequences_equal_separate_runs(kda):
    """A varlen call over packed sequences (one empty) gives, per sequence, exactly what a call
    on that sequence alone gives."""
    geo = SMALL
    lengths = [7, 0, 13, 1]
    inp = (kda_prefill_inputs if kda else prefill_inputs)(lengths, seed=65, geo=geo, random_conv_state=True)
    run = oracle.kda_prefill if kda else oracle.prefill
    a = (geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim, 0.3)
    packed = run(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"], inp["norm_w"], *a,
                 state_in=inp["state0"], conv_state_in=inp["conv_state0"])
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        one = run(inp["x"][s:e], inp["conv_w"], [0, e - s], inp["g"][s:e], inp["beta"][s:e], inp["z"][s:e],
                  inp["norm_w"], *a, state_in=inp["state0"][n:n + 1], conv_state_in=inp["conv_state0"][n:n + 1])
        assert torch.equal(one["out"], packed["out"][s:e])
        assert torch.equal(one["state"][0], packed["state"][n])
        assert torch.equal(one["conv_state"][0].view(torch.int16), packed["conv_state"][n].view(torch.int16))

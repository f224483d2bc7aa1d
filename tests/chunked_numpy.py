"""The chunk-wise (WY) form of the gated delta rule, in plain numpy fp64 (test helper).

This is a second, independently structured derivation of the same recurrence, following the
stage order the pegainfer PR #1152 page gives for its production prefill ("prepare -> cumsum ->
A -> solve -> recompute -> state -> output", Consumer / Shipped-line diff) with 64-token
chunks.  The sequential oracle must agree with it at any length, in particular across chunk
boundaries (GLM-5.3-Flash kernel TDD ledger, slice I4: "chunk path matches sequential state
and output" at 63/64/65).  It is used only to pin the oracle and to document the chunk algebra
that the CUDA kernels implement; it is never compared against the GPU directly.

Within one chunk of length L (tokens 1..L), with gamma_t = sum_{i<=t} g_i:
  A[t, j]  = beta_t exp(gamma_t - gamma_j) k_t . k_j          (j < t, else 0)
  T        = (I + A)^-1                                        (unit lower triangular)
  U        = T diag(beta) V,   W = T diag(beta exp(gamma)) K
  E        = U - W S0^T                                        (rows e_t^T)
  O        = q_scale [diag(exp(gamma)) Q S0^T + (mask_{j<=t} exp(gamma_t - gamma_j) Q K^T) E]
  S_L      = exp(gamma_L) S0 + E^T diag(exp(gamma_L - gamma)) K
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def l2n(x, eps):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def chunked_chain(q, k, v, g, beta, S0, q_scale, chunk=64):
    """q, k: [T, Dk] (already L2-normalised); v: [T, Dv]; g, beta: [T]; S0: [Dv, Dk]."""
    T = q.shape[0]
    S = S0.astype(np.float64).copy()
    O = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        Q, K, V, G, B = q[sl], k[sl], v[sl], g[sl], beta[sl]
        L = Q.shape[0]
        gam = np.cumsum(G)
        diff = gam[:, None] - gam[None, :]
        lower_strict = np.tril(np.ones((L, L)), -1)
        lower_incl = np.tril(np.ones((L, L)), 0)
        decay = np.exp(np.where(lower_incl > 0, diff, -np.inf))
        A = (B[:, None] * decay * (K @ K.T)) * lower_strict
        Tm = solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True)
        U = Tm @ (B[:, None] * V)
        W = Tm @ ((B * np.exp(gam))[:, None] * K)
        E = U - W @ S.T
        P = decay * (Q @ K.T) * lower_incl
        O[sl] = q_scale * ((np.exp(gam)[:, None] * Q) @ S.T + P @ E)
        S = np.exp(gam[-1]) * S + E.T @ (np.exp(gam[-1] - gam)[:, None] * K)
    return O, S


def chunked_chain_kda(q, k, v, g, beta, S0, q_scale, chunk=64):
    """The same chunk-wise form with a per-key-channel log decay (KDA).

    q, k: [T, Dk] (L2-normalised); v: [T, Dv]; g: [T, Dk] (already clamped); beta: [T];
    S0: [Dv, Dk].  Within a chunk, Gamma_t = sum_{i<=t} g_i is a vector over the key channels and
    every decay between tokens j <= t is the per-channel factor exp(Gamma_t - Gamma_j), taken
    from the difference directly (never as a product of exp(Gamma_t) and exp(-Gamma_j), which
    leaves the range of doubles over a long chunk):
      A[t, j] = beta_t sum_i k_ti k_ji exp(Gamma_ti - Gamma_ji)       (j < t)
      U = T diag(beta) V,   W = T diag(beta) (K * exp(Gamma)),   E = U - W S0^T
      P[t, j] = sum_i q_ti k_ji exp(Gamma_ti - Gamma_ji)              (j <= t)
      O = q_scale [(Q * exp(Gamma)) S0^T + P E]
      S_L = S0 diag(exp(Gamma_L)) + E^T (K * exp(Gamma_L - Gamma))
    """
    T = q.shape[0]
    S = S0.astype(np.float64).copy()
    O = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        Q, K, V, G, B = q[sl], k[sl], v[sl], g[sl], beta[sl]
        L = Q.shape[0]
        gam = np.cumsum(G, axis=0)                                  # [L, Dk]
        lower_incl = np.tril(np.ones((L, L)), 0) > 0
        diff = np.where(lower_incl[:, :, None], gam[:, None, :] - gam[None, :, :], -np.inf)
        decay = np.exp(diff)                                        # [t, j, i]
        A = B[:, None] * np.einsum("ti,ji,tji->tj", K, K, decay) * np.tril(np.ones((L, L)), -1)
        Tm = solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True)
        U = Tm @ (B[:, None] * V)
        W = Tm @ (B[:, None] * K * np.exp(gam))
        E = U - W @ S.T
        P = np.einsum("ti,ji,tji->tj", Q, K, decay)
        O[sl] = q_scale * ((Q * np.exp(gam)) @ S.T + P @ E)
        S = S * np.exp(gam[-1])[None, :] + E.T @ (K * np.exp(gam[-1][None, :] - gam))
    return O, S


def kda_intra_chunk_weights(X, K, gam, sub=16, dtype=np.float32):
    """M[t, j] = sum_i X_ti K_ji exp(Gamma_ti - Gamma_ji) for j <= t within one chunk, in `dtype`, formed
    the way a tensor-core kernel can: 16-token sub-blocks; a diagonal sub-block takes each factor
    exp(Gamma_ti - Gamma_ji) directly; an off-diagonal block (rows in sub-block a, columns in an
    earlier sub-block b) is one product (X_a * exp(Gamma_a - Gamma_r)) (K_b * exp(Gamma_r - Gamma_b))^T
    around r, the last token of sub-block b.  With g <= 0 every factor is a decay in (0, 1], so
    nothing overflows however strong the decay; a factor that underflows stands for a term below
    the precision of the sum.  Entries with j > t are zero."""
    L = X.shape[0]
    X, K, gam = X.astype(dtype), K.astype(dtype), gam.astype(dtype)
    M = np.zeros((L, L), dtype=dtype)
    for a0 in range(0, L, sub):
        a1 = min(L, a0 + sub)
        for t in range(a0, a1):  # the diagonal block, factor by factor
            for j in range(a0, t + 1):
                M[t, j] = np.sum(X[t] * K[j] * np.exp(gam[t] - gam[j]), dtype=dtype)
        for b0 in range(0, a0, sub):
            b1 = b0 + sub
            r = b1 - 1
            Xs = X[a0:a1] * np.exp(gam[a0:a1] - gam[r])
            Ks = K[b0:b1] * np.exp(gam[r] - gam[b0:b1])
            M[a0:a1, b0:b1] = Xs @ Ks.T
    return M


def chunked_chain_kda_fp32(q, k, v, g, beta, S0, q_scale, chunk=64, sub=16):
    """chunked_chain_kda carried out in fp32 with the sub-block weights of kda_intra_chunk_weights:
    the arithmetic precision and factorisation a chunked KDA kernel uses (fp32 state, fp32
    products).  Every other decay factor is taken against the chunk's start or end, so it too is
    at most 1: exp(Gamma_t) on Q and K, exp(Gamma_L - Gamma_t) on K in the state update."""
    f = np.float32
    T = q.shape[0]
    S = S0.astype(f).copy()
    O = np.zeros((T, v.shape[1]), dtype=f)
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        Q, K, V, G, B = (a[sl].astype(f) for a in (q, k, v, g, beta))
        L = Q.shape[0]
        gam = np.cumsum(G, axis=0, dtype=f)
        A = B[:, None] * kda_intra_chunk_weights(K, K, gam, sub) * np.tril(np.ones((L, L), dtype=f), -1)
        Tm = solve_triangular(np.eye(L, dtype=f) + A, np.eye(L, dtype=f), lower=True, unit_diagonal=True).astype(f)
        U = Tm @ (B[:, None] * V)
        W = Tm @ (B[:, None] * K * np.exp(gam))
        E = U - W @ S.T
        P = kda_intra_chunk_weights(Q, K, gam, sub)
        O[sl] = q_scale * ((Q * np.exp(gam)) @ S.T + P @ E)
        S = S * np.exp(gam[-1])[None, :] + E.T @ (K * np.exp(gam[-1][None, :] - gam))
    return O, S


def _bf16(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def tc_product(a, b, split_a=True, split_b=True):
    """a @ b as a bf16 tensor-core product with fp32 accumulation: each operand is its bf16
    rounding (hi) or, split, hi + lo with lo the bf16 rounding of the remainder; the products
    hi*hi, hi*lo and lo*hi are summed (lo*lo is below fp32) and the result is rounded to fp32."""
    ah, bh = _bf16(a), _bf16(b)
    r = ah @ bh
    if split_b:
        r = r + ah @ _bf16(b - bh)
    if split_a:
        r = r + _bf16(a - ah) @ bh
    return r.astype(np.float32).astype(np.float64)


TC_SPLIT_ALL = dict(T=True, Kg=True, S=True, R=True, E=True, Kd=True, Qg=True, S_o=True, P=True, E_o=True)


def chunked_chain_kda_tc(q, k, v, g, beta, S0, q_scale, split=TC_SPLIT_ALL, chunk=64):
    """The chunked KDA form with every contraction a bf16 tensor-core product (tc_product),
    everything else in fp32, in the order a kernel takes it per chunk:
      X = (K e^Gamma) S0^T            [split Kg, S]
      R = beta (V - X)                fp32 epilogue (beta never enters an operand)
      E = T R                         [split T, R]
      O = q_scale ((Q e^Gamma) S0^T + P E)    [Qg, S_o; P, E_o]  -- the output only
      S = S0 diag(e^Gamma_L) + E^T (K e^(Gamma_L - Gamma))     [E, Kd]
    `split` says which operands are bf16 hi + lo pairs (True) or plain bf16 (False)."""
    f32 = lambda x: np.asarray(x, dtype=np.float32).astype(np.float64)
    T = q.shape[0]
    S = f32(S0)
    O = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        Q, K, V, G, B = q[sl], k[sl], v[sl], g[sl], beta[sl]
        L = Q.shape[0]
        gam = f32(np.cumsum(G, axis=0))
        A = B[:, None] * kda_intra_chunk_weights(K, K, gam).astype(np.float64) * np.tril(np.ones((L, L)), -1)
        Tm = f32(solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True))
        X = tc_product(K * np.exp(gam), S.T, split["Kg"], split["S"])
        R = f32(B[:, None] * (V - X))
        E = tc_product(Tm, R, split["T"], split["R"])
        P = kda_intra_chunk_weights(Q, K, gam).astype(np.float64)
        O[sl] = q_scale * (tc_product(Q * np.exp(gam), S.T, split["Qg"], split["S_o"])
                           + tc_product(P, E, split["P"], split["E_o"]))
        S = f32(S * np.exp(gam[-1])[None, :]
                + tc_product(E.T, K * np.exp(gam[-1][None, :] - gam), split["E"], split["Kd"]))
    return O, S


def kda_gram_middle_reference(X, K, gam, ref=31):
    """M[t, j] = sum_i X_ti K_ji exp(Gamma_ti - Gamma_ji) (j <= t, else 0) as one bf16 hi / lo tensor-core
    product around the chunk's middle token: (X * exp(Gamma - Gamma_ref)) (K * exp(Gamma_ref - Gamma))^T.
    Valid while every |Gamma_t - Gamma_ref| stays far inside the fp32 range; entries above the
    diagonal are dropped by position (their factors may overflow)."""
    f32 = lambda x: np.asarray(x, dtype=np.float32).astype(np.float64)
    L = X.shape[0]
    r = min(ref, L - 1)
    e_row = f32(np.exp(f32(gam - gam[r])))
    e_col = f32(np.exp(f32(gam[r] - gam)))
    with np.errstate(over="ignore", invalid="ignore"):
        M = tc_product(f32(X * e_row), f32(K * e_col).T, True, True)
    return np.where(np.tril(np.ones((L, L), dtype=bool)), M, 0.0)


def chunked_chain_kda_tc_middle(q, k, v, g, beta, S0, q_scale, chunk=64):
    """chunked_chain_kda_tc (every state-path operand split, the output-only products plain) with A
    and P from kda_gram_middle_reference instead of the sub-block form."""
    f32 = lambda x: np.asarray(x, dtype=np.float32).astype(np.float64)
    T = q.shape[0]
    S = f32(S0)
    O = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        Q, K, V, G, B = q[sl], k[sl], v[sl], g[sl], beta[sl]
        L = Q.shape[0]
        gam = f32(np.cumsum(G.astype(np.float32), axis=0))
        A = B[:, None] * kda_gram_middle_reference(K, K, gam) * np.tril(np.ones((L, L)), -1)
        P = kda_gram_middle_reference(Q, K, gam)
        Tm = f32(solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True))
        X = tc_product(K * np.exp(gam), S.T, True, True)
        R = f32(B[:, None] * (V - X))
        E = tc_product(Tm, R, True, True)
        O[sl] = q_scale * (tc_product(Q * np.exp(gam), S.T, False, False) + tc_product(P, E, False, False))
        S = f32(S * np.exp(gam[-1])[None, :] + tc_product(E.T, K * np.exp(gam[-1][None, :] - gam), True, True))
    return O, S

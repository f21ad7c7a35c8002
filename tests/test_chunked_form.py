"""Pins the chunked (UT / WY) form of the gated delta rule that the
tensor-core kernels evaluate, against the sequential CPU oracle in fp64.

The form follows the chunkwise delta-rule algorithm of Yang et al.,
"Parallelizing Linear Transformers with the Delta Rule over Sequence Length"
(NeurIPS 2024), with the gates of "Gated Delta Networks" (ICLR 2025).  For one
(sequence, head) with C replayed tokens, G_t = sum_{s<=t} g_s and gamma_t = e^{G_t}:

  u_t = beta_t (v_t - gamma_t S0 k_t - sum_{s<t} e^{G_t-G_s} (k_t.k_s) u_s)   (forward substitution)
  o_t = scale (gamma_t S0 q_t + sum_{s<=t} e^{G_t-G_s} (q_t.k_s) u_s)
  S_C = gamma_C S0 + sum_s e^{G_C-G_s} u_s k_s^T

The verify kernel evaluates the outputs by effective queries, W = M (I + A)^{-1}
over the token system, and the fold kernel the new state through E' built from a
blocked (I + A)^{-1}; both rearrangements are restated below as well, together
with the fused step (fold, then the draft from the folded state).

These restatements live only here (never in the oracle); they show the algebra the
kernels rely on reproduces the recurrence, including at g = 0 / g = -20 and
beta near 0 / 1, where only differences G_t - G_s <= 0 are exponentiated.
"""
import math

import numpy as np
import pytest

import oracle


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def chunked(S0, K, V, g, beta, Q, q_pos, scale):
    C = K.shape[0]
    G = np.cumsum(g)
    P = K @ S0.T                                   # [C, dv]: (S0 k_t)
    U = np.zeros_like(V)
    for t in range(C):
        acc = np.zeros(V.shape[1])
        for s in range(t):
            acc += math.exp(G[t] - G[s]) * (K[t] @ K[s]) * U[s]
        U[t] = beta[t] * (V[t] - math.exp(G[t]) * P[t] - acc)
    O = []
    for q, p in zip(Q, q_pos):
        o = math.exp(G[p]) * (S0 @ q)
        for s in range(p + 1):
            o = o + math.exp(G[p] - G[s]) * (q @ K[s]) * U[s]
        O.append(scale * o)
    S_C = math.exp(G[-1]) * S0 + (U * np.exp(G[-1] - G)[:, None]).T @ K
    return np.array(O), S_C


@pytest.mark.parametrize("case", ["normal", "extreme", "no_buffer", "long"])
def test_chunked_form_matches_sequential(case):
    rng = np.random.default_rng({"normal": 1, "extreme": 2, "no_buffer": 3, "long": 4}[case])
    dk, dv = 16, 12
    L = {"normal": 7, "extreme": 9, "no_buffer": 0, "long": 60}[case]
    T = 5
    C = L + T
    S0 = rng.normal(0, 0.1, (dv, dk))
    K = unit(rng.normal(size=(C, dk)))
    V = rng.normal(size=(C, dv))
    Q = unit(rng.normal(size=(T, dk)))
    g = -np.log1p(np.exp(rng.normal(size=C)))
    beta = 1 / (1 + np.exp(-rng.normal(size=C)))
    if case == "extreme":
        g[::3] = 0.0
        g[1::4] = -20.0
        beta[::2] = 1 - 1e-4
        beta[1::5] = 1e-4
    d = oracle.Dims(B=1, H=1, dk=dk, dv=dv, T=T, cap=C, threshold=C, n_slot=1,
                    scale=1 / math.sqrt(dk))
    S = S0.copy()
    oracle.recur(d, S, K[:L], V[:L], g[:L], beta[:L])
    O_seq = oracle.recur(d, S, K[L:], V[L:], g[L:], beta[L:], q=Q)
    O_ch, S_ch = chunked(S0, K, V, g, beta, Q, list(range(L, C)), d.scale)
    np.testing.assert_allclose(O_ch, O_seq, rtol=0, atol=1e-10)
    np.testing.assert_allclose(S_ch, S, rtol=0, atol=1e-10)


# ------------------------------------------------------------------------------
# The two rearrangements the tensor-core kernels evaluate, restated here only.

def token_system(K, g, beta):
    """A[t][s] = beta_t e^{G_t - G_s} (k_t . k_s) for s < t, and G."""
    C = K.shape[0]
    G = np.cumsum(g)
    A = np.zeros((C, C))
    for t in range(C):
        for s in range(t):
            A[t, s] = beta[t] * math.exp(G[t] - G[s]) * (K[t] @ K[s])
    return A, G


def verify_effective_queries(S0, K, V, g, beta, Q, L, scale):
    """Outputs of the T draft tokens (buffer of L tokens first) by effective queries:
    W = M (I + A)^{-1}, qe = gamma_p q - sum_s W beta_s gamma_s k_s,
    ve = sum_s W beta_s v_s, o = scale (S0 qe + ve)."""
    C = K.shape[0]
    A, G = token_system(K, g, beta)
    T = Q.shape[0]
    M = np.zeros((T, C))
    for t2 in range(T):
        p = L + t2
        for s in range(p + 1):
            M[t2, s] = math.exp(G[p] - G[s]) * (Q[t2] @ K[s])
    W = M @ np.linalg.inv(np.eye(C) + A)
    gam = np.exp(G)
    out = []
    for t2 in range(T):
        p = L + t2
        qe = gam[p] * Q[t2] - (W[t2] * beta * gam) @ K
        ve = (W[t2] * beta) @ V
        out.append(scale * (S0 @ qe + ve))
    return np.array(out)


def blocked_inverse(A, blk):
    """(I + A)^{-1} for strictly lower-triangular A by blocks: each diagonal block by
    forward substitution, then the blocks below one block diagonal at a time,
    T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj."""
    C = A.shape[0]
    nb = (C + blk - 1) // blk
    Cp = nb * blk
    Ap = np.zeros((Cp, Cp))
    Ap[:C, :C] = A
    Ti = np.zeros((Cp, Cp))
    for b in range(nb):                            # diagonal blocks
        o = b * blk
        for j in range(blk):
            x = np.zeros(blk)
            x[j] = 1.0
            for r in range(j + 1, blk):
                x[r] = -Ap[o + r, o + j:o + r] @ x[j:r]
            Ti[o:o + blk, o + j] = x
    for d in range(1, nb):                         # block diagonals below
        for j in range(nb - d):
            i = j + d
            Y = np.zeros((blk, blk))
            for k in range(j, i):
                Y += Ap[i * blk:(i + 1) * blk, k * blk:(k + 1) * blk] @ Ti[k * blk:(k + 1) * blk, j * blk:(j + 1) * blk]
            Ti[i * blk:(i + 1) * blk, j * blk:(j + 1) * blk] = -Ti[i * blk:(i + 1) * blk, i * blk:(i + 1) * blk] @ Y
    return Ti[:C, :C]


def fold_through_inverse(S0, K, V, g, beta, blk):
    """S_L = gamma_{L-1} S0 + sum_s' (v_s' - gamma_s' S0 k_s') E'[s'] with
    E'[s'] = beta_s' sum_s Tinv[s][s'] D_s k_s, D_s = e^{G_{L-1} - G_s}."""
    A, G = token_system(K, g, beta)
    Ti = blocked_inverse(A, blk)
    D = np.exp(G[-1] - G)
    E = beta[:, None] * (Ti.T @ (D[:, None] * K))  # [L, dk]
    R = V - np.exp(G)[:, None] * (K @ S0.T)        # rows v_s' - gamma_s' S0 k_s'
    return math.exp(G[-1]) * S0 + R.T @ E


def _case(seed, L, T, dk=16, dv=12, extreme=False):
    rng = np.random.default_rng(seed)
    C = L + T
    S0 = rng.normal(0, 0.1, (dv, dk))
    K = unit(rng.normal(size=(C, dk)))
    V = rng.normal(size=(C, dv))
    Q = unit(rng.normal(size=(T, dk)))
    g = -np.log1p(np.exp(rng.normal(size=C)))
    beta = 1 / (1 + np.exp(-rng.normal(size=C)))
    if extreme:
        g[::3] = 0.0
        g[1::4] = -20.0
        beta[::2] = 1 - 1e-4
        beta[1::5] = 1e-4
    d = oracle.Dims(B=1, H=1, dk=dk, dv=dv, T=T, cap=C, threshold=C, n_slot=1,
                    scale=1 / math.sqrt(dk))
    return S0, K, V, Q, g, beta, d


@pytest.mark.parametrize("L,T,extreme", [(0, 5, False), (7, 5, False), (9, 4, True), (31, 16, False),
                                         (47, 1, True)])
def test_effective_query_verify_matches_sequential(L, T, extreme):
    S0, K, V, Q, g, beta, d = _case(10 + L, L, T, extreme=extreme)
    S = S0.copy()
    oracle.recur(d, S, K[:L], V[:L], g[:L], beta[:L])
    O_seq = oracle.recur(d, S, K[L:], V[L:], g[L:], beta[L:], q=Q)
    O_eq = verify_effective_queries(S0, K, V, g, beta, Q, L, d.scale)
    np.testing.assert_allclose(O_eq, O_seq, rtol=0, atol=1e-10)


@pytest.mark.parametrize("C,blk", [(1, 4), (5, 4), (16, 16), (37, 16), (48, 16), (63, 16)])
def test_blocked_inverse_is_the_inverse(C, blk):
    rng = np.random.default_rng(C)
    K = unit(rng.normal(size=(C, 16)))
    A, _ = token_system(K, -np.log1p(np.exp(rng.normal(size=C))), 1 / (1 + np.exp(-rng.normal(size=C))))
    Ti = blocked_inverse(A, blk)
    np.testing.assert_allclose(Ti @ (np.eye(C) + A), np.eye(C), rtol=0, atol=1e-12)
    assert np.allclose(np.triu(Ti, 1), 0.0)


@pytest.mark.parametrize("L,extreme", [(1, False), (16, False), (32, True), (47, False), (63, True)])
def test_fold_through_inverse_matches_sequential(L, extreme):
    S0, K, V, _, g, beta, d = _case(50 + L, L, 0, extreme=extreme)
    S = S0.copy()
    oracle.recur(d, S, K, V, g, beta)
    np.testing.assert_allclose(fold_through_inverse(S0, K, V, g, beta, 16), S, rtol=0, atol=1e-10)


def test_fused_step_draft_from_folded_state():
    """The fused step: fold the buffer, then verify the draft from S_L with the token
    system of the draft alone (G restarted), equals replaying buffer and draft."""
    L, T = 35, 16
    S0, K, V, Q, g, beta, d = _case(99, L, T)
    S = S0.copy()
    oracle.recur(d, S, K[:L], V[:L], g[:L], beta[:L])
    O_seq = oracle.recur(d, S, K[L:], V[L:], g[L:], beta[L:], q=Q)
    S_L = fold_through_inverse(S0, K[:L], V[:L], g[:L], beta[:L], 16)
    O_f = verify_effective_queries(S_L, K[L:], V[L:], g[L:], beta[L:], Q, 0, d.scale)
    np.testing.assert_allclose(O_f, O_seq, rtol=0, atol=1e-10)

"""Pins the chunked (UT / WY) form of the gated delta rule that the
tensor-core kernels evaluate, against the sequential CPU oracle in fp64.

The form follows the chunkwise delta-rule algorithm of Yang et al.,
"Parallelizing Linear Transformers with the Delta Rule over Sequence Length"
(NeurIPS 2024), with the gates of "Gated Delta Networks" (ICLR 2025).  For one
(sequence, head) with C replayed tokens, G_t = sum_{s<=t} g_s and gamma_t = e^{G_t}:

  u_t = beta_t (v_t - gamma_t S0 k_t - sum_{s<t} e^{G_t-G_s} (k_t.k_s) u_s)   (forward substitution)
  o_t = scale (gamma_t S0 q_t + sum_{s<=t} e^{G_t-G_s} (q_t.k_s) u_s)
  S_C = gamma_C S0 + sum_s e^{G_C-G_s} u_s k_s^T

This restatement lives only here (never in the oracle); it shows the algebra the
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

"""Chunk-parallel form of the KDA recurrence in numpy fp64 -- TEST INFRASTRUCTURE.

Used only to pin the token-by-token oracle (the two must agree to rounding).
The deep dive ("Kimi Delta Attention", section 06) states that prefill runs
the same state update chunk by chunk: tokens inside a chunk become matrix
products and only the chunk-boundary state is carried forward.  The pages do
not print the algebra; this is the plainest derivation from the recurrence of
section 03, written out step by step for one (sequence, head):

Within a chunk of c tokens with start state S0, let g_r = sum_{i<=r} log alpha_i
(per key channel) and Gamma_r = exp(g_r).  Unrolling the recurrence gives

    S_r = Diag(Gamma_r) S0 + sum_{i<=r} Diag(Gamma_r / Gamma_i) k_i u_i^T,
    u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r).

With K~ = K * exp(g), K^ = K * exp(-g), Q~ = Q * exp(g) (row r scaled by its
own g_r) this is the lower-triangular system

    (I + A) U = Diag(beta) (V - K~ S0),   A = Diag(beta) StrictLower(K~ K^T),

so with T = (I + A)^-1 Diag(beta), W = T K~, U0 = T V:  U = U0 - W S0.
Outputs are O = Q~ S0 + P U with P = LowerIncl(Q~ K^T), and the chunk-end
state is S_c = Diag(Gamma_c) S0 + K^end^T U with K^end = K * exp(g_c - g).
"""
from __future__ import annotations

import numpy as np


def prefill(q, k, v, log_alpha, beta, cu_seqlens=None, initial_state=None, chunk: int = 64):
    """Same contract as ``oracle.prefill`` (numpy inputs, fp64 outputs)."""
    q, k, v, la, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, T] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    out = np.zeros((T, H, dv))
    sf = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if initial_state is None else \
                np.asarray(initial_state, dtype=np.float64).reshape(N, H, dk, dv)[n, h].copy()
            for c0 in range(cu[n], cu[n + 1], chunk):
                c1 = min(c0 + chunk, cu[n + 1])
                Q, K, V, LA, B = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h], la[c0:c1, h], b[c0:c1, h]
                c = c1 - c0
                g = np.cumsum(LA, axis=0)                       # [c, dk]
                Kt, Kh, Qt = K * np.exp(g), K * np.exp(-g), Q * np.exp(g)
                Kend = K * np.exp(g[-1][None, :] - g)
                A = np.diag(B) @ np.tril(Kt @ Kh.T, -1)
                Tm = np.linalg.solve(np.eye(c) + A, np.diag(B))
                W, U0 = Tm @ Kt, Tm @ V
                U = U0 - W @ S
                P = np.tril(Qt @ Kh.T)
                out[c0:c1, h] = Qt @ S + P @ U
                S = np.exp(g[-1])[:, None] * S + Kend.T @ U
            sf[n, h] = S
    return out, sf

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


def backward(q, k, v, log_alpha, beta, cu_seqlens=None, initial_state=None, dout=None, dfinal=None,
             chunk: int = 64):
    """Reverse mode of the chunk form above, in numpy fp64 -- the chunk-level
    gradients a chunked backward kernel computes.  Same contract as
    ``oracle.backward`` (per-channel log alpha; returns dq, dk, dv, dlog_alpha,
    dbeta, dinitial_state).  The pages give no backward; this is the chain rule
    through each step of the chunk algebra, taken in reverse:

      across chunks (from the last, dS' the gradient of the chunk-end state):
        dU  = K^end dS' + P^T dO            dS = Diag(Gamma) dS' + Q~^T dO - W^T dU
      inside a chunk (dP = LowerIncl(dO U^T), M = (I + A)^-1, T = M Diag(beta)):
        dK^end = U dS'^T                     dGamma = rowsum(dS' * S)
        dQ~ = dO S^T + dP K^                 dW = -dU S^T,  dU0 = dU
        dT = dW K~^T + dU0 V^T               dV = T^T dU0
        dM = dT Diag(beta)                   dA = -M^T dM M^T (strictly lower part)
        dG = Diag(beta) dA                   dbeta = colsum(M * dT) + rowsum(StrictLower(G) * dA)
        dK~ = T^T dW + dG K^                 dK^ = dP^T Q~ + dG^T K~
      and through the decays (g_r = sum_{i<=r} log alpha_i, g_C the chunk's last):
        dK = dK~ e^g + dK^ e^-g + dK^end e^(g_C - g),  dQ = dQ~ e^g
        dg = dK~ K~ - dK^ K^ + dQ~ Q~ - dK^end K^end   (elementwise)
        dg_C = colsum(dK^end * K^end) + dGamma * Gamma
        dlog alpha_i = sum_{r >= i} dg_r + dg_C.
    """
    q, k, v, la, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    scalar_gate = la.ndim == 2
    if scalar_gate:
        la = np.repeat(la[:, :, None], dk, axis=2)
    cu = np.array([0, T] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    do_all = np.zeros((T, H, dv)) if dout is None else np.asarray(dout, dtype=np.float64).reshape(T, H, dv)
    g_out = {"dq": np.zeros((T, H, dk)), "dk": np.zeros((T, H, dk)), "dv": np.zeros((T, H, dv)),
             "dlog_alpha": np.zeros((T, H, dk)), "dbeta": np.zeros((T, H)),
             "dinitial_state": np.zeros((N, H, dk, dv))}
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if initial_state is None else \
                np.asarray(initial_state, dtype=np.float64).reshape(N, H, dk, dv)[n, h].copy()
            saved = []
            for c0 in range(cu[n], cu[n + 1], chunk):      # forward, keeping each chunk's pieces
                c1 = min(c0 + chunk, cu[n + 1])
                K, Q, V, LA, B = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h], la[c0:c1, h], b[c0:c1, h]
                c = c1 - c0
                g = np.cumsum(LA, axis=0)
                Kt, Kh, Qt = K * np.exp(g), K * np.exp(-g), Q * np.exp(g)
                Ke = K * np.exp(g[-1][None, :] - g)
                G = Kt @ Kh.T
                A = np.diag(B) @ np.tril(G, -1)
                M = np.linalg.inv(np.eye(c) + A)
                Tm = M @ np.diag(B)
                W, U0 = Tm @ Kt, Tm @ V
                P = np.tril(Qt @ Kh.T)
                U = U0 - W @ S
                saved.append((c0, c1, K, Q, V, B, g, Kt, Kh, Qt, Ke, G, M, Tm, W, P, U, S.copy()))
                S = np.exp(g[-1])[:, None] * S + Ke.T @ U
            dS = np.zeros((dk, dv)) if dfinal is None else \
                np.asarray(dfinal, dtype=np.float64).reshape(N, H, dk, dv)[n, h].copy()
            for (c0, c1, K, Q, V, B, g, Kt, Kh, Qt, Ke, G, M, Tm, W, P, U, S0) in reversed(saved):
                dO = do_all[c0:c1, h]
                Gam = np.exp(g[-1])
                dU = Ke @ dS + P.T @ dO
                dKe = U @ dS.T
                dGam = np.sum(dS * S0, axis=1)
                dP = np.tril(dO @ U.T)
                dQt = dO @ S0.T + dP @ Kh
                dW = -dU @ S0.T
                dT = dW @ Kt.T + dU @ V.T
                dV = Tm.T @ dU
                dM = dT @ np.diag(B)
                dA = np.tril(-M.T @ dM @ M.T, -1)
                dB = np.sum(M * dT, axis=0) + np.sum(np.tril(G, -1) * dA, axis=1)
                dG = np.diag(B) @ dA
                dKt = Tm.T @ dW + dG @ Kh
                dKh = dP.T @ Qt + dG.T @ Kt
                e, einv, eend = np.exp(g), np.exp(-g), np.exp(g[-1][None, :] - g)
                g_out["dk"][c0:c1, h] = dKt * e + dKh * einv + dKe * eend
                g_out["dq"][c0:c1, h] = dQt * e
                g_out["dv"][c0:c1, h] = dV
                g_out["dbeta"][c0:c1, h] = dB
                dg = dKt * Kt - dKh * Kh + dQt * Qt - dKe * Ke
                dgC = np.sum(dKe * Ke, axis=0) + dGam * Gam
                g_out["dlog_alpha"][c0:c1, h] = np.cumsum(dg[::-1], axis=0)[::-1] + dgC[None, :]
                dS = Gam[:, None] * dS + Qt.T @ dO - W.T @ dU
            g_out["dinitial_state"][n, h] = dS
    if scalar_gate:
        g_out["dlog_alpha"] = g_out["dlog_alpha"].sum(axis=2)
    return g_out

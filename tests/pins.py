"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` takes an oracle object (``prefill`` / ``decode_step`` methods,
see ``oracle.Oracle``) and raises AssertionError when the oracle disagrees
with the special case, closed form or invariant it states.  They are run
against the real oracle in ``test_oracle_pins.py`` and against builds with a
planted mistake in ``test_oracle_mutants.py`` (every mutant must fail at
least one pin).

Sources, all on the "Kimi Delta Attention" deep dive unless stated:
  * the KDA recurrence, section 03: S_t = (I - b k k^T) Diag(alpha) S + b k v^T,
    read right to left: decay rows, erase along k, write;
  * the read o_t = S_t^T q_t and the delta rule with its error-correcting
    write, section 02;
  * DeltaNet, Gated DeltaNet and KDA differ only in the forget rule
    (section 02's comparison table, section 03);
  * exact continuation from a restored boundary state, section 07;
  * chunked prefill and recurrent decode are the same state update, section 06;
  * variable-length batches, section 06 (the FlashKDA update).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

import oracle.chunked as chunked
import oracle.exact as exact

RNG_SEED = 1234


def _rand_case(rng, T, H, dk, dv, la_range=(0.01, 0.3), unit_k=True, unit_q=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    if unit_q:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    la = -rng.uniform(*la_range, size=(T, H, dk))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, la, b


def _close(a, b, tol, what):
    err = np.max(np.abs(np.asarray(a) - np.asarray(b))) if np.size(a) else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if np.size(b) else 1.0)
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol:.1e} x {scale:.3g}"
    return err


def pin_deltanet(O):
    """alpha = 1 (log alpha = 0) reduces KDA to the delta rule (DeltaNet),
    S_t = S_{t-1} + b k (v - S_{t-1}^T k)^T (deep dive, section 02)."""
    rng = np.random.default_rng(RNG_SEED)
    T, H, dk, dv = 40, 2, 6, 5
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    la[:] = 0.0
    s0 = rng.standard_normal((1, H, dk, dv)) * 0.3
    out, sf = O.prefill(q, k, v, la, b, None, s0)
    for h in range(H):
        S = s0[0, h].copy()
        for t in range(T):
            S = S + b[t, h] * np.outer(k[t, h], v[t, h] - S.T @ k[t, h])
            _close(out[t, h], S.T @ q[t, h], 1e-12, "DeltaNet output")
        _close(sf[0, h], S, 1e-12, "DeltaNet state")


def pin_gated_deltanet(O):
    """alpha the same on every channel reduces KDA to Gated DeltaNet,
    S_t = a_t (I - b k k^T) S_{t-1} + b k v^T with a scalar gate per head and
    token (deep dive, sections 02-03)."""
    rng = np.random.default_rng(RNG_SEED + 1)
    T, H, dk, dv = 40, 2, 6, 5
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    la[:] = la[:, :, :1]
    s0 = rng.standard_normal((1, H, dk, dv)) * 0.3
    out, sf = O.prefill(q, k, v, la, b, None, s0)
    for h in range(H):
        S = s0[0, h].copy()
        for t in range(T):
            a = np.exp(la[t, h, 0])
            kk = k[t, h]
            S = a * (np.eye(dk) - b[t, h] * np.outer(kk, kk)) @ S + b[t, h] * np.outer(kk, v[t, h])
            _close(out[t, h], S.T @ q[t, h], 1e-12, "GDN output")
        _close(sf[0, h], S, 1e-12, "GDN state")


def pin_scalar_gate(O):
    """A scalar gate given as log_alpha [T, H] (one per token and head) is
    Gated DeltaNet: S_t = a_t (I - b k k^T) S_{t-1} + b k v^T, prefill and
    decode step alike (deep dive, section 03: GDN multiplies a head's state by
    a scalar; KDA generalises it to Diag(alpha))."""
    rng = np.random.default_rng(RNG_SEED + 12)
    T, H, dk, dv = 30, 3, 5, 7
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    la2 = la[:, :, 0].copy()
    s0 = rng.standard_normal((1, H, dk, dv)) * 0.3
    out, sf = O.prefill(q, k, v, la2, b, None, s0)
    ref_out = np.zeros_like(out)
    for h in range(H):
        S = s0[0, h].copy()
        for t in range(T):
            kk = k[t, h]
            S = np.exp(la2[t, h]) * (np.eye(dk) - b[t, h] * np.outer(kk, kk)) @ S + b[t, h] * np.outer(kk, v[t, h])
            ref_out[t, h] = S.T @ q[t, h]
        _close(sf[0, h], S, 1e-12, "scalar-gate state")
    _close(out, ref_out, 1e-12, "scalar-gate output")
    # one decode step with a [N, H] gate
    st = s0[0][None].repeat(2, axis=0).reshape(2, H, dk, dv) + rng.standard_normal((2, H, dk, dv)) * 0.1
    qd, kd, vd, lad, bd = (x[:2] for x in (q, k, v, la2, b))
    od, sd = O.decode_step(qd, kd, vd, lad, bd, st)
    for n in range(2):
        for h in range(H):
            kk = kd[n, h]
            S = np.exp(lad[n, h]) * (np.eye(dk) - bd[n, h] * np.outer(kk, kk)) @ st[n, h] + bd[n, h] * np.outer(kk, vd[n, h])
            _close(sd[n, h], S, 1e-12, "scalar-gate decode state")
            _close(od[n, h], S.T @ qd[n, h], 1e-12, "scalar-gate decode output")


def pin_no_write(O):
    """beta = 0 writes nothing: S_t = Diag(exp(sum_{s<=t} log alpha_s)) S_0 in
    closed form and o_t = S_t^T q_t; with alpha = 1 as well S stays S_0."""
    rng = np.random.default_rng(RNG_SEED + 2)
    T, H, dk, dv = 33, 2, 5, 7
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv, la_range=(0.0, 0.5))
    b[:] = 0.0
    s0 = rng.standard_normal((1, H, dk, dv))
    out, sf = O.prefill(q, k, v, la, b, None, s0)
    G = np.exp(np.cumsum(la, axis=0))            # [T, H, dk]
    for h in range(H):
        for t in range(T):
            St = G[t, h][:, None] * s0[0, h]
            _close(out[t, h], St.T @ q[t, h], 1e-12, "no-write output")
        _close(sf[0, h], G[-1, h][:, None] * s0[0, h], 1e-12, "no-write state")
    out1, sf1 = O.prefill(q, k, v, np.zeros_like(la), b, None, s0)
    _close(sf1, s0, 0.0, "no-write, no-decay state")
    _close(out1, np.einsum("thi,hij->thj", q, s0[0]), 1e-13, "no-write, no-decay output")


def pin_exact_overwrite(O):
    """With ||k_t|| = 1 and beta_t = 1 the write replaces what the decayed memory
    held at k_t: S_t^T k_t = v_t exactly, since (I - k k^T) k = 0 (deep dive,
    section 02: read, measure the error, write the correction)."""
    rng = np.random.default_rng(RNG_SEED + 3)
    H, dk, dv = 3, 8, 6
    lens = [1, 2, 3, 5, 8, 13]
    T = sum(lens)
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv, la_range=(0.05, 0.8))
    b[:] = 1.0
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s0 = rng.standard_normal((len(lens), H, dk, dv))
    _, sf = O.prefill(q, k, v, la, b, cu, s0)
    for n in range(len(lens)):
        t = cu[n + 1] - 1
        for h in range(H):
            _close(sf[n, h].T @ k[t, h], v[t, h], 1e-13, "exact overwrite")


def pin_closed_forms(O):
    """One- and two-token closed forms, expanded by hand from the recurrence.

    T=1, S_0=0:  S_1 = b1 k1 v1^T,  o_1 = b1 (k1.q1) v1.
    T=2, S_0=0, D = Diag(alpha_2), c = k1^T D k2:
        S_2 = b1 (D k1) v1^T + b2 k2 (v2 - b1 c v1)^T
        o_2 = b1 (q2^T D k1) v1 + b2 (k2.q2) (v2 - b1 c v1).
    d_k != d_v, so a transposed state or read cannot pass."""
    rng = np.random.default_rng(RNG_SEED + 4)
    dk, dv = 4, 3
    q, k, v, la, b = _rand_case(rng, 2, 1, dk, dv, unit_k=False, unit_q=False)
    out, sf = O.prefill(q[:1], k[:1], v[:1], la[:1], b[:1])
    k1, v1, q1, b1 = k[0, 0], v[0, 0], q[0, 0], b[0, 0]
    _close(sf[0, 0], b1 * np.outer(k1, v1), 1e-14, "T=1 state")
    _close(out[0, 0], b1 * (k1 @ q1) * v1, 1e-14, "T=1 output")
    out, sf = O.prefill(q, k, v, la, b)
    k2, v2, q2, b2 = k[1, 0], v[1, 0], q[1, 0], b[1, 0]
    D = np.exp(la[1, 0])
    c = k1 @ (D * k2)
    e2 = v2 - b1 * c * v1
    _close(sf[0, 0], b1 * np.outer(D * k1, v1) + b2 * np.outer(k2, e2), 1e-14, "T=2 state")
    _close(out[1, 0], b1 * (q2 @ (D * k1)) * v1 + b2 * (k2 @ q2) * e2, 1e-14, "T=2 output")


def pin_chunked_form(O):
    """The chunk-parallel form (matrix products inside chunks, state carried
    between them; deep dive, section 06) equals the recurrence, for chunk
    sizes 1, 2, 16 and 64, with partial chunks and several sequences."""
    rng = np.random.default_rng(RNG_SEED + 5)
    H, dk, dv = 2, 16, 12
    lens = [200, 37, 1, 0, 130]
    T = sum(lens)
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv, la_range=(0.01, 0.3))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s0 = rng.standard_normal((len(lens), H, dk, dv)) * 0.1
    out, sf = O.prefill(q, k, v, la, b, cu, s0)
    for c in (1, 2, 16, 64):
        o2, s2 = chunked.prefill(q, k, v, la, b, cu, s0, chunk=c)
        _close(out, o2, 1e-12, f"chunked C={c} output")
        _close(sf, s2, 1e-12, f"chunked C={c} state")


def pin_continuation(O):
    """Restoring the state a prefix produced and continuing reproduces the
    uninterrupted run (deep dive, section 07), at every split point."""
    rng = np.random.default_rng(RNG_SEED + 6)
    T, H, dk, dv = 23, 2, 5, 4
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dk, dv))
    out, sf = O.prefill(q, k, v, la, b, None, s0)
    for m in range(0, T + 1):
        o1, s1 = O.prefill(q[:m], k[:m], v[:m], la[:m], b[:m], None, s0)
        o2, s2 = O.prefill(q[m:], k[m:], v[m:], la[m:], b[m:], None, s1)
        _close(np.concatenate([o1, o2]), out, 1e-13, f"continuation m={m} output")
        _close(s2, sf, 1e-13, f"continuation m={m} state")


def pin_varlen_isolation(O):
    """A packed varlen batch equals each sequence run on its own (no state
    leaks across cu_seqlens boundaries); empty sequences keep their state."""
    rng = np.random.default_rng(RNG_SEED + 7)
    H, dk, dv = 2, 4, 6
    lens = [5, 0, 1, 9, 3]
    T = sum(lens)
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s0 = rng.standard_normal((len(lens), H, dk, dv))
    out, sf = O.prefill(q, k, v, la, b, cu, s0)
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        o1, s1 = O.prefill(q[a:e], k[a:e], v[a:e], la[a:e], b[a:e], None, s0[n:n + 1])
        _close(out[a:e], o1, 0.0, f"varlen seq {n} output")
        _close(sf[n], s1[0], 0.0, f"varlen seq {n} state")
    _close(sf[1], s0[1], 0.0, "empty sequence keeps its state")


def pin_mode_duality(O):
    """T one-token decode steps equal one prefill of T tokens, outputs and
    state (deep dive, section 06: the same state update in both modes)."""
    rng = np.random.default_rng(RNG_SEED + 8)
    T, H, dk, dv = 17, 3, 5, 4
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dk, dv))
    out, sf = O.prefill(q, k, v, la, b, None, s0)
    S = s0.copy()
    for t in range(T):
        o, S = O.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1], S)
        _close(o[0], out[t], 0.0, f"decode step {t} output")
    _close(S, sf, 0.0, "decode final state")


def pin_linearity(O):
    """For fixed (k, alpha, beta) outputs and state are jointly linear in
    (V, S_0): scaling, superposition; and column j of the state depends only
    on column j of V and S_0 (a column permutation commutes with the run)."""
    rng = np.random.default_rng(RNG_SEED + 9)
    T, H, dk, dv = 19, 2, 6, 5
    q, k, v, la, b = _rand_case(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v.shape)
    s0 = rng.standard_normal((1, H, dk, dv))
    s02 = rng.standard_normal(s0.shape)
    o1, f1 = O.prefill(q, k, v, la, b, None, s0)
    o2, f2 = O.prefill(q, k, v2, la, b, None, s02)
    o3, f3 = O.prefill(q, k, 2.5 * v - 0.5 * v2, la, b, None, 2.5 * s0 - 0.5 * s02)
    _close(o3, 2.5 * o1 - 0.5 * o2, 1e-12, "superposition output")
    _close(f3, 2.5 * f1 - 0.5 * f2, 1e-12, "superposition state")
    perm = rng.permutation(dv)
    o4, f4 = O.prefill(q, k, v[..., perm], la, b, None, s0[..., perm])
    _close(o4, o1[..., perm], 0.0, "column permutation output")
    _close(f4, f1[..., perm], 0.0, "column permutation state")
    o5, f5 = O.prefill(q, k, v, la, b, None, s0, cols=(1, 3))
    _close(o5[..., 1:3], o1[..., 1:3], 0.0, "column subset output")
    _close(f5[..., 1:3], f1[..., 1:3], 0.0, "column subset state")


def pin_exact_rational(O):
    """Brute force in exact rational arithmetic on tiny inputs: the fp64
    oracle must agree to rounding (alpha given as rationals, log alpha = its
    fp64 logarithm)."""
    rng = np.random.default_rng(RNG_SEED + 10)
    T, dk, dv = 4, 3, 2

    def rat(lo, hi):
        return Fraction(int(rng.integers(lo, hi)), 16)

    q = [[rat(-16, 17) for _ in range(dk)] for _ in range(T)]
    k = [[rat(-16, 17) for _ in range(dk)] for _ in range(T)]
    v = [[rat(-32, 33) for _ in range(dv)] for _ in range(T)]
    al = [[Fraction(int(rng.integers(1, 16)), 16) for _ in range(dk)] for _ in range(T)]
    be = [Fraction(int(rng.integers(0, 17)), 16) for _ in range(T)]
    s0 = [[rat(-16, 17) for _ in range(dv)] for _ in range(dk)]
    eo, es = exact.prefill(q, k, v, al, be, s0)

    f = lambda m: np.array(m, dtype=np.float64)
    out, sf = O.prefill(f(q)[:, None], f(k)[:, None], f(v)[:, None],
                        np.log(f(al))[:, None], f(be)[:, None], None, f(s0)[None, None])
    _close(out[:, 0], f([[float(x) for x in r] for r in eo]), 1e-14, "exact output")
    _close(sf[0, 0], f([[float(x) for x in r] for r in es]), 1e-14, "exact state")


def pin_zero_state_default(O):
    """No initial state means the zero state; an empty sequence returns it."""
    rng = np.random.default_rng(RNG_SEED + 11)
    q, k, v, la, b = _rand_case(rng, 9, 2, 4, 3)
    o1, s1 = O.prefill(q, k, v, la, b, None, None)
    o2, s2 = O.prefill(q, k, v, la, b, None, np.zeros((1, 2, 4, 3)))
    _close(o1, o2, 0.0, "null initial state output")
    _close(s1, s2, 0.0, "null initial state state")
    o3, s3 = O.prefill(q[:0], k[:0], v[:0], la[:0], b[:0], None, None)
    assert o3.shape == (0, 2, 3)
    _close(s3, np.zeros((1, 2, 4, 3)), 0.0, "empty sequence, zero state")


def _fd_check(O, case, cu, coords=None, h=1e-6, tol=1e-7, seed=0):
    """Central finite differences of L = <wo, out> + <ws, final_state> against
    the oracle's reverse mode, on every input (or `coords` sampled ones)."""
    q, k, v, la, b, s0 = case
    rng = np.random.default_rng(seed)
    N = len(cu) - 1
    T, H = q.shape[:2]
    wo = rng.standard_normal((T, H, v.shape[2]))
    ws = rng.standard_normal((N, H, k.shape[2], v.shape[2]))
    g = O.backward(q, k, v, la, b, cu, s0, wo, ws)
    names = ["q", "k", "v", "log_alpha", "beta", "s0"]
    keys = ["dq", "dk", "dv", "dlog_alpha", "dbeta", "dinitial_state"]
    arrs = [q, k, v, la, b, s0]

    def loss(vals):
        o, sf = O.prefill(*vals[:5], cu, vals[5])
        return float((o * wo).sum() + (sf * ws).sum())

    for ai, (name, key) in enumerate(zip(names, keys)):
        idxs = list(np.ndindex(arrs[ai].shape))
        if coords is not None and len(idxs) > coords:
            idxs = [idxs[i] for i in rng.choice(len(idxs), coords, replace=False)]
        for idx in idxs:
            vals = [a.copy() for a in arrs]
            vals[ai][idx] += h
            lp = loss(vals)
            vals[ai][idx] -= 2 * h
            lm = loss(vals)
            fd = (lp - lm) / (2 * h)
            got = g[key][idx]
            assert abs(fd - got) <= tol * max(1.0, abs(fd)), \
                f"d/d{name}{idx}: reverse mode {got:.10g}, finite difference {fd:.10g}"


def pin_backward_finite_differences(O):
    """The reverse mode equals central finite differences of the forward
    oracle (the definition of the gradient) for every input, on two packed
    sequences, with d_k != d_v."""
    rng = np.random.default_rng(RNG_SEED + 20)
    q, k, v, la, b = _rand_case(rng, 9, 2, 4, 3)
    s0 = rng.standard_normal((2, 2, 4, 3)) * 0.3
    _fd_check(O, (q, k, v, la, b, s0), np.array([0, 5, 9], dtype=np.int32))


def pin_backward_across_checkpoints(O):
    """A sequence longer than the oracle's recompute segments (70 tokens):
    sampled finite differences, including inputs near the start."""
    rng = np.random.default_rng(RNG_SEED + 21)
    q, k, v, la, b = _rand_case(rng, 70, 1, 3, 2)
    s0 = rng.standard_normal((1, 1, 3, 2)) * 0.3
    _fd_check(O, (q, k, v, la, b, s0), np.array([0, 70], dtype=np.int32), coords=25, seed=1)


def pin_backward_scalar_gate(O):
    """With a scalar gate [T, H] the gate's gradient is that of the shared
    value: finite differences on the scalar gate itself."""
    rng = np.random.default_rng(RNG_SEED + 22)
    q, k, v, la, b = _rand_case(rng, 8, 2, 3, 4)
    s0 = rng.standard_normal((1, 2, 3, 4)) * 0.3
    _fd_check(O, (q, k, v, la[:, :, 0].copy(), b, s0), np.array([0, 8], dtype=np.int32), seed=2)


def pin_backward_no_write(O):
    """beta = 0 writes nothing, so neither k nor v can influence anything:
    their gradients are exactly zero (deep dive, section 03: beta scales
    the whole correction)."""
    rng = np.random.default_rng(RNG_SEED + 23)
    q, k, v, la, b = _rand_case(rng, 12, 2, 4, 3)
    b[:] = 0.0
    s0 = rng.standard_normal((1, 2, 4, 3))
    g = O.backward(q, k, v, la, b, None, s0, rng.standard_normal((12, 2, 3)), rng.standard_normal((1, 2, 4, 3)))
    assert np.all(g["dk"] == 0.0) and np.all(g["dv"] == 0.0), "beta = 0 but k or v has a gradient"


def pin_chunked_backward(O):
    """The reverse mode of the chunk form (oracle/chunked.py: the gradients a
    chunked backward computes, chunk by chunk through T = (I + A)^-1 Diag(beta),
    W, U0, P and the decays) equals the token-by-token reverse mode, for chunk
    sizes 1, 2, 16 and 64 with partial chunks, a ragged varlen batch, an
    initial state, output and final-state gradients, and the scalar gate."""
    rng = np.random.default_rng(RNG_SEED + 25)
    q, k, v, la, b = _rand_case(rng, 150, 2, 5, 4)
    cu = np.array([0, 1, 70, 150], dtype=np.int32)
    s0 = rng.standard_normal((3, 2, 5, 4)) * 0.2
    do = rng.standard_normal((150, 2, 4))
    dfin = rng.standard_normal((3, 2, 5, 4))
    ref = O.backward(q, k, v, la, b, cu, s0, do, dfin)
    for c in (1, 2, 16, 64):
        got = chunked.backward(q, k, v, la, b, cu, s0, do, dfin, chunk=c)
        for key in ref:
            _close(got[key], ref[key], 1e-12, f"chunked backward C={c} {key}")
    las = la[:, :, 0].copy()
    ref = O.backward(q, k, v, las, b, cu, s0, do, None)
    got = chunked.backward(q, k, v, las, b, cu, s0, do, None, chunk=16)
    for key in ref:
        _close(got[key], ref[key], 1e-12, f"chunked backward, scalar gate, {key}")


ALL_PINS = [pin_deltanet, pin_gated_deltanet, pin_scalar_gate, pin_no_write, pin_exact_overwrite,
            pin_closed_forms, pin_chunked_form, pin_continuation, pin_varlen_isolation,
            pin_mode_duality, pin_linearity, pin_exact_rational, pin_zero_state_default,
            pin_backward_finite_differences, pin_backward_across_checkpoints, pin_backward_scalar_gate,
            pin_backward_no_write, pin_chunked_backward]

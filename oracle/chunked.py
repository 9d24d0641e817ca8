"""Chunked (WY / UT) form of the gated delta rule, fp64 numpy.

TEST INFRASTRUCTURE ONLY.  This module is the oracle's second, independent
path: it reaches the per-token result of ``gdn_oracle.c`` by the chunked
route the pages describe, one chunk at a time, with library matmuls as its
only primitive.  It supplies the per-chunk intermediates (S, T, w, u, A, B)
that the device path's debug export is compared with, and the cross-checks
between the ladder inverse and forward substitution.  Nothing in the product
path may import it.

Notation (one batch row b and one value head j, chunk of C rows r, s):
  G_r   = g_0 + ... + g_r                 chunk-local inclusive cumsum
  gamma = exp(G),  gamma_C = exp(G_{C-1})  (the pages' "exp(g_last)")
  M_rs  = exp(G_r - G_s) for s <= r, else 0   (masked before the exp)
  S     = tril(diag(beta) (K K^T * M), -1)
  T     = (I + S)^-1                       the UT-transform inverse
  w     = T diag(beta * gamma) K,  u = T diag(beta) V
  Delta = u - w h                          ("u - w h" in the inter-chunk step)
  O     = diag(gamma) Q h + (Q K^T * M) Delta       (mask includes diagonal)
  h'    = gamma_C h + k_g^T Delta,  k_g = diag(exp(G_{C-1} - G)) K

Sources on the pages:
  * the inter-chunk step h_new = exp(g_last) h + k_g^T (u - w h)
    = (exp(g_last) I - k_g^T w) h + k_g^T u = A h + B: issue "GatedDeltaNet
    does not support ici_context_parallelism", section "The recurrence is
    affine, so it can be parallelized" (also PR "Shard the GatedDeltaNet
    sequence under ici_context_parallelism", description).
  * the composition law (A2, B2) o (A1, B1) = (A2 A1, A2 B1 + B2): same issue,
    same section.
  * the blockwise doubling ladder for (I + S)^-1 (with X the inverse at block
    size b, the inverse at 2b is X - X S_l X) and the analytic inverse
    backward dS = -(T^T dT T^T), strict-lower masked: PR "Fuse the Gated Delta
    Net inter-chunk scan into a Pallas TPU kernel", section "Changes",
    "Triangular inversion kernel".
  * the two-pass segment scan (fold each segment to one (A, B), exclusive
    prefix, replay): PR "Shard the GatedDeltaNet sequence ...", description.

The pages name w, u and k_g but never define them.  The definitions above
are the unique ones under which the inter-chunk step reproduces the
per-token rule: unrolling the rule over a chunk gives
(I + S) Delta = diag(beta) V - diag(beta gamma) K h, hence Delta = u - w h.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------- gates (a1)
def chunk_gates(g: np.ndarray):
    """Chunk-local cumsum G, gamma = exp(G) and the decay matrix M.

    M_rs = exp(G_r - G_s) for s <= r and 0 above the diagonal; the exponent
    is masked to 0 above the diagonal *before* exp so that no overflow or
    inf * 0 can arise.
    """
    g = np.asarray(g, dtype=np.float64)
    C = g.shape[0]
    G = np.cumsum(g)
    gamma = np.exp(G)
    low = np.tril(np.ones((C, C), dtype=bool))
    diff = np.where(low, G[:, None] - G[None, :], 0.0)
    M = np.where(low, np.exp(diff), 0.0)
    return G, gamma, M


# ------------------------------------------------------------ UT inverse (a3)
def ut_forward_substitution(S: np.ndarray) -> np.ndarray:
    """(I + S)^-1 for strictly-lower S, row by row (forward substitution).

    Row r of T satisfies T_r + sum_{s<r} S_rs T_s = e_r.
    """
    S = np.asarray(S, dtype=np.float64)
    C = S.shape[0]
    T = np.zeros((C, C))
    for r in range(C):
        row = np.zeros(C)
        row[r] = 1.0
        for s in range(r):
            row -= S[r, s] * T[s]
        T[r] = row
    return T


def ut_ladder(S: np.ndarray) -> np.ndarray:
    """(I + S)^-1 for strictly-lower S by the blockwise doubling ladder.

    Start from X = I (the inverse for diagonal blocks of size 1).  With X the
    inverse of I + S restricted to its diagonal blocks of size b, the inverse
    at size 2b is X - X S_l X, where S_l keeps only the lower-left b x b
    block of each 2b x 2b diagonal block of S.  Sizes that are not a power of
    two are padded with zero rows/columns (I + 0 inverts to I there).
    """
    S = np.asarray(S, dtype=np.float64)
    C = S.shape[0]
    P = 1
    while P < C:
        P *= 2
    Sp = np.zeros((P, P))
    Sp[:C, :C] = S
    X = np.eye(P)
    b = 1
    while b < P:
        Sl = np.zeros((P, P))
        for s0 in range(0, P, 2 * b):
            Sl[s0 + b:s0 + 2 * b, s0:s0 + b] = Sp[s0 + b:s0 + 2 * b, s0:s0 + b]
        X = X - X @ Sl @ X
        b *= 2
    return X[:C, :C]


# --------------------------------------------------------- one chunk, forward
def chunk_intermediates(Q, K, V, g, beta, use_ladder=True):
    """Per-chunk quantities that do not depend on the incoming state (a1-a4).

    Q, K: [C, dk]; V: [C, dv]; g, beta: [C].  Returns a dict with G, gamma,
    M, S, T, w, u, kg (= diag(exp(G_{C-1} - G)) K) and P (= Q K^T * M).
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    beta = np.asarray(beta, np.float64)
    G, gamma, M = chunk_gates(g)
    S = np.tril(beta[:, None] * (K @ K.T) * M, -1)
    T = ut_ladder(S) if use_ladder else ut_forward_substitution(S)
    w = T @ ((beta * gamma)[:, None] * K)
    u = T @ (beta[:, None] * V)
    kg = np.exp(G[-1] - G)[:, None] * K
    P = (Q @ K.T) * M
    return dict(G=G, gamma=gamma, M=M, S=S, T=T, w=w, u=u, kg=kg, P=P)


def chunk_affine(it):
    """(A_c, B_c) of one chunk: h' = A_c h + B_c with
    A_c = gamma_C I - k_g^T w and B_c = k_g^T u."""
    dk = it["w"].shape[1]
    gC = it["gamma"][-1]
    A = gC * np.eye(dk) - it["kg"].T @ it["w"]
    B = it["kg"].T @ it["u"]
    return A, B


def compose(second, first):
    """(A2, B2) o (A1, B1) = (A2 A1, A2 B1 + B2): apply `first`, then `second`."""
    A2, B2 = second
    A1, B1 = first
    return A2 @ A1, A2 @ B1 + B2


def identity_map(dk, dv):
    return np.eye(dk), np.zeros((dk, dv))


# ------------------------------------------------------------ one head, full
def _chunks(T, C):
    return [(c0, min(c0 + C, T)) for c0 in range(0, T, C)]


def head_fwd(q, k, v, g, beta, h0, C, use_ladder=True, keep=False):
    """Chunked forward of one head.  q, k: [T, dk]; v: [T, dv]; g, beta: [T];
    h0: [dk, dv] or None.  Returns (o [T, dv], hT [dk, dv]) and, with
    keep=True, also the list of per-chunk intermediates and entering states.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    h = np.zeros((dk, dv)) if h0 is None else np.array(h0, np.float64)
    o = np.zeros((T, dv))
    inter, states = [], []
    for c0, c1 in _chunks(T, C):
        it = chunk_intermediates(q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1],
                                 beta[c0:c1], use_ladder)
        states.append(h.copy())
        Delta = it["u"] - it["w"] @ h
        o[c0:c1] = it["gamma"][:, None] * (q[c0:c1] @ h) + it["P"] @ Delta
        h = it["gamma"][-1] * h + it["kg"].T @ Delta
        if keep:
            inter.append(it)
    if keep:
        return o, h, inter, states
    return o, h


def segment_bounds(n_chunks, n_segments):
    """Segment s holds chunks [floor(s N / S), floor((s+1) N / S))."""
    return [((s * n_chunks) // n_segments, ((s + 1) * n_chunks) // n_segments)
            for s in range(n_segments)]


def head_fwd_segmented(q, k, v, g, beta, h0, C, n_segments, drop_incoming=False):
    """Two-pass segment scan of one head.

    Pass 1 folds each segment's chunks, in order, into one (A, B) starting
    from the identity map.  The exclusive prefix gives each segment its
    entering state: h_in[0] = h0, h_in[s+1] = A_s h_in[s] + B_s, and the final
    state is h_in[n_segments].  Pass 2 replays each segment from h_in[s].
    drop_incoming=True replays every segment from a zero state (the failure
    the pages report for a path that skips the composition) and exists only
    as a negative control.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    ch = _chunks(T, C)
    its = [chunk_intermediates(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b]) for a, b in ch]
    segs = segment_bounds(len(ch), n_segments)
    pairs = []
    for s0, s1 in segs:
        AB = identity_map(dk, dv)
        for c in range(s0, s1):
            AB = compose(chunk_affine(its[c]), AB)
        pairs.append(AB)
    h_in = [np.zeros((dk, dv)) if h0 is None else np.array(h0, np.float64)]
    for A, B in pairs:
        h_in.append(A @ h_in[-1] + B)
    o = np.zeros((T, dv))
    for s, (s0, s1) in enumerate(segs):
        h = np.zeros((dk, dv)) if drop_incoming else h_in[s]
        for c in range(s0, s1):
            a, b = ch[c]
            it = its[c]
            Delta = it["u"] - it["w"] @ h
            o[a:b] = it["gamma"][:, None] * (q[a:b] @ h) + it["P"] @ Delta
            h = it["gamma"][-1] * h + it["kg"].T @ Delta
    return o, h_in[-1], pairs


def inclusive_prefix(As, Bs):
    """Inclusive prefix of affine maps: out[i] = (A_i, B_i) o ... o (A_0, B_0)."""
    outA, outB = [], []
    acc = None
    for A, B in zip(As, Bs):
        acc = (A, B) if acc is None else compose((A, B), acc)
        outA.append(acc[0])
        outB.append(acc[1])
    return np.array(outA), np.array(outB)


# ----------------------------------------------------------- one chunk, bwd
def chunk_bwd(Q, K, V, g, beta, h, dO, dh_out):
    """Gradients of one chunk given its entering state h, the output
    cotangent dO and the cotangent dh_out of the state it leaves.

    Returns dQ, dK, dV, dg, dbeta and dh_in (the cotangent of h).  Each line
    is the reverse of one line of the chunk forward; the inverse's backward
    is the analytic dS = -(T^T dT T^T), kept strictly lower; the gate
    cotangent dg is the reverse cumsum of the cotangent of G.
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    beta = np.asarray(beta, np.float64)
    C = K.shape[0]
    it = chunk_intermediates(Q, K, V, g, beta)
    G, gamma, M, T, w, u, kg, P = (it[x] for x in ("G", "gamma", "M", "T", "w", "u", "kg", "P"))
    gC = gamma[-1]
    KK = K @ K.T
    QK = Q @ K.T
    ef = np.exp(G[-1] - G)
    Delta = u - w @ h
    strict = np.tril(np.ones((C, C)), -1)
    incl = np.tril(np.ones((C, C)))

    dDelta = P.T @ dO + kg @ dh_out
    dh_in = gC * dh_out + Q.T @ (gamma[:, None] * dO) - w.T @ dDelta
    # O = diag(gamma) Q h + P Delta
    dQ = gamma[:, None] * (dO @ h.T)
    dgamma = np.sum(dO * (Q @ h), axis=1)
    dP = (dO @ Delta.T) * incl
    dQK = dP * M
    dM = dP * QK
    dQ = dQ + dQK @ K
    dK = dQK.T @ Q
    # h' = gamma_C h + kg^T Delta
    dgC = np.sum(dh_out * h)
    dkg = Delta @ dh_out.T
    dK = dK + ef[:, None] * dkg
    d_ef = np.sum(dkg * K, axis=1)
    # Delta = u - w h
    du = dDelta
    dw = -dDelta @ h.T
    # u = T diag(beta) V ; w = T diag(beta gamma) K
    bV = beta[:, None] * V
    bgK = (beta * gamma)[:, None] * K
    dT = du @ bV.T + dw @ bgK.T
    dbV = T.T @ du
    dV = beta[:, None] * dbV
    dbeta = np.sum(dbV * V, axis=1)
    dbgK = T.T @ dw
    dK = dK + (beta * gamma)[:, None] * dbgK
    dbg = np.sum(dbgK * K, axis=1)
    dbeta = dbeta + gamma * dbg
    dgamma = dgamma + beta * dbg
    # T = (I + S)^-1
    dS = -(T.T @ dT @ T.T) * strict
    # S = tril(diag(beta) (KK * M), -1)
    dbeta = dbeta + np.sum(dS * KK * M, axis=1)
    dKK = dS * beta[:, None] * M
    dM = dM + dS * beta[:, None] * KK
    dK = dK + dKK @ K + dKK.T @ K
    # gate cotangents, through G
    dG = gamma * dgamma
    dG[-1] += gC * dgC
    X = dM * M
    dG = dG + X.sum(axis=1) - X.sum(axis=0)
    Y = d_ef * ef
    dG[-1] += Y.sum()
    dG = dG - Y
    dg = np.cumsum(dG[::-1])[::-1]
    return dQ, dK, dV, dg, dbeta, dh_in


def head_bwd(q, k, v, g, beta, h0, dO, dhT, C):
    """Chunked backward of one head: forward to get each chunk's entering
    state, a reverse walk of the state cotangent, and the per-chunk
    gradients.  Returns dq, dk, dv, dg, dbeta, dh0 (this value head's
    contribution to dq and dk) plus the list of per-chunk leaving-state
    cotangents."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    T, dk_ = k.shape
    dv_ = v.shape[1]
    _, _, inter, states = head_fwd(q, k, v, g, beta, h0, C, keep=True)
    ch = _chunks(T, C)
    dh = np.zeros((dk_, dv_)) if dhT is None else np.array(dhT, np.float64)
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    dg = np.zeros(T)
    db = np.zeros(T)
    dh_leave = [None] * len(ch)
    for c in range(len(ch) - 1, -1, -1):
        a, b = ch[c]
        dh_leave[c] = dh
        dQ, dK, dV, dgc, dbc, dh = chunk_bwd(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b],
                                            states[c], dO[a:b], dh)
        dq[a:b], dkk[a:b], dvv[a:b], dg[a:b], db[a:b] = dQ, dK, dV, dgc, dbc
    return dq, dkk, dvv, dg, db, dh, dh_leave

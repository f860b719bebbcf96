"""numpy twins that pin the fp64 oracle -- TEST INFRASTRUCTURE ONLY.

Every function works on fp64 numpy arrays in the library's layouts:
* q, k [B, T, H, dk]; v [B, T, H, dv];
* g = log alpha [B, T, H], or [B, T, H, dk] for a per-key-channel (KDA) gate;
* beta [B, T, H];
* states in the transposed layout [B, H, dk, dv], that is S^T.
They are slow on purpose and written for small shapes, one (batch, head)
chain at a time, in the pages' notation.

Sources (page title, then section / equation):
* "TileLang 实战：KDA 从零到一 -- Gated DeltaNet" (the "TileLang page"):
  - the opening recurrence;
  - §1.1, the overwrite reading;
  - §2.2, the WY/UT representation (paper eqs 3-9);
  - §2.3, the gated chunk algorithm (paper eqs 11, 12);
  - §3, the four reference levels.
* "Gated Delta Network (GDN)": eqs 2-4 and 8-12; §4(b3), (d).
* "You Could Have Come Up With Kimi Delta Attention" (the "KDA page"): the
  chunkwise derivation with per-channel decay.
* "阅读笔记：DeltaNet 在 FLA 中的代码实现" (the "FLA notes"): forward Steps 1-5.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "matrix_recurrence", "deltanet_overwrite_form", "mamba2_closed_form",
    "chunkwise_gdn", "chunkwise_kda", "unit_lower_inverse_fwdsub", "unit_lower_inverse_blocked",
    "chunk_matrices_gdn",
]


def _retention(g_t: np.ndarray, dk: int) -> np.ndarray:
    """exp(log retention) as a d_k-vector (a scalar gate is broadcast over key channels)."""
    a = np.exp(np.asarray(g_t, dtype=np.float64))
    return np.broadcast_to(a, (dk,)) if a.ndim == 0 else a


def matrix_recurrence(q, k, v, g, beta, scale, S0=None):
    """The literal d_v x d_k recurrence, one token at a time.

    S_t = S_{t-1} Diag(a_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and
    o_t = scale * S_t q_t.  For GDN the retention a_t is the scalar alpha_t
    times the identity: the TileLang page's opening equation (also its ref_A,
    §3.1) and eq. 4 of the GDN page.  For KDA it is the per-channel Diag(gamma_t)
    that right-multiplies the state (KDA page: one retention factor per key
    column of S).  Returns (o, S^T) with the states as [B, H, dk, dv].
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    I = np.eye(dk)
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else S0[b, h].T.copy()
            for t in range(T):
                kt, vt, qt = k[b, t, h], v[b, t, h], q[b, t, h]
                a = _retention(g[b, t, h], dk)
                S = S @ (np.diag(a) @ (I - beta[b, t, h] * np.outer(kt, kt))) + beta[b, t, h] * np.outer(vt, kt)
                o[b, t, h] = scale * (S @ qt)
            ST[b, h] = S.T
    return o, ST


def deltanet_overwrite_form(q, k, v, beta, scale, S0=None):
    """DeltaNet (alpha = 1) written as 'subtract the old value, write the new one'.

    v_old = S k_t, v_new = beta v_t + (1 - beta) v_old, and
    S <- S - v_old k_t^T + v_new k_t^T (TileLang page §1.1, GDN page eq. 3).
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else S0[b, h].T.copy()
            for t in range(T):
                kt, vt, bt = k[b, t, h], v[b, t, h], beta[b, t, h]
                v_old = S @ kt
                v_new = bt * vt + (1.0 - bt) * v_old
                S = S - np.outer(v_old, kt) + np.outer(v_new, kt)
                o[b, t, h] = scale * (S @ q[b, t, h])
            ST[b, h] = S.T
    return o, ST


def mamba2_closed_form(q, k, v, g, scale):
    """Scalar-decay linear attention in its parallel (attention) form.

    S_t = alpha_t S_{t-1} + v_t k_t^T (GDN page eq. 2), started from zero,
    unrolls to o_t = scale * sum_{i<=t} (prod_{j=i+1..t} alpha_j) (k_i . q_t) v_i.
    The decay products come from differences of the cumulative log gate.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            L = np.cumsum(g[b, :, h])
            D = np.zeros((T, T))
            for t in range(T):
                D[t, : t + 1] = np.exp(L[t] - L[: t + 1])
            o[b, :, h] = scale * ((q[b, :, h] @ k[b, :, h].T) * D) @ v[b, :, h]
    return o


def unit_lower_inverse_fwdsub(L: np.ndarray) -> np.ndarray:
    """Inverse of a unit lower-triangular matrix by forward substitution, column by column.

    No pivoting is needed: det = 1 (TileLang page §2.3).
    """
    n = L.shape[0]
    X = np.zeros_like(L)
    for c in range(n):
        for r in range(n):
            s = 1.0 if r == c else 0.0
            for j in range(r):
                s -= L[r, j] * X[j, c]
            X[r, c] = s
    return X


def unit_lower_inverse_blocked(L: np.ndarray, bs: int = 16) -> np.ndarray:
    """Blocked inverse of a unit lower-triangular matrix.

    The bs x bs diagonal blocks are inverted by forward substitution.  The
    blocks below the diagonal come from T_ab = -T_aa sum_{b<=m<a} L_am T_mb,
    which is row a of L T = I (FLA notes, Step 2; TileLang page §4.2, the
    blocked recursion).
    """
    n = L.shape[0]
    nb = (n + bs - 1) // bs
    sl = [slice(i * bs, min(n, (i + 1) * bs)) for i in range(nb)]
    X = np.zeros_like(L)
    for a in range(nb):
        X[sl[a], sl[a]] = unit_lower_inverse_fwdsub(L[sl[a], sl[a]])
    for dist in range(1, nb):
        for a in range(dist, nb):
            b = a - dist
            acc = np.zeros((sl[a].stop - sl[a].start, sl[b].stop - sl[b].start))
            for m in range(b, a):
                acc += L[sl[a], sl[m]] @ X[sl[m], sl[b]]
            X[sl[a], sl[b]] = -X[sl[a], sl[a]] @ acc
    return X


def chunk_matrices_gdn(Kc, g_c, be):
    """Per-chunk quantities of the gated chunk algorithm (TileLang page §2.3).

    gamma^r = prod_{i<=r} alpha_i, taken as exp of the cumulative log gate.
    Gamma_ij = gamma_i / gamma_j for j <= i, else 0; the exponent is formed as
    a difference and masked before exp (TileLang page §4.1).
    A = diag(beta)(Gamma * K K^T).
    """
    Cn = Kc.shape[0]
    G = np.cumsum(g_c)
    gam = np.exp(G)
    Gam = np.zeros((Cn, Cn))
    for i in range(Cn):
        Gam[i, : i + 1] = np.exp(G[i] - G[: i + 1])
    A = np.diag(be) @ (Gam * (Kc @ Kc.T))
    return G, gam, Gam, A


def chunkwise_gdn(q, k, v, g, beta, scale, S0=None, C=64, solve="inv", block_dv=None):
    """Chunkwise gated delta rule, for the scalar gate.

    This is the TileLang page §2.3, paper eqs 11-12, per (batch, head) chain.
    The chain is cut into chunks of C tokens; the last chunk may be shorter.
    solve picks how the unit lower-triangular system
    (I + strictLower(A)) Delta = R, R = diag(beta)(V - diag(gamma) K S^T), is solved:
      "inv"       -- T = [I + strictLower(A)]^{-1} diag(beta) by a dense inverse,
                     then Delta = T V - T diag(gamma) K S^T (paper eqs 6-7 with
                     the gated inputs of §2.2.6; the page's ref_B);
      "fwdsub"    -- forward substitution on the rows of R, no T
                     (Delta[r] = R[r] - sum_{j<r} A[r, j] Delta[j]);
      "blocked16" -- T0 = (I + strictLower(A))^{-1} by the blocked inverse, then
                     W = T0 diag(beta) diag(gamma) K and U = T0 diag(beta) V,
                     and V_new = U - W S^T (FLA notes Steps 1-4; GDN page §4(d)).
    Output: O = (diag(gamma) Q) S^T + (Q K^T * Gamma) Delta, times scale.
    State: S <- gamma^C S + Delta^T diag(gamma^C / gamma) K.
    block_dv splits d_v into slices that are run independently, as the page's
    kernel mirror (ref_C, §3.3) does.
    Returns (o, S^T) with the states as [B, H, dk, dv].
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if block_dv is not None:
        o = np.zeros((B, T, H, dv))
        ST = np.zeros((B, H, dk, dv))
        for j0 in range(0, dv, block_dv):
            js = slice(j0, min(dv, j0 + block_dv))
            s0 = None if S0 is None else S0[..., js]
            oj, sj = chunkwise_gdn(q, k, v[..., js], g, beta, scale, s0, C, solve, None)
            o[..., js] = oj
            ST[..., js] = sj
        return o, ST
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else S0[b, h].T.copy()
            for c0 in range(0, T, C):
                sl = slice(c0, min(T, c0 + C))
                Qc, Kc, Vc = q[b, sl, h], k[b, sl, h], v[b, sl, h]
                g_c, be = g[b, sl, h], beta[b, sl, h]
                Cn = Kc.shape[0]
                G, gam, Gam, A = chunk_matrices_gdn(Kc, g_c, be)
                gC = gam[-1]
                Lm = np.eye(Cn) + np.tril(A, -1)
                if solve == "inv":
                    Tm = np.linalg.inv(Lm) @ np.diag(be)
                    Delta = Tm @ Vc - Tm @ (np.diag(gam) @ (Kc @ S.T))
                elif solve == "fwdsub":
                    R = be[:, None] * (Vc - (gam[:, None] * Kc) @ S.T)
                    Delta = np.zeros_like(R)
                    for r in range(Cn):
                        Delta[r] = R[r] - A[r, :r] @ Delta[:r]
                elif solve == "blocked16":
                    T0 = unit_lower_inverse_blocked(Lm, 16)
                    W = T0 @ (np.diag(be) @ np.diag(gam) @ Kc)
                    U = T0 @ (np.diag(be) @ Vc)
                    Delta = U - W @ S.T
                else:
                    raise ValueError(solve)
                o[b, sl, h] = scale * ((gam[:, None] * Qc) @ S.T + ((Qc @ Kc.T) * Gam) @ Delta)
                S = gC * S + Delta.T @ (np.exp(G[-1] - G)[:, None] * Kc)
            ST[b, h] = S.T
    return o, ST


def chunkwise_kda(q, k, v, g, beta, scale, S0=None, C=64):
    """Chunkwise KDA: the per-key-channel gate, brute force.

    This follows the KDA page's chunkwise derivation, in the transposed state
    h = S^T (dk x dv).  Inside a chunk, G[i, c] is the cumulative log decay of
    key channel c up to token i.  A write made at token j reaches token i
    decayed by the diagonal exp(G_i - G_j).
    * Causal key-key coefficients, strictly below the diagonal:
      A[i, j] = sum_c k_ic k_jc exp(G_ic - G_jc), j < i.
    * The errors E solve (I + diag(beta) strictLower(A)) E
      = diag(beta)(V - (K * exp(G)) h_in).
    * Read matrix, diagonal included, since token i reads after its own write:
      Aqk[i, j] = sum_c q_ic k_jc exp(G_ic - G_jc), j <= i.
    * O = scale ((Q * exp(G)) h_in + Aqk E).
    * h_out = diag(exp(G_C)) h_in + (K * exp(G_C - G))^T E.  The second factor
      is the keys decayed to the chunk end.
    Exponents are differences, formed only where j <= i.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for hh in range(H):
            h = np.zeros((dk, dv)) if S0 is None else S0[b, hh].copy()
            for c0 in range(0, T, C):
                sl = slice(c0, min(T, c0 + C))
                Qc, Kc, Vc = q[b, sl, hh], k[b, sl, hh], v[b, sl, hh]
                be = beta[b, sl, hh]
                G = np.cumsum(g[b, sl, hh], axis=0)          # [Cn, dk]
                Cn = Kc.shape[0]
                Akk = np.zeros((Cn, Cn))
                Aqk = np.zeros((Cn, Cn))
                for i in range(Cn):
                    for j in range(i + 1):
                        dec = np.exp(G[i] - G[j])
                        if j < i:
                            Akk[i, j] = np.sum(Kc[i] * Kc[j] * dec)
                        Aqk[i, j] = np.sum(Qc[i] * Kc[j] * dec)
                M = np.eye(Cn) + be[:, None] * Akk
                R = be[:, None] * (Vc - (Kc * np.exp(G)) @ h)
                E = np.linalg.solve(M, R)
                o[b, sl, hh] = scale * ((Qc * np.exp(G)) @ h + Aqk @ E)
                h = np.exp(G[-1])[:, None] * h + (Kc * np.exp(G[-1][None, :] - G)).T @ E
            ST[b, hh] = h
    return o, ST

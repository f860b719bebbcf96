"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

The oracle is the C token recurrence (oracle.recurrence).  Each test compares
it with something it shares no code with:
* an algebraically different formulation (the d x d matrix recurrence, the
  overwrite form of DeltaNet, the parallel form of scalar-decay attention, the
  chunkwise WY/UT algorithm);
* closed forms (pure decay, exact retrieval, orthonormal keys, axis-aligned
  KDA keys);
* a finite-difference gradient (the test-time SGD reading);
* the error magnitudes the TileLang page prints.
A plausible slip in the oracle fails one of them: a dropped term, a wrong sign
or index, a transposed operand, or a read before the write.
test_oracle_mutations.py checks that.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import reference as ref

HERE = os.path.dirname(os.path.abspath(__file__))


def _case(seed, B=2, T=13, H=2, dk=5, dv=3, unit_keys=True, kda=False, g_scale=1.0, h0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, 0.95, (B, T, H))
    gshape = (B, T, H, dk) if kda else (B, T, H)
    g = -g_scale * rng.uniform(0.0, 1.0, gshape)
    S0 = rng.standard_normal((B, H, dk, dv)) if h0 else None
    return q, k, v, g, beta, S0


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --- the recurrence itself ------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("kda", [False, True])
def test_rank1_oracle_equals_matrix_recurrence(seed, kda):
    # TileLang page, opening equation / ref_A; GDN page eq. 4; KDA page, Diag(gamma) right-multiplying S
    q, k, v, g, beta, S0 = _case(seed, kda=kda)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.7, S0)
    o2, s2 = ref.matrix_recurrence(q, k, v, g, beta, 0.7, S0)
    assert _rel(o1, o2) < 1e-13 and _rel(s1, s2) < 1e-13


def test_non_unit_keys_and_large_decay_range():
    # the identity holds for any keys; the eigenvalue bound of TileLang page §1.2 needs unit keys
    q, k, v, g, beta, S0 = _case(3, unit_keys=False, g_scale=8.0)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 1.3, S0)
    o2, s2 = ref.matrix_recurrence(q, k, v, g, beta, 1.3, S0)
    assert _rel(o1, o2) < 1e-12 and _rel(s1, s2) < 1e-12


def test_alpha_one_is_deltanet():
    # GDN page §6: alpha = 1 gives DeltaNet (eq. 3), here in its overwrite form (TileLang page §1.1)
    q, k, v, g, beta, S0 = _case(4)
    g = np.zeros_like(g)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.9, S0)
    o2, s2 = ref.deltanet_overwrite_form(q, k, v, beta, 0.9, S0)
    assert _rel(o1, o2) < 1e-13 and _rel(s1, s2) < 1e-13


def test_beta_zero_is_pure_decay():
    # beta -> 0: T -> 0, Delta -> 0, only the decay of the entry state remains (TileLang page §2.3)
    q, k, v, g, beta, S0 = _case(5)
    beta = np.zeros_like(beta)
    o, s = oracle.recurrence(q, k, v, g, beta, 0.8, S0)
    B, T, H, dk = q.shape
    G = np.cumsum(g, axis=1)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                expect = 0.8 * np.exp(G[b, t, h]) * (S0[b, h].T @ q[b, t, h])
                assert np.allclose(o[b, t, h], expect, rtol=1e-13, atol=1e-15)
            assert np.allclose(s[b, h], np.exp(G[b, -1, h]) * S0[b, h], rtol=1e-13, atol=1e-15)


def test_small_beta_first_order_is_mamba2():
    # to first order in beta = eps (S0 = 0), S_t / eps -> sum_i gamma_{i+1:t} v_i k_i^T,
    # the scalar-decay recurrence of GDN page eq. 2 (Mamba2), whose parallel form is independent code
    q, k, v, g, beta, _ = _case(6, h0=False)
    eps = 1e-7
    o, _ = oracle.recurrence(q, k, v, g, np.full_like(beta, eps), 0.6, None)
    om = ref.mamba2_closed_form(q, k, v, g, 0.6)
    assert _rel(o / eps, om) < 1e-5


def test_retrieval_is_exact_for_beta_one_unit_keys():
    # beta = 1 and |k| = 1: S_t k_t = v_t for any alpha (TileLang page §1.1; KDA page, immediate reconstruction)
    for kda in (False, True):
        q, k, v, g, beta, S0 = _case(7, g_scale=3.0, kda=kda)
        o, _ = oracle.recurrence(k, k, v, g, np.ones_like(beta), 1.0, S0)
        assert np.abs(o - v).max() < 1e-13


def test_orthonormal_keys_closed_form():
    # beta = 1, S0 = 0, orthonormal k_1..k_T (T <= dk): S_T k_i = gamma_{i+1:T} v_i,
    # because each write leaves the other keys' directions untouched (TileLang page §1.1)
    rng = np.random.default_rng(8)
    dk, dv, T = 8, 3, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :T].T.reshape(1, T, 1, dk)
    q = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv))
    g = -rng.uniform(0, 1, (1, T, 1))
    _, s = oracle.recurrence(q, k, v, g, np.ones((1, T, 1)), 1.0, None)
    S_T = s[0, 0].T
    for i in range(T):
        decay = np.exp(np.sum(g[0, i + 1:, 0]))
        assert np.allclose(S_T @ k[0, i, 0], decay * v[0, i, 0], atol=1e-14)


def test_householder_eigenstructure():
    # one step with v = 0 maps h0 to alpha (I - beta k k^T) h0; for a unit k its eigenvalues are
    # alpha(1 - beta) along k and alpha on the d_k - 1 orthogonal directions (TileLang page §1.2)
    rng = np.random.default_rng(9)
    dk = 6
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    alpha, beta = 0.8, 0.35
    M = np.zeros((dk, dk))
    for i in range(dk):
        h0 = np.zeros((1, 1, dk, 1))
        h0[0, 0, i, 0] = 1.0
        _, s = oracle.recurrence(np.zeros((1, 1, 1, dk)), k.reshape(1, 1, 1, dk), np.zeros((1, 1, 1, 1)),
                                 np.full((1, 1, 1), np.log(alpha)), np.full((1, 1, 1), beta), 1.0, h0)
        M[:, i] = s[0, 0, :, 0]
    assert np.allclose(M, M.T, atol=1e-15)
    w, U = np.linalg.eigh(M)
    assert np.allclose(w, np.sort([alpha * (1 - beta)] + [alpha] * (dk - 1)), atol=1e-14)
    assert abs(abs(U[:, 0] @ k) - 1.0) < 1e-12



def test_beta_two_is_a_reflection():
    # beta = 2 (the top of the (0, 2) range allowed with negative eigenvalues, GDN page §5 notes) with alpha = 1,
    # a unit key and v = 0 maps h0 to (I - 2 k k^T) h0: a Householder reflection, so two identical steps give
    # h0 back, one step flips the component along k and keeps the rest, and the Frobenius norm never changes
    rng = np.random.default_rng(11)
    dk, dv = 5, 3
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    h0 = rng.standard_normal((1, 1, dk, dv))
    kk = np.tile(k, (2, 1)).reshape(1, 2, 1, dk)
    _, s1 = oracle.recurrence(np.zeros((1, 1, 1, dk)), kk[:, :1], np.zeros((1, 1, 1, dv)), np.zeros((1, 1, 1)),
                              np.full((1, 1, 1), 2.0), 1.0, h0)
    _, s2 = oracle.recurrence(np.zeros((1, 2, 1, dk)), kk, np.zeros((1, 2, 1, dv)), np.zeros((1, 2, 1)),
                              np.full((1, 2, 1), 2.0), 1.0, h0)
    assert np.allclose(s2, h0, atol=1e-14)
    assert np.allclose(k @ s1[0, 0], -(k @ h0[0, 0]), atol=1e-14)
    perp = np.eye(dk) - np.outer(k, k)
    assert np.allclose(perp @ s1[0, 0], perp @ h0[0, 0], atol=1e-14)
    assert abs(np.linalg.norm(s1) - np.linalg.norm(h0)) < 1e-13

def test_test_time_sgd_identity():
    # S_t = S' - beta grad_S 1/2 |S k - v|^2 at S' = alpha S_{t-1} (TileLang page §1.3);
    # the gradient is taken by central finite differences, independent of any closed form
    rng = np.random.default_rng(10)
    dk, dv = 4, 3
    S0 = rng.standard_normal((dv, dk))
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    v = rng.standard_normal(dv)
    alpha, beta = 0.7, 0.4
    Sp = alpha * S0
    loss = lambda S: 0.5 * np.sum((S @ k - v) ** 2)
    grad = np.zeros_like(Sp)
    hstep = 1e-6
    for i in range(dv):
        for j in range(dk):
            E = np.zeros_like(Sp)
            E[i, j] = hstep
            grad[i, j] = (loss(Sp + E) - loss(Sp - E)) / (2 * hstep)
    expect = Sp - beta * grad
    _, s = oracle.recurrence(np.zeros((1, 1, 1, dk)), k.reshape(1, 1, 1, dk), v.reshape(1, 1, 1, dv),
                             np.full((1, 1, 1), np.log(alpha)), np.full((1, 1, 1), beta), 1.0,
                             S0.T.reshape(1, 1, dk, dv))
    assert np.allclose(s[0, 0].T, expect, atol=1e-8)


# --- the chunk algebra ------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("solve", ["inv", "fwdsub", "blocked16"])
def test_chunkwise_equals_recurrence(C, solve):
    # TileLang page §2.3 eqs 11-12 and FLA notes Steps 1-5 give the recurrence exactly, for any chunk
    # size, with the last chunk shorter than C (77 is a multiple of no C > 1 here)
    q, k, v, g, beta, S0 = _case(11 + C, B=1, T=77, H=2, dk=6, dv=5)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.5, S0)
    o2, s2 = ref.chunkwise_gdn(q, k, v, g, beta, 0.5, S0, C=C, solve=solve)
    assert _rel(o2, o1) < 1e-12 and _rel(s2, s1) < 1e-12


def test_kernel_mirror_dv_split_is_exact():
    # d_v columns of the state evolve independently (TileLang page §3.3, ref_C splits DV)
    q, k, v, g, beta, S0 = _case(12, B=1, T=40, H=1, dk=6, dv=8)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.5, S0)
    o2, s2 = ref.chunkwise_gdn(q, k, v, g, beta, 0.5, S0, C=8, solve="fwdsub", block_dv=3)
    assert _rel(o2, o1) < 1e-12 and _rel(s2, s1) < 1e-12


@pytest.mark.parametrize("C", [1, 3, 4, 16])
def test_kda_chunkwise_equals_recurrence(C):
    # KDA page, chunkwise form: per-channel diagonal decays, strictly lower key-key system, read incl. diagonal
    q, k, v, g, beta, S0 = _case(13 + C, B=1, T=37, H=2, dk=5, dv=4, kda=True, g_scale=2.0)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.5, S0)
    o2, s2 = ref.chunkwise_kda(q, k, v, g, beta, 0.5, S0, C=C)
    assert _rel(o2, o1) < 1e-12 and _rel(s2, s1) < 1e-12


def test_ut_matrix_properties():
    # I + strictLower(A) is unit lower triangular: det 1, no pivoting; its inverse by forward
    # substitution and by the 16x16 blocked recursion both satisfy (I + A) T = I (TileLang page §2.3)
    rng = np.random.default_rng(14)
    C, dk = 64, 32
    K = rng.standard_normal((C, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    g = -rng.uniform(0, 0.3, C)
    be = rng.uniform(0, 1, C)
    _, _, _, A = ref.chunk_matrices_gdn(K, g, be)
    L = np.eye(C) + np.tril(A, -1)
    assert abs(np.linalg.det(L) - 1.0) < 1e-12
    for T in (ref.unit_lower_inverse_fwdsub(L), ref.unit_lower_inverse_blocked(L, 16)):
        assert np.abs(L @ T - np.eye(C)).max() < 1e-13
        assert np.allclose(np.diag(T), 1.0) and np.allclose(np.triu(T, 1), 0.0)
    # the two ways of forming A agree (TileLang page §3.4: diag(beta) @ (Gamma * K K^T) vs (K * beta) @ K^T * Gamma)
    _, _, Gam, _ = ref.chunk_matrices_gdn(K, g, be)
    A2 = ((K * be[:, None]) @ K.T) * Gam
    assert np.abs(A - A2).max() < 1e-15


def test_printed_consistency_magnitudes():
    # the page's own case: B=2, H=2, N=12, dk=dv=4, C=4, block_DV=2, fp64; it prints only error sizes,
    # so the test reproduces their order of magnitude (within 16x), not values
    gold = json.load(open(os.path.join(HERE, "golden", "tilelang_page_consistency.json")))
    p = gold["printed"]
    rng = np.random.default_rng(15)
    B, H, N, d = 2, 2, 12, 4
    q = rng.standard_normal((B, N, H, d)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, N, H, d)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, N, H, d))
    g = np.log(rng.uniform(0.5, 1.0, (B, N, H)))
    beta = rng.uniform(0, 1, (B, N, H))
    oA, _ = oracle.recurrence(q, k, v, g, beta, 1.0, None)
    oB, _ = ref.chunkwise_gdn(q, k, v, g, beta, 1.0, None, C=4, solve="inv")
    oC, _ = ref.chunkwise_gdn(q, k, v, g, beta, 1.0, None, C=4, solve="fwdsub", block_dv=2)
    assert np.abs(oB - oA).max() <= 16 * p["chunkwise_ut_vs_recurrence_max_abs"]
    assert _rel(oB, oA) <= 16 * p["chunkwise_ut_vs_recurrence_rel_l2"]
    assert np.abs(oC - oA).max() <= 16 * p["kernel_mirror_vs_recurrence_max_abs"]
    assert _rel(oC, oA) <= 16 * p["kernel_mirror_vs_recurrence_rel_l2"]
    z = np.zeros_like(g)
    o1, _ = oracle.recurrence(q, k, v, z, beta, 1.0, None)
    o2, _ = ref.chunkwise_gdn(q, k, v, z, beta, 1.0, None, C=4, solve="inv")
    assert np.abs(o2 - o1).max() <= 16 * p["alpha_one_chunkwise_vs_recurrence_max_abs"]
    b12 = np.full_like(beta, 1e-12)
    o1, _ = oracle.recurrence(q, k, v, g, b12, 1.0, None)
    o2, _ = ref.chunkwise_gdn(q, k, v, g, b12, 1.0, None, C=4, solve="inv")
    assert np.abs(o2 - o1).max() <= 16 * p["beta_1e-12_chunkwise_vs_recurrence_max_abs"]


# --- KDA specifics ----------------------------------------------------------------------

def test_kda_with_equal_channels_is_gdn_bitwise():
    # a per-channel gate that is the same on every channel is the scalar gate (KDA page)
    q, k, v, g, beta, S0 = _case(16)
    gk = np.repeat(g[..., None], q.shape[-1], axis=-1)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.5, S0)
    o2, s2 = oracle.recurrence(q, k, v, gk, beta, 0.5, S0)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_kda_axis_aligned_keys_decouple_per_channel():
    # with one-hot keys k_t = e_{c_t} each key channel c (a row of S^T) evolves on its own:
    # decay by exp(g_c), and the written row moves towards v by beta (KDA page: retention per key column of S)
    rng = np.random.default_rng(17)
    dk, dv, T = 5, 3, 30
    c_t = rng.integers(0, dk, T)
    k = np.zeros((1, T, 1, dk))
    k[0, np.arange(T), 0, c_t] = 1.0
    q = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv))
    g = -rng.uniform(0, 2, (1, T, 1, dk))
    beta = rng.uniform(0, 1, (1, T, 1))
    h0 = rng.standard_normal((1, 1, dk, dv))
    o, s = oracle.recurrence(q, k, v, g, beta, 0.9, h0)
    rows = [h0[0, 0, c].copy() for c in range(dk)]
    for t in range(T):
        for c in range(dk):
            rows[c] = rows[c] * np.exp(g[0, t, 0, c])
        c = c_t[t]
        rows[c] = rows[c] + beta[0, t, 0] * (v[0, t, 0] - rows[c])
        expect = 0.9 * sum(q[0, t, 0, cc] * rows[cc] for cc in range(dk))
        assert np.allclose(o[0, t, 0], expect, atol=1e-13)
    assert np.allclose(s[0, 0], np.stack(rows), atol=1e-13)


# --- state hand-off and packed sequences ------------------------------------------------

def test_state_handoff_is_bitwise():
    # the state is the checkpoint: running T1 tokens then T - T1 with the state handed over is the same run
    q, k, v, g, beta, S0 = _case(18, B=1, T=29, H=2)
    o, s = oracle.recurrence(q, k, v, g, beta, 0.5, S0)
    T1 = 11
    oa, sa = oracle.recurrence(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], 0.5, S0)
    ob, sb = oracle.recurrence(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], 0.5, sa)
    assert np.array_equal(np.concatenate([oa, ob], axis=1), o) and np.array_equal(sb, s)


def test_packed_sequences_equal_separate_runs_bitwise():
    # GDN page §6: packed independent sequences reset the state at their boundaries; nothing leaks
    rng = np.random.default_rng(19)
    lens = [5, 0, 17, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Ttot = int(cu[-1])
    q, k, v, g, beta, _ = _case(20, B=1, T=Ttot, H=3)
    h0 = rng.standard_normal((len(lens), 3, 5, 3))
    o, s = oracle.recurrence(q, k, v, g, beta, 0.5, h0, cu_seqlens=cu)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        on, sn = oracle.recurrence(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], 0.5, h0[n:n + 1])
        assert np.array_equal(o[:, a:b], on) and np.array_equal(s[n], sn[0])
    # perturbing one sequence leaves the others bitwise unchanged
    v2 = v.copy()
    v2[:, cu[2]:cu[3]] += 1.0
    o2, s2 = oracle.recurrence(q, k, v2, g, beta, 0.5, h0, cu_seqlens=cu)
    keep = np.ones(Ttot, bool)
    keep[cu[2]:cu[3]] = False
    assert np.array_equal(o2[:, keep], o[:, keep])
    assert np.array_equal(np.delete(s2, 2, axis=0), np.delete(s, 2, axis=0))
    assert not np.array_equal(s2[2], s[2])


def test_oracle_rejects_bad_cu_seqlens():
    q, k, v, g, beta, _ = _case(21, B=1, T=10, H=1)
    for cu in ([0, 4, 3, 10], [1, 10], [0, 9]):
        with pytest.raises(ValueError):
            oracle.recurrence(q, k, v, g, beta, 1.0, None, cu_seqlens=np.array(cu, np.int32))

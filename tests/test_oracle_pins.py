"""Pins for the fp64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself -- a
hand-worked example, a closed form, a textbook reduction, brute-force
transition-matrix products, or an independent chunked-algebra model -- so that
a dropped term, a wrong sign or index or a transposed operand fails one of
them.  None of these tests needs a GPU.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import chunked_model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, T, H, dk, dv, N=1, s0=True, gate=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, H, dk)))) * gate
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = rng.standard_normal((N, H, dk, dv)) * 0.5 if s0 else None
    return q, k, v, g, beta, S0


# ---------------------------------------------------------------------------
# hand-worked example (tests/golden/delta_rule_d2.txt)
# ---------------------------------------------------------------------------
def _read_golden():
    toks, final = [], None
    with open(os.path.join(GOLDEN, "delta_rule_d2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("token"):
                parts = [list(map(float, p.split())) for p in line[5:].split("|")]
                toks.append(parts)
            elif line.startswith("final_state"):
                final = list(map(float, line.split()[1:]))
    return toks, final


def test_hand_worked_example():
    toks, final = _read_golden()
    T = len(toks)
    q = np.array([t[4] for t in toks])[:, None, :]
    k = np.array([t[0] for t in toks])[:, None, :]
    v = np.array([t[1] for t in toks])[:, None, :]
    beta = np.array([t[2][0] for t in toks])[:, None]
    g = np.log(np.array([t[3] for t in toks]))[:, None, :]
    o_exp = np.array([t[5] for t in toks])[:, None, :]
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, None, [0, T])
    np.testing.assert_allclose(o, o_exp, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_T.reshape(-1), final, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# brute force: products of transition matrices M_t = (I - b k k^T) Diag(alpha)
# ---------------------------------------------------------------------------
def _brute_force(q, k, v, g, beta, S0):
    """S_t = M_t ... M_1 S0 + sum_i M_t ... M_{i+1} b_i k_i v_i^T, as dense
    matrix products (no step-by-step state update); o_t = S_t^T q_t."""
    T, dk = k.shape
    dv = v.shape[1]
    Ms = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
          for t in range(T)]
    o = np.zeros((T, dv))
    S_t = None
    for t in range(T):
        prod = np.eye(dk)
        for j in range(t, -1, -1):
            prod = prod @ Ms[j]
        S_t = prod @ S0
        for i in range(t + 1):
            tail = np.eye(dk)
            for j in range(t, i, -1):
                tail = tail @ Ms[j]
            S_t = S_t + tail @ (beta[i] * np.outer(k[i], v[i]))
        o[t] = S_t.T @ q[t]
    return o, S_t


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_transition_products(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 9))
    dk = int(rng.integers(1, 5))
    dv = int(rng.integers(1, 5))
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))  # not normalised: keeps every term alive
    v = rng.standard_normal((T, dv))
    g = -np.abs(rng.standard_normal((T, dk)))
    beta = rng.uniform(0.05, 0.95, T)
    S0 = rng.standard_normal((dk, dv))
    o_bf, S_bf = _brute_force(q, k, v, g, beta, S0)
    o, S_T, _ = oracle.prefill(q[:, None], k[:, None], v[:, None], g[:, None],
                               beta[:, None], S0[None, None], [0, T])
    np.testing.assert_allclose(o[:, 0], o_bf, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_T[0, 0], S_bf, rtol=1e-12, atol=1e-12)


def test_brute_force_exact_rationals():
    """Same identity in exact rational arithmetic (alpha given as a rational,
    g = ln(alpha) for the oracle), on a 3-token, 2x3 case."""
    al = [[Fraction(1, 2), Fraction(3, 4)], [Fraction(1), Fraction(1, 3)],
          [Fraction(2, 5), Fraction(7, 8)]]
    ks = [[Fraction(1), Fraction(-2)], [Fraction(1, 2), Fraction(1, 3)],
          [Fraction(-1), Fraction(3, 2)]]
    vs = [[Fraction(1), Fraction(0), Fraction(-1)], [Fraction(2), Fraction(1, 2), Fraction(1)],
          [Fraction(0), Fraction(-3), Fraction(1, 4)]]
    qs = [[Fraction(1), Fraction(1)], [Fraction(0), Fraction(2)], [Fraction(-1), Fraction(1, 2)]]
    bs = [Fraction(1, 4), Fraction(3, 5), Fraction(1, 2)]
    S = [[Fraction(1, 10), Fraction(0), Fraction(-1, 5)], [Fraction(0), Fraction(3, 10), Fraction(0)]]
    S0 = np.array([[float(x) for x in r] for r in S])

    def mat(a):
        return [list(r) for r in a]

    def mul(A, B):
        return [[sum(A[i][t] * B[t][j] for t in range(len(B))) for j in range(len(B[0]))]
                for i in range(len(A))]

    def add(A, B):
        return [[A[i][j] + B[i][j] for j in range(len(A[0]))] for i in range(len(A))]

    outs = []
    for t in range(3):
        M = [[(1 if i == j else 0) - bs[t] * ks[t][i] * ks[t][j] for j in range(2)]
             for i in range(2)]
        M = [[M[i][j] * al[t][j] for j in range(2)] for i in range(2)]   # (I - b k k^T) Diag(a)
        W = [[bs[t] * ks[t][i] * vs[t][j] for j in range(3)] for i in range(2)]
        S = add(mul(M, mat(S)), W)
        outs.append([sum(S[i][j] * qs[t][i] for i in range(2)) for j in range(3)])
    q = np.array([[float(x) for x in r] for r in qs])[:, None]
    k = np.array([[float(x) for x in r] for r in ks])[:, None]
    v = np.array([[float(x) for x in r] for r in vs])[:, None]
    g = np.log(np.array([[float(x) for x in r] for r in al]))[:, None]
    beta = np.array([float(x) for x in bs])[:, None]
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, S0[None, None], [0, 3])
    np.testing.assert_allclose(o[:, 0], np.array([[float(x) for x in r] for r in outs]),
                               rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S_T[0, 0], np.array([[float(x) for x in r] for r in S]),
                               rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# invariants named by the pages
# ---------------------------------------------------------------------------
def test_delta_zero_leaves_state_unchanged():
    """v_new == v_old => delta = 0 => the write changes nothing; only the decay
    acts ("DeltaNet" section of the lineage essay)."""
    rng = np.random.default_rng(1)
    T, dk, dv = 6, 5, 3
    q, k, v, g, beta, S0 = _rand_case(rng, T, 1, dk, dv)
    S_prev = S0[0, 0]
    for t in range(T):
        Sd = np.exp(g[t, 0])[:, None] * S_prev
        v[t, 0] = Sd.T @ k[t, 0]              # the value already stored at k_t
        _, S_t, _ = oracle.prefill(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1],
                                   beta[:t + 1], S0, [0, t + 1])
        np.testing.assert_allclose(S_t[0, 0], Sd, rtol=1e-12, atol=1e-14)
        S_prev = S_t[0, 0]


def test_overwrite_with_unit_key():
    """beta = 1 with a unit-norm key overwrites the stored value: k^T S_t = v_t."""
    rng = np.random.default_rng(2)
    T, dk, dv = 7, 8, 6
    q, k, v, g, beta, S0 = _rand_case(rng, T, 1, dk, dv)
    beta[:] = 1.0
    for t in range(1, T + 1):
        _, S_t, _ = oracle.prefill(q[:t], k[:t], v[:t], g[:t], beta[:t], S0, [0, t])
        np.testing.assert_allclose(S_t[0, 0].T @ k[t - 1, 0], v[t - 1, 0],
                                   rtol=1e-12, atol=1e-12)


def test_interpolation_between_old_and_new():
    """0 < beta < 1, unit key: k^T S_t = (1 - beta) k^T S'_t + beta v_t."""
    rng = np.random.default_rng(3)
    T, dk, dv = 5, 6, 4
    q, k, v, g, beta, S0 = _rand_case(rng, T, 1, dk, dv)
    S_prev = S0[0, 0]
    for t in range(T):
        Sd = np.exp(g[t, 0])[:, None] * S_prev
        _, S_t, _ = oracle.prefill(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1],
                                   beta[:t + 1], S0, [0, t + 1])
        b = beta[t, 0]
        expect = (1 - b) * (Sd.T @ k[t, 0]) + b * v[t, 0]
        np.testing.assert_allclose(S_t[0, 0].T @ k[t, 0], expect, rtol=1e-12, atol=1e-12)
        S_prev = S_t[0, 0]


def test_linear_attention_reduction():
    """alpha = 1 (g = 0), S0 = 0 and orthonormal keys: the delta read is always
    zero, so KDA reduces to causal linear attention S = sum_i beta_i k_i v_i^T,
    o_t = sum_{i<=t} beta_i (q_t . k_i) v_i -- a masked dense matmul."""
    rng = np.random.default_rng(4)
    dk, dv = 16, 5
    T = dk
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm.T.copy()                                   # rows orthonormal
    q = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    beta = rng.uniform(0.1, 0.9, T)
    g = np.zeros((T, dk))
    o, S_T, _ = oracle.prefill(q[:, None], k[:, None], v[:, None], g[:, None],
                               beta[:, None], None, [0, T])
    mask = np.tril(np.ones((T, T)))
    o_lin = (mask * (q @ k.T)) @ (beta[:, None] * v)
    S_lin = k.T @ (beta[:, None] * v)
    np.testing.assert_allclose(o[:, 0], o_lin, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_T[0, 0], S_lin, rtol=1e-12, atol=1e-12)


def test_decay_only_closed_form():
    """beta = 0: no writes, S_t = Diag(exp(sum_{i<=t} g_i)) S0 and o_t = S_t^T q_t
    (cumulative per-channel decay, "Gated DeltaNet" section)."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 9, 2, 7, 3
    q, k, v, g, beta, S0 = _rand_case(rng, T, H, dk, dv)
    beta[:] = 0.0
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, S0, [0, T])
    cum = np.cumsum(g, axis=0)
    for h in range(H):
        for t in range(T):
            St = np.exp(cum[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S_T[0, h], np.exp(cum[-1, h])[:, None] * S0[0, h],
                                   rtol=1e-12, atol=1e-14)


def test_alpha_one_is_deltanet_and_alpha_zero_erases():
    """alpha = 1 gives the ungated delta rule; alpha = 0 (g = -inf) at step t
    erases memory so that S_t = beta_t k_t v_t^T ("Gated DeltaNet" section)."""
    rng = np.random.default_rng(6)
    T, dk, dv = 6, 4, 3
    q, k, v, g, beta, S0 = _rand_case(rng, T, 1, dk, dv)
    # alpha = 1: plain DeltaNet, S_t = S_{t-1} + b k (v - k^T S_{t-1})^T
    g0 = np.zeros_like(g)
    _, S_T, _ = oracle.prefill(q, k, v, g0, beta, S0, [0, T])
    S = S0[0, 0].copy()
    for t in range(T):
        kt = k[t, 0]
        S = S + beta[t, 0] * np.outer(kt, v[t, 0] - S.T @ kt)
    np.testing.assert_allclose(S_T[0, 0], S, rtol=1e-12, atol=1e-12)
    # alpha = 0 at the last step
    g1 = g.copy()
    g1[T - 1, 0, :] = -np.inf
    _, S_T, _ = oracle.prefill(q, k, v, g1, beta, S0, [0, T])
    np.testing.assert_allclose(S_T[0, 0], beta[T - 1, 0] * np.outer(k[T - 1, 0], v[T - 1, 0]),
                               rtol=1e-12, atol=1e-15)


def test_scalar_gate_special_case():
    """A gate that is equal on every channel is the scalar-gated (Gated DeltaNet)
    rule S_t = a_t (I - b k k^T) S_{t-1} + b k v^T, checked step by step."""
    rng = np.random.default_rng(7)
    T, dk, dv = 8, 6, 5
    q, k, v, g, beta, S0 = _rand_case(rng, T, 1, dk, dv)
    a = -np.abs(rng.standard_normal(T))
    g[:] = a[:, None, None]
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, S0, [0, T])
    S = S0[0, 0].copy()
    for t in range(T):
        kt, b = k[t, 0], beta[t, 0]
        S = math.exp(a[t]) * (np.eye(dk) - b * np.outer(kt, kt)) @ S + b * np.outer(kt, v[t, 0])
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_T[0, 0], S, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# the chunked algebra the kernels implement reaches the same result
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [16, 64, 128, 10_000])
def test_chunked_algebra_equals_recurrence(chunk):
    rng = np.random.default_rng(8)
    lengths = [1, 70, 200, 129]          # partial chunks and a 1-token sequence
    T, H, dk, dv = sum(lengths), 2, 16, 12
    q, k, v, g, beta, S0 = _rand_case(rng, T, H, dk, dv, N=len(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, S0, cu)
    o_c, S_c = chunked_model.prefill(q, k, v, g, beta, S0, cu, chunk)
    np.testing.assert_allclose(o_c, o, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(S_c, S_T, rtol=1e-10, atol=1e-11)


def test_padding_tokens_are_noops():
    """A token with g = 0, beta = 0 (and k = 0) leaves the state unchanged: the
    reading used to pad a ragged last chunk."""
    rng = np.random.default_rng(9)
    T, dk, dv = 12, 8, 8
    q, k, v, g, beta, S0 = _rand_case(rng, T, 1, dk, dv)
    _, S_a, _ = oracle.prefill(q, k, v, g, beta, S0, [0, T])
    pad = 5
    qp = np.concatenate([q, rng.standard_normal((pad, 1, dk))])
    kp = np.concatenate([k, np.zeros((pad, 1, dk))])
    vp = np.concatenate([v, rng.standard_normal((pad, 1, dv))])
    gp = np.concatenate([g, np.zeros((pad, 1, dk))])
    bp = np.concatenate([beta, np.zeros((pad, 1))])
    _, S_b, _ = oracle.prefill(qp, kp, vp, gp, bp, S0, [0, T + pad])
    np.testing.assert_array_equal(S_a, S_b)


# ---------------------------------------------------------------------------
# segmentation, packing, decode: the state is the whole checkpoint
# ---------------------------------------------------------------------------
def test_resume_from_state():
    rng = np.random.default_rng(10)
    T1, T2, H, dk, dv = 37, 50, 3, 8, 8
    q, k, v, g, beta, S0 = _rand_case(rng, T1 + T2, H, dk, dv)
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, S0, [0, T1 + T2])
    o1, S1, _ = oracle.prefill(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], S0, [0, T1])
    o2, S2, _ = oracle.prefill(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], S1, [0, T2])
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S_T, rtol=1e-12, atol=1e-13)


def test_packed_batch_equals_separate_sequences():
    rng = np.random.default_rng(11)
    lengths = [5, 0, 17, 3]
    T, H, dk, dv = sum(lengths), 2, 6, 4
    q, k, v, g, beta, S0 = _rand_case(rng, T, H, dk, dv, N=len(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S_T, _ = oracle.prefill(q, k, v, g, beta, S0, cu)
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        o_n, S_n, _ = oracle.prefill(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b],
                                     S0[n:n + 1], [0, b - a])
        np.testing.assert_array_equal(o[a:b], o_n)
        np.testing.assert_array_equal(S_T[n], S_n[0])
    # an empty sequence passes its initial state through
    np.testing.assert_array_equal(S_T[1], S0[1])


def test_decode_equals_prefill_of_one_more_token():
    rng = np.random.default_rng(12)
    T, B, H, dk, dv = 20, 3, 2, 8, 8
    q, k, v, g, beta, S0 = _rand_case(rng, B * (T + 1), H, dk, dv, N=B)
    q, k, v, g = (x.reshape(B, T + 1, H, -1) for x in (q, k, v, g))
    beta = beta.reshape(B, T + 1, H)
    o_full, S_full, _ = oracle.prefill(
        q.reshape(-1, H, dk), k.reshape(-1, H, dk), v.reshape(-1, H, dv),
        g.reshape(-1, H, dk), beta.reshape(-1, H), S0,
        np.arange(B + 1) * (T + 1))
    _, S_pre, _ = oracle.prefill(
        q[:, :T].reshape(-1, H, dk), k[:, :T].reshape(-1, H, dk),
        v[:, :T].reshape(-1, H, dv), g[:, :T].reshape(-1, H, dk),
        beta[:, :T].reshape(-1, H), S0, np.arange(B + 1) * T)
    o_d, S_d = oracle.decode_step(q[:, T], k[:, T], v[:, T], g[:, T], beta[:, T], S_pre)
    np.testing.assert_allclose(S_d, S_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o_d, o_full.reshape(B, T + 1, H, dv)[:, T], rtol=1e-12, atol=1e-13)


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(13)
    T, H, dk, dv = 40, 3, 8, 70          # 70 columns: three column blocks, ragged
    q, k, v, g, beta, S0 = _rand_case(rng, T, H, dk, dv)
    o1, S1, n1 = oracle.prefill(q, k, v, g, beta, S0, [0, T], nthreads=1)
    o8, S8, n8 = oracle.prefill(q, k, v, g, beta, S0, [0, T], nthreads=8)
    assert n1 == 1 and n8 >= 1
    np.testing.assert_array_equal(o1, o8)
    np.testing.assert_array_equal(S1, S8)


def test_rejects_bad_offsets():
    rng = np.random.default_rng(14)
    q, k, v, g, beta, S0 = _rand_case(rng, 6, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.prefill(q, k, v, g, beta, S0, [0, 7])
    with pytest.raises(ValueError):
        oracle.prefill(q, k, v, g, beta, np.zeros((2, 1, 4, 4)), [0, 4, 2])


# ---------------------------------------------------------------------------
# Gated DeltaNet (one gate per head): "Gated DeltaNet" section of the essay
# ---------------------------------------------------------------------------
def test_gdn_prefill_follows_the_scalar_gated_rule():
    """gdn_prefill with g [T, H] matches S_t = a_t S_{t-1} + k_t delta_t^T,
    delta_t = b_t (v_t - (a_t S_{t-1})^T k_t), written out per step in its
    'decay the old memory, then write the delta' order, over two sequences."""
    rng = np.random.default_rng(21)
    T, H, dk, dv = 11, 2, 5, 4
    q, k, v, _, beta, S0 = _rand_case(rng, T, H, dk, dv, N=2)
    g = -np.abs(rng.standard_normal((T, H)))
    cu = [0, 4, T]
    o, S_T, _ = oracle.gdn_prefill(q, k, v, g, beta, S0, cu)
    for n in range(2):
        for h in range(H):
            S = S0[n, h].copy()
            for t in range(cu[n], cu[n + 1]):
                a, b, kt = math.exp(g[t, h]), beta[t, h], k[t, h]
                delta = b * (v[t, h] - (a * S).T @ kt)
                S = a * S + np.outer(kt, delta)
                np.testing.assert_allclose(o[t, h], S.T @ q[t, h], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(S_T[n, h], S, rtol=1e-12, atol=1e-12)


def test_gdn_cumulative_decay():
    """With no writes (beta = 0) a value stored at the start is read at step t
    through the product of the gates a_1 ... a_t, one number for the whole
    head (the essay's cumulative-decay statement for Gated DeltaNet)."""
    rng = np.random.default_rng(22)
    T, H, dk, dv = 9, 3, 4, 6
    q, k, v, _, beta, S0 = _rand_case(rng, T, H, dk, dv)
    beta[:] = 0.0
    g = -np.abs(rng.standard_normal((T, H)))
    o, S_T, _ = oracle.gdn_prefill(q, k, v, g, beta, S0, [0, T])
    cum = np.cumsum(g, axis=0)
    for h in range(H):
        for t in range(T):
            np.testing.assert_allclose(o[t, h], math.exp(cum[t, h]) * (S0[0, h].T @ q[t, h]),
                                       rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S_T[0, h], math.exp(cum[-1, h]) * S0[0, h],
                                   rtol=1e-12, atol=1e-14)


def test_gdn_decode_matches_gdn_prefill_step():
    rng = np.random.default_rng(23)
    B, H, dk, dv = 3, 2, 4, 5
    q, k, v, _, beta, S0 = _rand_case(rng, B, H, dk, dv, N=B)
    g = -np.abs(rng.standard_normal((B, H)))
    o_d, S_d = oracle.gdn_decode_step(q[:, :, :], k, v, g, beta, S0)
    o_p, S_p, _ = oracle.gdn_prefill(q, k, v, g, beta, S0, list(range(B + 1)))
    np.testing.assert_allclose(o_d, o_p, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S_d, S_p, rtol=1e-13, atol=1e-14)

"""Pins for the fp64 oracle: closed forms, invariants, exact rational brute force.

Each test fixes a property of the gated delta rule with per-channel decay (the
reading of the KDA paragraph of "Kimi K3 on Fireworks: Fast RL at frontier
scale" that the oracle implements) by something other than the oracle itself:
a closed form, a special case with a known answer, a hand-derived worked
example, or exact rational arithmetic in a different (matrix-product) form.
Shapes use dk != dv wherever possible so that a transposed operand fails.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rng(seed):
    return np.random.default_rng(seed)


def _orthonormal_rows(n, d, rng):
    a = rng.standard_normal((d, d))
    qm, _ = np.linalg.qr(a)
    return qm[:n].copy()  # n orthonormal rows of length d


def _one_seq(x):
    """Add the head axis: [T, d] -> [T, 1, d]; [T] -> [T, 1]."""
    return np.asarray(x, dtype=np.float64)[:, None, ...]


def test_worked_example_by_hand():
    """Hand-stepped 2x2, two-token example (stored with its derivation)."""
    ex = json.load(open(os.path.join(GOLDEN, "worked_example_2x2.json")))
    q, k, v = (_one_seq(ex[n]) for n in ("q", "k", "v"))
    a, b = _one_seq(ex["alpha"]), _one_seq(ex["beta"])
    s0 = np.asarray(ex["init_state"])[None, None]
    cu = np.array([0, 2])
    o, fs = oracle.forward(q, k, v, a, b, cu, s0, scale=ex["scale"], gate_is_alpha=True)
    np.testing.assert_allclose(o[:, 0], ex["expected_o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(fs[0, 0], ex["expected_final_state"], rtol=0, atol=1e-14)
    # the same through log-gates: alpha = exp(g)
    o2, fs2 = oracle.forward(q, k, v, np.log(a), b, cu, s0, scale=ex["scale"])
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(fs2, fs, rtol=0, atol=1e-14)


def test_no_decay_no_write_keeps_state():
    """alpha = 1, beta = 0: S_t = S_0 exactly and o_t = S_0^T (scale q_t)."""
    rng = _rng(1)
    T, H, dk, dv = 7, 2, 5, 3
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = np.zeros((T, H, dk))
    b = np.zeros((T, H))
    s0 = rng.standard_normal((1, H, dk, dv))
    o, fs = oracle.forward(q, k, v, g, b, np.array([0, T]), s0, scale=0.7)
    assert np.array_equal(fs, s0)
    exp_o = np.einsum("hij,thi->thj", s0[0], 0.7 * q)
    np.testing.assert_allclose(o, exp_o, rtol=1e-13, atol=1e-13)


def test_pure_decay_closed_form():
    """beta = 0: S_t = Diag(prod_{s<=t} alpha_s) S_0 (decay acts on the dk rows)."""
    rng = _rng(2)
    T, dk, dv = 6, 5, 3
    q = rng.standard_normal((T, 1, dk))
    g = -rng.uniform(0.0, 0.7, size=(T, 1, dk))
    s0 = rng.standard_normal((1, 1, dk, dv))
    o, fs = oracle.forward(q, rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dv)), g,
                           np.zeros((T, 1)), np.array([0, T]), s0)
    cum = np.cumsum(g[:, 0], axis=0)  # [T, dk]
    for t in range(T):
        st = np.exp(cum[t])[:, None] * s0[0, 0]
        np.testing.assert_allclose(o[t, 0], st.T @ q[t, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fs[0, 0], np.exp(cum[-1])[:, None] * s0[0, 0], rtol=1e-12)


def test_accumulation_reduces_to_causal_linear_attention():
    """alpha = 1, S_0 = 0, orthonormal keys: o_t = sum_{s<=t} (q_t . k_s) beta_s v_s."""
    rng = _rng(3)
    T, dk, dv = 6, 8, 5
    k = _orthonormal_rows(T, dk, rng)[:, None, :]
    q = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    b = rng.uniform(0.1, 0.9, size=(T, 1))
    o, _ = oracle.forward(q, k, v, np.zeros((T, 1, dk)), b, np.array([0, T]), None, scale=1.0)
    for t in range(T):
        exp = sum((q[t, 0] @ k[s, 0]) * b[s, 0] * v[s, 0] for s in range(t + 1))
        np.testing.assert_allclose(o[t, 0], exp, rtol=1e-12, atol=1e-13)


def test_delta_rule_retrieval_and_overwrite():
    """beta = 1, alpha = 1, orthonormal keys, any S_0: S_t^T k_s = v_s for written s <= t;
    writing the same key twice keeps only the second value (inclusive output)."""
    rng = _rng(4)
    dk, dv, n = 8, 3, 5
    keys = _orthonormal_rows(n, dk, rng)
    vals = rng.standard_normal((n, dv))
    # write keys 0..n-1, then write key 2 again with a new value
    new_v2 = rng.standard_normal(dv)
    kk = np.concatenate([keys, keys[2:3]])
    vv = np.concatenate([vals, new_v2[None]])
    T = kk.shape[0]
    # query at token t is the key written at token t (inclusive output gives back v_t)
    o, fs = oracle.forward(kk[:, None], kk[:, None], vv[:, None], np.zeros((T, 1, dk)), np.ones((T, 1)),
                           np.array([0, T]), rng.standard_normal((1, 1, dk, dv)))
    np.testing.assert_allclose(o[:, 0], vv, rtol=1e-12, atol=1e-12)
    S = fs[0, 0]
    for s in range(n):
        want = new_v2 if s == 2 else vals[s]
        np.testing.assert_allclose(S.T @ keys[s], want, rtol=1e-12, atol=1e-12)


def test_basis_key_single_step():
    """k = e_m: row m becomes (1 - beta) alpha_m S0[m] + beta v, other rows alpha_i S0[i].
    Fixes that the delta step reads the decayed state and the sign of the correction."""
    rng = _rng(5)
    dk, dv, m = 4, 3, 2
    s0 = rng.standard_normal((dk, dv))
    alpha = rng.uniform(0.2, 0.9, size=dk)
    beta, v = 0.3, rng.standard_normal(dv)
    k = np.zeros(dk)
    k[m] = 1.0
    q = rng.standard_normal(dk)
    o, fs = oracle.forward(q[None, None], k[None, None], v[None, None], alpha[None, None],
                           np.array([[beta]]), np.array([0, 1]), s0[None, None], gate_is_alpha=True)
    want = alpha[:, None] * s0
    want[m] = (1 - beta) * alpha[m] * s0[m] + beta * v
    np.testing.assert_allclose(fs[0, 0], want, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(o[0, 0], want.T @ q, rtol=1e-13, atol=1e-13)


def test_reset_alpha_zero():
    """alpha_t0 = 0 (g = -inf) erases the state: outputs from t0 on equal a fresh run, bitwise."""
    rng = _rng(6)
    T, H, dk, dv, t0 = 12, 2, 6, 4, 5
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.0, 0.5, size=(T, H, dk))
    b = rng.uniform(0.0, 1.0, size=(T, H))
    g[t0] = -np.inf
    s0 = rng.standard_normal((1, H, dk, dv))
    o, fs = oracle.forward(q, k, v, g, b, np.array([0, T]), s0)
    o2, fs2 = oracle.forward(q[t0:], k[t0:], v[t0:], g[t0:], b[t0:], np.array([0, T - t0]), None)
    assert np.array_equal(o[t0:], o2)
    assert np.array_equal(fs, fs2)
    # alpha given directly (alpha_t0 = 0) resets the same way
    a = np.exp(g)
    o3, fs3 = oracle.forward(q, k, v, a, b, np.array([0, T]), s0, gate_is_alpha=True)
    o4, fs4 = oracle.forward(q[t0:], k[t0:], v[t0:], a[t0:], b[t0:], np.array([0, T - t0]), None,
                             gate_is_alpha=True)
    assert np.array_equal(o3[t0:], o4) and np.array_equal(fs3, fs4)


def _random_case(rng, T, H, dk, dv):
    q = rng.standard_normal((T, H, dk)) / math.sqrt(dk)
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = np.log(1.0 / (1.0 + np.exp(-(rng.standard_normal((T, H, dk)) + 3.0))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, b


@pytest.mark.parametrize("t_split", [1, 7, 16, 31])
def test_split_invariance_bitwise(t_split):
    """[0,t) then [t,T) with the carried state equals [0,T) bit for bit."""
    rng = _rng(7)
    T, H, dk, dv = 32, 3, 6, 5
    q, k, v, g, b = _random_case(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dk, dv)) * 0.1
    o, fs = oracle.forward(q, k, v, g, b, np.array([0, T]), s0)
    sl1, sl2 = slice(0, t_split), slice(t_split, T)
    o1, f1 = oracle.forward(q[sl1], k[sl1], v[sl1], g[sl1], b[sl1], np.array([0, t_split]), s0)
    o2, f2 = oracle.forward(q[sl2], k[sl2], v[sl2], g[sl2], b[sl2], np.array([0, T - t_split]), f1)
    assert np.array_equal(np.concatenate([o1, o2]), o)
    assert np.array_equal(f2, fs)


def test_varlen_packing_equals_separate_runs():
    rng = _rng(8)
    lens = [5, 0, 9, 1]
    H, dk, dv = 2, 4, 6
    T = sum(lens)
    q, k, v, g, b = _random_case(rng, T, H, dk, dv)
    s0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, fs = oracle.forward(q, k, v, g, b, cu, s0)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        on, fn = oracle.forward(q[sl], k[sl], v[sl], g[sl], b[sl], np.array([0, L]), s0[n:n + 1])
        assert np.array_equal(o[sl], on)
        assert np.array_equal(fs[n], fn[0])
    # a length-0 sequence returns its initial state unchanged
    assert np.array_equal(fs[1], s0[1])


def test_scale_is_linear_on_the_query():
    rng = _rng(9)
    T, H, dk, dv = 9, 2, 5, 3
    q, k, v, g, b = _random_case(rng, T, H, dk, dv)
    o1, f1 = oracle.forward(q, k, v, g, b, np.array([0, T]), None, scale=1.0)
    o2, f2 = oracle.forward(q, k, v, g, b, np.array([0, T]), None, scale=0.125)
    assert np.array_equal(o2, 0.125 * o1)  # power-of-two scale: exact
    assert np.array_equal(f1, f2)


def test_decode_and_replay_helpers_follow_forward():
    rng = _rng(10)
    H, dk, dv, N, slots_n = 2, 4, 3, 3, 5
    pool = rng.standard_normal((slots_n, H, dk, dv))
    slots = np.array([4, 0, 2])
    q, k, v, g, b = _random_case(rng, N, H, dk, dv)
    o, new_pool = oracle.decode(q, k, v, g, b, pool, slots, scale=0.5)
    for n in range(N):
        on, fn = oracle.forward(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1], b[n:n + 1],
                                np.array([0, 1]), pool[slots[n]][None], scale=0.5)
        assert np.array_equal(o[n], on[0]) and np.array_equal(new_pool[slots[n]], fn[0])
    assert np.array_equal(new_pool[[1, 3]], pool[[1, 3]])
    acc = [2, 0, 3]
    qa, ka, va, ga, ba = _random_case(rng, sum(acc), H, dk, dv)
    cu = np.concatenate([[0], np.cumsum(acc)])
    rp = oracle.replay(ka, va, ga, ba, cu, pool, slots)
    for n in range(N):
        sl = slice(cu[n], cu[n + 1])
        _, fn = oracle.forward(qa[sl], ka[sl], va[sl], ga[sl], ba[sl], np.array([0, acc[n]]),
                               pool[slots[n]][None])
        assert np.array_equal(rp[slots[n]], fn[0])


# ----------------------------------------------------------------------------------------------
# Exact rational arithmetic
# ----------------------------------------------------------------------------------------------

def _frac_matrix(rows, cols, rng, lo=-4, hi=4, den=8):
    return [[Fraction(int(rng.integers(lo, hi + 1)), den) for _ in range(cols)] for _ in range(rows)]


def _mm(a, b):
    return [[sum((a[i][p] * b[p][j] for p in range(len(b))), Fraction(0)) for j in range(len(b[0]))]
            for i in range(len(a))]


def _madd(a, b, s=1):
    return [[a[i][j] + s * b[i][j] for j in range(len(a[0]))] for i in range(len(a))]


def _transpose(a):
    return [list(r) for r in zip(*a)]


def _eye(n):
    return [[Fraction(int(i == j)) for j in range(n)] for i in range(n)]


def _diag(d):
    return [[d[i] if i == j else Fraction(0) for j in range(len(d))] for i in range(len(d))]


def _bruteforce_matrix_form(q, k, v, alpha, beta, s0, scale):
    """Recurrence as matrix products: S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T; o_t = S_t^T q."""
    dk = len(s0)
    S = [row[:] for row in s0]
    outs = []
    for t in range(len(k)):
        kc = [[x] for x in k[t]]                       # dk x 1
        house = _madd(_eye(dk), _mm(kc, _transpose(kc)), -beta[t])
        S = _madd(_mm(house, _mm(_diag(alpha[t]), S)), _mm(kc, [v[t]]), beta[t])
        qs = [[scale * x] for x in q[t]]
        outs.append([r[0] for r in _mm(_transpose(S), qs)])
    return outs, S


@pytest.mark.parametrize("seed,dk,dv,T", [(11, 4, 4, 8), (12, 4, 3, 7), (13, 3, 5, 6)])
def test_bruteforce_rational_matches_oracle(seed, dk, dv, T):
    rng = _rng(seed)
    q = _frac_matrix(T, dk, rng)
    k = _frac_matrix(T, dk, rng)
    v = _frac_matrix(T, dv, rng)
    alpha = [[Fraction(int(rng.integers(1, 9)), 8) for _ in range(dk)] for _ in range(T)]
    beta = [Fraction(int(rng.integers(0, 9)), 8) for _ in range(T)]
    s0 = _frac_matrix(dk, dv, rng)
    scale = Fraction(3, 4)
    outs, S = _bruteforce_matrix_form(q, k, v, alpha, beta, s0, scale)
    f = lambda m: np.array([[float(x) for x in r] for r in m])
    o, fs = oracle.forward(f(q)[:, None], f(k)[:, None], f(v)[:, None], f(alpha)[:, None],
                           np.array([float(x) for x in beta])[:, None], np.array([0, T]),
                           f(s0)[None, None], scale=float(scale), gate_is_alpha=True)
    np.testing.assert_allclose(o[:, 0], f(outs), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fs[0, 0], f(S), rtol=1e-13, atol=1e-13)


def _chunked_wy(q, k, v, alpha, beta, s0, scale, C):
    """The 64-token chunked form the CUDA kernel evaluates, in exact rationals, for chunk size C.

    Per chunk with state S (prefix products A_r = prod_{j<=r} alpha_j, A_C its last row):
      Kbar = K*A, Qbar = scale*Q*A, Ktil = K/A, Khat = K*A_C/A,
      M[r,i] = beta_r Kbar_r.Ktil_i (i<r), P[r,i] = Qbar_r.Ktil_i (i<=r), T = (I+M)^-1,
      W = T diag(beta) Kbar, Utl = T diag(beta) V, U = Utl - W S,
      O = Qbar S + P U, S <- Diag(A_C) S + Khat^T U.
    """
    dk, dv = len(s0), len(s0[0])
    S = [r[:] for r in s0]
    outs = []
    for c0 in range(0, len(k), C):
        idx = list(range(c0, min(c0 + C, len(k))))
        n = len(idx)
        A, acc = [], [Fraction(1)] * dk
        for t in idx:
            acc = [acc[c] * alpha[t][c] for c in range(dk)]
            A.append(acc)
        AC = A[-1]
        Kbar = [[k[t][c] * A[r][c] for c in range(dk)] for r, t in enumerate(idx)]
        Qbar = [[scale * q[t][c] * A[r][c] for c in range(dk)] for r, t in enumerate(idx)]
        Ktil = [[k[t][c] / A[r][c] for c in range(dk)] for r, t in enumerate(idx)]
        Khat = [[k[t][c] * AC[c] / A[r][c] for c in range(dk)] for r, t in enumerate(idx)]
        dot = lambda a, b: sum((x * y for x, y in zip(a, b)), Fraction(0))
        M = [[beta[idx[r]] * dot(Kbar[r], Ktil[i]) if i < r else Fraction(0) for i in range(n)]
             for r in range(n)]
        P = [[dot(Qbar[r], Ktil[i]) if i <= r else Fraction(0) for i in range(n)] for r in range(n)]
        # T = (I + M)^-1 by forward substitution (unit lower triangular)
        Tm = [[Fraction(0)] * n for _ in range(n)]
        for r in range(n):
            for m in range(n):
                Tm[r][m] = Fraction(int(r == m)) - sum((M[r][i] * Tm[i][m] for i in range(r)),
                                                       Fraction(0))
        Tb = [[Tm[r][i] * beta[idx[i]] for i in range(n)] for r in range(n)]
        W = _mm(Tb, Kbar)
        Utl = _mm(Tb, [v[t] for t in idx])
        U = _madd(Utl, _mm(W, S), -1)
        O = _madd(_mm(Qbar, S), _mm(P, U))
        outs.extend(O)
        S = _madd(_mm(_diag(AC), S), _mm(_transpose(Khat), U))
    return outs, S


@pytest.mark.parametrize("C", [1, 3, 4, 8])
def test_chunked_wy_identities_exact(C):
    """The chunked WY form used on the GPU equals the token recurrence exactly."""
    rng = _rng(20 + C)
    T, dk, dv = 10, 4, 3
    q = _frac_matrix(T, dk, rng)
    k = _frac_matrix(T, dk, rng)
    v = _frac_matrix(T, dv, rng)
    alpha = [[Fraction(int(rng.integers(1, 9)), 8) for _ in range(dk)] for _ in range(T)]
    beta = [Fraction(int(rng.integers(0, 9)), 8) for _ in range(T)]
    s0 = _frac_matrix(dk, dv, rng)
    scale = Fraction(1, 2)
    o_ref, s_ref = _bruteforce_matrix_form(q, k, v, alpha, beta, s0, scale)
    o_chk, s_chk = _chunked_wy(q, k, v, alpha, beta, s0, scale, C)
    assert o_chk == o_ref
    assert s_chk == s_ref


# ---------------------------------------------------------------------------------------------
# Optional input preprocessing (fused in the library behind flags): L2-normalised q / k rows,
# alpha = sigmoid(x_g) (the log-gate logsigmoid(x)), beta = sigmoid(x_beta).
# ---------------------------------------------------------------------------------------------
PREP_ALL = oracle.PREP_L2NORM_Q | oracle.PREP_L2NORM_K | oracle.PREP_SIGMOID_GATE | oracle.PREP_SIGMOID_BETA


def test_prep_closed_forms():
    x = np.array([[[3.0, 4.0, 0.0, 0.0], [0.0, 0.0, 5.0, 12.0]]])
    g = np.array([[[0.0, 40.0, -40.0, np.log(3.0)]] * 2]).reshape(1, 2, 4)
    b = np.array([[0.0, np.log(3.0)]])
    q2, k2, g2, b2 = oracle.prep(x, x, g, b, PREP_ALL, eps=0.0)
    np.testing.assert_allclose(q2[0, 0], [0.6, 0.8, 0.0, 0.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(k2[0, 1], [0.0, 0.0, 5 / 13, 12 / 13], rtol=0, atol=1e-15)
    # sigmoid(0) = 1/2, sigmoid(log 3) = 3/4, sigmoid(40) ~ 1, sigmoid(-40) ~ e^-40
    np.testing.assert_allclose(g2[0, 0], [0.5, 1.0, np.exp(-40.0), 0.75], rtol=1e-12, atol=0)
    np.testing.assert_allclose(b2[0], [0.5, 0.75], rtol=1e-15, atol=0)
    # only the flagged inputs change
    q3, k3, g3, b3 = oracle.prep(x, x, g, b, oracle.PREP_L2NORM_K, eps=0.0)
    assert np.array_equal(q3, x) and np.array_equal(g3, g) and np.array_equal(b3, b)


def test_prep_invariants():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 3, 16))
    g = rng.standard_normal((5, 3, 16)) * 4
    b = rng.standard_normal((5, 3))
    q1, k1, g1, b1 = oracle.prep(x, x, g, b, PREP_ALL, eps=0.0)
    q2, _, g2, b2 = oracle.prep(7.5 * x, x, -g, -b, PREP_ALL, eps=0.0)
    np.testing.assert_allclose(q2, q1, rtol=1e-14, atol=1e-15)          # scale invariance
    np.testing.assert_allclose(np.linalg.norm(k1, axis=-1), 1.0, rtol=1e-14)  # unit rows
    np.testing.assert_allclose(g1 + g2, 1.0, rtol=0, atol=1e-15)       # sigmoid(x) + sigmoid(-x) = 1
    np.testing.assert_allclose(b1 + b2, 1.0, rtol=0, atol=1e-15)
    # with eps > 0 the norm shrinks below one, more for short rows
    _, k_eps, _, _ = oracle.prep(x, x, g, b, oracle.PREP_L2NORM_K, eps=1.0)
    assert np.all(np.linalg.norm(k_eps, axis=-1) < 1.0)


def test_prep_forward_reduces_to_plain_forward():
    """Gate limits and fixed points of the preprocessing give the plain recurrence."""
    rng = _rng(21)
    T, H, dk, dv = 13, 2, 8, 6
    cu = np.array([0, 9, 13])
    q, k = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk))
    v, beta = rng.standard_normal((T, H, dv)), rng.standard_normal((T, H))
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)            # unit rows: L2 flag is a no-op (eps = 0)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    s0 = rng.standard_normal((2, H, dk, dv)) * 0.1
    xg_inf = np.full(k.shape, np.inf)                              # sigmoid(+inf) = 1: no decay
    o_a, s_a = oracle.forward(q, k, v, xg_inf, np.zeros_like(beta), cu, s0,
                              prep_flags=PREP_ALL, prep_eps=0.0)
    o_b, s_b = oracle.forward(q, k, v, np.zeros(k.shape), np.full(beta.shape, 0.5), cu, s0)
    np.testing.assert_allclose(o_a, o_b, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s_a, s_b, rtol=1e-13, atol=1e-13)
    # sigmoid(-inf) = 0 erases the state: equals a fresh start with no decay afterwards
    xg = np.full(k.shape, np.inf)
    xg[0] = -np.inf
    o_c, _ = oracle.forward(q, k, v, xg, beta, cu, s0, prep_flags=oracle.PREP_SIGMOID_GATE)
    o_d, _ = oracle.forward(q, k, v, np.zeros(k.shape), beta, cu, np.zeros_like(s0))
    np.testing.assert_allclose(o_c[:9], o_d[:9], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------------------------------------
# Backward (reverse mode of the recurrence): pinned against the forward by central finite
# differences, against a closed form, and by linearity.
# ------------------------------------------------------------------------------------------------

def _bwd_case(seed, lens=(5, 3, 0, 4), H=2, dk=3, dv=4):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = len(lens)
    d = dict(q=rng.standard_normal((T, H, dk)), k=rng.standard_normal((T, H, dk)),
             v=rng.standard_normal((T, H, dv)), g=-np.abs(rng.standard_normal((T, H, dk))) * 0.5,
             b=rng.uniform(0.1, 0.9, (T, H)), s0=rng.standard_normal((N, H, dk, dv)) * 0.3)
    Wo, Ws = rng.standard_normal((T, H, dv)), rng.standard_normal((N, H, dk, dv))
    return cu, d, Wo, Ws


@pytest.mark.parametrize("gate_is_alpha", [False, True])
def test_backward_matches_finite_differences_of_forward(gate_is_alpha):
    """L = sum(o * Wo) + sum(final * Ws): every gradient the backward returns equals the
    central difference of the forward's L (step 1e-6, fp64) to 1e-7 relative."""
    cu, d, Wo, Ws = _bwd_case(11 + gate_is_alpha)
    if gate_is_alpha:
        d["g"] = np.exp(d["g"])
    sc = 0.7

    def loss(q, k, v, g, b, s0):
        o, fs = oracle.forward(q, k, v, g, b, cu, s0, scale=sc, gate_is_alpha=gate_is_alpha)
        return float((o * Wo).sum() + (fs * Ws).sum())

    G = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["b"], cu, d["s0"], Wo, Ws, scale=sc,
                        gate_is_alpha=gate_is_alpha)
    h = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("b", "dbeta"), ("s0", "d_init")):
        arr = d[name]
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = dict(d), dict(d)
            plus[name] = arr.copy()
            plus[name][idx] += h
            minus[name] = arr.copy()
            minus[name][idx] -= h
            num[idx] = (loss(**plus) - loss(**minus)) / (2 * h)
        err = np.abs(num - G[key]).max() / np.abs(num).max()
        assert err < 1e-7, (name, err)


def test_backward_closed_form_without_delta_step():
    """beta = 0: S_t = Diag(A_t) S_0 with A_t the running product of exp(g), o_t = S_t^T (s q_t).
    Then dq_t = s Diag(A_t) S_0 do_t, d_init = sum_t Diag(A_t) (s q_t) do_t^T,
    dg_{u,i} = sum_{t >= u} s q_{t,i} A_{t,i} (S_0 do_t)_i, dk = dv = 0."""
    rng = np.random.default_rng(5)
    T, H, dk, dv, s = 6, 1, 3, 2, 0.9
    q, k, v = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.0, 0.7, (T, H, dk))
    b = np.zeros((T, H))
    s0 = rng.standard_normal((1, H, dk, dv))
    do = rng.standard_normal((T, H, dv))
    G = oracle.backward(q, k, v, g, b, np.array([0, T]), s0, do, None, scale=s)
    A = np.exp(np.cumsum(g[:, 0, :], axis=0))            # [T, dk]
    S0 = s0[0, 0]
    S0do = do[:, 0, :] @ S0.T                            # [T, dk]: (S_0 do_t)
    np.testing.assert_allclose(G["dq"][:, 0, :], s * A * S0do, rtol=1e-12, atol=1e-12)
    dinit = sum(np.outer(A[t] * s * q[t, 0], do[t, 0]) for t in range(T))
    np.testing.assert_allclose(G["d_init"][0, 0], dinit, rtol=1e-12, atol=1e-12)
    contrib = s * q[:, 0, :] * A * S0do                  # [T, dk], term of token t
    dg = np.cumsum(contrib[::-1], axis=0)[::-1]          # sum over t >= u
    np.testing.assert_allclose(G["dg"][:, 0, :], dg, rtol=1e-12, atol=1e-12)
    assert np.abs(G["dk"]).max() == 0.0 and np.abs(G["dv"]).max() == 0.0


def test_backward_is_linear_in_the_output_gradients_and_empty_sequences_pass_through():
    cu, d, Wo, Ws = _bwd_case(7)
    G1 = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["b"], cu, d["s0"], Wo, Ws)
    G2 = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["b"], cu, d["s0"], -2.5 * Wo, -2.5 * Ws)
    for key in G1:
        np.testing.assert_allclose(G2[key], -2.5 * G1[key], rtol=1e-12, atol=1e-12)
    # sequence 2 is empty: its initial-state gradient is the final-state gradient
    np.testing.assert_array_equal(G1["d_init"][2], Ws[2])


# ------------------------------------------------------------------------------------------------
# Short convolution of the input projections (depthwise, causal, width W, then SiLU), with
# the convolution state carried across calls.
# ------------------------------------------------------------------------------------------------

def _silu(x):
    return x / (1.0 + np.exp(-x))


def test_conv_matches_numpy_convolve_per_channel():
    """Each channel is numpy's valid-mode convolution of [state, x] with the reversed
    weights (w[W-1] weighs the current token), one value per token, then SiLU."""
    rng = np.random.default_rng(21)
    lens, H, C, W = [7, 0, 3, 5], 2, 3, 4
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = rng.standard_normal((T, H, C))
    w = rng.standard_normal((H, C, W))
    st = rng.standard_normal((len(lens), W - 1, H, C))
    y, so = oracle.conv(x, w, cu, st)
    for n in range(len(lens)):
        b, e = cu[n], cu[n + 1]
        for h in range(H):
            for c in range(C):
                full = np.concatenate([st[n, :, h, c], x[b:e, h, c]])
                if e > b:  # (numpy's valid mode swaps operands when the input is shorter than w)
                    ref = np.convolve(full, w[h, c, ::-1], mode="valid")   # one value per token
                    np.testing.assert_allclose(y[b:e, h, c], _silu(ref), rtol=1e-12, atol=1e-12)
                np.testing.assert_array_equal(so[n, :, h, c], full[len(full) - (W - 1):])


def test_conv_impulse_response_and_zero_state():
    """A unit impulse at token 0 with no state gives SiLU(w reversed) on tokens 0..W-1, then SiLU(0) = 0."""
    W, T = 4, 7
    x = np.zeros((T, 1, 1))
    x[0, 0, 0] = 1.0
    w = np.array([[[0.5, -1.0, 2.0, 3.0]]])
    y, so = oracle.conv(x, w, np.array([0, T]))
    np.testing.assert_allclose(y[:W, 0, 0], _silu(w[0, 0, ::-1]), rtol=1e-14)
    np.testing.assert_array_equal(y[W:, 0, 0], np.zeros(T - W))
    np.testing.assert_array_equal(so[0, :, 0, 0], np.zeros(W - 1))


def test_conv_state_carries_across_a_split():
    """conv over a sequence == conv over its first part, then the rest from the carried state."""
    rng = np.random.default_rng(22)
    T, H, C, W = 11, 2, 5, 4
    x = rng.standard_normal((T, H, C))
    w = rng.standard_normal((H, C, W))
    st = rng.standard_normal((1, W - 1, H, C))
    y, so = oracle.conv(x, w, np.array([0, T]), st)
    for cut in (1, 2, 3, 6):
        y1, s1 = oracle.conv(x[:cut], w, np.array([0, cut]), st)
        y2, s2 = oracle.conv(x[cut:], w, np.array([0, T - cut]), s1)
        np.testing.assert_array_equal(np.concatenate([y1, y2]), y)
        np.testing.assert_array_equal(s2, so)



def test_backward_with_preprocessing_matches_finite_differences():
    """With every preprocessing flag the backward returns the gradients with respect to the
    raw inputs: central differences of the forward with the same flags (1e-6 relative)."""
    cu, d, Wo, Ws = _bwd_case(31, lens=(4, 3), H=1, dk=3, dv=2)
    d["g"] = np.random.default_rng(3).standard_normal(d["g"].shape) + 2.0   # raw gate logits
    d["b"] = np.random.default_rng(4).standard_normal(d["b"].shape)          # raw beta logits
    sc, flags, eps = 0.8, 15, 1e-3

    def loss(q, k, v, g, b, s0):
        o, fs = oracle.forward(q, k, v, g, b, cu, s0, scale=sc, prep_flags=flags, prep_eps=eps)
        return float((o * Wo).sum() + (fs * Ws).sum())

    G = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["b"], cu, d["s0"], Wo, Ws, scale=sc, prep_flags=flags,
                        prep_eps=eps)
    h = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("b", "dbeta"), ("s0", "d_init")):
        arr = d[name]
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = dict(d), dict(d)
            plus[name] = arr.copy()
            plus[name][idx] += h
            minus[name] = arr.copy()
            minus[name][idx] -= h
            num[idx] = (loss(**plus) - loss(**minus)) / (2 * h)
        err = np.abs(num - G[key]).max() / np.abs(num).max()
        assert err < 1e-6, (name, err)

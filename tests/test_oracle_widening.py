"""Pins of the oracle's widening rows (CPU only): one set of hyperplanes per head, the hard-hash
limit beta -> infinity, and the exact angular attention that a P-bit hard hash estimates.

Each test names the passage it rests on.  The independent routes are numpy: the product-form
brute force of the soft kernel (shared with the core pins), integer bucket ids and collision
counts for the hard hash, and the matrix form arccos(Qhat Khat^T) for angular attention.
"""
import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import _attention_bruteforce, _rand, _unit_rows


# ------------------------------------------------------------------ per-head hyperplanes

@pytest.mark.parametrize("causal", [False, True])
def test_per_head_forward_equals_bruteforce(causal):
    """Each head hashes with its own W[h] (the pages are silent; reading: [H, L, P, d]).  B = 2 so
    that indexing W by (b, h) instead of h would read the wrong set."""
    B, H, N, d, P, L, beta = 2, 3, 11, 8, 2, 3, 4.0
    Q, K, V = (_rand((B, H, N, d), s) for s in (300, 301, 302))
    W = _rand((H, L, P, d), 303)
    O = oracle.forward(Q, K, V, W, beta, causal)
    for b in range(B):
        for h in range(H):
            bf = _attention_bruteforce(Q[b, h], K[b, h], V[b, h], W[h], beta, causal)
            np.testing.assert_allclose(O[b, h], bf, rtol=1e-11, atol=1e-12)
    # and a shared W is the per-head form with every head's set equal
    Os = oracle.forward(Q, K, V, W[1], beta, causal)
    Op = oracle.forward(Q, K, V, np.broadcast_to(W[1], W.shape), beta, causal)
    np.testing.assert_array_equal(Os, Op)


@pytest.mark.parametrize("causal", [False, True])
def test_per_head_backward_finite_differences(causal):
    """Central differences of sum(O * dO), O from the per-head product-form brute force, with
    respect to every entry of Q, K, V, and of beta per (b, h)."""
    B, H, N, d, P, L, beta = 1, 2, 6, 4, 2, 2, 3.0
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (310, 311, 312, 313))
    W = _rand((H, L, P, d), 314)
    dQ, dK, dV, db = oracle.backward(Q, K, V, dO, W, beta, causal, want_dbeta=True)

    def loss(Qx, Kx, Vx, bt=beta):
        return sum(float((_attention_bruteforce(Qx[0, h], Kx[0, h], Vx[0, h], W[h], bt, causal)
                          * dO[0, h]).sum()) for h in range(H))

    eps = 1e-6
    for which, g in enumerate((dQ, dK, dV)):
        fd = np.zeros_like(g)
        for idx in np.ndindex(*Q.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += eps
            lp = loss(*args)
            args[which][idx] -= 2 * eps
            fd[idx] = (lp - loss(*args)) / (2 * eps)
        assert np.abs(fd - g).max() <= 1e-6 * np.abs(g).max() + 1e-9, which
    for h in range(H):
        def lh(bt):
            return float((_attention_bruteforce(Q[0, h], K[0, h], V[0, h], W[h], bt, causal) * dO[0, h]).sum())
        fd = (lh(beta + eps) - lh(beta - eps)) / (2 * eps)
        assert abs(fd - db[0, h]) <= 1e-6 * max(1.0, abs(fd)), (h, fd, db[0, h])


def test_per_head_decode_reproduces_the_causal_forward():
    """Decode steps (the recurrent form of Algorithm 2) with per-head W give the causal forward."""
    B, H, N, d, P, L = 1, 3, 9, 8, 3, 2
    Q, K, V = (_rand((B, H, N, d), s) for s in (320, 321, 322))
    W = _rand((H, L, P, d), 323)
    ref = oracle.forward(Q, K, V, W, 10.0, True)
    state = np.zeros((B, H, L << P, d + 1))
    for t in range(N):
        o = oracle.decode_step(Q[:, :, t], K[:, :, t], V[:, :, t], W, 10.0, state)
        np.testing.assert_array_equal(o, ref[:, :, t])


# ------------------------------------------------------------------ hard hashing (beta = inf)

def _bucket_ids(X, W):
    """Integer corner ids sum_t [w_{l,t} . x > 0] 2^t, [M, L] (bit t set means v_{r,t} = +1)."""
    Z = np.einsum("lpd,md->mlp", W, X)
    return ((Z > 0).astype(np.int64) << np.arange(W.shape[1])).sum(axis=2)


def _hard_counts(Xq, Xk, W):
    """c_ij = number of tables in which q_i and k_j land in the same corner."""
    return (_bucket_ids(Xq, W)[:, None, :] == _bucket_ids(Xk, W)[None, :, :]).sum(axis=2)


@pytest.mark.parametrize("causal", [False, True])
def test_hard_hash_equals_collision_counting(causal):
    """beta -> infinity is hard hashing ("Soft corner assignments make hashing differentiable");
    each table then adds V_j to the query's bucket iff h(q) = h(k_j), so the read-out is the
    collision-count average sum_j c_ij V_j / sum_j c_ij."""
    B, H, N, d, P, L = 1, 2, 16, 8, 3, 4
    Q = _rand((B, H, N, d), 330)
    K = Q + 0.05 * _rand((B, H, N, d), 331)      # every query shares buckets with its own key
    V = _rand((B, H, N, d), 332)
    W = _rand((L, P, d), 333)
    O = oracle.forward(Q, K, V, W, math.inf, causal)
    for h in range(H):
        c = _hard_counts(Q[0, h], K[0, h], W).astype(float)
        if causal:
            c = np.tril(c)
        assert np.all(c.sum(axis=1) > 0)
        np.testing.assert_allclose(O[0, h], (c @ V[0, h]) / c.sum(axis=1, keepdims=True),
                                   rtol=1e-12, atol=1e-13)


def test_hard_hash_is_the_large_beta_limit():
    """The soft features saturate to the hard corners: at beta = 1e9 and |u| >= 1e-6 every other
    corner's logit is at least 2000 below the winner's, so exp() underflows to 0 and the soft
    oracle's output equals the hard one exactly."""
    B, H, N, d, P, L = 1, 1, 12, 8, 3, 2
    Q, K, V = (_rand((B, H, N, d), s) for s in (340, 341, 342))
    W = _rand((L, P, d), 343)
    U = np.tanh(np.einsum("lpd,md->mlp", W, _unit_rows(np.concatenate([Q[0, 0], K[0, 0]]))))
    assert np.abs(U).min() >= 1e-6
    np.testing.assert_array_equal(oracle.forward(Q, K, V, W, 1e9, False),
                                  oracle.forward(Q, K, V, W, math.inf, False))
    phs, _ = oracle.features(Q[0, 0], W, 1e9)
    phh, _ = oracle.features(Q[0, 0], W, math.inf)
    np.testing.assert_array_equal(phs, phh)
    assert set(np.unique(phh)) <= {0.0, 1.0} and np.all(phh.sum(axis=2) == 1.0)


def test_hard_hash_ties_split_evenly():
    """Reading: a projection that is exactly 0 keeps the limit sigma(0) = 1/2 of the soft bit, so
    the two corners that differ only in that bit get half the row each; a zero row is uniform."""
    d, P = 4, 2
    W = np.zeros((1, P, d))
    W[0, 0, 0] = 1.0                              # bit 0 reads x_0
    W[0, 1, 1] = 1.0                              # bit 1 reads x_1
    x = np.array([[0.0, 2.0, 1.0, 0.0],           # bit 0 tied, bit 1 = +1: corners 2 and 3
                  [-1.0, 0.0, 0.0, 0.0],          # bit 0 = -1, bit 1 tied: corners 0 and 2
                  [0.0, 0.0, 0.0, 0.0]])          # zero row: uniform
    ph, _ = oracle.features(x, W, math.inf)
    np.testing.assert_array_equal(ph[0, 0], [0.0, 0.0, 0.5, 0.5])
    np.testing.assert_array_equal(ph[1, 0], [0.5, 0.0, 0.5, 0.0])
    np.testing.assert_array_equal(ph[2, 0], [0.25] * 4)
    # the soft features agree on the tied bits at any beta (sigma(0) = 1/2 exactly)
    phs, _ = oracle.features(x, W, 1e9)
    np.testing.assert_array_equal(phs, ph)


def test_hard_hash_empty_buckets_give_no_output():
    """With hard hashing a query can meet no key in any table; its ratio is 0/0 (NaN in the
    oracle) while the other rows are unaffected."""
    d = 2
    W = np.array([[[1.0, 0.0]]])                  # L = P = 1: the sign of x_0
    K = np.array([[[[1.0, 0.3], [2.0, -1.0], [0.5, 0.5]]]])
    V = _rand(K.shape, 350)
    Q = np.array([[[[-1.0, 0.0], [1.0, 1.0], [3.0, 0.1]]]])
    O = oracle.forward(Q, K, V, W, math.inf, False)
    assert np.all(np.isnan(O[0, 0, 0]))
    np.testing.assert_allclose(O[0, 0, 1:], np.broadcast_to(V[0, 0].mean(axis=0), (2, d)), atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_hard_hash_backward(causal):
    """A hard hash is piecewise constant: no gradient reaches Q, K or beta; V gets
    dV_j = sum_i c_ij dO_i / den_i (over i >= j when causal)."""
    B, H, N, d, P, L = 1, 1, 14, 6, 2, 3
    Q = _rand((B, H, N, d), 360)
    K = Q + 0.05 * _rand((B, H, N, d), 361)
    V, dO = _rand((B, H, N, d), 362), _rand((B, H, N, d), 363)
    W = _rand((L, P, d), 364)
    dQ, dK, dV, db = oracle.backward(Q, K, V, dO, W, math.inf, causal, want_dbeta=True)
    assert np.all(dQ == 0) and np.all(dK == 0) and np.all(db == 0)
    c = _hard_counts(Q[0, 0], K[0, 0], W).astype(float)
    if causal:
        c = np.tril(c)
    ref = c.T @ (dO[0, 0] / c.sum(axis=1, keepdims=True))
    np.testing.assert_allclose(dV[0, 0], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_hard_hash_estimates_angular_attention(causal):
    """"A hash collision estimates a powered angular kernel": over many independent Gaussian
    tables, c_ij / L -> (1 - theta_ij / pi)^P, so the hard-hash read-out tends to P-powered
    angular attention.  At L = 200000 tables the collision rates are within ~1e-3 of the kernel."""
    B, H, N, d, P, L = 1, 1, 6, 8, 2, 200000
    Q, K, V = (_rand((B, H, N, d), s) for s in (370, 371, 372))
    W = _rand((L, P, d), 373)
    O = oracle.forward(Q, K, V, W, math.inf, causal)
    A = oracle.angular_forward(Q, K, V, P, causal)
    assert np.abs(O - A).max() < 0.02
    # a different power is clearly further away
    assert np.abs(oracle.angular_forward(Q, K, V, 2 * P, causal) - A).max() > 0.05


# ------------------------------------------------------------------ angular attention

def _angular_matrix_form(Q, K, V, gamma, causal):
    """numpy: S = (1 - arccos(clip(Qhat Khat^T)) / pi)^gamma, zero rows at cosine 0."""
    C = np.clip(_unit_rows(Q) @ _unit_rows(K).T, -1.0, 1.0)
    S = (1.0 - np.arccos(C) / np.pi) ** gamma
    if causal:
        S = np.tril(S)
    return (S @ V) / S.sum(axis=1, keepdims=True)


def test_angular_two_keys_closed_form():
    """Slides, "Choose a nonnegative kernel that can be sketched" (Eqs. 3-4): keys at angles pi/3
    and pi/2 from the query have kernel 2/3 and 1/2; with gamma = 2 the weights are 4/9 and 1/4,
    so O = (16/25, 9/25); with gamma = 1, O = (4/7, 3/7)."""
    Q = np.zeros((1, 1, 2, 4))                    # the oracle takes as many queries as keys:
    Q[..., 0] = 1.0                               # row 1 repeats the query
    K = np.zeros((1, 1, 2, 4))
    K[0, 0, 0, :2] = [0.5, math.sqrt(3) / 2]
    K[0, 0, 1, 1] = 3.0
    V = np.zeros((1, 1, 2, 4))
    V[0, 0, 0, 0] = V[0, 0, 1, 1] = 1.0
    np.testing.assert_allclose(oracle.angular_forward(Q, K, V, 2, False)[0, 0, 0, :2], [16 / 25, 9 / 25],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.angular_forward(Q, K, V, 1, False)[0, 0, 0, :2], [4 / 7, 3 / 7],
                               rtol=0, atol=1e-15)


def test_angular_kernel_at_zero_right_and_straight_angles():
    """The kernel is 1, 1/2 and 0 at angles 0, pi/2 and pi; orthogonal pairs score 2^-gamma."""
    gamma = 3
    Q = np.zeros((1, 1, 3, 3))                    # three copies of one query
    Q[..., 0] = 2.0
    K = np.array([[[[1.0, 0, 0], [0, 1.0, 0], [-1.0, 0, 0]]]])
    V = np.eye(3)[None, None]
    o = oracle.angular_forward(Q, K, V, gamma, False)[0, 0, 0]
    w = np.array([1.0, 2.0 ** -gamma, 0.0])
    np.testing.assert_allclose(o, w / w.sum(), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("gamma", [1, 3, 8, 2.5])
def test_angular_equals_matrix_form(causal, gamma):
    """The oracle's row loop against the numpy matrix form, with a ragged N and a zero row."""
    B, H, N, d = 2, 2, 13, 8
    Q, K, V = (_rand((B, H, N, d), s) for s in (380, 381, 382))
    Q[1, 0, 5] = 0.0
    K[0, 1, 2] = 0.0
    O = oracle.angular_forward(Q, K, V, gamma, causal)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(O[b, h], _angular_matrix_form(Q[b, h], K[b, h], V[b, h], gamma, causal),
                                       rtol=1e-12, atol=1e-13)
    rows = [0, 4, 12]
    np.testing.assert_array_equal(oracle.angular_forward(Q, K, V, gamma, causal, rows=rows), O[:, :, rows])


def test_angular_invariances():
    """Positive rescaling of any row changes nothing (the kernel reads only angles); flipping a
    key's sign moves its angle to pi - theta and does change the output; gamma = 0 and a zero
    query both give the plain mean of the values; causal row 0 is V_0."""
    B, H, N, d = 1, 1, 9, 6
    Q, K, V = (_rand((B, H, N, d), s) for s in (390, 391, 392))
    O = oracle.angular_forward(Q, K, V, 3, False)
    s = np.exp(_rand((B, H, N, 1), 393))
    np.testing.assert_allclose(oracle.angular_forward(Q * s, K / s, V, 3, False), O, rtol=1e-12, atol=1e-13)
    K2 = K.copy()
    K2[0, 0, 3] *= -1.0
    assert np.abs(oracle.angular_forward(Q, K2, V, 3, False) - O).max() > 1e-3
    np.testing.assert_allclose(oracle.angular_forward(Q, K, V, 0, False)[0, 0],
                               np.broadcast_to(V[0, 0].mean(axis=0), (N, d)), atol=1e-14)
    Qz = Q.copy()
    Qz[0, 0, 2] = 0.0
    np.testing.assert_allclose(oracle.angular_forward(Qz, K, V, 3, False)[0, 0, 2], V[0, 0].mean(axis=0),
                               atol=1e-14)
    np.testing.assert_allclose(oracle.angular_forward(Q, K, V, 3, True)[0, 0, 0], V[0, 0, 0], atol=1e-15)


def test_soft_race_error_falls_with_beta_and_tables():
    """The error bound's two terms ("The claimed bound separates bias and sampling error",
    Theorem 2): the soft-hash bias falls as beta grows, the sampling error as L grows.  Against
    P-powered angular attention: large beta beats small beta at many tables, many tables beat few
    at large beta."""
    B, H, N, d, P = 1, 1, 32, 16, 2
    Q, K, V = (_rand((B, H, N, d), s) for s in (400, 401, 402))
    A = oracle.angular_forward(Q, K, V, P, False)

    def err(beta, L):
        O = oracle.forward(Q, K, V, _rand((L, P, d), 403), beta, False)
        return float(np.sqrt(((O - A) ** 2).sum() / N))

    assert err(50.0, 4096) < 0.5 * err(0.5, 4096)
    assert err(50.0, 4096) < 0.5 * err(50.0, 8)


# ------------------------------------------------------------------ d(loss)/d(W)

@pytest.mark.parametrize("causal", [False, True])
def test_dW_finite_differences_shared(causal):
    """The hyperplanes W are the layer's other parameter next to beta (their rows give
    u = tanh(W xhat), "Soft corner assignments make hashing differentiable"): d(sum O * dO)/dW,
    summed over (b, h) for a shared W, against central differences of the product-form brute
    force on every entry."""
    B, H, N, d, P, L, beta = 1, 2, 7, 4, 2, 2, 3.0
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (410, 411, 412, 413))
    W = _rand((L, P, d), 414)
    *_, dW = oracle.backward(Q, K, V, dO, W, beta, causal, want_dW=True)
    got = dW.sum(axis=(0, 1))

    def loss(Wx):
        return sum(float((_attention_bruteforce(Q[0, h], K[0, h], V[0, h], Wx, beta, causal) * dO[0, h]).sum())
                   for h in range(H))

    eps = 1e-6
    fd = np.zeros_like(W)
    for idx in np.ndindex(*W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[idx] += eps
        Wm[idx] -= eps
        fd[idx] = (loss(Wp) - loss(Wm)) / (2 * eps)
    assert np.abs(fd - got).max() <= 1e-6 * np.abs(fd).max() + 1e-9


@pytest.mark.parametrize("causal", [False, True])
def test_dW_finite_differences_per_head(causal):
    """Per-head W: head h's gradient is the sum over the batch of its (b, h) terms (B = 2)."""
    B, H, N, d, P, L, beta = 2, 2, 5, 4, 2, 1, 2.0
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (420, 421, 422, 423))
    W = _rand((H, L, P, d), 424)
    *_, dW = oracle.backward(Q, K, V, dO, W, beta, causal, want_dW=True)
    got = dW.sum(axis=0)  # [H, L, P, d]
    eps = 1e-6
    for h in range(H):
        def loss(Wx):
            return sum(float((_attention_bruteforce(Q[b, h], K[b, h], V[b, h], Wx, beta, causal)
                              * dO[b, h]).sum()) for b in range(B))
        fd = np.zeros_like(W[h])
        for idx in np.ndindex(*W[h].shape):
            Wp, Wm = W[h].copy(), W[h].copy()
            Wp[idx] += eps
            Wm[idx] -= eps
            fd[idx] = (loss(Wp) - loss(Wm)) / (2 * eps)
        assert np.abs(fd - got[h]).max() <= 1e-6 * np.abs(fd).max() + 1e-9, h


@pytest.mark.parametrize("causal", [False, True])
def test_dW_sums_every_token_whatever_rows(causal):
    """Like d(loss)/d(beta), dW covers every token even when dQ, dK, dV are asked for a few rows;
    at beta = +inf (hard hashing) it is zero."""
    B, H, N, d, P, L = 1, 2, 13, 6, 3, 2
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (430, 431, 432, 433))
    W = _rand((L, P, d), 434)
    full = oracle.backward(Q, K, V, dO, W, 4.0, causal, want_dbeta=True, want_dW=True)
    part = oracle.backward(Q, K, V, dO, W, 4.0, causal, rows=[2, 9], want_dbeta=True, want_dW=True)
    np.testing.assert_allclose(part[3], full[3], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(part[4], full[4], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(part[0], full[0][:, :, [2, 9]])
    *_, dWh = oracle.backward(Q, K, V, dO, W, math.inf, causal, want_dW=True)
    assert np.all(dWh == 0)

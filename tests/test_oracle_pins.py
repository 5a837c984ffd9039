"""Pins of the float64 oracle to facts the pages and the mathematics fix (CPU only).

Each test names the passage it rests on.  The independent routes used here (numpy) share no
code with the oracle: the brute-force kernel uses the product-form identity of the soft bucket
probabilities, not the oracle's softmax over explicit hypercube corners and its sketches.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _unit_rows(X):
    n = np.linalg.norm(X, axis=-1, keepdims=True)
    return np.where(n > 0, X / np.where(n > 0, n, 1.0), 0.0)


def _bit_probs(X, W, beta):
    """(p, 1 - p) with p[m, l, t] = sigmoid(2 beta tanh(w_{l,t} . xhat_m)), the probability of
    corner bit +1; 1 - p is evaluated as sigmoid(-2 beta u) so that it keeps its digits."""
    U = np.tanh(np.einsum("lpd,md->mlp", W, _unit_rows(X)))
    return _sigmoid(2.0 * beta * U), _sigmoid(-2.0 * beta * U)


def _kernel_bruteforce(Xq, Xk, W, beta):
    """S_ij = sum_l phi(q_i) . phi(k_j) through the product form: for each table,
    phi(q).phi(k) = prod_t [p_t(q) p_t(k) + (1 - p_t(q)) (1 - p_t(k))]."""
    pq, mq = _bit_probs(Xq, W, beta)
    pk, mk = _bit_probs(Xk, W, beta)
    agree = pq[:, None] * pk[None, :] + mq[:, None] * mk[None, :]
    return agree.prod(axis=3).sum(axis=2)


def _attention_bruteforce(Q, K, V, W, beta, causal):
    """O_i = sum_j S_ij V_j / sum_j S_ij (paper Eq. 3 with the implicit RACE kernel)."""
    S = _kernel_bruteforce(Q, K, W, beta)
    if causal:
        S = np.tril(S)
    return (S @ V) / S.sum(axis=1, keepdims=True)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ------------------------------------------------------------------ read-out with given features

def test_worked_example_global_ratio(golden_dir):
    """Slides, 'Backup: bucket masses change the answer': 4.3 / 0.95 = 4.5263, not 4.3030."""
    g = json.load(open(os.path.join(golden_dir, "race_worked_example.json")))
    phiK = np.array(g["phiK"])[None]           # [L=1, N=2, R=2]
    phiQ = np.array(g["phiQ"])[None]           # [L=1, M=1, R=2]
    V = np.array(g["V"])
    O, mass, content = oracle.readout_given_phi(phiK, V, phiQ)
    np.testing.assert_allclose(mass[0], g["mass"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(content[0, :, 0], g["content"], rtol=0, atol=1e-14)
    assert abs(O[0, 0] - g["O"]) < 1e-13
    assert round(O[0, 0], 4) == g["O_rounded_as_printed"]
    # per-bucket means mixed by phi(Q) is the other operator the pages warn about
    assert abs(O[0, 0] - g["per_bucket_means_variant"]) > 0.2
    # the equivalent pairwise weights phi(Q).phi(K_j)
    w = phiQ[0, 0] @ phiK[0].T
    np.testing.assert_allclose(w, g["pairwise_weights"], atol=1e-15)


def test_linear_attention_example(golden_dir):
    """Visual walkthrough, Step 5 example: S = [10, 4, 5], Z = [4, 2, 2], out = 14/6."""
    g = json.load(open(os.path.join(golden_dir, "linear_attention_example.json")))
    phiK = np.array(g["phiK"], dtype=float)[None]
    phiQ = np.array(g["phiQ"], dtype=float)[None]
    V = np.array(g["V"], dtype=float)
    O, mass, content = oracle.readout_given_phi(phiK, V, phiQ)
    np.testing.assert_allclose(content[0, :, 0], g["S"], atol=0)
    np.testing.assert_allclose(mass[0], g["Z"], atol=0)
    assert O[0, 0] == pytest.approx(g["num"] / g["den"], abs=1e-15)


def test_readout_given_phi_causal_is_prefix():
    """Slides, 'Causality is a prefix update': query t reads the sketch after key t is added."""
    rng = np.random.default_rng(3)
    L, N, R, dv = 2, 9, 4, 3
    phiK = rng.random((L, N, R))
    phiQ = rng.random((L, N, R))
    V = rng.standard_normal((N, dv))
    O, _, _ = oracle.readout_given_phi(phiK, V, phiQ, causal=True)
    for t in range(N):
        w = sum(phiQ[l, t] @ phiK[l, : t + 1].T for l in range(L))
        np.testing.assert_allclose(O[t], w @ V[: t + 1] / w.sum(), rtol=1e-13)


# ------------------------------------------------------------------ features (Algorithm 1)

@pytest.mark.parametrize("P,beta", [(1, 10.0), (2, 0.7), (3, 10.0), (6, 3.0), (8, 10.0)])
def test_features_product_form_and_simplex(P, beta):
    """Reading notes 2.4: phi_r = prod_t sigmoid(2 beta u_t v_{r,t}); phi is a probability vector."""
    X = _rand((17, 24), 1 + P)
    X[5] = 0.0  # zero row: xhat = 0, u = 0, uniform buckets
    W = _rand((3, P, 24), 2 + P)
    phi, u = oracle.features(X, W, beta)
    np.testing.assert_allclose(u, np.tanh(np.einsum("lpd,md->mlp", W, _unit_rows(X))), atol=1e-15)
    p, m = _bit_probs(X, W, beta)
    R = 1 << P
    bits = (np.arange(R)[:, None] >> np.arange(P)[None, :]) & 1          # [R, P]
    prod = np.where(bits[None, None], p[:, :, None, :], m[:, :, None, :]).prod(axis=3)
    np.testing.assert_allclose(phi, prod, rtol=1e-12, atol=1e-300)
    assert np.all(phi >= 0)
    np.testing.assert_allclose(phi.sum(axis=2), 1.0, atol=1e-14)
    np.testing.assert_allclose(phi[5], 1.0 / R, atol=1e-15)


def test_features_beta_zero_uniform():
    """Slides, soft corners: beta -> 0 gives uniform buckets."""
    X = _rand((5, 16), 7)
    W = _rand((2, 3, 16), 8)
    phi, _ = oracle.features(X, W, 0.0)
    np.testing.assert_allclose(phi, 1.0 / 8, atol=1e-16)


def test_features_large_beta_is_hard_hash():
    """Slides, soft corners: beta -> infinity recovers h(x) = sign(W x)."""
    X = _rand((50, 16), 9)
    W = _rand((4, 3, 16), 10)
    phi, u = oracle.features(X, W, 1e6)
    signs = (u > 0).astype(int)
    idx = (signs * (1 << np.arange(3))).sum(axis=2)                        # [M, L]
    onehot = np.zeros_like(phi)
    np.put_along_axis(onehot, idx[..., None], 1.0, axis=2)
    np.testing.assert_allclose(phi, onehot, atol=1e-12)


def test_counterexample_bound():
    """Slides, 'Backup: Lemma 10 omits the soft-hash bias': Q = K unit, P = 2, beta = 0.1 gives
    phi . phi <= max_r phi_r <= e^0.4 / 4 < 0.373 for every table."""
    x = _rand((1, 32), 11)
    x /= np.linalg.norm(x)
    W = _rand((2000, 2, 32), 12)
    phi, _ = oracle.features(x, W, 0.1)
    sq = (phi[0] ** 2).sum(axis=1)
    assert np.all(sq <= phi[0].max(axis=1) + 1e-15)
    assert phi[0].max() <= math.exp(0.4) / 4 + 1e-15
    assert sq.max() < 0.373


@pytest.mark.parametrize("theta,P", [(math.pi / 2, 3), (math.pi / 3, 2), (math.pi / 4, 3)])
def test_hard_hash_collision_rate(theta, P):
    """Slides, 'A hash collision estimates a powered angular kernel': with hard hashing the
    collision probability over Gaussian tables is (1 - theta/pi)^P; orthogonal pairs 2^-P."""
    d, T = 16, 100000
    q = np.zeros(d)
    q[0] = 1.0
    k = np.zeros(d)
    k[0], k[1] = math.cos(theta), math.sin(theta)
    W = _rand((T, P, d), 13 + P)
    phq, _ = oracle.features(q[None], W, 1e4)
    phk, _ = oracle.features(k[None], W, 1e4)
    coll = (phq[0] * phk[0]).sum(axis=1)                                   # per table
    target = (1.0 - theta / math.pi) ** P
    sigma = math.sqrt(target * (1.0 - target) / T)
    assert abs(coll.mean() - target) < 5 * sigma
    if abs(theta - math.pi / 2) < 1e-12:
        assert abs(target - 2.0 ** -P) < 1e-15


# ------------------------------------------------------------------ forward (Algorithms 1 and 2)

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("beta,P,L", [(10.0, 2, 2), (1.0, 3, 2), (4.0, 1, 5)])
def test_forward_equals_bruteforce(causal, beta, P, L):
    """Slides, 'Normalize after combining the tables': the sketch read-out equals
    O_i = sum_j S_ij V_j / sum_j S_ij with S_ij = sum_l phi(Q_i) . phi(K_j) (causal: j <= i)."""
    B, H, N, d = 1, 2, 40, 16
    Q, K, V = (_rand((B, H, N, d), s) for s in (20, 21, 22))
    W = _rand((L, P, d), 23)
    O = oracle.forward(Q, K, V, W, beta, causal)
    for h in range(H):
        ref = _attention_bruteforce(Q[0, h], K[0, h], V[0, h], W, beta, causal)
        np.testing.assert_allclose(O[0, h], ref, rtol=1e-12, atol=1e-12)


def test_forward_c1_shape_bruteforce():
    """The tiny float32 workload's shape (N=256, d=64, (P,L)=(2,2), beta=10), both modes."""
    Q, K, V = (_rand((1, 1, 256, 64), s) for s in (30, 31, 32))
    W = _rand((2, 2, 64), 33)
    for causal in (False, True):
        O = oracle.forward(Q, K, V, W, 10.0, causal)
        ref = _attention_bruteforce(Q[0, 0], K[0, 0], V[0, 0], W, 10.0, causal)
        np.testing.assert_allclose(O[0, 0], ref, rtol=1e-11, atol=1e-12)


def test_output_in_convex_hull():
    """Slides, 'Choose a nonnegative kernel': outputs are convex combinations of values."""
    Q, K, V = (_rand((1, 1, 64, 8), s) for s in (40, 41, 42))
    W = _rand((2, 3, 8), 43)
    O = oracle.forward(Q, K, V, W, 10.0, False)[0, 0]
    assert np.all(O <= V[0, 0].max(axis=0) + 1e-12) and np.all(O >= V[0, 0].min(axis=0) - 1e-12)
    Oc = oracle.forward(Q, K, V, W, 10.0, True)[0, 0]
    hi = np.maximum.accumulate(V[0, 0], axis=0)
    lo = np.minimum.accumulate(V[0, 0], axis=0)
    assert np.all(Oc <= hi + 1e-12) and np.all(Oc >= lo - 1e-12)


def test_single_token_and_first_causal_row():
    """Visual walkthrough, Step 6 case B: one token attends to itself, out = v_1; the first causal
    row is that case (update before read)."""
    Q, K, V = (_rand((1, 1, 1, 8), s) for s in (50, 51, 52))
    W = _rand((3, 2, 8), 53)
    for causal in (False, True):
        np.testing.assert_allclose(oracle.forward(Q, K, V, W, 10.0, causal), V, rtol=1e-13)
    Q, K, V = (_rand((1, 1, 30, 8), s) for s in (54, 55, 56))
    np.testing.assert_allclose(oracle.forward(Q, K, V, W, 10.0, True)[0, 0, 0], V[0, 0, 0], rtol=1e-13)


def test_causal_last_row_is_noncausal_row():
    """Algorithm 2 includes the current token, so the last causal row sees every key."""
    Q, K, V = (_rand((1, 2, 33, 8), s) for s in (60, 61, 62))
    W = _rand((2, 2, 8), 63)
    Oc = oracle.forward(Q, K, V, W, 10.0, True)
    On = oracle.forward(Q, K, V, W, 10.0, False)
    np.testing.assert_allclose(Oc[:, :, -1], On[:, :, -1], rtol=1e-12)


def test_beta_zero_gives_mean_of_values():
    """Uniform buckets make every pair weight equal: O = mean of V (causal: prefix mean)."""
    Q, K, V = (_rand((1, 1, 20, 8), s) for s in (70, 71, 72))
    W = _rand((2, 2, 8), 73)
    np.testing.assert_allclose(oracle.forward(Q, K, V, W, 0.0, False)[0, 0],
                               np.broadcast_to(V[0, 0].mean(axis=0), (20, 8)), rtol=1e-12)
    pref = np.cumsum(V[0, 0], axis=0) / np.arange(1, 21)[:, None]
    np.testing.assert_allclose(oracle.forward(Q, K, V, W, 0.0, True)[0, 0], pref, rtol=1e-12)


def test_row_scale_invariance_and_zero_row():
    """Reading taken: Q and K rows are L2-normalised first, so positive rescaling of any row leaves
    O unchanged; a zero query row has uniform buckets and reads the plain mean of V."""
    Q, K, V = (_rand((1, 1, 24, 8), s) for s in (80, 81, 82))
    W = _rand((2, 3, 8), 83)
    O = oracle.forward(Q, K, V, W, 10.0, False)
    s = np.exp(_rand((1, 1, 24, 1), 84))
    np.testing.assert_allclose(oracle.forward(Q * s, K / s, V, W, 10.0, False), O, rtol=1e-12)
    Q[0, 0, 3] = 0.0
    O0 = oracle.forward(Q, K, V, W, 10.0, False)
    np.testing.assert_allclose(O0[0, 0, 3], V[0, 0].mean(axis=0), rtol=1e-12)
    # the `normalize` switch is live: without it the raw rows are projected
    assert np.abs(oracle.forward(Q * 3, K, V, W, 10.0, False, normalize=False) -
                  oracle.forward(Q, K, V, W, 10.0, False, normalize=False)).max() > 1e-3


def test_rows_subset_matches_full():
    Q, K, V, dO = (_rand((2, 1, 37, 8), s) for s in (90, 91, 92, 93))
    W = _rand((2, 2, 8), 94)
    rows = np.array([0, 5, 6, 20, 36])
    for causal in (False, True):
        O = oracle.forward(Q, K, V, W, 10.0, causal)
        np.testing.assert_array_equal(oracle.forward(Q, K, V, W, 10.0, causal, rows=rows), O[:, :, rows])
        full = oracle.backward(Q, K, V, dO, W, 10.0, causal)
        part = oracle.backward(Q, K, V, dO, W, 10.0, causal, rows=rows)
        for a, b in zip(full, part):
            np.testing.assert_allclose(b, a[:, :, rows], rtol=1e-13, atol=1e-15)


def test_bf16_bits_are_widened_exactly():
    import torch
    from linear_lsh_sketch_gb300.workloads import as_oracle_array
    x = torch.randn(1, 1, 16, 8).to(torch.bfloat16)
    W = _rand((1, 2, 8), 95)
    a = oracle.forward(as_oracle_array(x), as_oracle_array(x), as_oracle_array(x), W, 10.0, False)
    b = oracle.forward(x.double().numpy(), x.double().numpy(), x.double().numpy(), W, 10.0, False)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ backward (chain rule)

def _loss(Q, K, V, dO, W, beta, causal):
    return float((oracle.forward(Q, K, V, W, beta, causal) * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("beta,P,L", [(10.0, 2, 2), (2.0, 3, 1)])
def test_backward_finite_differences_every_entry(causal, beta, P, L):
    """Central differences of loss = sum(O * dO) with respect to every entry of Q, K and V."""
    B, H, N, d = 1, 2, 10, 6
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (100, 101, 102, 103))
    W = _rand((L, P, d), 104)
    grads = oracle.backward(Q, K, V, dO, W, beta, causal)
    h = 1e-6
    for which, g in zip(range(3), grads):
        fd = np.zeros_like(g)
        for idx in np.ndindex(*Q.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            lp = _loss(*args, dO, W, beta, causal)
            args[which][idx] -= 2 * h
            lm = _loss(*args, dO, W, beta, causal)
            fd[idx] = (lp - lm) / (2 * h)
        scale = np.abs(g).max()
        assert np.abs(fd - g).max() <= 1e-6 * scale + 1e-9, which


@pytest.mark.parametrize("causal", [False, True])
def test_backward_directional_c1_shape(causal):
    """Directional derivatives on the tiny float32 workload's shape (N=256, d=64, (P,L)=(2,2))."""
    Q, K, V, dO = (_rand((1, 1, 256, 64), s) for s in (110, 111, 112, 113))
    W = _rand((2, 2, 64), 114)
    dQ, dK, dV = oracle.backward(Q, K, V, dO, W, 10.0, causal)
    h = 1e-6
    for s in range(3):
        tq, tk, tv = (_rand(Q.shape, 120 + 3 * s + i) for i in range(3))
        lp = _loss(Q + h * tq, K + h * tk, V + h * tv, dO, W, 10.0, causal)
        lm = _loss(Q - h * tq, K - h * tk, V - h * tv, dO, W, 10.0, causal)
        fd = (lp - lm) / (2 * h)
        an = (dQ * tq).sum() + (dK * tk).sum() + (dV * tv).sum()
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an))


def test_zero_row_gradient_is_zero():
    """Reading taken: the normalisation has no derivative at a zero row; its gradient is 0."""
    Q, K, V, dO = (_rand((1, 1, 12, 8), s) for s in (130, 131, 132, 133))
    Q[0, 0, 4] = 0.0
    K[0, 0, 7] = 0.0
    W = _rand((2, 2, 8), 134)
    dQ, dK, _ = oracle.backward(Q, K, V, dO, W, 10.0, False)
    assert np.all(dQ[0, 0, 4] == 0) and np.all(dK[0, 0, 7] == 0)


# ------------------------------------------------------------------ d(loss)/d(beta)

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("beta,P,L", [(10.0, 2, 2), (2.0, 3, 1), (5.0, 1, 3)])
def test_dbeta_finite_differences(causal, beta, P, L):
    """beta is trained with the layer ("RACE Attention" slides, "Soft corner assignments make
    hashing differentiable"): d(sum O * dO)/d(beta) per (b, h) against central differences of the
    independent product-form brute force (paper Eq. 3 with the implicit RACE kernel)."""
    B, H, N, d = 1, 2, 10, 6
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (140, 141, 142, 143))
    W = _rand((L, P, d), 144)
    *_, db = oracle.backward(Q, K, V, dO, W, beta, causal, want_dbeta=True)
    h = 1e-6
    for b in range(B):
        for hh in range(H):
            def loss(bt):
                O = _attention_bruteforce(Q[b, hh], K[b, hh], V[b, hh], W, bt, causal)
                return float((O * dO[b, hh]).sum())
            fd = (loss(beta + h) - loss(beta - h)) / (2 * h)
            assert abs(fd - db[b, hh]) <= 1e-6 * max(1.0, abs(fd)), (b, hh, fd, db[b, hh])


@pytest.mark.parametrize("causal", [False, True])
def test_dbeta_sums_every_token_whatever_rows(causal):
    """d(loss)/d(beta) covers every token even when only some rows' dQ, dK, dV are asked for, and
    asking for it leaves dQ, dK, dV unchanged."""
    Q, K, V, dO = (_rand((2, 1, 33, 8), s) for s in (150, 151, 152, 153))
    W = _rand((3, 2, 8), 154)
    full = oracle.backward(Q, K, V, dO, W, 7.0, causal, want_dbeta=True)
    plain = oracle.backward(Q, K, V, dO, W, 7.0, causal)
    rows = np.array([0, 5, 17, 32])
    part = oracle.backward(Q, K, V, dO, W, 7.0, causal, rows=rows, want_dbeta=True)
    np.testing.assert_array_equal(full[3], part[3])
    for a, p, q in zip(full[:3], part[:3], plain):
        np.testing.assert_array_equal(a, q)
        np.testing.assert_array_equal(a[:, :, rows], p)


# ------------------------------------------------------------------ causal decode step

@pytest.mark.parametrize("P,L", [(2, 2), (3, 3)])
def test_decode_steps_reproduce_the_causal_forward(P, L):
    """Algorithm 2 is a recurrence ("Causality is a prefix update of the same statistics"): adding
    one key at a time to an empty prefix sketch and reading with the same token's query gives the
    causal forward, row for row (the same sums in the same order: bit for bit)."""
    B, H, N, d = 2, 2, 23, 8
    Q, K, V = (_rand((B, H, N, d), s) for s in (160, 161, 162))
    W = _rand((L, P, d), 163)
    ref = oracle.forward(Q, K, V, W, 10.0, True)
    state = np.zeros((B, H, L << P, d + 1))
    for t in range(N):
        o = oracle.decode_step(Q[:, :, t], K[:, :, t], V[:, :, t], W, 10.0, state)
        np.testing.assert_array_equal(o, ref[:, :, t])


def test_decode_continues_a_prefill_sketch():
    """The state after a prompt is the prompt's non-causal sketch [A | B] (the sum over its keys),
    so decoding on from it matches the causal forward of prompt + continuation; the independent
    product-form brute force checks the same rows."""
    B, H, N0, N, d, P, L = 1, 2, 15, 21, 8, 3, 2
    Q, K, V = (_rand((B, H, N, d), s) for s in (170, 171, 172))
    W = _rand((L, P, d), 173)
    _, state = oracle.forward(Q[:, :, :N0], K[:, :, :N0], V[:, :, :N0], W, 10.0, False, want_sketch=True)
    state = np.ascontiguousarray(state)
    ref = oracle.forward(Q, K, V, W, 10.0, True)
    for t in range(N0, N):
        o = oracle.decode_step(Q[:, :, t], K[:, :, t], V[:, :, t], W, 10.0, state)
        np.testing.assert_allclose(o, ref[:, :, t], rtol=1e-12, atol=1e-12)
        for h in range(H):
            bf = _attention_bruteforce(Q[0, h, :t + 1], K[0, h, :t + 1], V[0, h, :t + 1], W, 10.0, True)[-1]
            np.testing.assert_allclose(o[0, h], bf, rtol=1e-10, atol=1e-12)

"""float64 CPU oracle of one RACE attention layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may import this
package. It shares no code with the GPU library and the GPU library never calls it.

Sources: "RACE Attention" slides (paper Algorithm 1, frames "Soft corner assignments make
hashing differentiable", "Each bucket stores mass and a weighted value sum", "Normalize after
combining the tables"; paper Algorithm 2, frame "Causality is a prefix update of the same
statistics") and the reading notes, sections 2.4-2.6; the hard-hash limit and the angular kernel
it collides with (frames "A hash collision estimates a powered angular kernel" and "Choose a
nonnegative kernel that can be sketched"; reading notes 2.3 and 3.1).  The C source states every
step.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None
_i64 = ctypes.c_int64
_dp = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.race_oracle_max_p.restype = ctypes.c_int
        L.race_oracle_features.argtypes = [_i64, _i64, _vp, _vp, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_int, _vp, _vp]
        L.race_oracle_readout_given_phi.argtypes = [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                                    _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp]
        L.race_oracle_forward.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_int, ctypes.c_int, _vp, _i64, _vp, _vp, ctypes.c_int]
        L.race_oracle_backward.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp,
                                           _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                           ctypes.c_int, ctypes.c_int, _vp, _i64, _vp, _vp, _vp, _vp,
                                           _vp, ctypes.c_int]
        L.race_oracle_decode_step.argtypes = [_i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                              ctypes.c_int, _vp, _vp]
        L.race_oracle_angular_forward.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp,
                                                  ctypes.c_double, ctypes.c_int, _vp, _i64, _vp,
                                                  ctypes.c_int]
        for f in ("race_oracle_features", "race_oracle_readout_given_phi", "race_oracle_forward",
                  "race_oracle_backward", "race_oracle_decode_step", "race_oracle_angular_forward"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _tokens(a):
    """Token tensor as (contiguous array, element code). bf16 arrives as uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, 0
    if a.dtype == np.float32:
        return a, 1
    if a.dtype == np.uint16:
        return a, 2
    raise TypeError("oracle token tensors must be float64, float32 or bf16 bits (uint16)")


def _check(status, what):
    if status != 0:
        raise ValueError("%s failed with status %d" % (what, status))


def _hash(W, H):
    """Hyperplanes as (float64 array, per_head, L, P): W is [L, P, d] shared by every head, or
    [H, L, P, d], one set per head."""
    W = _f64(W)
    if W.ndim == 3:
        return W, 0, W.shape[0], W.shape[1]
    assert W.ndim == 4 and W.shape[0] == H, "W must be [L, P, d] or [H, L, P, d]"
    return W, 1, W.shape[1], W.shape[2]


def features(X, W, beta, normalize=True):
    """Bucket probabilities of rows X [M, d] for W [L, P, d]: returns (phi [M, L, R], u [M, L, P]).
    beta = inf gives the hard hash (one corner per table; a zero projection splits evenly)."""
    X = _f64(X)
    W = _f64(W)
    M, d = X.shape
    L, P, _ = W.shape
    R = 1 << P
    phi = np.empty((M, L, R))
    u = np.empty((M, L, P))
    _check(lib().race_oracle_features(M, d, _ptr(X), _ptr(W), L, P, float(beta), int(normalize),
                                      _ptr(phi), _ptr(u)), "features")
    return phi, u


def readout_given_phi(phiK, V, phiQ, causal=False):
    """Sketch + global-ratio read-out with bucket probabilities given directly.

    phiK [L, N, R], V [N, dv], phiQ [L, M, R]. Returns (O [M, dv], mass [L, R], content [L, R, dv]).
    """
    phiK, V, phiQ = _f64(phiK), _f64(V), _f64(phiQ)
    L, N, R = phiK.shape
    M = phiQ.shape[1]
    dv = V.shape[1]
    O = np.empty((M, dv))
    mass = np.empty((L, R))
    content = np.empty((L, R, dv))
    _check(lib().race_oracle_readout_given_phi(N, M, dv, L, R, _ptr(phiK), _ptr(V), _ptr(phiQ),
                                               int(causal), _ptr(O), _ptr(mass), _ptr(content)),
           "readout_given_phi")
    return O, mass, content


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.size


def forward(Q, K, V, W, beta, causal, normalize=True, rows=None, want_sketch=False, nthreads=0):
    """O for Q, K, V [B, H, N, d] (float64/float32/bf16-bits). rows: sorted token rows to output.
    W: [L, P, d] shared, or [H, L, P, d] per head.  beta = inf: hard hashing."""
    Q, e = _tokens(Q)
    K, e2 = _tokens(K)
    V, e3 = _tokens(V)
    assert e == e2 == e3 and Q.shape == K.shape == V.shape
    B, H, N, d = Q.shape
    W, ph, L, P = _hash(W, H)
    r, nr = _rows(rows)
    nout = nr if r is not None else N
    O = np.empty((B, H, nout, d))
    sk = np.empty((B, H, L << P, d + 1)) if (want_sketch and not causal) else None
    _check(lib().race_oracle_forward(B, H, N, d, e, _ptr(Q), _ptr(K), _ptr(V), _ptr(W), ph, L, P,
                                     float(beta), int(causal), int(normalize), _ptr(r), nr,
                                     _ptr(O), _ptr(sk), int(nthreads)), "forward")
    return (O, sk) if want_sketch else O


def backward(Q, K, V, dO, W, beta, causal, normalize=True, rows=None, nthreads=0, want_dbeta=False,
             want_dW=False):
    """(dQ, dK, dV) for the output O and its cotangent dO; rows as in `forward`.  With
    want_dbeta also d(loss)/d(beta) per (b, h) [B, H], and with want_dW d(loss)/d(W) per (b, h)
    [B, H, L, P, d], both summed over every token and appended in that order.  W and beta as in
    `forward` (a hard hash passes no gradient to Q, K, beta or W)."""
    Q, e = _tokens(Q)
    K, _ = _tokens(K)
    V, _ = _tokens(V)
    dO, e4 = _tokens(dO)
    assert e == e4
    B, H, N, d = Q.shape
    W, ph, L, P = _hash(W, H)
    r, nr = _rows(rows)
    nout = nr if r is not None else N
    dQ = np.empty((B, H, nout, d))
    dK = np.empty((B, H, nout, d))
    dV = np.empty((B, H, nout, d))
    db = np.zeros((B, H)) if want_dbeta else None
    dW = np.zeros((B, H, L, P, d)) if want_dW else None
    _check(lib().race_oracle_backward(B, H, N, d, e, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(W),
                                      ph, L, P, float(beta), int(causal), int(normalize), _ptr(r), nr,
                                      _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(db), _ptr(dW), int(nthreads)),
           "backward")
    return (dQ, dK, dV) + ((db,) if want_dbeta else ()) + ((dW,) if want_dW else ())


def decode_step(q, k, v, W, beta, state, normalize=True):
    """One causal decode step per (b, h): state [B, H, L*R, d+1] float64 (updated in place) gains
    key k / value v, then query q reads it.  q, k, v: [B, H, d].  Returns o [B, H, d]."""
    q, e = _tokens(q)
    k, e2 = _tokens(k)
    v, e3 = _tokens(v)
    assert e == e2 == e3 and q.shape == k.shape == v.shape and q.ndim == 3
    B, H, d = q.shape
    W, ph, L, P = _hash(W, H)
    assert state.dtype == np.float64 and state.flags.c_contiguous and state.shape == (B, H, L << P, d + 1)
    o = np.empty((B, H, d))
    _check(lib().race_oracle_decode_step(B, H, d, e, _ptr(q), _ptr(k), _ptr(v), _ptr(W), ph, L, P, float(beta),
                                         int(normalize), _ptr(state), _ptr(o)), "decode_step")
    return o


def angular_forward(Q, K, V, gamma, causal, rows=None, nthreads=0):
    """Angular attention O_i = sum_j S_ij V_j / sum_j S_ij with S_ij = (1 - theta_ij / pi)^gamma
    (j <= i when causal), O(N^2): the kernel a gamma-bit hard hash collides with."""
    Q, e = _tokens(Q)
    K, e2 = _tokens(K)
    V, e3 = _tokens(V)
    assert e == e2 == e3 and Q.shape == K.shape == V.shape
    B, H, N, d = Q.shape
    r, nr = _rows(rows)
    O = np.empty((B, H, nr if r is not None else N, d))
    _check(lib().race_oracle_angular_forward(B, H, N, d, e, _ptr(Q), _ptr(K), _ptr(V), float(gamma),
                                             int(causal), _ptr(r), nr, _ptr(O), int(nthreads)),
           "angular_forward")
    return O

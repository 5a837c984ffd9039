"""Named workloads and seeded synthetic inputs.

Holds no arithmetic of the method: only shapes and random draws, shared by the tests, the
benchmark and the smoke check.  The shapes are those of the pages' operator timings (one
attention layer, batch 1, 4 heads, d = 128, up to 12M tokens) plus smaller parity cases.

Draw recipe (one torch.Generator on the target device, seeded once, draws in this order):
  1. W  ~ N(0, 1), float32 [L, P, d]
  2. Q, K: i.i.d. N(0, 1); or, when `clusters` > 0, for each (b, h) in order: centroids
     C ~ N(0, 1) [clusters, d], then Q rows = C[idx_q] + 0.3 N(0, 1) and K rows = C[idx_k] +
     0.3 N(0, 1) with idx_q, idx_k uniform over the centroids (drawn: idx_q, noise_q, idx_k,
     noise_k).  Q and K share the centroids of their (b, h).
  3. V  ~ N(0, 1);  4. dO ~ N(0, 1).
Large tensors are drawn one (b, h) slice at a time in float32 and rounded to the workload dtype
(round to nearest even), so peak memory stays one float32 slice above the result.
"""
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    P: int
    L: int
    beta: float
    causal: bool
    dtype: str          # "f32" or "bf16"
    clusters: int = 0   # 0: i.i.d. Q and K; > 0: clustered Q and K (see module docstring)

    @property
    def R(self):
        return 1 << self.P

    @property
    def LR(self):
        return self.L << self.P

    @property
    def tokens(self):
        return self.B * self.N

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2

    def scaled(self, **kw):
        return replace(self, **kw)

    def describe(self):
        kind = "causal" if self.causal else "non-causal"
        qk = ("clustered Q/K (%d centroids + 0.3 noise)" % self.clusters) if self.clusters else "iid N(0,1)"
        return ("%s RACE fwd+bwd, %s, B%d H%d N%d d%d (P,L)=(%d,%d) R=%d beta=%g, %s"
                % (kind, self.dtype, self.B, self.H, self.N, self.d, self.P, self.L, self.R, self.beta, qk))


CONFIGS = {
    # tiny float32 parity case (brute force and finite differences are feasible)
    "c1_f32_tiny": Workload("c1_f32_tiny", 1, 1, 256, 64, 2, 2, 10.0, False, "f32"),
    # bf16 non-causal, clustered Q/K
    "c2_bf16_65k": Workload("c2_bf16_65k", 1, 4, 65536, 64, 3, 3, 10.0, False, "bf16", 16),
    # bf16 causal, the shape of a 1024-token language-model layer
    "c3_bf16_causal_lm": Workload("c3_bf16_causal_lm", 8, 12, 1024, 64, 4, 4, 10.0, True, "bf16"),
    # bf16 non-causal, L*R = 256 (dense contraction regime)
    "c4_bf16_1m_lr256": Workload("c4_bf16_1m_lr256", 1, 4, 1048576, 128, 6, 4, 10.0, False, "bf16", 64),
    # bf16 causal 12M-token stress test: one layer, batch 1, 4 heads, d = 128
    "c5_bf16_causal_12m": Workload("c5_bf16_causal_12m", 1, 4, 12000000, 128, 3, 3, 10.0, True, "bf16"),
}


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _token_tensor(w, gen, device):
    out = torch.empty((w.B, w.H, w.N, w.d), dtype=w.torch_dtype, device=device)
    for b in range(w.B):
        for h in range(w.H):
            out[b, h].copy_(_normal((w.N, w.d), gen, device))
    return out


def _clustered_pair(w, gen, device):
    Q = torch.empty((w.B, w.H, w.N, w.d), dtype=w.torch_dtype, device=device)
    K = torch.empty_like(Q)
    for b in range(w.B):
        for h in range(w.H):
            C = _normal((w.clusters, w.d), gen, device)
            iq = torch.randint(0, w.clusters, (w.N,), generator=gen, device=device)
            Q[b, h].copy_(C[iq] + 0.3 * _normal((w.N, w.d), gen, device))
            ik = torch.randint(0, w.clusters, (w.N,), generator=gen, device=device)
            K[b, h].copy_(C[ik] + 0.3 * _normal((w.N, w.d), gen, device))
    return Q, K


def make_inputs(w, seed=0, device="cpu", need_grad_inputs=True):
    """Seeded {W, Q, K, V, dO} for workload w on `device` (see the module docstring)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    W = _normal((w.L, w.P, w.d), gen, device).contiguous()
    if w.clusters:
        Q, K = _clustered_pair(w, gen, device)
    else:
        Q = _token_tensor(w, gen, device)
        K = _token_tensor(w, gen, device)
    V = _token_tensor(w, gen, device)
    out = {"W": W, "Q": Q, "K": K, "V": V}
    if need_grad_inputs:
        out["dO"] = _token_tensor(w, gen, device)
    return out


def as_oracle_array(t):
    """Exact host copy of a token tensor for the float64 oracle (bf16 as its raw bit pattern)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()

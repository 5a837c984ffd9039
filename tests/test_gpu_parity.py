"""GPU parity: the library (called through its C ABI) against the float64 oracle on the same
seeded inputs.  Small shapes span several token tiles and a ragged tail; the named workloads
run at full size (sampled rows where the oracle would take too long)."""
import math

import numpy as np
import pytest
import torch

import linear_lsh_sketch_gb300 as race
from linear_lsh_sketch_gb300.workloads import CONFIGS, Workload, make_inputs
import oracle
from linear_lsh_sketch_gb300.workloads import as_oracle_array
from parity import TOL, assert_close, gpu_run, inputs_on_gpu, oracle_run

pytestmark = pytest.mark.gpu


def W_(name, B, H, N, d, P, L, causal, dtype, beta=10.0, clusters=0):
    return Workload(name, B, H, N, d, P, L, beta, causal, dtype, clusters)


SMALL = [
    W_("ragged", 1, 2, 100, 64, 2, 2, False, "f32"),
    W_("ragged_c", 1, 2, 100, 64, 2, 2, True, "f32"),
    W_("d128", 1, 1, 77, 128, 3, 3, False, "f32"),
    W_("d128_c", 1, 1, 77, 128, 3, 3, True, "f32"),
    W_("lr256", 1, 1, 70, 32, 6, 4, False, "f32"),
    W_("lr64_c", 2, 1, 130, 64, 4, 4, True, "f32"),
    W_("p1_l16", 1, 2, 45, 16, 1, 16, True, "f32"),
    W_("p8", 1, 1, 50, 8, 8, 1, False, "f32"),
    W_("bf_ragged", 1, 2, 1000, 64, 3, 3, False, "bf16"),
    W_("bf_ragged_c", 1, 2, 1000, 64, 3, 3, True, "bf16"),
    W_("bf_d128_c", 1, 2, 555, 128, 3, 3, True, "bf16"),
    W_("bf_lr256", 1, 2, 300, 128, 6, 4, False, "bf16", clusters=8),
    W_("bf_lr64_c", 2, 3, 257, 64, 4, 4, True, "bf16"),
    # causal bf16 with L R = 48 at d = 128: forward on tcgen05, backward on the CUDA-core kernels
    # (the tcgen05 backward's TMEM holds L R > 32 only at d = 64)
    W_("bf_d128_lr48_c", 1, 2, 300, 128, 4, 3, True, "bf16"),
    # L R = 64 at d = 64 with P = 6, 5, 3, 2 (run-time L) on the tcgen05 backward
    W_("bf_p6_l1_c", 1, 2, 333, 64, 6, 1, True, "bf16"),
    W_("bf_p5_l2_c", 1, 1, 300, 64, 5, 2, True, "bf16"),
    W_("bf_p3_l8_c", 1, 1, 260, 64, 3, 8, True, "bf16"),
    W_("bf_p2_l12_c", 1, 1, 200, 64, 2, 12, True, "bf16"),
    # shapes of the tcgen05 paths: bucket counts 2 .. 64, tables 1 .. 16, ragged tails, d 64 / 128
    W_("bf_p1_l16_c", 1, 2, 700, 64, 1, 16, True, "bf16"),
    W_("bf_p5_l1_c", 1, 1, 333, 128, 5, 1, True, "bf16"),
    W_("bf_p4_l2_c", 2, 1, 400, 128, 4, 2, True, "bf16"),
    W_("bf_p2_l3_c", 1, 2, 260, 64, 2, 3, True, "bf16"),
    W_("bf_p2_l5_c", 1, 1, 129, 128, 2, 5, True, "bf16"),
    W_("bf_p1_l16", 1, 2, 700, 64, 1, 16, False, "bf16"),
    W_("bf_p5_l5", 1, 1, 515, 64, 5, 5, False, "bf16"),
    W_("bf_p6_l2", 1, 2, 390, 128, 6, 2, False, "bf16", clusters=4),
    W_("bf_p3_l10", 1, 1, 260, 128, 3, 10, False, "bf16"),
    W_("beta0", 1, 1, 64, 32, 2, 2, False, "f32", beta=0.0),
    # near the hard-hash limit while every bucket probability stays a normal float32
    W_("beta_sharp", 1, 1, 64, 32, 2, 2, True, "f32", beta=12.0),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_shapes(w):
    inp = inputs_on_gpu(w, seed=1)
    assert_close(w, gpu_run(w, inp), oracle_run(w, inp), w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token(causal, dtype):
    """N = 1: the token attends only to itself, so O = V and dV = dO exactly; O does not depend
    on Q or K, whose exact gradient is zero (a pure rounding residue here, only checked finite)."""
    w = W_("one_token", 2, 1, 1, 64, 3, 2, causal, dtype)
    inp = inputs_on_gpu(w, seed=1)
    O, dQ, dK, dV = gpu_run(w, inp)
    V = inp["V"].double().cpu().numpy()
    dO = inp["dO"].double().cpu().numpy()
    tol = 1e-6 if dtype == "f32" else 1e-2
    np.testing.assert_allclose(O, V, rtol=tol, atol=tol)
    np.testing.assert_allclose(dV, dO, rtol=tol, atol=tol)
    assert np.all(np.isfinite(dQ)) and np.all(np.isfinite(dK))


def test_c1_full():
    w = CONFIGS["c1_f32_tiny"]
    inp = inputs_on_gpu(w, seed=0)
    assert_close(w, gpu_run(w, inp), oracle_run(w, inp), w.name)


@pytest.mark.parametrize("name", ["c2_bf16_65k", "c3_bf16_causal_lm"])
def test_config_full(name):
    w = CONFIGS[name]
    inp = make_inputs(w, seed=0, device="cuda")
    assert_close(w, gpu_run(w, inp), oracle_run(w, inp), w.name)


def test_zero_rows_and_state_reuse():
    """A zero Q/K row has uniform buckets (and zero gradient); bwd with the saved sketch equals
    bwd that recomputes it, bit for bit."""
    w = W_("zero_rows", 1, 2, 96, 64, 3, 2, True, "f32")
    inp = inputs_on_gpu(w, seed=2)
    inp["Q"][0, 0, 5] = 0
    inp["K"][0, 1, 40] = 0
    a = gpu_run(w, inp, with_state=True)
    b = gpu_run(w, inp, with_state=False)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert np.all(a[1][0, 0, 5] == 0) and np.all(a[2][0, 1, 40] == 0)
    assert_close(w, a, oracle_run(w, inp), w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic(causal):
    w = W_("det", 1, 4, 3000, 64, 3, 3, causal, "bf16")
    inp = inputs_on_gpu(w, seed=3)
    a = gpu_run(w, inp)
    b = gpu_run(w, inp)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_outputs_16_byte_aligned(causal):
    """Outputs that are 16- but not 32-byte aligned (the ABI's minimum) take the narrow store path;
    the values equal those written to aligned outputs bit for bit."""
    w = W_("align", 1, 2, 700, 128, 3, 3, causal, "bf16")
    inp = inputs_on_gpu(w, seed=8)
    args = (inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal)
    n = inp["Q"].numel()

    def shifted():
        buf = torch.empty(n + 64, dtype=inp["Q"].dtype, device="cuda")
        t = buf[8:8 + n].view(inp["Q"].shape)
        assert t.data_ptr() % 32 == 16
        return t

    O = race.race_attn_fwd(*args)
    ref = (O,) + race.race_attn_bwd(*args, inp["dO"], O=O)
    O2 = race.race_attn_fwd(*args, O=shifted())
    got = (O2,) + race.race_attn_bwd(*args, inp["dO"], O=O2, dQ=shifted(), dK=shifted(), dV=shifted())
    torch.cuda.synchronize()
    for x, y in zip(ref, got):
        assert torch.equal(x, y)


def test_beta_zero_mean():
    """beta = 0: uniform buckets, O = mean of V (causal: prefix mean)."""
    for causal in (False, True):
        w = W_("b0", 1, 1, 200, 32, 2, 2, causal, "f32", beta=0.0)
        inp = inputs_on_gpu(w, seed=4)
        O = race.race_attn_fwd(inp["Q"], inp["K"], inp["V"], inp["W"], 0.0, 2, 2, causal).double().cpu()
        V = inp["V"].double().cpu()[0, 0]
        ref = V.cumsum(0) / torch.arange(1, 201, dtype=torch.float64)[:, None] if causal else V.mean(0).expand(200, 32)
        assert (O[0, 0] - ref).abs().max() < 1e-5


@pytest.mark.parametrize("w", [
    W_("sk_bf_d64", 1, 2, 1000, 64, 3, 3, False, "bf16"),
    W_("sk_bf_d128_lr256", 1, 2, 700, 128, 6, 4, False, "bf16", clusters=8),
    W_("sk_bf_p2_l5", 2, 1, 333, 128, 2, 5, False, "bf16"),
    W_("sk_bf_p5_l5", 1, 1, 515, 64, 5, 5, False, "bf16"),
], ids=lambda w: w.name)
def test_noncausal_sketch_state(w):
    """The saved non-causal sketch [A | B] = Phi_K^T [V | 1] (sketch rows L * R, d + 1 columns)
    against the oracle's, normwise: relative L2 error over each (b, h) sketch."""
    inp = inputs_on_gpu(w, seed=6)
    shape = race.make_shape(w.B, w.H, w.N, w.d, w.torch_dtype)
    state = torch.empty(race.race_attn_state_bytes(shape, w.L, w.P, w.causal), dtype=torch.uint8, device="cuda")
    race.race_attn_fwd(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal, state=state)
    torch.cuda.synchronize()
    got = state.view(torch.float32).double().cpu().numpy().reshape(w.B, w.H, w.LR, w.d + 1)
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V")}
    _, ref = oracle.forward(a["Q"], a["K"], a["V"], inp["W"].double().cpu().numpy(), w.beta, False,
                            want_sketch=True)
    for b in range(w.B):
        for h in range(w.H):
            e = np.linalg.norm(got[b, h] - ref[b, h]) / np.linalg.norm(ref[b, h])
            assert e <= 1e-2, "%s sketch (%d, %d) error %.3e" % (w.name, b, h, e)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_match_oracle(dtype):
    """Causal decode, one token per call from an empty prefix (the recurrence of Algorithm 2,
    "Causality is a prefix update of the same statistics"), against the oracle's decode step on
    the same inputs: every step's output and the final sketch."""
    w = W_("decode", 2, 3, 40, 64, 3, 2, True, dtype)
    inp = inputs_on_gpu(w, seed=11)
    Q, K, V, W = inp["Q"], inp["K"], inp["V"], inp["W"]
    B, H, N, d = Q.shape
    LR = w.L << w.P
    state = torch.zeros((B, H, LR, d + 1), dtype=torch.float32, device="cuda")
    ref_state = np.zeros((B, H, LR, d + 1))
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V")}
    Wd = W.double().cpu().numpy()
    tol = 2e-5 if dtype == "f32" else 1e-2
    for t in range(N):
        tok = [x[:, :, t:t + 1].contiguous() for x in (Q, K, V)]
        o = race.race_attn_decode(*tok, W, w.beta, w.L, w.P, state)
        ref = oracle.decode_step(a["Q"][:, :, t], a["K"][:, :, t], a["V"][:, :, t], Wd, w.beta, ref_state)
        got = o[:, :, 0].double().cpu().numpy()
        assert np.abs(got - ref).max() <= tol * np.abs(ref).max(), t
    got_state = state.double().cpu().numpy()
    assert np.abs(got_state - ref_state).max() <= 1e-5 * np.abs(ref_state).max()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_after_prefill(dtype):
    """The state race_attn_fwd (causal = 0) leaves for a prompt is the prompt's sketch; decoding
    on from it gives the causal forward of prompt + continuation (oracle rows)."""
    w = W_("prefill", 1, 2, 60, 64, 3, 3, True, dtype)
    inp = inputs_on_gpu(w, seed=12)
    Q, K, V, W = inp["Q"], inp["K"], inp["V"], inp["W"]
    B, H, N, d = Q.shape
    N0, LR = 45, w.L << w.P
    pre = [x[:, :, :N0].contiguous() for x in (Q, K, V)]
    shape = race.make_shape(B, H, N0, d, w.torch_dtype)
    raw = torch.empty(race.race_attn_state_bytes(shape, w.L, w.P, False), dtype=torch.uint8, device="cuda")
    race.race_attn_fwd(*pre, W, w.beta, w.L, w.P, False, state=raw)
    state = raw.view(torch.float32).view(B, H, LR, d + 1)
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V")}
    ref = oracle.forward(a["Q"], a["K"], a["V"], W.double().cpu().numpy(), w.beta, True)
    tol = 1e-5 if dtype == "f32" else 2e-2
    for t in range(N0, N):
        tok = [x[:, :, t:t + 1].contiguous() for x in (Q, K, V)]
        o = race.race_attn_decode(*tok, W, w.beta, w.L, w.P, state)[:, :, 0].double().cpu().numpy()
        assert np.abs(o - ref[:, :, t]).max() <= tol * np.abs(ref[:, :, t]).max(), t


def _sampled_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=n, replace=False).tolist())
    rows.update([0, 1, N // 2, N - 2, N - 1])
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("w", [
    # one (b, h) split into 304 segments of 3 token tiles each, the last one ragged
    W_("mc_bf_d128_c", 1, 1, 3 * 304 * 128 - 51, 128, 3, 3, True, "bf16"),
    W_("mc_bf_d64_c", 1, 2, 3 * 152 * 128 + 300, 64, 2, 5, True, "bf16"),
    W_("mc_bf_d128_p5_c", 2, 1, 4 * 152 * 128 + 1, 128, 5, 1, True, "bf16"),
    W_("mc_bf_d128", 1, 1, 6 * 304 * 128 - 51, 128, 3, 3, False, "bf16"),
], ids=lambda w: w.name)
def test_multichunk_segments(w):
    """Several token tiles per segment: every barrier phase of the per-chunk pipelines turns over
    more than once (small shapes give each segment a single tile)."""
    inp = inputs_on_gpu(w, seed=9)
    rows = _sampled_rows(w.N, 64, 9)
    assert_close(w, gpu_run(w, inp, rows=rows), oracle_run(w, inp, rows=rows), w.name)


class _HeadErrors:
    """Accumulates, per (b, h), the parity measures over the rows compared so far: the normwise
    max error of O (max |O - O_ref| / max |O_ref|) and the relative L2 error of each gradient."""

    def __init__(self):
        self.o_diff = self.o_ref = 0.0
        self.sq = {g: [0.0, 0.0] for g in ("dQ", "dK", "dV")}
        self.rows = 0

    def add_O(self, got, ref):
        assert np.all(np.isfinite(got))
        self.o_diff = max(self.o_diff, float(np.abs(got - ref).max()))
        self.o_ref = max(self.o_ref, float(np.abs(ref).max()))
        self.rows += got.shape[0]

    def add_grad(self, name, got, ref):
        assert np.all(np.isfinite(got))
        self.sq[name][0] += float(((got - ref) ** 2).sum())
        self.sq[name][1] += float((ref ** 2).sum())

    def check(self, w, label):
        to, tg = TOL[w.dtype]
        eo = self.o_diff / self.o_ref
        assert eo <= to, "%s: O error %.3e > %.1e" % (label, eo, to)
        eg = {}
        for g, (num, den) in self.sq.items():
            eg[g] = math.sqrt(num / den)
            assert eg[g] <= tg, "%s: %s error %.3e > %.1e" % (label, g, eg[g], tg)
        return eo, eg


def _full_size_check(w, rows_of_chunk, nchunks):
    """The workload at full size on the GPU (one forward and one backward, the launch
    configuration the benchmark times), then every (b, h) through the float64 oracle on the rows
    `rows_of_chunk(k)` for k < nchunks, one host thread per (b, h, chunk) (the oracle releases
    the interpreter lock).  Each (b, h) must meet the tolerances on its own."""
    import concurrent.futures
    import os

    inp = make_inputs(w, seed=0, device="cuda")
    got = gpu_run(w, inp, keep_on_device=True)
    W = inp["W"].double().cpu().numpy()
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    host = {}
    for b, h in heads:  # one (b, h) slice of each input at a time on the host
        host[(b, h)] = {k: as_oracle_array(inp[k][b:b + 1, h:h + 1]) for k in ("Q", "K", "V", "dO")}
    del inp
    err = {bh: _HeadErrors() for bh in heads}

    def task(bh, k):
        rows = rows_of_chunk(k)
        a = host[bh]
        O = oracle.forward(a["Q"], a["K"], a["V"], W, w.beta, w.causal, rows=rows, nthreads=1)[0, 0]
        g = oracle.backward(a["Q"], a["K"], a["V"], a["dO"], W, w.beta, w.causal, rows=rows, nthreads=1)
        return bh, rows, O, [x[0, 0] for x in g]

    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        futs = [ex.submit(task, bh, k) for bh in heads for k in range(nchunks)]
        for f in concurrent.futures.as_completed(futs):
            (b, h), rows, O, grads = f.result()
            idx = torch.as_tensor(rows, device="cuda")
            e = err[(b, h)]
            e.add_O(got[0][b, h, idx].double().cpu().numpy(), O)
            for name, t, r in zip(("dQ", "dK", "dV"), got[1:], grads):
                e.add_grad(name, t[b, h, idx].double().cpu().numpy(), r)
    return err


@pytest.mark.slow
def test_c4_full_size_every_head_every_row():
    """The 1M-token L R = 256 non-causal workload at full size: all 4 heads, every row of O, dQ,
    dK and dV against the float64 oracle (the read-out rows split over host threads; each call
    rebuilds the head's sketch in the same key order)."""
    w = CONFIGS["c4_bf16_1m_lr256"]
    nchunks = 4
    bounds = np.linspace(0, w.N, nchunks + 1).astype(np.int64)
    err = _full_size_check(w, lambda k: np.arange(bounds[k], bounds[k + 1], dtype=np.int64), nchunks)
    for (b, h), e in err.items():
        assert e.rows == w.N
        e.check(w, "%s head (b=%d, h=%d), all %d rows" % (w.name, b, h, w.N))


@pytest.mark.slow
def test_c5_full_size_every_head():
    """The 12M-token causal workload at full size: all 4 heads, on every row of the first and last
    2^20 tokens and a seeded 1 % sample of the rows between, against the float64 oracle's literal
    token recurrence.  Heads 2 and 3 start at element offsets 3.07e9 and 4.61e9, past 2^31 and
    2^32, so 64-bit addressing is covered."""
    w = CONFIGS["c5_bf16_causal_12m"]
    edge = 1 << 20
    rng = np.random.default_rng(2024)
    middle = np.sort(rng.choice(np.arange(edge, w.N - edge), size=(w.N - 2 * edge) // 100, replace=False))
    rows = np.concatenate([np.arange(edge), middle, np.arange(w.N - edge, w.N)]).astype(np.int64)
    err = _full_size_check(w, lambda k: rows, 1)
    for (b, h), e in err.items():
        off = ((b * w.H + h) * w.N + int(rows[-1])) * w.d
        assert e.rows == rows.size
        e.check(w, "%s head (b=%d, h=%d): rows 0..%d, %d sampled, %d..%d (last element offset %d)"
                % (w.name, b, h, edge - 1, middle.size, w.N - edge, w.N - 1, off))


# d(loss)/d(beta): one workload per backward kernel family (CUDA-core non-causal / causal,
# tcgen05 non-causal / causal, the tcgen05 causal backward at L R = 64), ragged tails and several
# segments.
DBETA = [
    W_("db_f32", 1, 2, 100, 64, 2, 2, False, "f32"),
    W_("db_f32_c", 1, 2, 100, 64, 2, 2, True, "f32"),
    W_("db_bf_nc", 1, 2, 1000, 64, 3, 3, False, "bf16"),
    W_("db_bf_lr256", 1, 2, 300, 128, 6, 4, False, "bf16", clusters=8),
    W_("db_bf_c5", 1, 2, 5555, 128, 3, 3, True, "bf16"),
    W_("db_bf_c5_p2", 2, 1, 700, 64, 2, 3, True, "bf16"),
    W_("db_bf_lr64_c", 2, 3, 257, 64, 4, 4, True, "bf16"),
]


@pytest.mark.parametrize("w", DBETA, ids=lambda w: w.name)
def test_dbeta_matches_oracle(w):
    """d(sum O * dO)/d(beta) per (b, h) against the oracle (whose value is pinned to finite
    differences of the brute force).  Tolerance relative to the largest |value|: 1e-4 for float32
    tensors, 5e-2 for bfloat16 (the gradient tolerance).  Asking for it leaves dQ, dK, dV bit for
    bit unchanged, and a second call gives the same bits."""
    inp = inputs_on_gpu(w, seed=4)
    args = (inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal, inp["dO"])
    plain = race.race_attn_bwd(*args)
    with_db = race.race_attn_bwd(*args, want_dbeta=True)
    again = race.race_attn_bwd(*args, want_dbeta=True)
    torch.cuda.synchronize()
    for x, y in zip(plain, with_db[:3]):
        assert torch.equal(x, y)
    assert torch.equal(with_db[3], again[3])
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V", "dO")}
    W = inp["W"].double().cpu().numpy()
    *_, ref = oracle.backward(a["Q"], a["K"], a["V"], a["dO"], W, w.beta, w.causal, want_dbeta=True)
    got = with_db[3].double().cpu().numpy()
    assert np.all(np.isfinite(got))
    tol = 1e-4 if w.dtype == "f32" else 5e-2
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err <= tol, "%s dbeta error %.3e > %.1e (got %s, oracle %s)" % (w.name, err, tol, got, ref)


DW = [
    (W_("dw_f32", 1, 2, 100, 64, 2, 2, False, "f32"), False),
    (W_("dw_f32_c", 1, 2, 100, 64, 2, 2, True, "f32"), False),
    (W_("dw_f32_ph_c", 2, 3, 70, 32, 3, 2, True, "f32"), True),
    (W_("dw_bf_nc", 1, 2, 1000, 64, 3, 3, False, "bf16"), False),
    (W_("dw_bf_lr256", 1, 2, 300, 128, 6, 4, False, "bf16", clusters=8), False),
    (W_("dw_bf_c5", 1, 2, 5555, 128, 3, 3, True, "bf16"), False),
    (W_("dw_bf_c5_ph", 2, 3, 700, 128, 3, 3, True, "bf16"), True),
    (W_("dw_bf_lr64_c", 2, 3, 257, 64, 4, 4, True, "bf16"), False),
]


@pytest.mark.parametrize("w,per_head", DW, ids=lambda x: x.name if hasattr(x, "name") else ("ph" if x else "shared"))
def test_dW_matches_oracle(w, per_head):
    """d(sum O * dO)/d(W) per (b, h), [B, H, L, P, d], against the oracle's (pinned to finite
    differences of the brute force).  Tolerance on the relative L2 error of the whole tensor: 1e-4
    for float32 tensors, 5e-2 for bfloat16 (the gradient tolerance).  Asking for it leaves dQ,
    dK, dV and d(loss)/d(beta) bit for bit unchanged, and a second call gives the same bits."""
    inp = inputs_on_gpu(w, seed=5)
    if per_head:
        inp["W"] = _per_head_w(w, 62)
    args = (inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal, inp["dO"])
    plain = race.race_attn_bwd(*args, want_dbeta=True)
    with_dw = race.race_attn_bwd(*args, want_dbeta=True, want_dW=True)
    again = race.race_attn_bwd(*args, want_dW=True)
    torch.cuda.synchronize()
    for x, y in zip(plain, with_dw[:4]):
        assert torch.equal(x, y)
    assert torch.equal(with_dw[4], again[3])
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V", "dO")}
    W = inp["W"].double().cpu().numpy()
    *_, ref = oracle.backward(a["Q"], a["K"], a["V"], a["dO"], W, w.beta, w.causal, want_dW=True)
    got = with_dw[4].double().cpu().numpy()
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    tol = 1e-4 if w.dtype == "f32" else 5e-2
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= tol, "%s dW error %.3e > %.1e" % (w.name, err, tol)


# One set of hyperplanes per head (W [H, L, P, d]); B = 2 so that reading W by (b, h) instead of
# by h would fail.  One workload per kernel family.
PER_HEAD = [
    W_("ph_f32", 2, 3, 100, 64, 2, 2, False, "f32"),
    W_("ph_f32_c", 2, 3, 100, 64, 2, 2, True, "f32"),
    W_("ph_bf_nc", 2, 3, 700, 64, 3, 3, False, "bf16"),
    W_("ph_bf_lr256", 2, 2, 300, 128, 6, 4, False, "bf16", clusters=8),
    W_("ph_bf_c5", 2, 3, 700, 128, 3, 3, True, "bf16"),
    W_("ph_bf_lr64_c", 2, 3, 257, 64, 4, 4, True, "bf16"),
]


def _per_head_w(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((w.H, w.L, w.P, w.d), generator=g, dtype=torch.float32).cuda()


@pytest.mark.parametrize("w", PER_HEAD, ids=lambda w: w.name)
def test_per_head_w(w):
    """Head h hashes with W[h]: forward and backward against the oracle's per-head layout, and
    a per-head W whose heads are all equal gives the shared-W results bit for bit."""
    inp = inputs_on_gpu(w, seed=6)
    inp["W"] = _per_head_w(w, 60)
    assert_close(w, gpu_run(w, inp), oracle_run(w, inp), w.name)
    shared = dict(inp, W=inp["W"][1].contiguous())
    same = dict(inp, W=inp["W"][1].expand(w.H, -1, -1, -1).contiguous())
    for x, y in zip(gpu_run(w, shared), gpu_run(w, same)):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_per_head_w(dtype):
    """Decode steps with one hyperplane set per head against the oracle's decode step."""
    w = W_("decode_ph", 2, 3, 20, 64, 3, 2, True, dtype)
    inp = inputs_on_gpu(w, seed=13)
    Q, K, V = inp["Q"], inp["K"], inp["V"]
    W = _per_head_w(w, 61)
    B, H, N, d = Q.shape
    state = torch.zeros((B, H, w.L << w.P, d + 1), dtype=torch.float32, device="cuda")
    ref_state = np.zeros((B, H, w.L << w.P, d + 1))
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V")}
    Wd = W.double().cpu().numpy()
    tol = 2e-5 if dtype == "f32" else 1e-2
    for t in range(N):
        tok = [x[:, :, t:t + 1].contiguous() for x in (Q, K, V)]
        o = race.race_attn_decode(*tok, W, w.beta, w.L, w.P, state)
        ref = oracle.decode_step(a["Q"][:, :, t], a["K"][:, :, t], a["V"][:, :, t], Wd, w.beta, ref_state)
        assert np.abs(o[:, :, 0].double().cpu().numpy() - ref).max() <= tol * np.abs(ref).max(), t


# Hard hashing (beta = +inf).  Every Q and K row keeps each projection |w . xhat| >= 1e-3 away
# from 0 (rows are redrawn until it does), so that the float32 projections on the GPU and the
# float64 ones of the oracle give the same signs; each key is its query plus a little noise, so
# that every query meets at least its own key in some table (no 0/0 rows).
HARD = [
    W_("hard_f32", 2, 2, 100, 64, 2, 3, False, "f32", beta=math.inf),
    W_("hard_f32_c", 2, 2, 100, 64, 2, 3, True, "f32", beta=math.inf),
    W_("hard_bf_nc", 1, 2, 700, 64, 3, 3, False, "bf16", beta=math.inf),
    W_("hard_bf_c5", 1, 2, 700, 128, 3, 3, True, "bf16", beta=math.inf),
    W_("hard_bf_lr64_c", 1, 2, 257, 64, 4, 4, True, "bf16", beta=math.inf),
]


def _hard_inputs(w, seed):
    inp = make_inputs(w, seed=seed, device="cpu")
    g = torch.Generator().manual_seed(seed + 1000)
    Wd = inp["W"].double()
    Q = inp["Q"].float()

    def margins(X):  # smallest |w . xhat| per row, on the values as rounded to the tensors' dtype
        Xr = X.to(w.torch_dtype).double()
        Xh = Xr / Xr.norm(dim=-1, keepdim=True)
        return torch.einsum("lpd,bhnd->bhnlp", Wd, Xh).abs().flatten(3).min(dim=3).values

    def own_key_missed(Q, K):  # q_i and k_i share no corner in any table
        sq = torch.einsum("lpd,bhnd->bhnlp", Wd, Q.to(w.torch_dtype).double()) > 0
        sk = torch.einsum("lpd,bhnd->bhnlp", Wd, K.to(w.torch_dtype).double()) > 0
        return ~(sq == sk).all(dim=4).any(dim=3)

    K = Q + 0.05 * torch.randn(Q.shape, generator=g)
    for _ in range(100):
        bad = (margins(Q) < 1e-3) | (margins(K) < 1e-3) | own_key_missed(Q, K)
        if not bad.any():
            break
        n = int(bad.sum())
        Q[bad] = torch.randn((n, w.d), generator=g)
        K[bad] = Q[bad] + 0.05 * torch.randn((n, w.d), generator=g)
    assert not bad.any()
    inp["Q"], inp["K"] = Q.to(w.torch_dtype), K.to(w.torch_dtype)
    return {k: v.cuda() for k, v in inp.items()}


@pytest.mark.parametrize("w", HARD, ids=lambda w: w.name)
def test_hard_hash(w):
    """beta = +inf: O and dV against the oracle's hard hash (sign bits); dQ, dK, d(loss)/d(beta)
    and d(loss)/d(W) exactly zero."""
    inp = _hard_inputs(w, seed=7)
    args = (inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal)
    O = race.race_attn_fwd(*args)
    dQ, dK, dV, db, dW = race.race_attn_bwd(*args, inp["dO"], O=O, want_dbeta=True, want_dW=True)
    torch.cuda.synchronize()
    assert torch.all(dQ == 0) and torch.all(dK == 0) and torch.all(db == 0) and torch.all(dW == 0)
    got = (O.double().cpu().numpy(), dQ.double().cpu().numpy(), dK.double().cpu().numpy(),
           dV.double().cpu().numpy())
    ref = oracle_run(w, inp)
    to, tg = TOL[w.dtype]
    assert np.all(np.isfinite(got[0])) and np.all(np.isfinite(got[3]))
    assert np.abs(got[0] - ref[0]).max() <= to * np.abs(ref[0]).max()
    assert np.linalg.norm(got[3] - ref[3]) <= tg * np.linalg.norm(ref[3])
    assert np.all(ref[1] == 0) and np.all(ref[2] == 0)


ANGULAR = [
    W_("ang_f32", 2, 2, 77, 64, 3, 1, False, "f32"),
    W_("ang_f32_c", 1, 3, 100, 32, 3, 1, True, "f32"),
    W_("ang_bf", 1, 2, 300, 128, 3, 1, False, "bf16"),
    W_("ang_bf_c", 2, 1, 129, 64, 3, 1, True, "bf16"),
]


@pytest.mark.parametrize("gamma", [0.0, 1.0, 3.0, 8.0, 2.5])
@pytest.mark.parametrize("w", ANGULAR, ids=lambda w: w.name)
def test_angular_matches_oracle(w, gamma):
    """Exact angular attention (Eqs. 3-4) against the oracle's, with a zero Q row and a zero K
    row; the float32 tolerance 1e-5 holds because the angle is formed stably (2 atan2 of the
    half-chords), not as arccos of a rounded cosine."""
    inp = inputs_on_gpu(w, seed=9)
    inp["Q"][0, 0, 5] = 0
    inp["K"][0, 0, 3] = 0
    O = race.race_attn_angular(inp["Q"], inp["K"], inp["V"], gamma, w.causal)
    torch.cuda.synchronize()
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V")}
    ref = oracle.angular_forward(a["Q"], a["K"], a["V"], gamma, w.causal)
    got = O.double().cpu().numpy()
    tol = TOL[w.dtype][0]
    assert np.abs(got - ref).max() <= tol * np.abs(ref).max()
    again = race.race_attn_angular(inp["Q"], inp["K"], inp["V"], gamma, w.causal)
    assert torch.equal(O, again)


def test_angular_near_parallel_and_antipodal():
    """Keys at angles 1e-4 and pi - 1e-4 from the query: the weights (1 - theta/pi)^8 are
    1 - 2.5e-4 and 1.3e-35, which a float32 arccos of the cosine gets wrong by far more than the
    float32 tolerance."""
    d = 64
    q = torch.zeros(d)
    q[0] = 1.0
    e = 1e-4
    k0 = torch.zeros(d)
    k0[0], k0[1] = math.cos(e), math.sin(e)
    k1 = -k0
    K = torch.stack([k0, k1, k0 * 2.0])
    Q = torch.stack([q, q * 3.0, -q])
    V = torch.randn((3, d), generator=torch.Generator().manual_seed(5))
    Qg, Kg, Vg = (x[None, None].contiguous().cuda() for x in (Q, K, V))
    O = race.race_attn_angular(Qg, Kg, Vg, 8.0, False)
    a = {k: as_oracle_array(x) for k, x in (("Q", Qg), ("K", Kg), ("V", Vg))}
    ref = oracle.angular_forward(a["Q"], a["K"], a["V"], 8.0, False)
    assert np.abs(O.double().cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()


def test_race_error_against_angular_falls_with_beta_and_tables():
    """The error bound's two terms ("The claimed bound separates bias and sampling error",
    Theorem 2), measured on the GPU against P-powered angular attention.  Sampling error: at
    beta = 50 one table is far worse than 16.  Soft-hash bias: with the output averaged over 32
    independent 16-table draws, so that sampling noise is small, beta = 2 beats beta = 0.5.  On
    these seeded inputs the float64 oracle gives 0.146 vs 0.539 and 0.019 vs 0.050; beyond
    beta ~ 2 the averaged error sits on the remaining sampling noise."""
    P, N, d, L, M = 2, 512, 64, 16, 32
    g = torch.Generator().manual_seed(21)
    Q, K, V = (torch.randn((1, 1, N, d), generator=g).cuda() for _ in range(3))
    A = race.race_attn_angular(Q, K, V, float(P), False)

    def rms(O):
        return float(((O - A) ** 2).sum().sqrt() / math.sqrt(N))

    def single(beta, Lx):
        W = torch.randn((Lx, P, d), generator=torch.Generator().manual_seed(22)).cuda()
        return rms(race.race_attn_fwd(Q, K, V, W, beta, Lx, P, False))

    def averaged(beta):
        acc = torch.zeros_like(A)
        for m in range(M):
            W = torch.randn((L, P, d), generator=torch.Generator().manual_seed(100 + m)).cuda()
            acc += race.race_attn_fwd(Q, K, V, W, beta, L, P, False)
        return rms(acc / M)

    assert single(50.0, 16) < 0.5 * single(50.0, 1)
    assert averaged(2.0) < 0.6 * averaged(0.5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_hard_hash(dtype):
    """Decode steps at beta = +inf against the oracle's hard-hash decode step (inputs as in
    test_hard_hash: sign margins >= 1e-3, each query meets its own key)."""
    w = W_("decode_hard", 2, 2, 24, 64, 3, 3, True, dtype, beta=math.inf)
    inp = _hard_inputs(w, seed=14)
    Q, K, V, W = inp["Q"], inp["K"], inp["V"], inp["W"]
    B, H, N, d = Q.shape
    state = torch.zeros((B, H, w.L << w.P, d + 1), dtype=torch.float32, device="cuda")
    ref_state = np.zeros((B, H, w.L << w.P, d + 1))
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V")}
    Wd = W.double().cpu().numpy()
    tol = 2e-5 if dtype == "f32" else 1e-2
    for t in range(N):
        tok = [x[:, :, t:t + 1].contiguous() for x in (Q, K, V)]
        o = race.race_attn_decode(*tok, W, w.beta, w.L, w.P, state)
        ref = oracle.decode_step(a["Q"][:, :, t], a["K"][:, :, t], a["V"][:, :, t], Wd, w.beta, ref_state)
        assert np.abs(o[:, :, 0].double().cpu().numpy() - ref).max() <= tol * np.abs(ref).max(), t
    assert np.abs(state.double().cpu().numpy() - ref_state).max() <= 1e-5 * np.abs(ref_state).max()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_count_equivalence(causal, dtype):
    """The decomposition a multi-GPU run would use, on one GPU: each sequence is cut into segments
    whose sketch sums are combined (non-causal) or scanned (causal) in a fixed order, and the
    planner picks the segment count from B * H (about two CTAs per SM over all (b, h)).  One
    sequence alone (B * H = 1: 157 segments at N = 20000) and the same sequence as one of 8 heads
    (32 segments) give the same O, dQ, dK, dV up to float32 rounding (bf16 outputs: a last-bit
    flip of the rounded value)."""
    w8 = W_("split8", 1, 8, 20000, 64, 3, 3, causal, dtype)
    inp = inputs_on_gpu(w8, seed=15)
    full = gpu_run(w8, inp)
    w1 = W_("split1", 1, 1, 20000, 64, 3, 3, causal, dtype)
    one = {k: (v[:, 3:4].contiguous() if v.dim() == 4 else v) for k, v in inp.items()}
    alone = gpu_run(w1, one)
    tol = 1e-5 if dtype == "f32" else 1e-2
    for name, a, b in zip(("O", "dQ", "dK", "dV"), full, alone):
        e = np.abs(a[:, 3:4] - b).max() / np.abs(b).max()
        assert e <= tol, "%s %s differs by %.2e across split counts" % (name, dtype, e)

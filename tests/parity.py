"""Helpers shared by the GPU parity tests: run the library through its C ABI, run the oracle on
the same seeded inputs, and compare with the tolerances the workloads state.

Tolerances (float64 oracle as reference):
  float32 tensors: max |O - O_ref| / max |O_ref| <= 1e-5 and, for each gradient,
                   ||g - g_ref||_2 / ||g_ref||_2 <= 1e-5;
  bfloat16 tensors: the same measures with 2e-2 on O and 5e-2 on the gradients.
"""
import numpy as np
import torch

import linear_lsh_sketch_gb300 as race
import oracle
from linear_lsh_sketch_gb300.workloads import as_oracle_array, make_inputs

TOL = {"f32": (1e-5, 1e-5), "bf16": (2e-2, 5e-2)}


def gpu_run(w, inp, with_state=True, rows=None, heads=None, keep_on_device=False):
    """Forward then backward through the C ABI; returns float64 host copies (O, dQ, dK, dV),
    optionally only token `rows` of the first `heads` heads, or, with keep_on_device, the four
    device tensors themselves."""
    dev = inp["Q"].device
    state = None
    if with_state:
        nb = race.race_attn_state_bytes(race.make_shape(w.B, w.H, w.N, w.d, w.torch_dtype), w.L, w.P,
                                        w.causal)
        state = torch.empty(nb, dtype=torch.uint8, device=dev)
    O = race.race_attn_fwd(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal, state=state)
    dQ, dK, dV = race.race_attn_bwd(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal,
                                    inp["dO"], O=O, state=state)
    torch.cuda.synchronize()
    if keep_on_device:
        return O, dQ, dK, dV
    out = []
    for t in (O, dQ, dK, dV):
        if heads is not None:
            t = t[:, :heads]
        if rows is not None:
            t = t[:, :, torch.as_tensor(rows, device=t.device)]
        out.append(t.double().cpu().numpy())
    return tuple(out)


def oracle_run(w, inp, rows=None, nthreads=0):
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V", "dO")}
    W = inp["W"].double().cpu().numpy()
    O = oracle.forward(a["Q"], a["K"], a["V"], W, w.beta, w.causal, rows=rows, nthreads=nthreads)
    dQ, dK, dV = oracle.backward(a["Q"], a["K"], a["V"], a["dO"], W, w.beta, w.causal, rows=rows,
                                 nthreads=nthreads)
    return O, dQ, dK, dV


def errors(got, ref):
    O, dQ, dK, dV = got
    Or, dQr, dKr, dVr = ref
    eo = np.abs(O - Or).max() / np.abs(Or).max()
    # a gradient that is exactly zero (e.g. dQ, dK at beta = 0) is compared in absolute terms
    eg = [np.linalg.norm(g - r) / (np.linalg.norm(r) if np.linalg.norm(r) > 0 else 1.0)
          for g, r in ((dQ, dQr), (dK, dKr), (dV, dVr))]
    return eo, eg


def assert_close(w, got, ref, label=""):
    to, tg = TOL[w.dtype]
    for x in got:
        assert np.all(np.isfinite(x)), "non-finite output " + label
    eo, eg = errors(got, ref)
    assert eo <= to, "%s O error %.3e > %.1e" % (label, eo, to)
    for name, e in zip(("dQ", "dK", "dV"), eg):
        assert e <= tg, "%s %s error %.3e > %.1e" % (label, name, e, tg)
    return eo, eg


def inputs_on_gpu(w, seed=0):
    inp = make_inputs(w, seed=seed, device="cpu")
    return {k: v.cuda() for k, v in inp.items()}

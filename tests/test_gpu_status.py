"""The device status word every workspace carries (GPU): a degenerate denominator and a bounded
wait that runs out are both reported to the caller, and the context stays usable afterwards.

The failure is made without faulting anything: a test hook makes the causal tcgen05 forward skip
its first tile request, so its waits run out after their time bound and the kernel takes its
abort path (drain, free tensor memory, return)."""
import numpy as np
import pytest
import torch

import linear_lsh_sketch_gb300 as race
from linear_lsh_sketch_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _run_fwd(w, inp, beta=None):
    shape = race.make_shape(w.B, w.H, w.N, w.d, w.torch_dtype)
    ws = torch.empty(race.race_attn_workspace_bytes(shape, w.L, w.P, w.causal, 0), dtype=torch.uint8,
                     device="cuda")
    O = race.race_attn_fwd(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta if beta is None else beta, w.L, w.P,
                           w.causal, workspace=ws)
    return O, race.race_attn_status(ws)


# one workload per forward kernel family: CUDA-core non-causal / causal (float32), tcgen05
# non-causal read-out and causal chunk kernel (bfloat16)
FAMILIES = [
    Workload("st_f32", 1, 2, 64, 64, 2, 1, 10.0, False, "f32"),
    Workload("st_f32_c", 1, 2, 64, 64, 2, 1, 10.0, True, "f32"),
    Workload("st_bf_nc", 1, 2, 200, 64, 2, 1, 10.0, False, "bf16"),
    Workload("st_bf_c", 1, 2, 200, 128, 2, 1, 10.0, True, "bf16"),
]


@pytest.mark.parametrize("w", FAMILIES, ids=lambda w: w.name)
def test_numeric_status(w):
    """Every query row equal to one vector q and every key row equal to -q, at beta = 1000: in
    every table the keys sit in the corner opposite the queries', so each query's corners hold no
    key mass in float32 (the products of sigmoid(-2 beta |u|) underflow), den = 0 and the row is
    0/0 -- the walkthrough's Step 6 case A.  The status word reports RACE_ERR_NUMERIC; at
    beta = 10 the same inputs give finite outputs and RACE_OK."""
    inp = {k: v.cuda() for k, v in make_inputs(w, seed=3, device="cpu").items()}
    q = inp["Q"][:, :, :1].float()
    inp["Q"] = q.expand_as(inp["Q"]).contiguous().to(w.torch_dtype)
    inp["K"] = (-q).expand_as(inp["K"]).contiguous().to(w.torch_dtype)
    O, st = _run_fwd(w, inp)
    assert st == 0 and torch.isfinite(O.float()).all()
    O, st = _run_fwd(w, inp, beta=1000.0)
    assert st == race.RACE_ERR_NUMERIC
    assert not torch.isfinite(O.float()).all()
    assert race.race_attn_strerror(st) != "unknown status"


def test_bounded_wait_runs_out_and_context_survives():
    """With the first tile request withheld, the causal bf16 tcgen05 forward's waits run out: the
    call reports RACE_ERR_DEVICE_TIMEOUT (through race_attn_status, and through
    race_attn_noalloc_status for the allocation-free entry point); the next calls on the same
    context run normally and reproduce the regular output bit for bit."""
    w = Workload("withhold", 1, 1, 300, 128, 3, 3, 10.0, True, "bf16")
    inp = {k: v.cuda() for k, v in make_inputs(w, seed=5, device="cpu").items()}
    ref, st = _run_fwd(w, inp)
    assert st == 0
    race.race_attn_test_withhold_first_load(True)
    try:
        _, st = _run_fwd(w, inp)
        assert st == race.RACE_ERR_DEVICE_TIMEOUT
        race.race_attn_fwd_noalloc(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal)
        assert race.race_attn_noalloc_status() == race.RACE_ERR_DEVICE_TIMEOUT
    finally:
        race.race_attn_test_withhold_first_load(False)
    again, st = _run_fwd(w, inp)
    assert st == 0 and torch.equal(again, ref)
    O = race.race_attn_fwd_noalloc(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal)
    assert race.race_attn_noalloc_status() == 0
    assert torch.equal(O, ref)

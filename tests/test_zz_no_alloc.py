"""The forward entry point that allocates nothing, against the regular forward (GPU).

race_attn_fwd_noalloc exists for callers that may not allocate device memory (an allocator
that owns the whole device, or a loop that must never allocate): it runs the same forward
kernels on the library's built-in static scratch buffer instead of a caller workspace.  This
file is named to be collected last, so a run that stops at the first failure has run every
other test before it.
"""
import pytest
import torch

import linear_lsh_sketch_gb300 as race
from linear_lsh_sketch_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

# the same normwise-max tolerance on O as the parity tests
TOL = {"f32": 1e-5, "bf16": 2e-2}

CASES = [
    Workload("noalloc_causal_bf16", 1, 4, 3000, 128, 3, 3, 10.0, True, "bf16"),
    Workload("noalloc_f32", 2, 2, 777, 64, 2, 2, 10.0, False, "f32"),
    Workload("noalloc_lr256_bf16", 1, 2, 1500, 128, 6, 4, 10.0, False, "bf16", 8),
]


def _err(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).abs().max() / b.abs().max())


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_regular_forward_on_two_calls(w):
    """Two calls in a row (the second sees what the first left in the shared scratch) match the
    regular forward, report a clean status, and allocate nothing: torch's allocator and the
    device's free memory are unchanged across the second call, whose output buffer is given."""
    race.race_attn_noalloc_init()
    inp = {k: v.cuda() for k, v in make_inputs(w, seed=7, device="cpu").items()}
    ref = race.race_attn_fwd(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal)
    torch.cuda.synchronize()
    assert torch.isfinite(ref.float()).all()
    O = torch.empty_like(ref)
    for call in range(2):
        if call == 1:
            torch.cuda.synchronize()
            allocs = torch.cuda.memory_stats()["allocation.all.allocated"]
            free = torch.cuda.mem_get_info()[0]
        race.race_attn_fwd_noalloc(inp["Q"], inp["K"], inp["V"], inp["W"], w.beta, w.L, w.P, w.causal, O=O)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.memory_stats()["allocation.all.allocated"] == allocs
            assert torch.cuda.mem_get_info()[0] == free
        assert race.race_attn_noalloc_status() == 0
        assert _err(O, ref) <= TOL[w.dtype]


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = Workload("noalloc_too_big", 1, 64, 65536, 128, 6, 4, 10.0, False, "bf16")
    shape = race.make_shape(w.B, w.H, w.N, w.d, w.torch_dtype)
    assert race.race_attn_workspace_bytes(shape, w.L, w.P, w.causal, 0) > race.RACE_NOALLOC_SCRATCH_BYTES
    t = torch.empty((1, 64, 65536, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((4, 6, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(race.RaceAttnError) as exc:
        race.race_attn_fwd_noalloc(t, t, t, W, 10.0, 4, 6, False, O=t)
    assert exc.value.status == race.RACE_ERR_SCRATCH_LIMIT

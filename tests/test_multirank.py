"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas) aggregate the step time as the
max over ranks and report the whole job's throughput; each rank draws its own inputs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from linear_lsh_sketch_gb300.workloads import CONFIGS, make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, ws, local = bench.env_rank()
        ms = bench.max_over_ranks(times[r], dist, "cpu")
        value = bench.weak_scaling_tokens_per_s(ws, 1000, ms)
        w = CONFIGS["c1_f32_tiny"]
        q = make_inputs(w, seed=r, device="cpu")["Q"]
        gathered = [torch.empty_like(q) for _ in range(ws)]
        dist.all_gather(gathered, q)
        same_inputs = all(torch.equal(gathered[0], g) for g in gathered[1:])
        out.put((r, ws, local, ms, value, same_inputs))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_aggregate_max_time():
    world, times = 2, [3.0, 5.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, ws, local, ms, value, same_inputs) in enumerate(res):
        assert (rank, ws, local) == (r, world, r)
        assert ms == max(times)                      # the slowest replica sets the step time
        assert value == pytest.approx(world * 1000 / (max(times) / 1000.0))
        assert not same_inputs                       # replicas run independent seeded inputs


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.env_rank() == (0, 1, 0)
    assert bench.weak_scaling_tokens_per_s(1, 12_000_000, 50.0) == pytest.approx(2.4e8)


def test_kernel_table():
    """Per-kernel shares and HBM fractions from a profile: compulsory bytes per (token, head)
    times the tokens, over the time per launch; kernels without a byte count get no fraction."""
    import bench
    from linear_lsh_sketch_gb300.workloads import CONFIGS

    w = CONFIGS["c5_bf16_causal_12m"]
    prof = {"tc5_causal_fwd": (2, 18.0), "combine": (4, 0.2), "tc5_causal_bwd_kv": (2, 34.0)}
    t = bench.kernel_table(prof, w, 6800.0)
    assert abs(sum(r["share"] for r in t.values()) - 1.0) < 1e-12
    fwd = t["tc5_causal_fwd"]
    # reads Q and V and the keys' stored feature rows (L R = 24 bf16), writes O
    want = (3 * w.d * 2 + 24 * 2) * w.B * w.H * w.N / (9.0 / 1000.0) / 1e9
    assert abs(fwd["achieved_gbs"] - want) < 1e-6 * want and abs(fwd["frac"] - want / 6800.0) < 1e-12
    # its share of the step's algorithmic bytes: Q, K, V in and O out
    alg = 4 * w.d * 2 * w.B * w.H * w.N / (9.0 / 1000.0) / 1e9
    assert abs(fwd["alg_gbs"] - alg) < 1e-6 * alg
    assert "frac" not in t["combine"] and t["combine"]["ms_per_launch"] == 0.05

"""Host-side logic of the engine-step executor and of the multi-rank bench
path, on the CPU (no GPU, gloo for the 2-rank case)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_deltanet_linear_build_gb300 import stack, synth


@pytest.mark.parametrize("budget", [2048, 1000, 513])
def test_pack_prefill_steps_covers_every_prompt_once(budget):
    lengths = [int(x) for x in synth.serving_mix_lengths(4)]
    steps = stack.pack_prefill_steps(lengths, budget)
    seen = {s: 0 for s in range(len(lengths))}
    for st in steps:
        assert 0 < st.tokens <= budget
        slots = [g.seq for g in st.segments]
        assert slots == list(range(slots[0], slots[0] + len(slots)))
        for g in st.segments:
            assert g.start == seen[g.seq], "segments continue where the last one ended"
            seen[g.seq] += g.length
    assert [seen[s] for s in range(len(lengths))] == lengths
    # All steps but the last are full.
    assert all(st.tokens == budget for st in steps[:-1])


def test_serving_mix_lengths_range():
    L = synth.serving_mix_lengths(4)
    assert len(L) == 32 and L.min() >= 512 and L.max() <= 1024


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.init_dist(world, "gloo")
    w, r, _ = bench.dist_env()
    mx = bench.reduce_over_ranks(10.0 + r, "max", d)
    sm = bench.reduce_over_ranks(100.0 * (r + 1), "sum", d)
    out[r] = (w, mx, sm, bench.rank_lengths_seed(r))
    d.destroy_process_group()


def test_bench_rank_reductions_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][:3] == (2, 11.0, 300.0) and res[1][:3] == (2, 11.0, 300.0)
    assert res[0][3] != res[1][3], "ranks serve different sequences"

"""bench.py's N > 1 host logic on CPU with two gloo ranks: each rank draws its own
batch (weak scaling, no data-path collective) and the reported time is the max
over ranks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_28_gb300 import workload as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    seed = bench.rank_seed(wl.DEFAULT_SEEDS["llama70b_layer"], r)
    batch = wl.make("llama70b_layer", seed=seed, with_pools=False)
    bench.barrier(w)
    t = bench.reduce_max(1.0 + r, w)          # rank-local "time"
    total = bench.reduce_max(float(batch.logical_tokens), w)
    out[r] = (seed, int(batch.logical_tokens), t, total, local)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_and_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    seeds = {res[r][0] for r in range(world)}
    assert len(seeds) == world                              # each rank its own batch
    assert res[0][1] != res[1][1]
    assert all(res[r][2] == 2.0 for r in range(world))      # max over ranks
    assert all(res[r][3] == max(res[0][1], res[1][1]) for r in range(world))
    assert [res[r][4] for r in range(world)] == [0, 1]


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.rank_seed(1, 0) == 1 and np.unique([bench.rank_seed(1, r) for r in range(8)]).size == 8


def test_decode_time_sample_is_stratified():
    """The decode kernel's mean over K timed steps from events on step 0 and the middle of
    each later block of 8: step 0 counts once, the other samples stand for the rest."""
    assert bench.sampled_steps(1) == [0]
    assert bench.sampled_steps(20) == [0, 4, 12]
    s = bench.sampled_steps(2000)
    assert s[0] == 0 and len(s) == 1 + 250 and all(i % 8 == 4 for i in s[1:])
    # equal times give that time; a slow first step weighs 1/K, not 1/len(sample)
    assert bench.mean_decode_ms({0: 3.0, 4: 3.0, 12: 3.0}, 20) == 3.0
    got = bench.mean_decode_ms({0: 230.0, 4: 210.0, 12: 210.0}, 20)
    assert abs(got - (230.0 + 19 * 210.0) / 20) < 1e-9
    assert bench.mean_decode_ms({0: 7.0}, 1) == 7.0

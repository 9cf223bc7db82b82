"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2): each rank
runs an independent shard (own seed, no data-path collective); the step time
is the max over ranks and the token count the sum over ranks."""
from __future__ import annotations

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_setup()
    assert (r, w) == (rank, world)
    from workloads import CONFIGS, draw_metadata
    import numpy as np
    cfg = CONFIGS["C2"]
    seed = bench.shard_seed(cfg.seed, r)
    meta = draw_metadata(cfg, np.random.default_rng(seed))
    tokens = bench.step_accounting(cfg, meta)["tokens"]
    fake_ms = 10.0 + 5.0 * r  # rank 1 is the slow one
    t_max = bench.max_over_ranks(fake_ms, w)
    tok_all = bench.sum_over_ranks(tokens, w)
    q.put((r, seed, tokens, t_max, tok_all))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, t0, m0, a0), (r1, s1, t1, m1, a1) = res
    assert s0 != s1                      # independent shards
    assert m0 == m1 == 15.0              # max over ranks
    assert a0 == a1 == t0 + t1           # whole-job tokens


def test_step_accounting_matches_the_per_item_formula():
    import numpy as np
    import bench
    from workloads import CONFIGS, draw_metadata
    cfg = CONFIGS["C2"]
    meta = draw_metadata(cfg, np.random.default_rng(2))
    acct = bench.step_accounting(cfg, meta)
    lens = np.minimum(np.diff(meta.query_start_loc), cfg.Q)
    # per (live request, head): 69 376 + 3 074 n bytes at K = V = 128, W = 4
    live = meta.state_indices > 0
    per_layer = cfg.H * sum(69376 + 3074 * int(n) for n in lens[live])
    per_layer += cfg.H * 2 * cfg.K * int(lens[~live].sum())
    per_layer += 3 * cfg.H * cfg.K * 4 * 2 + 4 * cfg.H + 4 * cfg.H * cfg.K
    assert acct["verify_layer_bytes"] == per_layer
    acc = np.minimum(meta.num_accepted, lens)
    commit = cfg.L * cfg.H * sum(131072 + 1024 * int(a) for a, l in zip(acc, live) if l and a > 0)
    assert acct["commit_bytes"] == commit
    assert acct["tokens"] == int(lens[live].sum())

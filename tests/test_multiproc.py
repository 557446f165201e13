"""The multi-rank path on CPU (gloo, world size 2): ranks verify disjoint
shards of one global batch with global Philox sequence ids, so together
they emit exactly what one call over the whole batch emits; the benchmark's
timing takes the slowest rank. No GPU is used: the oracle stands in for the
per-rank verify call, and the collectives below only check the results."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from oracle import oracle as orc

WORLD = 2


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def make_batch(B=8, K=4, V=60, seed=3):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 2, (B, K + 1, V))
    drf = tgt[:, :K] + rng.normal(0, 1, (B, K, V))
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    return tgt, drf, tok


def worker(rank, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        tgt, drf, tok = make_batch()
        B = tgt.shape[0] // WORLD
        sl = slice(rank * B, (rank + 1) * B)
        ids = bench.shard_seq_ids(rank, B, "cpu").numpy().astype(np.uint64)
        out = orc.verify(tgt[sl], drf[sl], tok[sl], 1.0, 1, seed=21, seq_ids=ids)
        mine = torch.from_numpy(np.concatenate([out["tokens"].ravel(), out["n_accepted"]]))
        gathered = [torch.empty_like(mine) for _ in range(WORLD)]
        dist.all_gather(gathered, mine)
        slowest = bench.max_over_ranks(1.0 + rank, "cpu", WORLD)
        # the bench line's whole-job rates: rank r verified 10 + r rows and
        # 1000 * (r + 1) bytes in (r + 1) ms
        rates = bench.job_rates(10 + rank, 1000 * (rank + 1), 1.0 + rank, "cpu", WORLD)
        if rank == 0:
            results.put((torch.stack(gathered).numpy(), slowest, rates))
    finally:
        dist.destroy_process_group()


def test_shards_with_global_ids_equal_one_call_and_time_is_the_slowest_rank():
    orc.build()  # once, before the ranks load it
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, port, results)) for r in range(WORLD)]
    for p in procs:
        p.start()
    gathered, slowest, rates = results.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    tgt, drf, tok = make_batch()
    B, K1 = tgt.shape[0], tgt.shape[1]
    full = orc.verify(tgt, drf, tok, 1.0, 1, seed=21)
    Bs = B // WORLD
    for r in range(WORLD):
        toks = gathered[r][:Bs * K1].reshape(Bs, K1)
        n = gathered[r][Bs * K1:]
        assert (toks == full["tokens"][r * Bs:(r + 1) * Bs]).all()
        assert (n == full["n_accepted"][r * Bs:(r + 1) * Bs]).all()
    assert slowest == float(WORLD)
    # rows and bytes of both ranks over the slowest rank's 2 ms
    assert rates["ms_max"] == 2.0
    assert np.isclose(rates["rows_per_s"], (10 + 11) / 2e-3)
    assert np.isclose(rates["gbs"], (1000 + 2000) / 2e-3 / 1e9)

"""Multi-process host logic on CPU (gloo, world size 2).

The scan shards over independent (batch, channel) units with no data-path
exchange: each rank runs its own block of channels, and only the benchmark's
bookkeeping (max of step times, sum of units) is reduced across ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from selective_state_space_146_b300 import dist as dh


def test_shard_range_partitions_units():
    for total in (0, 1, 7, 64, 12288):
        for world in (1, 2, 3, 8):
            spans = [dh.shard_range(total, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0 and a0 <= a1
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from selective_state_space_146_b300 import inputs
    inp = inputs.selective_inputs(2, 12, 16, 64, "f32", seed=4)
    total = 2 * 12
    lo, hi = dh.shard_range(total, rank, world)
    rows = []
    for c in range(lo, hi):
        b, d = divmod(c, 12)
        y, s = oracle.selective_scan(inp["u"][b:b + 1, d:d + 1], inp["delta"][b:b + 1, d:d + 1],
                                     inp["A"][d:d + 1], inp["B"][b:b + 1], inp["C"][b:b + 1],
                                     inp["D"][d:d + 1], inp["z"][b:b + 1, d:d + 1],
                                     inp["delta_bias"][d:d + 1])
        rows.append(y[0, 0])
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), np.stack(rows))
    t_max = dh.max_over_ranks(float(rank + 1))
    n_sum = dh.sum_over_ranks(float(hi - lo))
    np.save(os.path.join(out_dir, f"red{rank}.npy"), np.array([t_max, n_sum]))
    dh.barrier()
    dist.destroy_process_group()


def test_two_rank_sharded_scan_matches_single_process(tmp_path):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from selective_state_space_146_b300 import inputs
    inp = inputs.selective_inputs(2, 12, 16, 64, "f32", seed=4)
    y, _ = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["z"], inp["delta_bias"])
    got = np.concatenate([np.load(tmp_path / f"rank{r}.npy") for r in range(2)])
    np.testing.assert_array_equal(got, y.reshape(24, 64))
    for r in range(2):
        t_max, n_sum = np.load(tmp_path / f"red{r}.npy")
        assert t_max == 2.0 and n_sum == 24.0


def test_reductions_are_identity_without_process_group():
    assert dh.max_over_ranks(3.5) == 3.5
    assert dh.sum_over_ranks(2.0) == 2.0
    assert dh.env_world()[2] >= 1

"""The N>1 path on CPU: two gloo ranks, spawned as processes.

* the max-over-ranks timing and the whole-job rate of the benchmark;
* sharding the (b, h) units by head needs no collective: each rank's
  gradients equal the single-process ones for its heads, bit for bit;
* sharding by batch row needs one sum of dR, du, dv over the ranks; the
  per-row gradients are still bit-exact.
The attention itself is the float64 oracle here (the CUDA path is the same
per rank).
"""
import os
import socket

import numpy as np
import pytest

import oracle
import rxl_inputs as gen
from long_context_lm_rel_gb300.multirank import max_over_ranks, replica_seed, shard, whole_job_rate

WORLD = 2
B, H, L, M, DH, SCALE = 2, 4, 24, 20, 16, 0.25


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, H, L, DH))
    k = rng.standard_normal((B, H, M + L, DH))
    v = rng.standard_normal((B, H, M + L, DH))
    r = rng.standard_normal((H, M + L, DH)) * 0.7
    u = rng.standard_normal((H, DH)) * 0.1
    vb = rng.standard_normal((H, DH)) * 0.1
    do = rng.standard_normal((B, H, L, DH))
    return q, k, v, r, u, vb, do


def _oracle(q, k, v, r, u, vb, do):
    o, lse = oracle.fwd(q, k, v, r, u, vb, SCALE, nthreads=1)
    g = oracle.bwd(q, k, v, r, u, vb, do, SCALE, nthreads=1)
    return o, lse, g


def _worker(rank, port, result_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=WORLD)
    try:
        # timing: the job takes as long as its slowest rank
        t = max_over_ranks(1.5 + rank, WORLD)
        assert t == 2.5, t
        assert abs(whole_job_rate(10.0, WORLD, t) - 8.0) < 1e-12

        q, k, v, r, u, vb, do = _problem()
        # by head: no collective, every output complete on its rank
        h0, h1 = shard(H, rank, WORLD)
        hs = slice(h0, h1)
        o, lse, g = _oracle(q[:, hs], k[:, hs], v[:, hs], r[hs], u[hs], vb[hs], do[:, hs])
        np.savez(os.path.join(result_dir, f"head{rank}.npz"), o=o, lse=lse, **g)
        # by batch row: dR, du, dv summed over the ranks
        b0, b1 = shard(B, rank, WORLD)
        bs = slice(b0, b1)
        o, lse, g = _oracle(q[bs], k[bs], v[bs], r, u, vb, do[bs])
        import torch
        for name in ("dr", "du", "dvb"):
            t = torch.from_numpy(np.ascontiguousarray(g[name]))
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
            g[name] = t.numpy()
        np.savez(os.path.join(result_dir, f"batch{rank}.npz"), o=o, lse=lse, **g)
    finally:
        dist.destroy_process_group()


def test_shard_covers_units_once():
    for n in range(0, 40):
        for world in range(1, 9):
            parts = [shard(n, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard(4, 2, 2)
    assert len({replica_seed(0, r) for r in range(8)}) == 8


def test_single_rank_helpers_need_no_process_group():
    assert max_over_ranks(3.25, 1) == 3.25
    assert whole_job_rate(5.0, 1, 2.0) == 2.5
    with pytest.raises(ValueError):
        whole_job_rate(5.0, 1, 0.0)


def test_two_gloo_ranks_shard_the_units(tmp_path):
    pytest.importorskip("torch.distributed")
    import torch.multiprocessing as mp
    oracle.load()  # build the C oracle once, before the ranks start
    mp.start_processes(_worker, args=(_free_port(), str(tmp_path)), nprocs=WORLD, join=True,
                       start_method="spawn")
    q, k, v, r, u, vb, do = _problem()
    o, lse, g = _oracle(q, k, v, r, u, vb, do)
    full = dict(o=o, lse=lse, **g)
    for rank in range(WORLD):
        h0, h1 = shard(H, rank, WORLD)
        part = np.load(tmp_path / f"head{rank}.npz")
        for name in ("o", "lse", "dq", "dk", "dv"):
            assert np.array_equal(part[name], full[name][:, h0:h1]), name
        for name in ("dr", "du", "dvb"):
            assert np.array_equal(part[name], full[name][h0:h1]), name
        b0, b1 = shard(B, rank, WORLD)
        part = np.load(tmp_path / f"batch{rank}.npz")
        for name in ("o", "lse", "dq", "dk", "dv"):
            assert np.array_equal(part[name], full[name][b0:b1]), name
        for name in ("dr", "du", "dvb"):
            np.testing.assert_allclose(part[name], full[name], rtol=1e-12, atol=1e-12)


def test_replica_inputs_differ_by_rank():
    import dataclasses
    w0 = dataclasses.replace(gen.CFG1, seed=replica_seed(0, 0))
    w1 = dataclasses.replace(gen.CFG1, seed=replica_seed(0, 1))
    assert not np.array_equal(gen.segment_inputs(w0)["q"], gen.segment_inputs(w1)["q"])

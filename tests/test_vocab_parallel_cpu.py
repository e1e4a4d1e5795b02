"""The vocabulary-parallel exchange on CPU: two gloo ranks each hold half of
the columns of every row.  Each rank reduces its block to per-row pairs (the
oracle stands in for the device kernel here), the pairs are exchanged with
the package's exchange_pairs (an all-gather, shard-major in rank order), and
the merged pairs and the finished blocks must equal the single-process
results on whole rows."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows(seed=41, M=37, N=1000):
    rng = np.random.default_rng(seed)
    x = rng.normal(scale=4.0, size=(M, N))
    x[3, :] = -np.inf          # an all -inf row: NaN after the finish
    x[5, :600] = -np.inf       # rank 0's block of row 5 holds no mass
    x[7, 123] = 40.0           # a spike in rank 0's block
    return x


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from memory_bound_row_gb300 import exchange_pairs

        x = _rows()
        cuts = [0, 600, x.shape[1]]
        block = np.ascontiguousarray(x[:, cuts[rank]:cuts[rank + 1]])
        mine = torch.from_numpy(oracle.softmax_partial_f64(block, "f64"))
        gathered = exchange_pairs(mine)
        assert gathered.shape == (world,) + tuple(mine.shape)
        assert torch.equal(gathered[rank], mine)
        merged = oracle.merge_pairs_f64(gathered.numpy())
        y = oracle.softmax_finish_f64(block, "f64", merged)
        out[rank] = (merged, y)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_pairs_and_finish_their_blocks():
    import oracle

    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x = _rows()
    whole_pairs = oracle.softmax_partial_f64(x, "f64")
    whole = oracle.softmax_f64(x, "f64")
    m0, y0 = out[0]
    m1, y1 = out[1]
    assert np.array_equal(m0, m1, equal_nan=True)               # every rank merges to the same pairs
    assert np.array_equal(m0[:, 0], whole_pairs[:, 0])          # the max is exact
    ok = ~np.isnan(whole_pairs[:, 1])
    assert np.allclose(m0[ok, 1], whole_pairs[ok, 1], rtol=1e-14, atol=0)
    y = np.concatenate([y0, y1], axis=1)
    assert np.array_equal(np.isnan(y), np.isnan(whole))
    assert np.all(np.isnan(y[3]))
    fin = ~np.isnan(whole)
    assert np.allclose(y[fin], whole[fin], rtol=1e-13, atol=1e-300)

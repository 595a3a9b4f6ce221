"""Host logic of decode context parallelism (moonmath-ai/amd-kernels README,
"Use / MLA decode": a rank holds the positions p % cp_world == cp_rank, and the
ranks' shares are merged after an exchange), on the CPU: the rank page tables
that ``split_kv_mla_gb300.dcp`` builds against the oracle's own sharding, and
the exchange step with world size 2 over gloo, whose gathered shares (computed
by the oracle) must merge to the unsharded decode."""
import dataclasses
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import oracle
from split_kv_mla_gb300 import dcp
from split_kv_mla_gb300 import inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("lens,world", [
    ([9, 1, 0, 6], 2),
    ([11, 2, 7, 3], 3),
    ([1, 1, 1], 4),
    ([0, 0], 2),
    ([40], 1),
    ([17, 5], 8),
])
def test_shard_page_table_matches_the_oracle_sharding(lens, world):
    inp = gen.dense_inputs(len(lens), 1, 1, lens, seed=7 + world, d_v=8, d_rope=0,
                           extra_slots=3)
    for k in range(world):
        sl, si, sp, glen = dcp.shard_page_table(inp.seq_lens, inp.kv_indices, inp.kv_indptr,
                                                k, world)
        ref, rglen = oracle.dcp_shard(inp, k, world)
        assert torch.equal(sl, ref.seq_lens)
        assert torch.equal(si, ref.kv_indices)
        assert torch.equal(sp, ref.kv_indptr)
        assert torch.equal(glen, rglen)
        assert sl.dtype == si.dtype == sp.dtype == torch.int32


def test_shard_page_table_ignores_slots_past_seq_len():
    # request 0 owns 6 slots but only 4 are live; its dead slots stay out
    idx = torch.arange(10, dtype=torch.int32)
    ptr = torch.tensor([0, 6, 10], dtype=torch.int32)
    lens = torch.tensor([4, 4], dtype=torch.int32)
    sl, si, sp, _ = dcp.shard_page_table(lens, idx, ptr, 1, 2)
    assert sl.tolist() == [2, 2]
    assert si.tolist() == [1, 3, 7, 9]
    assert sp.tolist() == [0, 2, 4]


def test_shard_page_table_rejects_bad_rank():
    t = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        dcp.shard_page_table(t, t, torch.zeros(2, dtype=torch.int32), 2, 2)
    with pytest.raises(ValueError):
        dcp.shard_page_table(t, t, torch.zeros(2, dtype=torch.int32), 0, 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), OMP_NUM_THREADS="1")
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import oracle as orc
        from split_kv_mla_gb300 import dcp as d
        from split_kv_mla_gb300 import inputs as g
        inp = g.dense_inputs(3, 3, 2, [13, 2, 8], seed=5, d_v=32, d_rope=8, extra_slots=2)
        sl, si, sp, glen = d.shard_page_table(inp.seq_lens, inp.kv_indices, inp.kv_indptr,
                                              rank, world)
        shard = dataclasses.replace(inp, seq_lens=sl, kv_indices=si, kv_indptr=sp)
        o, lse = orc.dcp_decode(shard, glen, rank, world)
        parts, lses = d.all_gather_shares(torch.from_numpy(o), torch.from_numpy(lse))
        mo, ml = orc.dcp_merge_ranks(parts.numpy(), lses.numpy())
        ro, rl = orc.dense_decode(inp)
        fin = np.isfinite(rl)
        out[rank] = (tuple(parts.shape), float(np.max(np.abs(mo - ro))),
                     float(np.max(np.abs(ml[fin] - rl[fin]))),
                     bool(np.array_equal(np.isfinite(ml), fin)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_exchange_and_merge_gloo(world):
    # world 4: the 2-key request has no positions on ranks 2 and 3, whose
    # shares are then empty (o = 0, lse = -inf) and must merge away
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == list(range(world))
    for shape, o_err, l_err, fin_ok in res.values():
        assert shape == (world, 9, 2, 32)
        assert o_err <= 1e-12 and l_err <= 1e-12 and fin_ok


def test_bench_dcp_workload_is_rank_0_share():
    sys.path.insert(0, ROOT)
    import bench
    kind, inp, desc = bench.make_workload("dcp3-c0")
    assert kind == "dcp" and "rank 0 of 3" in desc
    assert inp.dcp_world == 3 and int(inp.dcp_glen[0]) == 256
    assert inp.total_keys == 86                     # positions 0, 3, ..., 255
    assert bench.kv_bytes_per_call(kind, inp) == 86 * 576
    with pytest.raises(SystemExit):
        bench.make_workload("dcp1-c0")

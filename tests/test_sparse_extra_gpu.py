"""Sparse top-k decode over a second (compressed) cache on the GPU
(``mla_sparse_decode_extra``; flashinfer
cake_sparse_mla_sm120_dsv4_nvfp4_plan_splits: ``extra_topk`` candidates per
token in the second cache) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle
from split_kv_mla_gb300 import inputs as gen
from split_kv_mla_gb300 import mla

from gpu_util import compare, sample_items

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    mla.load()


def _run(inp, splits=None, ws=None, max_splits=0):
    plan = mla.mla_sparse_decode_plan(inp.num_tokens, inp.num_heads, inp.topk, mla.sm_count(),
                                      max_splits, extra_topk=inp.extra_topk)
    if splits is not None:
        plan = mla.mla_plan_force_splits(plan, splits)
    o, lse = mla.mla_sparse_decode_extra(plan, inp.q_nope.cuda(), inp.q_pe.cuda(),
                                         inp.pool.cuda(), inp.indices.cuda(),
                                         inp.extra_pool.cuda(), inp.extra_indices.cuda(),
                                         inp.scale, inp.kv_scale, workspace_t=ws)
    torch.cuda.synchronize()
    return o, lse, plan


@pytest.mark.parametrize("T,H,topk,extra,rows,xrows,inv", [
    (3, 64, 100, 37, 500, 200, 0.2),
    (2, 64, 5, 1, 40, 3, 0.0),
    (24, 128, 2046, 6, 8192, 64, 0.1),
    (5, 16, 0, 300, 16, 1000, 0.0),
    (4, 32, 513, 511, 4096, 4096, 0.3),
    (1, 64, 2048, 512, 131072, 32768, 0.0),
    (8, 64, 2048, 512, 131072, 32768, 0.0),
])
def test_two_caches_against_oracle(T, H, topk, extra, rows, xrows, inv):
    inp = gen.sparse_extra_inputs(T, H, topk, extra, rows, xrows, seed=T * 31 + extra,
                                  invalid_frac=inv)
    o, lse, plan = _run(inp)
    ro, rl = oracle.sparse_extra_decode(inp)
    compare(o, lse, ro, rl, f"T={T} H={H} topk={topk}+{extra} ns={plan.num_splits}")


def test_c4x_64_tokens_sampled():
    inp = gen.workload_c4x(64)
    o, lse, plan = _run(inp)
    sel = sample_items(64 * 64, 96, seed=5)
    ro, rl = _oracle_items(inp, sel)
    compare(o.reshape(-1, 448)[torch.as_tensor(sel)], lse.reshape(-1)[torch.as_tensor(sel)],
            ro, rl, f"c4x-64 ns={plan.num_splits}")


def _oracle_items(inp, sel):
    # the oracle over the sampled tokens only, then the sampled heads
    toks = sorted(set(int(i) // inp.num_heads for i in sel))
    sub = gen.SparseInputs(num_tokens=len(toks), num_heads=inp.num_heads, topk=inp.topk,
                           q_nope=inp.q_nope[toks], q_pe=inp.q_pe[toks], pool=inp.pool,
                           indices=inp.indices[toks].contiguous(), scale=inp.scale,
                           kv_scale=inp.kv_scale, extra_pool=inp.extra_pool,
                           extra_indices=inp.extra_indices[toks].contiguous())
    o, lse = oracle.sparse_extra_decode(sub)
    pos = {t: i for i, t in enumerate(toks)}
    rows = [pos[int(i) // inp.num_heads] * inp.num_heads + int(i) % inp.num_heads for i in sel]
    return o.reshape(-1, inp.d_v)[rows], lse.reshape(-1)[rows]


@pytest.mark.parametrize("splits", [1, 3, 7, 40])
def test_forced_split_counts(splits):
    inp = gen.sparse_extra_inputs(3, 64, 700, 150, 3000, 900, seed=splits, invalid_frac=0.1)
    o, lse, plan = _run(inp, splits=splits)
    assert plan.num_splits == splits
    ro, rl = oracle.sparse_extra_decode(inp)
    compare(o, lse, ro, rl, f"ns={splits}")


def test_token_with_no_valid_candidate():
    inp = gen.sparse_extra_inputs(3, 64, 64, 32, 300, 100, seed=9)
    inp.indices[1] = -1
    inp.extra_indices[1] = -1
    o, lse, _ = _run(inp)
    assert torch.all(o[1] == 0) and torch.all(torch.isneginf(lse[1]))
    ro, rl = oracle.sparse_extra_decode(inp)
    compare(o, lse, ro, rl, "empty token")


@pytest.mark.parametrize("rows_per_cta", [32, 16])
def test_second_cache_on_several_head_blocks(rows_per_cta):
    # H=128: four 32-row or eight 16-row head blocks, each gathering its own
    # rows of both caches
    inp = gen.sparse_extra_inputs(4, 128, 1024, 256, 8192, 2048, seed=3)
    plan = mla.mla_sparse_decode_plan(4, 128, 1024, mla.sm_count(), extra_topk=256)
    plan.rows_per_cta = rows_per_cta
    plan.head_blocks = plan.grid_x = 128 // rows_per_cta
    o, lse = mla.mla_sparse_decode_extra(plan, inp.q_nope.cuda(), inp.q_pe.cuda(),
                                         inp.pool.cuda(), inp.indices.cuda(),
                                         inp.extra_pool.cuda(), inp.extra_indices.cuda(),
                                         inp.scale, inp.kv_scale)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_extra_decode(inp)
    compare(o, lse, ro, rl, f"H=128 second cache, {rows_per_cta} rows per CTA")


def test_out_of_range_second_cache_slot_sets_error_word():
    inp = gen.sparse_extra_inputs(2, 64, 64, 16, 300, 50, seed=4)
    inp.extra_indices[0, 3] = 50            # one past the second cache
    plan = mla.mla_sparse_decode_plan(2, 64, 64, mla.sm_count(), extra_topk=16)
    ws = mla.workspace(plan)
    mla.mla_workspace_reset(ws)
    mla.mla_sparse_decode_extra(plan, inp.q_nope.cuda(), inp.q_pe.cuda(), inp.pool.cuda(),
                                inp.indices.cuda(), inp.extra_pool.cuda(),
                                inp.extra_indices.cuda(), inp.scale, inp.kv_scale,
                                workspace_t=ws)
    assert mla.mla_read_device_error(ws) & 1    # MLA_DEVERR_BAD_SLOT


def test_plan_must_match_extra_topk():
    inp = gen.sparse_extra_inputs(2, 64, 64, 16, 300, 50, seed=4)
    plan = mla.mla_sparse_decode_plan(2, 64, 80, mla.sm_count())   # same total, no extra
    with pytest.raises(mla.MlaError):
        mla.mla_sparse_decode_extra(plan, inp.q_nope.cuda(), inp.q_pe.cuda(), inp.pool.cuda(),
                                    inp.indices.cuda(), inp.extra_pool.cuda(),
                                    inp.extra_indices.cuda(), inp.scale, inp.kv_scale)

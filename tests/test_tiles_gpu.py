"""GPU: both query-row tiles above 16 rows per request.

Requests of more than 16 (head x draft) rows run as 32-row or 16-row head
blocks, whichever the planner finds faster.  Every case here runs the plan at
both tiles with the same split count, checks each against the fp64 oracle, and
checks that the two differ by no more than a few output roundings (the tiles
group rows differently, so the per-tile choices -- the query's third e4m3 term,
lazy rescaling -- may round differently).
"""
import pytest
import torch

from oracle import oracle
from split_kv_mla_gb300 import inputs as gen
from split_kv_mla_gb300 import mla

from gpu_util import compare, run_dense, run_sparse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    mla.load()


def _with_tile(plan, rpc):
    p = mla.mla_plan_t.from_buffer_copy(plan)
    rows = p.q_len * p.num_heads
    p.rows_per_cta = rpc
    p.head_blocks = -(-rows // rpc)
    p.grid_x = p.head_blocks
    return p


def _close(a, b):
    d = (a.float() - b.float()).abs().max().item()
    assert d <= 2 ** -5, d


@pytest.mark.parametrize("batch,q_len,heads,lens,ns", [
    (1, 1, 64, [3000], 8),                # H=64, one request
    (2, 4, 16, [1500, 700], 4),           # 64 draft x head rows, ragged windows
    (3, 1, 128, [2000, 37, 900], 2),      # eight 16-row head blocks, a short request
    (1, 2, 32, [5000], 16),               # two draft rows of 32 heads
    (2, 1, 48, [129, 1], 1),              # a ragged last head block, one split
    (1, 3, 7, [640], 3),                  # 21 rows: two 16-row or one 32-row head block
])
def test_dense_tiles_agree_with_oracle_and_each_other(batch, q_len, heads, lens, ns):
    inp = gen.dense_inputs(batch, q_len, heads, lens, seed=70 + heads + ns)
    base = mla.mla_plan_force_splits(
        mla.mla_decode_plan(batch, q_len, heads, inp.total_keys, mla.sm_count()), ns)
    ro, rl = oracle.dense_decode(inp)
    outs = []
    for rpc in (16, 32):
        o, lse, _ = run_dense(inp, plan=_with_tile(base, rpc))
        compare(o, lse, ro, rl, f"dense rows_per_cta={rpc}")
        outs.append((o, lse))
    _close(outs[0][0], outs[1][0])


@pytest.mark.parametrize("tokens,heads,topk,ns", [
    (2, 64, 300, 2), (1, 64, 2048, 16), (5, 128, 777, 4), (3, 32, 129, 1),
])
def test_sparse_tiles_agree_with_oracle_and_each_other(tokens, heads, topk, ns):
    inp = gen.sparse_inputs(tokens, heads, topk, pool_rows=6000, seed=90 + ns,
                            invalid_frac=0.1)
    base = mla.mla_plan_force_splits(
        mla.mla_sparse_decode_plan(tokens, heads, topk, mla.sm_count()), ns)
    ro, rl = oracle.sparse_decode(inp)
    outs = []
    for rpc in (16, 32):
        o, lse, _ = run_sparse(inp, plan=_with_tile(base, rpc))
        compare(o, lse, ro, rl, f"sparse rows_per_cta={rpc}")
        outs.append(o)
    _close(outs[0], outs[1])


def test_planner_tile_on_small_h64_decode_matches_oracle():
    # the planner's own choice (16-row tiles for short work at 64 heads)
    inp = gen.dense_inputs(2, 1, 64, [2048, 1999], seed=5)
    o, lse, plan = run_dense(inp)
    assert plan.rows_per_cta == 16 and plan.head_blocks == 4
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, "planner tile")


@pytest.mark.parametrize("rpc", [16, 32])
def test_many_head_blocks_per_request(rpc):
    # 8 draft rows x 128 heads = 1024 rows per request: 64 or 32 head blocks,
    # ragged windows, a short request and a forced split count
    inp = gen.dense_inputs(2, 8, 128, [900, 5], seed=77 + rpc)
    base = mla.mla_plan_force_splits(
        mla.mla_decode_plan(2, 8, 128, inp.total_keys, mla.sm_count()), 3)
    plan = _with_tile(base, rpc)
    assert plan.head_blocks == 1024 // rpc
    o, lse, _ = run_dense(inp, plan=plan)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, f"1024 rows per request, rows_per_cta={rpc}")

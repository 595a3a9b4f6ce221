"""GPU: seeded random shapes against the fp64 oracle.

Each case draws a dense or sparse call at random -- batch, draft rows, heads,
ragged lengths (some empty), top-k with invalid entries, a forced split count
and, above 16 rows per request, a forced query-row tile -- and checks the
result against the oracle at the parity bar.  The draws are seeded, so a
failure names a reproducible case.
"""
import numpy as np
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


def _tile(plan, rpc):
    p = mla.mla_plan_t.from_buffer_copy(plan)
    rows = p.q_len * p.num_heads
    p.rows_per_cta = rpc
    p.head_blocks = p.grid_x = -(-rows // rpc)
    return p


def _shape_plan(plan, rng, keys):
    ns = int(rng.integers(1, min(64, max(1, keys // 64) + 2) + 1))
    p = mla.mla_plan_force_splits(plan, ns)
    rows = p.q_len * p.num_heads
    if rows > 16 and rng.random() < 0.5:
        p = _tile(p, 32 if p.rows_per_cta == 16 else 16)
    return p


@pytest.mark.parametrize("seed", range(48))
def test_random_dense_calls(seed):
    rng = np.random.default_rng(1000 + seed)
    batch = int(rng.integers(1, 6))
    q_len = int(rng.integers(1, 5))
    heads = int(rng.choice([1, 3, 8, 16, 20, 32, 48, 64, 128]))
    while q_len * heads > 256:
        q_len -= 1
    lens = [int(x) for x in rng.integers(0, 2500, size=batch)]
    lens[int(rng.integers(0, batch))] = int(rng.choice([0, 1, 127, 128, 129]))
    if sum(lens) == 0:
        lens[0] = 1   # the oracle takes a non-empty page table (empty calls: below)
    inp = gen.dense_inputs(batch, q_len, heads, lens, seed=2000 + seed,
                           extra_slots=int(rng.integers(0, 40)))
    plan = mla.mla_decode_plan(batch, q_len, heads, inp.total_keys, mla.sm_count())
    plan = _shape_plan(plan, rng, max(lens))
    o, lse, _ = run_dense(inp, plan=plan)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, f"dense seed {seed}: B={batch} q={q_len} H={heads} lens={lens} "
                            f"ns={plan.num_splits} rpc={plan.rows_per_cta}")


@pytest.mark.parametrize("seed", range(32))
def test_random_sparse_calls(seed):
    rng = np.random.default_rng(3000 + seed)
    tokens = int(rng.integers(1, 6))
    heads = int(rng.choice([16, 32, 64, 128]))
    topk = int(rng.integers(1, 900))
    inp = gen.sparse_inputs(tokens, heads, topk, pool_rows=int(rng.integers(topk, 6000)),
                            seed=4000 + seed, invalid_frac=float(rng.choice([0.0, 0.1, 0.5])))
    plan = mla.mla_sparse_decode_plan(tokens, heads, topk, mla.sm_count())
    plan = _shape_plan(plan, rng, topk)
    o, lse, _ = run_sparse(inp, plan=plan)
    ro, rl = oracle.sparse_decode(inp)
    compare(o, lse, ro, rl, f"sparse seed {seed}: T={tokens} H={heads} topk={topk} "
                            f"ns={plan.num_splits} rpc={plan.rows_per_cta}")


@pytest.mark.parametrize("batch,q_len,heads,ns", [(3, 1, 16, 1), (2, 2, 64, 4), (1, 4, 7, 2)])
def test_call_with_no_key_at_all(batch, q_len, heads, ns):
    # every request empty (an empty page table): o = 0 and lse = -inf, no error
    inp = gen.dense_inputs(batch, q_len, heads, [0] * batch, seed=5, extra_slots=4)
    assert inp.total_keys == 0
    plan = mla.mla_plan_force_splits(
        mla.mla_decode_plan(batch, q_len, heads, 0, mla.sm_count()), ns)
    ws = mla.workspace(plan)
    o, lse, _ = run_dense(inp, plan=plan, ws=ws)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    assert mla.mla_read_device_error(ws) == 0


@pytest.mark.parametrize("seed", range(16))
def test_random_second_cache_calls(seed):
    rng = np.random.default_rng(5000 + seed)
    tokens = int(rng.integers(1, 5))
    heads = int(rng.choice([16, 32, 64, 128]))
    topk = int(rng.integers(0, 700))
    extra = int(rng.integers(1 if topk == 0 else 0, 300))
    rows = int(rng.integers(max(topk, 1), 5000))
    xrows = int(rng.integers(max(extra, 1), 3000))
    inp = gen.sparse_extra_inputs(tokens, heads, topk, extra, rows, xrows, seed=6000 + seed,
                                  invalid_frac=float(rng.choice([0.0, 0.2])))
    plan = mla.mla_sparse_decode_plan(tokens, heads, topk, mla.sm_count(), extra_topk=extra)
    plan = _shape_plan(plan, rng, topk + extra)
    o, lse = mla.mla_sparse_decode_extra(plan, inp.q_nope.cuda(), inp.q_pe.cuda(),
                                         inp.pool.cuda(), inp.indices.cuda(),
                                         inp.extra_pool.cuda(), inp.extra_indices.cuda(),
                                         inp.scale, inp.kv_scale)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_extra_decode(inp)
    compare(o, lse, ro, rl, f"second cache seed {seed}: T={tokens} H={heads} topk={topk} "
                            f"extra={extra} ns={plan.num_splits} rpc={plan.rows_per_cta}")

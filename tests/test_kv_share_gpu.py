"""GPU: head blocks that share every gathered KV block through a thread-block
cluster and TMA multicast (plan.kv_share 2 or 4) give exactly the bits of the
unshared launch (kv_share 1) -- only the data movement differs -- and meet the
oracle.  Shapes cover 2 and 4 sharing CTAs, a ragged last head block (its rows
beyond the request are idle), empty splits, forced split counts and the sparse
path.
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


def _unshared(plan):
    p = mla.mla_plan_t.from_buffer_copy(plan)
    p.kv_share = 1
    return p


@pytest.mark.parametrize("batch,q_len,heads,lens,ns,share", [
    (2, 1, 64, [3000, 1700], 0, 2),
    (3, 4, 16, [2000, 5, 1300], 0, 2),
    (2, 1, 128, [700, 1], 0, 4),
    (1, 3, 40, [1537], 0, 4),      # 120 rows: 4 head blocks, the last one 24 rows
    (2, 1, 128, [900, 2500], 13, 4),
    (1, 1, 64, [5000], 40, 2),
])
def test_dense_shared_gather_is_bit_exact(batch, q_len, heads, lens, ns, share):
    inp = gen.dense_inputs(batch, q_len, heads, lens, seed=500 + heads + ns, extra_slots=9)
    plan = mla.mla_decode_plan(batch, q_len, heads, inp.total_keys, mla.sm_count())
    if ns:
        plan = mla.mla_plan_force_splits(plan, ns)
    assert plan.kv_share == share
    o1, l1, _ = run_dense(inp, plan=plan)
    o2, l2, _ = run_dense(inp, plan=_unshared(plan))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl = oracle.dense_decode(inp)
    compare(o1, l1, ro, rl, f"shared x{share}")


@pytest.mark.parametrize("tokens,heads,topk,share", [
    (3, 64, 2048, 2),
    (2, 128, 1024, 4),
    (5, 64, 300, 2),
])
def test_sparse_shared_gather_is_bit_exact(tokens, heads, topk, share):
    inp = gen.sparse_inputs(tokens, heads, topk, pool_rows=6000, seed=600 + heads,
                            invalid_frac=0.1)
    plan = mla.mla_sparse_decode_plan(tokens, heads, topk, mla.sm_count(), 0)
    assert plan.kv_share == share
    o1, l1, _ = run_sparse(inp, plan=plan)
    o2, l2, _ = run_sparse(inp, plan=_unshared(plan))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl = oracle.sparse_decode(inp)
    compare(o1, l1, ro, rl, f"sparse shared x{share}")


def test_shared_gather_bad_slot_is_reported_once_and_skipped():
    inp = gen.dense_inputs(2, 1, 64, [400, 300], seed=31)
    plan = mla.mla_decode_plan(2, 1, 64, inp.total_keys, mla.sm_count())
    assert plan.kv_share == 2
    ws = mla.workspace(plan)
    inp.kv_indices[5] = inp.pool.shape[0] + 3
    run_dense(inp, plan=plan, ws=ws)
    assert mla.mla_read_device_error(ws) == mla.MLA_DEVERR_BAD_SLOT

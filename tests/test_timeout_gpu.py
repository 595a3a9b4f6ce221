"""GPU: a pipeline wait that runs out ends the call with an error status, not a
hang or a fault, and leaves the device usable.

mla_debug_wait_limit lowers the bound of the split kernel's pipeline waits to a
few hundred cycles, so the first waits of every CTA give up while its copies and
MMAs are still in flight.  Each CTA must then stop issuing, wait (with the full
bound) for what it already issued, report MLA_DEVERR_TIMEOUT in the workspace
error word and exit; the call returns.  With the bound restored, the next call
on the same workspace (after mla_workspace_reset) matches the fp64 oracle and
reports no error.  Dense 16- and 32-row kernels and the sparse kernel, one and
several splits.
"""
import pytest
import torch

from oracle import oracle
from split_kv_mla_gb300 import inputs as gen
from split_kv_mla_gb300 import mla

from gpu_util import compare, run_dense, run_sparse

pytestmark = pytest.mark.gpu

SHORT_BOUND = 300   # SM cycles: far below any copy's latency


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    mla.load()


def _timeout_then_normal(run, inp, plan, ref):
    ws = mla.workspace(plan)
    prev = mla.mla_debug_wait_limit(SHORT_BOUND)
    try:
        run(inp, plan=plan, ws=ws)          # synchronises: the call returns
    finally:
        mla.mla_debug_wait_limit(0)
    assert prev > SHORT_BOUND
    assert mla.mla_read_device_error(ws) & mla.MLA_DEVERR_TIMEOUT
    mla.mla_workspace_reset(ws)
    o, lse, _ = run(inp, plan=plan, ws=ws)
    assert mla.mla_read_device_error(ws) == 0
    compare(o, lse, ref[0], ref[1], "after a timed-out call")


@pytest.mark.parametrize("heads,q_len,ns", [(16, 1, 0), (16, 1, 1), (64, 1, 0), (16, 4, 3)])
def test_dense_timeout_is_reported_and_the_device_stays_usable(heads, q_len, ns):
    inp = gen.dense_inputs(3, q_len, heads, [2500, 900, 1700], seed=61 + heads + ns)
    plan = mla.mla_decode_plan(inp.batch, q_len, heads, inp.total_keys, mla.sm_count())
    if ns:
        plan = mla.mla_plan_force_splits(plan, ns)
    _timeout_then_normal(run_dense, inp, plan, oracle.dense_decode(inp))


def test_sparse_timeout_is_reported_and_the_device_stays_usable():
    inp = gen.sparse_inputs(4, 64, 2048, pool_rows=9000, seed=67)
    plan = mla.mla_sparse_decode_plan(4, 64, 2048, mla.sm_count())
    _timeout_then_normal(run_sparse, inp, plan, oracle.sparse_decode(inp))


def test_default_bound_is_restored():
    prev = mla.mla_debug_wait_limit(0)
    assert mla.mla_debug_wait_limit(0) == prev
    assert prev >= 10 ** 9

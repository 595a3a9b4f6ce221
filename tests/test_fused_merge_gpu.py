"""GPU: the split-K merge fused into the split kernel (plan.merge_cluster 2 or 4).

The CTAs of a (request, head block) tile form clusters of merge_cluster
consecutive splits that merge their partials through each other's shared
memory; with several clusters per tile, the last cluster to finish merges the
clusters' results from the workspace.  Each case is checked against the fp64
oracle and against the same plan with the separate reduce kernel
(merge_cluster 1), and the arrival tickets in the workspace header must be back
at zero after every call.
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


def _with(plan, ns=None, mc=None):
    p = mla.mla_plan_force_splits(plan, ns) if ns else mla.mla_plan_t.from_buffer_copy(plan)
    if mc is not None:
        p.merge_cluster = mc
    return p


def _tickets_clear(ws):
    head = ws[:mla.MLA_WORKSPACE_HEADER_BYTES].view(torch.int32)
    return int(head[64:].abs().sum().item()) == 0


@pytest.mark.parametrize("batch,q_len,heads,lens,ns,mc", [
    (8, 1, 16, [4096] * 8, 16, 4),       # c1-like: four clusters per tile
    (8, 1, 16, [4096] * 8, 4, 4),        # one cluster per tile
    (3, 1, 16, [2000, 37, 1500], 8, 2),  # clusters of two, a short request
    (2, 4, 16, [3000, 900], 8, 4),       # draft rows on the 32-row kernel
    (2, 1, 64, [5000, 128], 8, 4),       # two head blocks, empty splits
    (1, 1, 128, [6000], 4, 2),           # four head blocks
    (2, 1, 5, [700, 1], 4, 4),           # ragged head block, a one-key request
    (1, 1, 16, [300], 16, 4),            # more splits than blocks
])
def test_dense_fused_merge_matches_oracle_and_reduce(batch, q_len, heads, lens, ns, mc):
    inp = gen.dense_inputs(batch, q_len, heads, lens, seed=800 + ns + mc, extra_slots=5)
    base = mla.mla_decode_plan(batch, q_len, heads, inp.total_keys, mla.sm_count())
    fused = _with(base, ns, mc)
    assert fused.merge_cluster == mc
    ws = mla.workspace(fused)
    o1, l1, _ = run_dense(inp, plan=fused, ws=ws)
    assert _tickets_clear(ws)
    o1b, l1b, _ = run_dense(inp, plan=fused, ws=ws)       # the same workspace again
    assert torch.equal(o1, o1b) and torch.equal(l1, l1b)
    assert _tickets_clear(ws)
    assert mla.mla_read_device_error(ws) == 0
    o2, l2, _ = run_dense(inp, plan=_with(fused, mc=1))
    ro, rl = oracle.dense_decode(inp)
    compare(o1, l1, ro, rl, f"fused ns={ns} mc={mc}")
    compare(o2, l2, ro, rl, f"reduce ns={ns}")
    d = (o1.float() - o2.float()).abs().max().item()
    assert d <= 2 ** -7, d


@pytest.mark.parametrize("tokens,heads,topk,ns,mc", [
    (1, 64, 2048, 16, 4), (8, 64, 2048, 8, 4), (3, 64, 300, 2, 2), (2, 16, 1024, 8, 2),
])
def test_sparse_fused_merge(tokens, heads, topk, ns, mc):
    inp = gen.sparse_inputs(tokens, heads, topk, pool_rows=8000, seed=900 + ns,
                            invalid_frac=0.1)
    base = mla.mla_sparse_decode_plan(tokens, heads, topk, mla.sm_count())
    plan = _with(base, ns, mc)
    ws = mla.workspace(plan)
    o, lse, _ = run_sparse(inp, plan=plan, ws=ws)
    assert _tickets_clear(ws)
    ro, rl = oracle.sparse_decode(inp)
    compare(o, lse, ro, rl, f"sparse fused ns={ns} mc={mc}")


def test_dcp_fp32_share_through_the_fused_merge():
    inp = gen.dense_inputs(2, 2, 16, [1900, 1300], seed=33)
    from split_kv_mla_gb300 import dcp
    d = {k: getattr(inp, k).cuda() for k in ("seq_lens", "kv_indices", "kv_indptr")}
    sl, si, sp, glen = dcp.shard_page_table(d["seq_lens"], d["kv_indices"], d["kv_indptr"], 1, 2)
    plan = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, si.numel(), mla.sm_count())
    plan = _with(plan, 8, 4)
    o, lse = mla.mla_decode_dcp(plan, inp.q_lat.cuda(), inp.q_pe.cuda(), inp.pool.cuda(), sl, si,
                                sp, inp.scale, inp.kv_scale, glen, 1, 2, out_dtype=torch.float32)
    p1 = _with(plan, mc=1)
    o2, l2 = mla.mla_decode_dcp(p1, inp.q_lat.cuda(), inp.q_pe.cuda(), inp.pool.cuda(), sl, si,
                                sp, inp.scale, inp.kv_scale, glen, 1, 2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (o - o2).abs().max().item() <= 1e-5
    fin = torch.isfinite(l2)
    assert torch.equal(torch.isfinite(lse), fin)
    assert (lse[fin] - l2[fin]).abs().max().item() <= 1e-5


def test_planner_keeps_the_reduce_kernel():
    # measured on GB300 the fused merge never beat the reduce kernel
    for args in [(8, 1, 16, 8 * 8192), (1, 1, 16, 256), (64, 1, 128, 64 * 16896),
                 (2, 2, 16, 1400), (1, 1, 64, 131072)]:
        plan = mla.mla_decode_plan(*args, mla.sm_count())
        assert plan.merge_cluster == 1, args
        assert mla.mla_plan_force_splits(plan, 4).merge_cluster == 1


def test_graph_replay_of_the_fused_merge():
    inp = gen.workload_c1(q_len=1, seq=2048)
    base = mla.mla_decode_plan(8, 1, 16, inp.total_keys, mla.sm_count())
    plan = _with(base, 16, 4)
    o_ref, l_ref, _ = run_dense(inp, plan=plan)
    d = {k: getattr(inp, k).cuda() for k in ("q_lat", "q_pe", "pool", "seq_lens", "kv_indices",
                                               "kv_indptr")}
    o = torch.empty_like(d["q_lat"])
    lse = torch.empty(o.shape[0], o.shape[1], dtype=torch.float32, device="cuda")
    ws = mla.workspace(plan)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                mla.mla_decode(plan, d["q_lat"], d["q_pe"], d["pool"], d["seq_lens"],
                               d["kv_indices"], d["kv_indptr"], inp.scale, inp.kv_scale,
                               o_lat=o, lse=lse, workspace_t=ws, stream=s)
    for _ in range(4):
        o.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert _tickets_clear(ws)

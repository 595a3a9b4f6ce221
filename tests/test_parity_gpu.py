"""GPU parity: libmla (through its C ABI) against the fp64 oracle.

Small and mid-size cases are compared element by element; the full-size
workloads are compared on sampled (row, head) items that the oracle computes
one by one, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from split_kv_mla_gb300 import inputs as gen
from split_kv_mla_gb300 import mla

from gpu_util import compare, run_dense, run_sparse, sample_items

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    mla.load()


# ---- dense: element-by-element --------------------------------------------------

def test_c0_single_request():
    inp = gen.workload_c0()
    o, lse, _ = run_dense(inp)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, "c0")


@pytest.mark.parametrize("q_len", [1, 4])
def test_c1_full_size(q_len):
    inp = gen.workload_c1(q_len=q_len)
    o, lse, plan = run_dense(inp)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, f"c1 q_len={q_len} ns={plan.num_splits}")


@pytest.mark.parametrize("batch,q_len,heads,lens", [
    (1, 1, 1, [1]),
    (2, 1, 16, [129, 127]),
    (3, 2, 5, [0, 1, 300]),
    (4, 4, 16, [3, 4, 5, 1000]),
    (2, 7, 3, [6, 530]),
    (5, 1, 64, [128, 256, 383, 1, 2049]),
    (2, 1, 128, [700, 1]),
    (1, 3, 40, [1537]),
])
def test_dense_ragged_shapes(batch, q_len, heads, lens):
    inp = gen.dense_inputs(batch, q_len, heads, lens, seed=100 + batch * 7 + q_len,
                           extra_slots=17)
    o, lse, plan = run_dense(inp)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, f"ragged {batch}x{q_len}x{heads} {lens} ns={plan.num_splits}")


def test_variable_length_batch_small():
    lens = gen.variable_lengths(12, 1, 3000, seed=5)
    inp = gen.dense_inputs(12, 1, 128, lens, seed=6)
    o, lse, _ = run_dense(inp)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, "varlen small")


# ---- dense: full-size sampled ------------------------------------------------------

@pytest.mark.parametrize("batch,seq", [(1, 131072), (2, 65536), (8, 131072), (16, 131072)])
def test_c2_split_heavy_sampled(batch, seq):
    inp = gen.workload_c2(batch, seq)
    o, lse, plan = run_dense(inp)
    items = sample_items(batch * 64, 24, seed=batch)
    ro, rl = oracle.dense_decode(inp, items)
    o_s = o.reshape(-1, 512)[torch.as_tensor(items, device=o.device)]
    l_s = lse.reshape(-1)[torch.as_tensor(items, device=o.device)]
    compare(o_s, l_s, ro, rl, f"c2 ({batch},{seq}) ns={plan.num_splits}")


def test_c3_variable_length_sampled():
    inp = gen.workload_c3()
    o, lse, plan = run_dense(inp)
    items = sample_items(64 * 128, 48, seed=3)
    ro, rl = oracle.dense_decode(inp, items)
    idx = torch.as_tensor(items, device=o.device)
    compare(o.reshape(-1, 512)[idx], lse.reshape(-1)[idx], ro, rl, f"c3 ns={plan.num_splits}")
    assert torch.isfinite(lse).all()


# ---- sparse ----------------------------------------------------------------------------

@pytest.mark.parametrize("tokens", [1, 8])
def test_c4_sparse_full(tokens):
    inp = gen.workload_c4(tokens)
    o, lse, plan = run_sparse(inp)
    ro, rl = oracle.sparse_decode(inp)
    compare(o, lse, ro, rl, f"c4 T={tokens} ns={plan.num_splits}")


@pytest.mark.parametrize("tokens", [24, 64])
def test_c4_sparse_sampled(tokens):
    inp = gen.workload_c4(tokens)
    o, lse, plan = run_sparse(inp)
    items = sample_items(tokens * 64, 32, seed=tokens)
    ro, rl = oracle.sparse_decode(inp, items)
    idx = torch.as_tensor(items, device=o.device)
    compare(o.reshape(-1, 448)[idx], lse.reshape(-1)[idx], ro, rl, f"c4 T={tokens}")


def test_sparse_invalid_entries_and_small_topk():
    inp = gen.sparse_inputs(5, 64, 300, pool_rows=4000, seed=9, invalid_frac=0.25)
    inp.indices[3, :] = -1
    o, lse, _ = run_sparse(inp)
    ro, rl = oracle.sparse_decode(inp)
    compare(o, lse, ro, rl, "sparse invalid")
    assert torch.all(o[3] == 0) and torch.all(torch.isneginf(lse[3]))


def test_sparse_forced_single_split():
    inp = gen.workload_c4(2)
    o, lse, plan = run_sparse(inp, max_splits=1)
    assert plan.num_splits == 1
    ro, rl = oracle.sparse_decode(inp)
    compare(o, lse, ro, rl, "sparse ns=1")


# ---- invariants ----------------------------------------------------------------------------

def test_deterministic_run_to_run():
    inp = gen.workload_c1(q_len=4, seq=3000)
    o1, l1, _ = run_dense(inp)
    o2, l2, _ = run_dense(inp)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_long_first_ordering_is_bit_exact():
    # variable lengths over more CTAs than one wave: serving the longest
    # requests first must not change a single bit
    lens = gen.variable_lengths(48, 16, 3000, seed=8)
    inp = gen.dense_inputs(48, 1, 128, lens, seed=8)
    plan = mla.mla_decode_plan(inp.batch, 1, 128, inp.total_keys, mla.sm_count())
    assert plan.long_first == 1
    o1, l1, _ = run_dense(inp, plan=plan)
    plan.long_first = 0
    o2, l2, _ = run_dense(inp, plan=plan)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    sel = sample_items(48 * 128, 64, seed=2)
    ro, rl = oracle.dense_decode(inp, sel)
    compare(o1.reshape(-1, 512)[torch.as_tensor(sel)], l1.reshape(-1)[torch.as_tensor(sel)],
            ro, rl, "long first")


def test_page_table_permutation_is_bit_exact():
    inp = gen.dense_inputs(3, 2, 16, [900, 1300, 77], seed=12, extra_slots=40)
    o1, l1, _ = run_dense(inp)
    n = inp.pool.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    inp.pool = inp.pool[perm].contiguous()
    inp.kv_indices = inv[inp.kv_indices.long()].to(torch.int32)
    o2, l2, _ = run_dense(inp)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_count_does_not_change_the_answer_beyond_tolerance():
    inp = gen.workload_c1(q_len=1, seq=4096, batch=2)
    ro, rl = oracle.dense_decode(inp)
    base = mla.mla_decode_plan(2, 1, 16, inp.total_keys, mla.sm_count())
    for ns in (1, 2, 7, 32, 256):
        plan = mla.mla_plan_force_splits(base, ns)
        o, lse, _ = run_dense(inp, plan=plan)
        compare(o, lse, ro, rl, f"forced ns={ns}")


def test_masked_keys_read_no_pool_row():
    # NaN bytes (e4m3fn 0x7f) in every pool row that no key names, row 0
    # included: masked keys (past each request's length in a split's last
    # block) must not bring them in
    import dataclasses
    inp = gen.dense_inputs(3, 1, 16, [1000, 77, 600], seed=61, extra_slots=50)
    idx = inp.kv_indices.clone()
    used = torch.zeros(inp.pool.shape[0], dtype=torch.bool)
    used[idx.long()] = True
    spare = int(torch.nonzero(~used)[0])
    idx[idx == 0] = spare                      # row 0 named by no key
    used = torch.zeros_like(used)
    used[idx.long()] = True
    assert not used[0] and int((~used).sum()) == 50
    pool = inp.pool.clone()
    pool[~used] = 0x7F
    inp2 = dataclasses.replace(inp, pool=pool, kv_indices=idx)
    plan = mla.mla_plan_force_splits(
        mla.mla_decode_plan(3, 1, 16, inp.total_keys, mla.sm_count()), 3)
    o, lse, _ = run_dense(inp2, plan=plan)
    assert torch.isfinite(o.float()).all()
    ro, rl = oracle.dense_decode(inp2)
    compare(o, lse, ro, rl, "NaN bytes in unnamed rows")


def test_invalid_sparse_entries_read_no_pool_row():
    # NaN bytes in every pool row no valid entry names, row 0 included; the
    # invalid (-1) entries and a short top-k must not bring them in
    import dataclasses
    inp = gen.sparse_inputs(4, 64, 300, pool_rows=2000, seed=62, invalid_frac=0.3)
    idx = inp.indices.clone()
    used = torch.zeros(inp.pool.shape[0], dtype=torch.bool)
    used[idx[idx >= 0].long()] = True
    spare = int(torch.nonzero(~used)[0])
    idx[idx == 0] = spare
    used = torch.zeros_like(used)
    used[idx[idx >= 0].long()] = True
    assert not used[0] and int((idx < 0).sum()) > 0
    pool = inp.pool.clone()
    pool[~used] = 0x7F
    inp2 = dataclasses.replace(inp, pool=pool, indices=idx)
    o, lse, _ = run_sparse(inp2)
    assert torch.isfinite(o.float()).all()
    ro, rl = oracle.sparse_decode(inp2)
    compare(o, lse, ro, rl, "NaN bytes in unnamed rows, sparse")


@pytest.mark.parametrize("rows,ns,d_v", [
    (37, 19, 512),     # four split groups (above 16 splits)
    (37, 7, 512),      # one group
    (300, 12, 512),    # above 8 splits but more than 128 rows: one group
    (120, 12, 448),    # above 8 splits, at most 128 rows: four groups
    (5, 65, 512),      # four groups, past the first 64 splits' loads
    (3, 256, 504),     # the largest split count; columns not a multiple of 512
    (4, 9, 8),         # four groups over a narrow row
])
def test_splitk_reduce_matches_oracle_merge(rows, ns, d_v):
    g = torch.Generator().manual_seed(4 + ns)
    parts = torch.randn(rows, ns, d_v, generator=g)
    lses = torch.randn(rows, ns, generator=g) * 6
    lses[min(3, rows - 1), :] = -float("inf")        # a row with no key at all
    if rows > 5:
        lses[5, 2:] = -float("inf")
    o, l = mla.mla_splitk_reduce(parts.cuda(), lses.cuda(), out_scale=0.25)
    torch.cuda.synchronize()
    ro = np.zeros((rows, d_v))
    rl = np.zeros(rows)
    for r in range(rows):
        ro[r], rl[r] = oracle.merge(parts[r].double().numpy(), lses[r].double().numpy(), 0.25)
    compare(o, l, ro, rl, "reduce")


def test_cuda_graph_replay_matches_eager():
    inp = gen.workload_c1(q_len=1, seq=2048)
    o_ref, l_ref, plan = run_dense(inp)
    d = {k: v.cuda() for k, v in dict(
        q_lat=inp.q_lat, q_pe=inp.q_pe, pool=inp.pool, seq_lens=inp.seq_lens,
        kv_indices=inp.kv_indices, kv_indptr=inp.kv_indptr).items()}
    o = torch.empty_like(d["q_lat"])
    lse = torch.empty(o.shape[0], o.shape[1], dtype=torch.float32, device="cuda")
    ws = mla.workspace(plan)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mla.mla_decode(plan, d["q_lat"], d["q_pe"], d["pool"], d["seq_lens"],
                           d["kv_indices"], d["kv_indptr"], inp.scale, inp.kv_scale,
                           o_lat=o, lse=lse, workspace_t=ws, stream=s)
    for _ in range(3):
        o.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


# ---- device error word ---------------------------------------------------------------------

def test_bad_slot_sets_error_word_without_fault():
    inp = gen.dense_inputs(2, 1, 16, [300, 200], seed=13)
    plan = mla.mla_decode_plan(2, 1, 16, inp.total_keys, mla.sm_count())
    ws = mla.workspace(plan)
    inp.kv_indices[7] = inp.pool.shape[0] + 5   # out of range: skipped, flagged
    run_dense(inp, plan=plan, ws=ws)
    assert mla.mla_read_device_error(ws) & mla.MLA_DEVERR_BAD_SLOT
    mla.mla_workspace_reset(ws)
    assert mla.mla_read_device_error(ws) == 0
    # the context is still usable
    good = gen.workload_c0()
    o, lse, _ = run_dense(good)
    ro, rl = oracle.dense_decode(good)
    compare(o, lse, ro, rl, "after bad slot")


def test_bad_length_sets_error_word():
    inp = gen.dense_inputs(2, 1, 16, [30, 20], seed=14)
    inp.seq_lens[1] = 25   # longer than its kv_indptr range
    plan = mla.mla_decode_plan(2, 1, 16, inp.total_keys, mla.sm_count())
    ws = mla.workspace(plan)
    run_dense(inp, plan=plan, ws=ws)
    assert mla.mla_read_device_error(ws) & mla.MLA_DEVERR_BAD_LENGTH


def test_rejects_cpu_tensors():
    inp = gen.workload_c0()
    plan = mla.mla_decode_plan(1, 1, 16, 256, mla.sm_count())
    with pytest.raises(ValueError):
        mla.mla_decode(plan, inp.q_lat, inp.q_pe, inp.pool, inp.seq_lens, inp.kv_indices,
                       inp.kv_indptr, inp.scale, inp.kv_scale)

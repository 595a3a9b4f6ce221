"""Decode context parallelism on the GPU (moonmath-ai/amd-kernels README, "MLA
absorbed decode" and "Use / MLA decode"): every rank's share from
``mla_decode_dcp`` against the oracle's share, and the shares merged by
``mla_dcp_lse_merge_ranks`` against the oracle's UNSHARDED decode.  One GPU
holds every rank: the ranks run one after another (no rank waits on another),
and their shares are stacked rank-major as an all-gather would leave them.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from split_kv_mla_gb300 import dcp
from split_kv_mla_gb300 import inputs as gen
from split_kv_mla_gb300 import mla

from gpu_util import LSE_ABS, O_MAX_ABS, O_REL_RMS, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    mla.load()


def _rank_share(inp, d, k, world, dtype=torch.float32, splits=None):
    sl, si, sp, glen = dcp.shard_page_table(d["seq_lens"], d["kv_indices"], d["kv_indptr"],
                                            k, world)
    plan = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, si.numel(), mla.sm_count())
    if splits is not None:
        plan = mla.mla_plan_force_splits(plan, splits)
    o, lse = mla.mla_decode_dcp(plan, d["q_lat"], d["q_pe"], d["pool"], sl, si, sp,
                                inp.scale, inp.kv_scale, glen, k, world, out_dtype=dtype)
    return o, lse, plan


def _compare_double_rounded(o, lse, ro, rl, what):
    """bf16 shares are rounded once before the merge and once after it, so the
    max-abs bar grows by half a bf16 ulp of the largest output, 2^-8 max|o|;
    the relative-RMS and LSE bars are unchanged."""
    on = o.float().cpu().double().numpy().reshape(ro.shape)
    ln = lse.cpu().double().numpy().reshape(rl.shape)
    diff = on - ro
    bound = O_MAX_ABS + 2.0 ** -8 * float(np.max(np.abs(ro)))
    assert float(np.max(np.abs(diff))) <= bound, what
    assert float(np.sqrt(np.mean(diff ** 2)) / np.sqrt(np.mean(ro ** 2))) <= O_REL_RMS, what
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(ln), fin), what
    assert float(np.max(np.abs(ln[fin] - rl[fin]))) <= LSE_ABS, what


def _to_cuda(inp):
    return dict(q_lat=inp.q_lat.cuda(), q_pe=inp.q_pe.cuda(), pool=inp.pool.cuda(),
                seq_lens=inp.seq_lens.cuda(), kv_indices=inp.kv_indices.cuda(),
                kv_indptr=inp.kv_indptr.cuda())


@pytest.mark.parametrize("batch,q_len,heads,lens,world", [
    (2, 1, 16, [1000, 37], 2),
    (3, 4, 16, [4097, 5, 2], 3),
    (1, 4, 64, [8192], 4),
    (4, 2, 128, [513, 1, 0, 300], 2),
    (2, 1, 16, [20000, 3], 8),
    (8, 4, 16, [8192] * 8, 2),
])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rank_shares_and_their_merge(batch, q_len, heads, lens, world, dtype):
    inp = gen.dense_inputs(batch, q_len, heads, lens, seed=200 + world * 3 + q_len,
                           extra_slots=11)
    d = _to_cuda(inp)
    parts, lses = [], []
    for k in range(world):
        o, lse, plan = _rank_share(inp, d, k, world, dtype)
        torch.cuda.synchronize()
        assert o.dtype == dtype
        shard, glen = oracle.dcp_shard(inp, k, world)
        ro, rl = oracle.dcp_decode(shard, glen, k, world)
        compare(o, lse, ro, rl, f"rank {k}/{world} ns={plan.num_splits}")
        parts.append(o)
        lses.append(lse)
    parts, lses = torch.stack(parts), torch.stack(lses)
    mo, ml = mla.mla_dcp_lse_merge_ranks(parts, lses)
    torch.cuda.synchronize()
    ro, rl = oracle.dense_decode(inp)
    if dtype == torch.float32:
        compare(mo, ml, ro, rl, f"merged world={world}")
    else:
        _compare_double_rounded(mo, ml, ro, rl, f"merged bf16 shares world={world}")
    # the merge alone, against the oracle merge of exactly these shares
    po, pl = oracle.dcp_merge_ranks(parts.double().cpu().numpy(), lses.double().cpu().numpy())
    compare(mo, ml, po, pl, f"merge of the GPU shares world={world}")


@pytest.mark.parametrize("splits", [1, 3])
def test_fp32_share_with_forced_splits(splits):
    # one split writes the fp32 share from the split kernel itself; several go
    # through the split-K reduce's fp32 output
    inp = gen.dense_inputs(3, 4, 16, [700, 9, 2], seed=31 + splits, extra_slots=7)
    d = _to_cuda(inp)
    for k in range(2):
        o, lse, plan = _rank_share(inp, d, k, 2, torch.float32, splits=splits)
        torch.cuda.synchronize()
        assert plan.num_splits == splits
        shard, glen = oracle.dcp_shard(inp, k, 2)
        ro, rl = oracle.dcp_decode(shard, glen, k, 2)
        compare(o, lse, ro, rl, f"fp32 share rank {k} ns={splits}")


def test_one_rank_is_bit_identical_to_mla_decode():
    inp = gen.dense_inputs(3, 4, 16, [700, 3, 1500], seed=17, extra_slots=5)
    d = _to_cuda(inp)
    plan = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, inp.total_keys,
                               mla.sm_count())
    o_ref, l_ref = mla.mla_decode(plan, d["q_lat"], d["q_pe"], d["pool"], d["seq_lens"],
                                  d["kv_indices"], d["kv_indptr"], inp.scale, inp.kv_scale)
    for glen in (d["seq_lens"].clone(), None):
        o, lse = mla.mla_decode_dcp(plan, d["q_lat"], d["q_pe"], d["pool"], d["seq_lens"],
                                    d["kv_indices"], d["kv_indptr"], inp.scale, inp.kv_scale,
                                    glen, 0, 1)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("world", [1, 5, 16, 17, 40])
def test_merge_kernel_against_the_oracle_merge(world, dtype):
    g = torch.Generator().manual_seed(world)
    rows, d_v = 45, 512
    # shares of the magnitude decode outputs have (|o| < 2, where half a bf16
    # ulp of the merged output stays below the max-abs bar)
    parts = (torch.randn(world, rows, d_v, generator=g) * 0.25).to(dtype)
    lses = torch.randn(world, rows, generator=g) * 8
    lses[:, 3] = -float("inf")            # no rank saw a key
    lses[1:, 7] = -float("inf")           # only rank 0 did
    o, l = mla.mla_dcp_lse_merge_ranks(parts.cuda(), lses.cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.dcp_merge_ranks(parts.double().numpy(), lses.double().numpy())
    compare(o, l, ro, rl, f"merge world={world}")
    assert torch.all(o[3] == 0)
    # weight 1 on rank 0 and 0 elsewhere: rank 0's row, rounded to bf16
    assert torch.equal(o[7].cpu(), parts[0, 7].to(torch.bfloat16))


def test_merge_keeps_leading_row_dims():
    parts = torch.randn(3, 2, 4, 16, 512, device="cuda").to(torch.bfloat16)
    lses = torch.randn(3, 2, 4, 16, device="cuda")
    o, l = mla.mla_dcp_lse_merge_ranks(parts, lses)
    assert o.shape == (2, 4, 16, 512) and l.shape == (2, 4, 16)


def test_dcp_rejections():
    inp = gen.dense_inputs(1, 1, 16, [64], seed=3)
    d = _to_cuda(inp)
    plan = mla.mla_decode_plan(1, 1, 16, inp.total_keys, mla.sm_count())
    args = (plan, d["q_lat"], d["q_pe"], d["pool"], d["seq_lens"], d["kv_indices"],
            d["kv_indptr"], inp.scale, inp.kv_scale)
    with pytest.raises(mla.MlaError):       # DCP needs glen whenever cp_world > 1
        mla.mla_decode_dcp(*args, None, 0, 2)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_dcp(*args, d["seq_lens"], 2, 2)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_dcp(*args, d["seq_lens"], 0, 0)
    with pytest.raises(ValueError):          # only bf16 and fp32 shares
        mla.mla_decode_dcp(*args, d["seq_lens"], 0, 2, out_dtype=torch.float16)
    bad = torch.zeros(2, 5, 100, dtype=torch.bfloat16, device="cuda")   # d_v not a multiple of 8
    with pytest.raises(mla.MlaError):
        mla.mla_dcp_lse_merge_ranks(bad, torch.zeros(2, 5, device="cuda"))


def test_splits_then_reduce_equals_the_one_call():
    inp = gen.dense_inputs(2, 4, 16, [3000, 900], seed=23, extra_slots=3)
    d = _to_cuda(inp)
    sl, si, sp, glen = dcp.shard_page_table(d["seq_lens"], d["kv_indices"], d["kv_indptr"], 1, 2)
    plan = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, si.numel(), mla.sm_count())
    plan = mla.mla_plan_force_splits(plan, 4)
    # the one call with the separate reduce is exactly split kernel + reduce
    # (a fused merge associates the same terms differently)
    plan.merge_cluster = 1
    args = (plan, d["q_lat"], d["q_pe"], d["pool"], sl, si, sp, inp.scale, inp.kv_scale,
            glen, 1, 2)
    ws = mla.workspace(plan)
    o1, l1 = mla.mla_decode_dcp(*args, workspace_t=ws, out_dtype=torch.float32)
    mla.mla_decode_dcp_splits(*args, workspace_t=ws, out_dtype=torch.float32)
    op, lp = mla.mla_workspace_partials(plan, ws)
    o2, l2 = mla.mla_splitk_reduce(op, lp, out_scale=inp.kv_scale)
    torch.cuda.synchronize()
    assert torch.equal(o2, o1.reshape(o2.shape).to(torch.bfloat16))
    assert torch.equal(l2, l1.reshape(-1))

"""The no-allocation dense decode entry point, through the C ABI.

Callers that cannot allocate device memory (no cudaMalloc available or allowed
where they run) use mla_decode_noalloc, whose scratch is a static array inside
the library.  Its output must match mla_decode's, within the parity tolerances,
on two calls in a row (the second call finds the first call's leftovers in the
shared scratch).  This file is collected last so that a run stopping at the
first failure has run every other test before it.
"""
import pytest
import torch

from split_kv_mla_gb300 import inputs as gen
from split_kv_mla_gb300 import mla

from gpu_util import O_MAX_ABS, O_REL_RMS, LSE_ABS

pytestmark = pytest.mark.gpu


def _close(o, l, o_ref, l_ref):
    d = (o.float() - o_ref.float())
    assert torch.isfinite(o.float()).all()
    assert d.abs().max().item() <= O_MAX_ABS
    rms = d.pow(2).mean().sqrt() / o_ref.float().pow(2).mean().sqrt()
    assert rms.item() <= O_REL_RMS
    fin = torch.isfinite(l_ref)
    assert torch.equal(torch.isfinite(l), fin)
    if fin.any():
        assert (l[fin] - l_ref[fin]).abs().max().item() <= LSE_ABS


def _device(inp):
    return [t.cuda() for t in (inp.q_lat, inp.q_pe, inp.pool, inp.seq_lens, inp.kv_indices,
                               inp.kv_indptr)]


def test_noalloc_matches_mla_decode_on_two_calls_in_a_row():
    mla.load()
    sms = mla.sm_count()
    cases = [gen.workload_c1(q_len=1, seq=4096, seed=21),
             gen.dense_inputs(3, 4, 16, [2000, 35, 999], seed=22)]
    runs = []
    for inp in cases:  # references from mla_decode first
        plan = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, inp.total_keys, sms)
        assert plan.num_splits > 1  # the scratch holds partials
        assert plan.workspace_bytes <= mla.MLA_NOALLOC_SCRATCH_BYTES
        args = _device(inp)
        o_ref, l_ref = mla.mla_decode(plan, *args, inp.scale, inp.kv_scale)
        runs.append((inp, plan, args, o_ref, l_ref))
    torch.cuda.synchronize()
    outs = []
    for inp, plan, args, o_ref, l_ref in runs:  # then two no-alloc calls back to back
        o = torch.empty_like(o_ref)
        l = torch.empty_like(l_ref)
        mla.mla_decode_noalloc(plan, *args, inp.scale, inp.kv_scale, o, l)
        outs.append((o, l))
    torch.cuda.synchronize()
    for (o, l), (_, _, _, o_ref, l_ref) in zip(outs, runs):
        _close(o, l, o_ref, l_ref)


def test_noalloc_rejects_plans_beyond_its_scratch():
    mla.load()
    inp = gen.workload_c0()
    q_lat, q_pe, pool, lens, idx, ptr = _device(inp)
    o = torch.empty_like(q_lat)
    # a shape whose partials need more than the scratch holds
    big = mla.mla_plan_force_splits(mla.mla_decode_plan(64, 1, 128, 64 * 4096, mla.sm_count()),
                                    256)
    assert big.workspace_bytes > mla.MLA_NOALLOC_SCRATCH_BYTES
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_noalloc(big, q_lat, q_pe, pool, lens, idx, ptr, inp.scale,
                               inp.kv_scale, o)
    assert e.value.status == -4
    # a plan whose workspace_bytes field was edited down is judged by its shape,
    # not by the field: still too big for the scratch
    big.workspace_bytes = 1024
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_noalloc(big, q_lat, q_pe, pool, lens, idx, ptr, inp.scale,
                               inp.kv_scale, o)
    assert e.value.status == -4

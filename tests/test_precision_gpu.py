"""GPU parity at the edges of the kernel's number formats.

The split kernel feeds the tensor cores e4m3 operands only: each query row and
each probability enters the MMA as two e4m3 terms (a high part and a scaled
residual).  These inputs put numbers where such a pair is weakest, and check
the result against the fp64 oracle with the same bar as every other parity
test (max-abs 1e-2 and relative RMS 5e-3 on o, 1e-3 on the base-2 LSE):

* one query row spanning a wide dynamic range: a single column 2^8, 2^10 or
  2^12 times the others, in the latent or the RoPE part; the RoPE part 32x
  larger or smaller than the latent part; a latent part near zero;
* softmax shapes: queries scaled x30 (sharply peaked), keys that are nearly
  identical (nearly tied logits), and one key whose logit exceeds the rest by
  about 12, 17, 21, 26 and 52 (base 2), so that every other key's weight
  falls deep into the small-number range of the probability pair.

Each case runs on the 16-row kernel (H=16), the 32-row kernel (H=64, and H=16
with four draft rows) and, for the query cases, the sparse path.
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


QUERY_CASES = {
    "outlier-lat-2^8": lambda i: gen.plant_query_outliers(i, 2.0 ** 8, 1),
    "outlier-lat-2^10": lambda i: gen.plant_query_outliers(i, 2.0 ** 10, 2),
    "outlier-lat-2^12": lambda i: gen.plant_query_outliers(i, 2.0 ** 12, 3),
    "outlier-pe-2^10": lambda i: gen.plant_query_outliers(i, 2.0 ** 10, 4, part="pe"),
    "outlier-pe-2^12": lambda i: gen.plant_query_outliers(i, 2.0 ** 12, 5, part="pe"),
    "pe-x32": lambda i: gen.scale_query_parts(i, pe=32.0),
    "pe-x1/32": lambda i: gen.scale_query_parts(i, pe=1.0 / 32),
    "lat-near-zero": lambda i: gen.scale_query_parts(i, lat=2.0 ** -10),
    "sharp-x30": lambda i: gen.scale_query_parts(i, lat=30.0, pe=30.0),
}

KEY_CASES = {
    "near-tied": lambda i: gen.near_tied_pool(i, 7),
    "dominant-0.35": lambda i: gen.plant_dominant_key(gen.share_query_across_heads(i), 0.35, 8),
    "dominant-0.5": lambda i: gen.plant_dominant_key(gen.share_query_across_heads(i), 0.5, 9),
    "dominant-0.6": lambda i: gen.plant_dominant_key(gen.share_query_across_heads(i), 0.6, 10),
    "dominant-0.75": lambda i: gen.plant_dominant_key(gen.share_query_across_heads(i), 0.75, 11),
    "dominant-1.5": lambda i: gen.plant_dominant_key(gen.share_query_across_heads(i), 1.5, 12),
}

DENSE_SHAPES = {
    "rows16": (2, 1, 16, [4000, 1700]),     # 16 query rows per CTA
    "rows32": (2, 1, 64, [3000, 900]),      # 32 query rows per CTA
    "draft4": (2, 4, 16, [2500, 1300]),     # 64 rows: draft positions on the 32-row kernel
}


def _dense(shape, seed):
    b, q, h, lens = DENSE_SHAPES[shape]
    return gen.dense_inputs(b, q, h, lens, seed=seed, extra_slots=11)


@pytest.mark.parametrize("shape", list(DENSE_SHAPES))
@pytest.mark.parametrize("case", list(QUERY_CASES) + list(KEY_CASES))
def test_dense_format_edges(shape, case):
    inp = _dense(shape, seed=40 + len(case))
    build = QUERY_CASES.get(case) or KEY_CASES[case]
    inp = build(inp)
    o, lse, plan = run_dense(inp)
    ro, rl = oracle.dense_decode(inp)
    compare(o, lse, ro, rl, f"{shape} {case} ns={plan.num_splits}")


@pytest.mark.parametrize("case", list(QUERY_CASES))
def test_sparse_format_edges(case):
    inp = gen.sparse_inputs(3, 64, 2048, pool_rows=20000, seed=70 + len(case))
    inp = QUERY_CASES[case](inp)
    o, lse, plan = run_sparse(inp)
    ro, rl = oracle.sparse_decode(inp)
    compare(o, lse, ro, rl, f"sparse {case} ns={plan.num_splits}")


def test_dense_forced_splits_with_a_dominant_key():
    # the dominant key's split outweighs the others: the merge weights then span
    # the full fp32 range
    inp = gen.plant_dominant_key(gen.share_query_across_heads(_dense("rows16", 90)), 0.75, 13)
    ro, rl = oracle.dense_decode(inp)
    base = mla.mla_decode_plan(inp.batch, inp.q_len, inp.num_heads, inp.total_keys,
                               mla.sm_count())
    for ns in (1, 5, 31):
        o, lse, _ = run_dense(inp, plan=mla.mla_plan_force_splits(base, ns))
        compare(o, lse, ro, rl, f"dominant key, ns={ns}")

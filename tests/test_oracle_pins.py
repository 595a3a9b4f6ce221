"""Pins for the fp64 oracle: each test ties it to something other than itself.

* number formats: every e4m3fn byte and every bf16 pattern against torch's own
  casts (a library routine), plus values fixed by the OCP E4M3 definition;
* softmax/LSE: an independent pure-Python brute force on tiny inputs, and
  closed forms (one key, identical keys, zero query, two keys with a known
  logit gap, a dominant key);
* split-K merge: split-count invariance and associativity
  (hip_mha_decoding_num_partitions: partitions merged by the split-K reducer;
  moonmath-ai/amd-kernels README, "Numerics": fixed merge association);
* page table: permutation invariance of pool rows (README, "Constraints /
  MLA decode": any permutation or subset of slots is legal);
* draft window: row t of a q_len=4 call equals a q_len=1 call on the request
  truncated to S - 4 + t + 1 keys (README, "Use / MLA decode");
* sparse variant: with a full index row it is the dense definition at
  448 + 64 columns; negative (invalid) entries are skipped;
* decode context parallelism (README, "Use / MLA decode", DCP): the ranks'
  shares merged equal the unsharded decode (softmax over a union of disjoint
  key sets), one rank is the plain decode, and each share equals a pure-Python
  enumeration of the rank's visible global positions.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from split_kv_mla_gb300 import inputs as gen

TOL = 1e-12


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.array_equal(a[~fin], b[~fin])
    if fin.any():
        err = np.max(np.abs(a[fin] - b[fin]) / np.maximum(1.0, np.abs(b[fin])))
        assert err <= tol, err


# ---- number formats -------------------------------------------------------------

def test_e4m3fn_every_byte_matches_torch_cast():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3fn_to_double(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])
    # signed zeros
    assert math.copysign(1.0, got[0x80]) == -1.0


@pytest.mark.parametrize("byte,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x3C, 1.5), (0x40, 2.0), (0x7E, 448.0), (0xFE, -448.0),
    (0xB8, -1.0), (0x77, 240.0)])
def test_e4m3fn_values_from_format_definition(byte, value):
    # OCP E4M3: bias 7, subnormal m*2^-9, max normal S.1111.110 = 448
    assert oracle.e4m3fn_to_double(byte) == value


def test_e4m3fn_nan_encodings():
    assert math.isnan(oracle.e4m3fn_to_double(0x7F))
    assert math.isnan(oracle.e4m3fn_to_double(0xFF))


def test_bf16_every_pattern_matches_torch_cast():
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = pats.view(torch.bfloat16).to(torch.float64).numpy()
    sample = list(range(0, 65536, 7)) + [0x0000, 0x8000, 0x3F80, 0x7F80, 0xFF80, 0x0001]
    got = np.array([oracle.bf16_to_double(h) for h in sample])
    exp = ref[np.array(sample)]
    assert np.array_equal(np.isnan(got), np.isnan(exp))
    m = ~np.isnan(exp)
    assert np.array_equal(got[m], exp[m])


# ---- brute force on tiny inputs ---------------------------------------------------

@pytest.mark.parametrize("q_len,lens,dims", [
    (1, [5, 8], (512, 64)),
    (3, [4, 7], (512, 64)),
    (2, [1, 3], (16, 8)),
    (4, [2, 6], (8, 0)),
])
def test_dense_oracle_matches_brute_force(q_len, lens, dims):
    d_v, d_r = dims
    inp = gen.dense_inputs(len(lens), q_len, 2, lens, seed=11 + q_len, d_v=d_v,
                           d_rope=d_r, extra_slots=3)
    o, lse = oracle.dense_decode(inp)
    ob, lb = oracle.brute_force_dense(inp)
    _close(o, ob)
    _close(lse, lb)


def test_sparse_oracle_matches_brute_force_with_invalid_entries():
    inp = gen.sparse_inputs(3, 2, 6, pool_rows=20, seed=5, invalid_frac=0.3)
    inp.indices[2, :] = -1  # a token with no valid entry
    o, lse = oracle.sparse_decode(inp)
    ob, lb = oracle.brute_force_sparse(inp)
    _close(o, ob)
    _close(lse, lb)
    assert np.all(o[2] == 0.0) and np.all(np.isneginf(lse[2]))


def test_selected_items_equal_full_call():
    inp = gen.dense_inputs(3, 2, 4, [9, 17, 5], seed=3)
    o, lse = oracle.dense_decode(inp)
    sel = np.array([0, 5, 7, 13, 23])
    os_, ls_ = oracle.dense_decode(inp, sel)
    R, H = 6, 4
    np.testing.assert_array_equal(os_, o.reshape(R * H, -1)[sel])
    np.testing.assert_array_equal(ls_, lse.reshape(-1)[sel])


# ---- closed forms ----------------------------------------------------------------

def _row(vals_u8, width):
    t = torch.zeros(width, dtype=torch.uint8)
    t[: len(vals_u8)] = torch.tensor(vals_u8, dtype=torch.uint8)
    return t


def test_single_key_returns_its_v_row_and_logit():
    inp = gen.dense_inputs(1, 1, 1, [1], seed=21)
    o, lse = oracle.dense_decode(inp)
    slot = int(inp.kv_indices[0])
    k = inp.pool[slot, 0].view(torch.float8_e4m3fn).to(torch.float64).numpy() * inp.kv_scale
    q = np.concatenate([inp.q_lat[0, 0].to(torch.float64).numpy(),
                        inp.q_pe[0, 0].to(torch.float64).numpy()])
    s = inp.scale * float(np.dot(q, k))
    _close(o[0, 0], k[:512])
    _close(lse[0, 0], s / math.log(2.0))


def test_identical_keys_give_that_row_and_log2_n_shift():
    n = 13
    inp = gen.dense_inputs(1, 1, 2, [n], seed=22)
    inp.pool[:] = inp.pool[int(inp.kv_indices[0])]  # every slot holds the same bytes
    o, lse = oracle.dense_decode(inp)
    k = inp.pool[0, 0].view(torch.float8_e4m3fn).to(torch.float64).numpy() * inp.kv_scale
    for h in range(2):
        q = np.concatenate([inp.q_lat[0, h].to(torch.float64).numpy(),
                            inp.q_pe[0, h].to(torch.float64).numpy()])
        s = inp.scale * float(np.dot(q, k))
        _close(o[0, h], k[:512])
        # natural-log form: LSE = ln(n) + logit
        _close(lse[0, h] * math.log(2.0), math.log(n) + s)


def test_zero_query_gives_mean_of_v_rows():
    inp = gen.dense_inputs(1, 1, 1, [10], seed=23)
    inp.q_lat.zero_()
    inp.q_pe.zero_()
    o, lse = oracle.dense_decode(inp)
    rows = inp.pool[inp.kv_indices.long(), 0].view(torch.float8_e4m3fn).to(
        torch.float64).numpy() * inp.kv_scale
    _close(o[0, 0], rows[:, :512].mean(axis=0))
    _close(lse[0, 0], math.log2(10))


def test_two_keys_with_known_logit_gap():
    # q has a single 1.0 in latent column 0, so s_j = scale * kv_scale * K_j[0].
    width = 576
    pool = torch.stack([_row([0x48, 0x38, 0xB8], width),    # K[0] = 4, V[1]=1, V[2]=-1
                        _row([0x38, 0xC0, 0x40], width)])   # K[0] = 1, V[1]=-2, V[2]=2
    q_lat = torch.zeros(512, dtype=torch.bfloat16)
    q_lat[0] = 1.0
    q_pe = torch.zeros(64, dtype=torch.bfloat16)
    scale, kv = 0.5, 0.25
    o, lse = oracle.attend(q_lat, q_pe, pool, [0, 1], scale, kv)
    gap = scale * kv * (4.0 - 1.0)
    w0 = 1.0 / (1.0 + math.exp(-gap))
    w1 = 1.0 - w0
    _close(o[0], kv * (w0 * 4.0 + w1 * 1.0))
    _close(o[1], kv * (w0 * 1.0 + w1 * -2.0))
    _close(o[2], kv * (w0 * -1.0 + w1 * 2.0))
    _close(lse, math.log2(math.exp(scale * kv * 4.0) + math.exp(scale * kv * 1.0)))


def test_dominant_key_without_overflow():
    # logits far beyond exp()'s range: result is the argmax row, LSE its logit
    width = 576
    pool = torch.stack([_row([0x7E, 0x38], width), _row([0x38, 0xC0], width)])
    q_lat = torch.zeros(512, dtype=torch.bfloat16)
    q_lat[0] = 2.0 ** 100
    q_pe = torch.zeros(64, dtype=torch.bfloat16)
    o, lse = oracle.attend(q_lat, q_pe, pool, [1, 0, 1], 1.0, 1.0)
    assert o[0] == 448.0 and o[1] == 1.0
    _close(lse, 448.0 * 2.0 ** 100 / math.log(2.0))


def test_no_key_gives_zero_and_minus_inf():
    inp = gen.dense_inputs(2, 3, 2, [0, 2], seed=24)
    o, lse = oracle.dense_decode(inp)
    # request 0 has no key at all; request 1 (S=2, q_len=3): t=0 sees 0 keys
    assert np.all(o[0:3] == 0.0) and np.all(np.isneginf(lse[0:3]))
    assert np.all(o[3] == 0.0) and np.all(np.isneginf(lse[3]))
    assert np.all(np.isfinite(lse[4:6]))


# ---- split-K merge -----------------------------------------------------------------

@pytest.mark.parametrize("ns", [1, 2, 3, 5, 8, 37, 40])
def test_split_count_invariance(ns):
    inp = gen.dense_inputs(1, 1, 1, [37], seed=31)
    full_o, full_l = oracle.attend(inp.q_lat[0, 0], inp.q_pe[0, 0], inp.pool.view(-1, 576),
                                   inp.kv_indices, inp.scale, inp.kv_scale)
    op, lp = oracle.split_partials(inp.q_lat[0, 0], inp.q_pe[0, 0], inp.pool.view(-1, 576),
                                   inp.kv_indices, inp.scale, inp.kv_scale, ns)
    if ns > 37:
        assert np.isneginf(lp[-1]) and np.all(op[-1] == 0)
    mo, ml = oracle.merge(op, lp)
    _close(mo, full_o)
    _close(ml, full_l)


def test_merge_is_associative():
    rng = np.random.default_rng(7)
    parts = rng.standard_normal((5, 32))
    lses = rng.standard_normal(5) * 4
    whole_o, whole_l = oracle.merge(parts, lses)
    a_o, a_l = oracle.merge(parts[:2], lses[:2])
    b_o, b_l = oracle.merge(parts[2:], lses[2:])
    left_o, left_l = oracle.merge(np.stack([a_o, b_o]), np.array([a_l, b_l]))
    c_o, c_l = oracle.merge(parts[1:4], lses[1:4])
    right_o, right_l = oracle.merge(np.stack([parts[0], c_o, parts[4]]),
                                    np.array([lses[0], c_l, lses[4]]))
    _close(left_o, whole_o)
    _close(left_l, whole_l)
    _close(right_o, whole_o)
    _close(right_l, whole_l)


def test_merge_closed_forms():
    a = np.array([[1.0, 2.0], [3.0, -2.0]])
    o, l = oracle.merge(a, np.array([5.0, 5.0]))
    _close(o, [2.0, 0.0])
    _close(l, 6.0)
    o, l = oracle.merge(a, np.array([-np.inf, 1.5]), out_scale=2.0)
    _close(o, [6.0, -4.0])
    _close(l, 1.5)
    o, l = oracle.merge(a, np.array([-np.inf, -np.inf]))
    assert np.all(o == 0.0) and np.isneginf(l)


# ---- page table and draft window ----------------------------------------------------

def test_pool_permutation_invariance():
    inp = gen.dense_inputs(2, 2, 3, [11, 6], seed=41, extra_slots=5)
    o, lse = oracle.dense_decode(inp)
    n = inp.pool.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    inp.pool = inp.pool[perm].contiguous()          # new row i = old row perm[i]
    inp.kv_indices = inv[inp.kv_indices.long()].to(torch.int32)
    o2, lse2 = oracle.dense_decode(inp)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_draft_window_equals_truncated_single_query():
    S, q_len = 12, 4
    inp = gen.dense_inputs(1, q_len, 2, [S], seed=51)
    o, lse = oracle.dense_decode(inp)
    for t in range(q_len):
        n = S - q_len + t + 1
        sub = gen.DenseInputs(
            batch=1, q_len=1, num_heads=2, q_lat=inp.q_lat[t:t + 1].clone(),
            q_pe=inp.q_pe[t:t + 1].clone(), pool=inp.pool,
            seq_lens=torch.tensor([n], dtype=torch.int32),
            kv_indices=inp.kv_indices[:n].clone(),
            kv_indptr=torch.tensor([0, n], dtype=torch.int32),
            scale=inp.scale, kv_scale=inp.kv_scale)
        os_, ls_ = oracle.dense_decode(sub)
        np.testing.assert_array_equal(o[t], os_[0])
        np.testing.assert_array_equal(lse[t], ls_[0])


def test_sparse_with_full_rows_is_dense_at_448_plus_64():
    inp = gen.sparse_inputs(2, 3, 9, pool_rows=30, seed=61)
    o, lse = oracle.sparse_decode(inp)
    dense = gen.DenseInputs(
        batch=2, q_len=1, num_heads=3, q_lat=inp.q_nope, q_pe=inp.q_pe,
        pool=inp.pool.view(30, 1, 512), seq_lens=torch.tensor([9, 9], dtype=torch.int32),
        kv_indices=inp.indices.reshape(-1).clone(),
        kv_indptr=torch.tensor([0, 9, 18], dtype=torch.int32),
        scale=inp.scale, kv_scale=inp.kv_scale)
    od, ld = oracle.dense_decode(dense)
    np.testing.assert_array_equal(o, od)
    np.testing.assert_array_equal(lse, ld)


# ---- rejections ------------------------------------------------------------------------

def test_out_of_range_slot_is_rejected():
    inp = gen.dense_inputs(1, 1, 1, [4], seed=71)
    inp.kv_indices[2] = inp.pool.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.dense_decode(inp)


def test_nan_byte_is_rejected():
    inp = gen.dense_inputs(1, 1, 1, [4], seed=72)
    inp.pool[int(inp.kv_indices[1]), 0, 3] = 0x7F
    with pytest.raises(oracle.OracleError):
        oracle.dense_decode(inp)


# ---- decode context parallelism -----------------------------------------------------

@pytest.mark.parametrize("q_len,world,lens", [
    (1, 2, [9, 1, 0, 6]),
    (4, 3, [11, 2, 7, 3]),
    (3, 4, [13, 5, 1, 8]),
])
def test_dcp_shares_merge_to_the_unsharded_decode(q_len, world, lens):
    inp = gen.dense_inputs(len(lens), q_len, 2, lens, seed=61 + world, extra_slots=4)
    o_ref, lse_ref = oracle.dense_decode(inp)
    parts, lses = [], []
    for k in range(world):
        shard, glen = oracle.dcp_shard(inp, k, world)
        o_k, l_k = oracle.dcp_decode(shard, glen, k, world)
        parts.append(o_k)
        lses.append(l_k)
    o, lse = oracle.dcp_merge_ranks(np.stack(parts), np.stack(lses))
    _close(o, o_ref)
    _close(lse, lse_ref)


def test_dcp_single_rank_is_the_plain_decode():
    inp = gen.dense_inputs(3, 3, 2, [10, 2, 5], seed=71)
    o_ref, lse_ref = oracle.dense_decode(inp)
    o, lse = oracle.dcp_decode(inp, inp.seq_lens.clone(), 0, 1)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, lse_ref)


@pytest.mark.parametrize("q_len,world", [(1, 2), (4, 3), (2, 5)])
def test_dcp_share_matches_brute_force(q_len, world):
    inp = gen.dense_inputs(2, q_len, 2, [9, 4], seed=81 + q_len, d_v=16, d_rope=8,
                           extra_slots=2)
    for k in range(world):
        shard, glen = oracle.dcp_shard(inp, k, world)
        o, lse = oracle.dcp_decode(shard, glen, k, world)
        ob, lb = oracle.brute_force_dcp(inp, k, world)
        _close(o, ob)
        _close(lse, lb)


def test_dcp_rank_without_visible_keys_gives_zero_and_minus_inf():
    # global length 2 with q_len 2: row 0 sees position 0 only, so rank 1 of 2
    # (positions 1, 3, ...) has nothing for row 0 and position 1 for row 1
    inp = gen.dense_inputs(1, 2, 2, [2], seed=91)
    shard, glen = oracle.dcp_shard(inp, 1, 2)
    o, lse = oracle.dcp_decode(shard, glen, 1, 2)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ---- sparse decode with a second (compressed) cache ---------------------------------

def _brute_force_sparse_extra(inp):
    main = oracle._torch_decode_rows(inp.pool)
    extra = oracle._torch_decode_rows(inp.extra_pool)
    qn = inp.q_nope.to(torch.float64).tolist()
    qp = inp.q_pe.to(torch.float64).tolist()
    T, H = inp.num_tokens, inp.num_heads
    o = np.zeros((T, H, inp.d_v))
    lse = np.zeros((T, H))
    for t in range(T):
        rows = [main[s] for s in inp.indices[t].tolist() if s >= 0]
        rows += [extra[s] for s in inp.extra_indices[t].tolist() if s >= 0]
        for h in range(H):
            o[t, h], lse[t, h] = oracle.brute_force_row(qn[t][h] + qp[t][h], rows, inp.d_v,
                                                        inp.scale, inp.kv_scale)
    return o, lse


def test_sparse_extra_matches_brute_force():
    inp = gen.sparse_extra_inputs(3, 2, 5, 3, pool_rows=12, extra_rows=7, seed=13,
                                  invalid_frac=0.25, d_v=24, d_rope=8)
    inp.indices[1, :] = -1              # a token whose candidates are all in the second cache
    inp.extra_indices[2, :] = -1        # a token whose candidates are all in the main cache
    o, lse = oracle.sparse_extra_decode(inp)
    ob, lb = _brute_force_sparse_extra(inp)
    _close(o, ob)
    _close(lse, lb)


def test_sparse_extra_with_no_valid_second_candidate_is_the_main_decode():
    inp = gen.sparse_extra_inputs(4, 3, 16, 6, pool_rows=40, extra_rows=9, seed=17)
    inp.extra_indices[:] = -1
    o, lse = oracle.sparse_extra_decode(inp)
    ro, rl = oracle.sparse_decode(inp)
    np.testing.assert_array_equal(o, ro)
    np.testing.assert_array_equal(lse, rl)


def test_sparse_extra_equals_one_cache_holding_the_same_rows():
    # the second cache holds copies of main-pool rows; pointing at the copies
    # must equal listing the originals after the main candidates
    inp = gen.sparse_extra_inputs(3, 2, 8, 5, pool_rows=30, extra_rows=5, seed=19)
    src = torch.tensor([3, 17, 29, 0, 11])
    inp.extra_pool = inp.pool[src].clone()
    perm = torch.tensor([[4, 0, 2, 1, 3], [1, 1, 0, 4, 2], [3, -1, 2, 0, -1]], dtype=torch.int32)
    inp.extra_indices = perm
    o, lse = oracle.sparse_extra_decode(inp)
    orig = torch.where(perm >= 0, src[perm.clamp(min=0).long()].to(torch.int32),
                       torch.full_like(perm, -1))
    one = gen.SparseInputs(num_tokens=3, num_heads=2, topk=13, q_nope=inp.q_nope, q_pe=inp.q_pe,
                           pool=inp.pool, indices=torch.cat([inp.indices, orig], 1).contiguous(),
                           scale=inp.scale, kv_scale=inp.kv_scale)
    ro, rl = oracle.sparse_decode(one)
    np.testing.assert_array_equal(o, ro)
    np.testing.assert_array_equal(lse, rl)

"""Host-side checks of libmla that need no GPU: the library builds for sm_103a,
loads, exports every entry point its header declares, plans from shapes alone,
and rejects bad arguments before touching the device."""
import ctypes
import os
import shutil

import pytest

from split_kv_mla_gb300 import build as mla_build
from split_kv_mla_gb300 import mla

HERE = os.path.dirname(os.path.abspath(__file__))
needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mla_build.LIB):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("library not built and nvcc not available")
        mla_build.build()
    import torch  # noqa: F401  (loads libcudart for the dynamic linker)
    return mla.load()


@needs_nvcc
def test_build_is_up_to_date():
    assert os.path.exists(mla_build.build())


@needs_nvcc
def test_gather_rate_probe_builds():
    # the measurement program behind profiles/gather_rate_576B_rows.md compiles
    # for sm_103a (it runs on a GPU only)
    from split_kv_mla_gb300 import gather_rate
    assert os.path.exists(gather_rate.build())


def test_trace_tool_matches_the_trace_buffer_layout():
    # trace.py reads the traced kernel's stamp buffer with its own copy of the
    # layout constants; they must be the ones the kernel is compiled with
    import re
    from split_kv_mla_gb300 import trace
    hdr = open(os.path.join(os.path.dirname(mla_build.__file__), "csrc",
                            "mla_internal.h")).read()
    const = {m.group(1): int(m.group(2))
             for m in re.finditer(r"constexpr int (kTrace\w+) = (\d+);", hdr)}
    assert (const["kTraceSlots"], const["kTraceCtas"], const["kTraceBlockCtas"],
            const["kTraceBlocks"], const["kTraceBlockEvents"]) == (
        trace.SLOTS, trace.MAX_CTAS, trace.BLOCK_CTAS, trace.BLOCKS, trace.BLOCK_EVENTS)
    assert len(trace.EVENTS) == trace.BLOCK_EVENTS
    assert len(trace.PHASES) <= trace.SLOTS


@needs_nvcc
def test_traced_build_compiles():
    # the clock-stamped build behind the phase timelines compiles for sm_103a
    from split_kv_mla_gb300 import trace
    assert os.path.exists(trace.build_traced())


def test_every_declared_symbol_is_exported(lib):
    names = mla.declared_symbols()
    assert {"mla_decode_plan", "mla_decode", "mla_sparse_decode", "mla_splitk_reduce",
            "mla_sparse_decode_plan"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(-7, 1):
        s = mla.status_string(code)
        assert s and s != "unknown status"
    assert mla.status_string(-99) == "unknown status"


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(HERE, "golden", name)):
        line = line.split("#", 1)[0].strip()
        if line:
            rows.append([int(x) for x in line.split()])
    return rows


def test_wave_fill_rule_reproduces_printed_mi355x_sweep(lib):
    # hip_mha_decoding_num_partitions, "Phase 0 sweep": MI355X constants
    for batch, keys, heads, expected in _golden_rows("wave_fill_mi355x.txt"):
        got = mla.mla_wave_fill_splits(batch, keys, heads, 256, 32, 256, 5, 256, 16)
        assert got == expected, (batch, keys, heads, got, expected)


def test_wave_fill_small_heads_exception(lib):
    # num_heads <= 16: np = min(two_wave, pages)
    assert mla.mla_wave_fill_splits(4, 32768, 16, 256, 32, 256, 5, 256, 16) == 128
    assert mla.mla_wave_fill_splits(8, 1024, 16, 256, 32, 256, 5, 256, 16) == 4
    # bs=1 two_wave = 512 clamps to the 256 cap
    assert mla.mla_wave_fill_splits(1, 131072, 16, 256, 32, 256, 5, 256, 16) == 256


@pytest.mark.parametrize("batch,q_len,heads,keys", [
    (1, 1, 16, 256), (8, 1, 16, 8192 * 8), (8, 4, 16, 8192 * 8), (1, 1, 64, 131072),
    (2, 1, 64, 131072), (8, 1, 64, 8 * 131072), (16, 1, 64, 16 * 131072),
    (64, 1, 128, 1081344), (3, 7, 5, 10), (1, 1, 1, 0), (0, 1, 16, 0)])
def test_dense_plan_invariants(lib, batch, q_len, heads, keys):
    p = mla.mla_decode_plan(batch, q_len, heads, keys, 152)
    assert 1 <= p.num_splits <= mla.MLA_MAX_SPLITS
    assert p.head_blocks * p.rows_per_cta >= q_len * heads
    assert (p.grid_x, p.grid_y, p.grid_z) == (p.head_blocks, p.num_splits, batch)
    assert (p.batch, p.q_len, p.num_heads, p.d_v, p.d_rope, p.total_keys) == (
        batch, q_len, heads, 512, 64, keys)
    items = batch * q_len * heads
    expect = mla.MLA_WORKSPACE_HEADER_BYTES
    if p.num_splits > 1:
        def up(x):
            return -(-x // 256) * 256
        expect += up(items * p.num_splits * 512 * 4) + up(items * p.num_splits * 4)
    assert p.workspace_bytes == expect
    # a plan is a pure function of its arguments
    q = mla.mla_decode_plan(batch, q_len, heads, keys, 152)
    assert p.as_dict() == q.as_dict()


def test_force_splits_recomputes_grid_and_workspace(lib):
    p = mla.mla_decode_plan(8, 1, 16, 8 * 8192, 152)
    for ns in (1, 3, 256):
        q = mla.mla_plan_force_splits(p, ns)
        assert q.num_splits == ns and q.grid_y == ns
        items = 8 * 16
        up = lambda x: -(-x // 256) * 256  # noqa: E731
        expect = mla.MLA_WORKSPACE_HEADER_BYTES + (
            (up(items * ns * 512 * 4) + up(items * ns * 4)) if ns > 1 else 0)
        assert q.workspace_bytes == expect
    with pytest.raises(mla.MlaError):
        mla.mla_plan_force_splits(p, 0)
    with pytest.raises(mla.MlaError):
        mla.mla_plan_force_splits(p, 257)


def test_plan_rejections(lib):
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan(1, 1, 16, 10, 152, d_v=448)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan(1, 1, 129, 10, 152)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan(1, 1, 0, 10, 152)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan(1, 0, 16, 10, 152)
    with pytest.raises(mla.MlaError):
        mla.mla_sparse_decode_plan(4, 64, 2048, 152, d_v=512)


def test_plans_cap_requests_and_tokens_at_the_grid_limit(lib):
    # requests (tokens) are the split grid's z dimension, at most 65535
    assert mla.mla_decode_plan(65535, 1, 16, 65535 * 64, 152).grid_z == 65535
    assert mla.mla_sparse_decode_plan(65535, 64, 2048, 152).grid_z == 65535
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_plan(65536, 1, 16, 65536 * 64, 152)
    assert e.value.status == -2
    with pytest.raises(mla.MlaError) as e:
        mla.mla_sparse_decode_plan(65536, 64, 2048, 152)
    assert e.value.status == -2
    # a plan edited past the limit is refused before any launch
    q = mla.mla_plan_t.from_buffer_copy(mla.mla_decode_plan(4, 1, 16, 256, 152))
    q.batch = q.grid_z = 70000
    assert _call_decode(lib, q, ws_bytes=1 << 30, batch=70000) == -1


def test_sparse_plan_max_splits(lib):
    p = mla.mla_sparse_decode_plan(1, 64, 2048, 152)
    assert p.num_splits >= 1 and p.total_keys == 2048
    q = mla.mla_sparse_decode_plan(1, 64, 2048, 152, max_splits=1)
    assert q.num_splits == 1


def _call_decode(lib, plan, ptr=0x10000, ws_bytes=1 << 20, batch=1, q_len=1, heads=16):
    P = ctypes.c_void_p
    return lib.mla_decode(ctypes.byref(plan) if plan is not None else None,
                          P(ptr), P(ptr), P(ptr), 10, P(ptr), P(ptr), P(ptr), batch, q_len,
                          heads, 0.1, 1.0, P(ptr), None, P(0x100000), ws_bytes, None)


def test_decode_argument_checks_run_before_the_device(lib):
    plan = mla.mla_decode_plan(1, 1, 16, 256, 152)
    assert _call_decode(lib, None) == -1
    assert _call_decode(lib, plan, heads=8) == -1          # plan/shape mismatch
    assert _call_decode(lib, plan, ptr=0x10004) == -3      # misaligned
    assert _call_decode(lib, plan, ws_bytes=16) == -4      # workspace too small
    bad = mla.mla_decode_plan(1, 1, 16, 256, 152)
    bad.num_splits = 0
    assert _call_decode(lib, bad) == -1
    # a zero-size batch is a no-op even without a device
    empty = mla.mla_decode_plan(0, 1, 16, 0, 152)
    assert _call_decode(lib, empty, batch=0) == 0


def test_reduce_argument_checks(lib):
    P = ctypes.c_void_p
    assert lib.mla_splitk_reduce(P(0x1000), P(0x1000), 4, 0, 512, 1.0, P(0x1000), None, None) == -1
    assert lib.mla_splitk_reduce(P(0x1000), P(0x1000), 4, 257, 512, 1.0, P(0x1000), None, None) == -2
    assert lib.mla_splitk_reduce(P(0x1000), P(0x1000), 4, 2, 12, 1.0, P(0x1000), None, None) == -2
    assert lib.mla_splitk_reduce(P(0x1004), P(0x1000), 4, 2, 512, 1.0, P(0x1000), None, None) == -3
    assert lib.mla_splitk_reduce(None, None, 0, 2, 512, 1.0, None, None, None) == 0


def test_plans_use_the_tcgen05_variant(lib):
    for batch, q_len, heads, keys in [(8, 1, 16, 8 * 8192), (1, 1, 16, 131072),
                                      (64, 1, 128, 1081344), (3, 7, 5, 10)]:
        p = mla.mla_decode_plan(batch, q_len, heads, keys, 152)
        assert p.variant == 2
        assert mla.mla_plan_force_splits(p, 7).variant == 2
    assert mla.mla_sparse_decode_plan(2, 128, 1024, 152).variant == 2


def test_decode_rejects_unknown_variant(lib):
    for variant in (0, 1, 3, 4):
        plan = mla.mla_plan_force_splits(mla.mla_decode_plan(1, 1, 16, 4096, 152), 4)
        plan.variant = variant
        assert _call_decode(lib, plan, ws_bytes=plan.workspace_bytes) == -1, variant


def test_every_plan_gathers_its_own_rows(lib):
    # each CTA gathers its own KV rows (no cluster sharing): kv_share is 1
    for batch, q_len, heads, keys in [(8, 1, 16, 8 * 8192), (8, 4, 16, 8 * 8192),
                                      (2, 1, 64, 131072), (64, 1, 128, 1081344),
                                      (1, 3, 40, 1537), (3, 7, 5, 10)]:
        assert mla.mla_decode_plan(batch, q_len, heads, keys, 152).kv_share == 1
    for heads in (16, 64, 128):
        assert mla.mla_sparse_decode_plan(4, heads, 2048, 152).kv_share == 1


def test_decode_rejects_kv_share_other_than_one(lib):
    p64 = mla.mla_decode_plan(1, 1, 64, 4096, 152)
    for share in (0, 2, 4, 8):
        q = mla.mla_plan_t.from_buffer_copy(p64)
        q.kv_share = share
        assert _call_decode(lib, q, ws_bytes=q.workspace_bytes, heads=64) == -1, share


def test_decode_rejects_a_plan_whose_fields_disagree(lib):
    # the kernels index the workspace and outputs by the plan's geometry, so a
    # plan edited out of step with its shape is refused before any launch
    base = mla.mla_plan_force_splits(mla.mla_decode_plan(2, 1, 64, 8192, 152), 4)
    other_tile = 32 if base.rows_per_cta == 16 else 16
    edits = [("workspace_bytes", base.workspace_bytes - 256),      # stale size
             ("workspace_bytes", base.workspace_bytes + 256),
             ("grid_y", 5), ("grid_x", 1), ("grid_z", 3), ("head_blocks", 1),
             ("rows_per_cta", other_tile), ("rows_per_cta", 8), ("block_n", 64)]
    for field, value in edits:
        q = mla.mla_plan_t.from_buffer_copy(base)
        setattr(q, field, value)
        rc = _call_decode(lib, q, ws_bytes=1 << 30, batch=2, heads=64)
        assert rc == -1, (field, value, rc)
    # the untouched plan passes every host check (and then needs a device)
    assert _call_decode(lib, base, ws_bytes=1 << 30, batch=2, heads=64) not in (-1, -3, -4)


@pytest.mark.parametrize("tokens,rows_per_cta,splits", [
    (1, 16, 16), (2, 16, 16), (4, 16, 9), (8, 16, 4), (12, 32, 6), (16, 32, 4), (24, 32, 3),
    (32, 32, 2), (64, 32, 1)])
def test_sparse_plan_matches_the_measured_best_tile_and_split(tokens, rows_per_cta, splits):
    # 64 heads, top-k 2048, 152 SMs: the tile and split count that forced sweeps
    # of the sparse workload measured fastest (or within 3 %) on GB300
    p = mla.mla_sparse_decode_plan(tokens, 64, 2048, 152)
    assert (p.rows_per_cta, p.num_splits) == (rows_per_cta, splits)
    assert p.head_blocks == 64 // rows_per_cta


@pytest.mark.parametrize("batch,q_len,heads,keys_per_request,rows_per_cta", [
    (1, 1, 64, 256, 16), (1, 1, 64, 1024, 16), (1, 1, 64, 4096, 16), (2, 1, 64, 2048, 16),
    (4, 1, 64, 1024, 16), (1, 1, 32, 2048, 16), (1, 4, 16, 8192, 16), (2, 1, 128, 1024, 16),
    (8, 4, 16, 8192, 32), (1, 1, 64, 131072, 32), (2, 1, 64, 65536, 32),
    (8, 1, 64, 131072, 32), (64, 1, 128, 16896, 32), (8, 1, 16, 8192, 16)])
def test_dense_tile_follows_the_measured_best(batch, q_len, heads, keys_per_request,
                                              rows_per_cta):
    # Above 16 rows the planner weighs 16-row tiles (twice the head blocks)
    # against 32-row ones; a forced sweep on GB300 measured these shapes
    # fastest at the given tile (the small ones 25-35 % faster at 16 rows)
    p = mla.mla_decode_plan(batch, q_len, heads, batch * keys_per_request, 152)
    assert p.rows_per_cta == rows_per_cta
    assert p.head_blocks == -(-(q_len * heads) // rows_per_cta)


def test_plans_may_carry_either_tile_above_16_rows(lib):
    # a 64-head plan is accepted with 16 or 32 rows per CTA (geometry in step);
    # 32 rows for a request of at most 16 rows is refused
    for rpc in (16, 32):
        q = mla.mla_plan_force_splits(mla.mla_decode_plan(2, 1, 64, 8192, 152), 4)
        q.rows_per_cta, q.head_blocks, q.grid_x = rpc, 64 // rpc, 64 // rpc
        assert _call_decode(lib, q, ws_bytes=1 << 30, batch=2, heads=64) not in (-1, -3, -4)
    q = mla.mla_decode_plan(2, 1, 16, 8192, 152)
    q.rows_per_cta = 32
    assert _call_decode(lib, q, ws_bytes=1 << 30, batch=2, heads=16) == -1


def test_long_first_only_when_the_grid_outlasts_a_wave():
    # B=64 H=128 (256 CTAs > one wave): longest requests first; c1 (128 CTAs): not
    assert mla.mla_decode_plan(64, 1, 128, 64 * 16896, 152).long_first == 1
    assert mla.mla_decode_plan(8, 1, 16, 8 * 8192, 152).long_first == 0
    assert mla.mla_decode_plan(1, 1, 64, 131072, 152).long_first == 0
    assert mla.mla_decode_plan(300, 1, 128, 300 * 4096, 152).long_first == 0   # batch > 256
    assert mla.mla_sparse_decode_plan(64, 64, 2048, 152).long_first == 0


@pytest.mark.parametrize("batch,q_len,heads,keys_per_request,splits", [
    (8, 1, 16, 8192, 16),       # c1 q_len=1
    (8, 4, 16, 8192, 8),        # c1 q_len=4
    (8, 1, 64, 131072, 9),      # c2 8x131072 (one wave)
    (1, 1, 64, 131072, 74),     # c2 1x131072 (48.99 us; 69 splits 50.76)
    (1, 1, 64, 65536, 74),      # 32.71 us; 64 splits 34.01
    (4, 1, 64, 16384, 19),      # 33.06 us; 16 splits 34.46
    (2, 1, 64, 65536, 37),      # c2 2x65536
    (16, 1, 64, 131072, 9),     # c2 16x131072
    (64, 1, 128, 16896, 1),     # c3's shape (mean length)
    (8, 1, 16, 131072, 19),     # longer H=16 contexts: a full wave
    (8, 1, 16, 65536, 19),
    (16, 1, 16, 131072, 19),
    (64, 1, 16, 16384, 2),
])
def test_dense_plan_stays_within_the_measured_best(batch, q_len, heads, keys_per_request,
                                                   splits):
    # split counts that a forced-split sweep on GB300 measured fastest (within
    # 1 %) for each workload (152 SMs); a planner change that moves them needs
    # a new sweep
    p = mla.mla_decode_plan(batch, q_len, heads, batch * keys_per_request, 152)
    assert p.num_splits == splits

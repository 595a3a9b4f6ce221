"""fp64 CPU oracle for absorbed-MLA decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module.  The library's
product path never touches it (the CUDA binding fails loudly instead of falling
back here).

Two independent implementations live here:

* ``mla_oracle.c`` (compiled with gcc, OpenMP over query rows x heads): the
  plain fp64 definition, see that file's header for the formulas and the
  passages they follow (moonmath-ai/amd-kernels README: "MLA absorbed decode",
  "Use / MLA decode", "Numerics"; hip_mha_decoding_num_partitions: the split-K
  merge; "[Perf] pa_decode_sparse ..." issue: the sparse top-k variant).
* ``brute_force_*`` below: pure-Python loops over Python floats for tiny
  inputs, decoding bytes with torch's own ``float8_e4m3fn`` / ``bfloat16``
  casts.  It shares nothing with the C file except the definition itself, so
  agreement between the two pins the C decode, indexing and softmax.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmla_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``oracle/_build/libmla_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # MLA_ORACLE_LIB points the wrappers at another build of mla_oracle.c
        # (the mutation test uses it to check that planted mistakes are caught).
        override = os.environ.get("MLA_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        c_i32, c_i64, c_dbl, c_p = (ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_double, ctypes.c_void_p)
        lib.oracle_e4m3fn_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3fn_to_double.restype = c_dbl
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = c_dbl
        lib.oracle_attend.argtypes = [c_p, c_p, ctypes.c_int, ctypes.c_int, c_p, c_i64,
                                      c_p, c_i64, c_dbl, c_dbl, c_p, c_p]
        lib.oracle_attend.restype = ctypes.c_int
        lib.oracle_merge.argtypes = [c_p, c_p, ctypes.c_int, ctypes.c_int, c_dbl, c_p, c_p]
        lib.oracle_merge.restype = ctypes.c_int
        lib.oracle_dense_decode.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32, c_p, c_p,
                                            c_p, c_i64, c_p, c_p, c_p, c_dbl, c_dbl,
                                            c_p, c_i64, c_p, c_p]
        lib.oracle_dense_decode.restype = ctypes.c_int
        lib.oracle_sparse_decode.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32, c_p, c_p,
                                             c_p, c_i64, c_p, c_dbl, c_dbl, c_p, c_i64,
                                             c_p, c_p]
        lib.oracle_sparse_decode.restype = ctypes.c_int
        lib.oracle_dcp_decode.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32, c_p, c_p,
                                          c_p, c_i64, c_p, c_p, c_p, c_p, c_i32, c_i32,
                                          c_dbl, c_dbl, c_p, c_p]
        lib.oracle_dcp_decode.restype = ctypes.c_int
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


_RC = {-1: "bad argument", -2: "slot out of range", -3: "NaN input"}


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(f"oracle returned {rc} ({_RC.get(rc, 'unknown')})")


def _ptr(t) -> int:
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _u16(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16)


def _u8(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.uint8:
        t = t.view(torch.uint8)
    return t.contiguous()


# ---- scalar formats ---------------------------------------------------------

def e4m3fn_to_double(b: int) -> float:
    return _load().oracle_e4m3fn_to_double(int(b) & 0xFF)


def bf16_to_double(h: int) -> float:
    return _load().oracle_bf16_to_double(int(h) & 0xFFFF)


# ---- one row / merge --------------------------------------------------------

def attend(q_lat: torch.Tensor, q_pe: torch.Tensor, pool: torch.Tensor,
           slots: Sequence[int] | torch.Tensor, scale: float,
           kv_scale: float) -> Tuple[np.ndarray, float]:
    """One query row (bf16 [d_v], [d_rope]) over explicit slots -> (o fp64 [d_v], lse2)."""
    lib = _load()
    ql, qp = _u16(q_lat.reshape(-1)), _u16(q_pe.reshape(-1))
    pl = _u8(pool).reshape(pool.shape[0], -1)
    sl = torch.as_tensor(slots, dtype=torch.int32).contiguous().reshape(-1)
    d_v, d_r = ql.numel(), qp.numel()
    assert pl.shape[1] == d_v + d_r
    o = np.zeros(d_v, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _check(lib.oracle_attend(_ptr(ql), _ptr(qp), d_v, d_r, _ptr(pl), pl.shape[0],
                             _ptr(sl), sl.numel(), float(scale), float(kv_scale),
                             _ptr(o), _ptr(lse)))
    return o, float(lse[0])


def merge(o_parts: np.ndarray, lse2_parts: np.ndarray,
          out_scale: float = 1.0) -> Tuple[np.ndarray, float]:
    """LSE merge of partials o_parts [ns, d_v] (normalized), lse2_parts [ns] (base 2)."""
    lib = _load()
    op = np.ascontiguousarray(o_parts, dtype=np.float64)
    lp = np.ascontiguousarray(lse2_parts, dtype=np.float64).reshape(-1)
    ns, d_v = op.shape
    o = np.zeros(d_v, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _check(lib.oracle_merge(_ptr(op), _ptr(lp), ns, d_v, float(out_scale),
                            _ptr(o), _ptr(lse)))
    return o, float(lse[0])


# ---- whole calls ------------------------------------------------------------

def dense_decode(inp, sel: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 dense decode of a ``DenseInputs``.

    Returns o [B*q_len, H, d_v] and lse2 [B*q_len, H]; with ``sel`` (flat
    ``row*H + h`` item indices) returns o [n_sel, d_v] and lse2 [n_sel].
    """
    lib = _load()
    ql, qp = _u16(inp.q_lat), _u16(inp.q_pe)
    pl = _u8(inp.pool)
    R, H = inp.batch * inp.q_len, inp.num_heads
    n = R * H if sel is None else len(sel)
    o = np.zeros((n, inp.d_v), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    s = None if sel is None else np.ascontiguousarray(sel, dtype=np.int64)
    lens = inp.seq_lens.to(torch.int32).contiguous()
    idx = inp.kv_indices.to(torch.int32).contiguous()
    ptr = inp.kv_indptr.to(torch.int32).contiguous()
    _check(lib.oracle_dense_decode(
        inp.batch, inp.q_len, H, inp.d_v, inp.d_rope, _ptr(ql), _ptr(qp), _ptr(pl),
        pl.shape[0], _ptr(lens), _ptr(idx), _ptr(ptr), inp.scale, inp.kv_scale,
        None if s is None else _ptr(s), 0 if s is None else len(s), _ptr(o), _ptr(lse)))
    if sel is None:
        return o.reshape(R, H, inp.d_v), lse.reshape(R, H)
    return o, lse


def sparse_decode(inp, sel: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 sparse top-k decode of a ``SparseInputs`` -> o [T, H, d_v], lse2 [T, H]."""
    lib = _load()
    qn, qp = _u16(inp.q_nope), _u16(inp.q_pe)
    pl = _u8(inp.pool)
    T, H = inp.num_tokens, inp.num_heads
    n = T * H if sel is None else len(sel)
    o = np.zeros((n, inp.d_v), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    s = None if sel is None else np.ascontiguousarray(sel, dtype=np.int64)
    idx = inp.indices.to(torch.int32).contiguous()
    _check(lib.oracle_sparse_decode(
        T, H, inp.topk, inp.d_v, inp.d_rope, _ptr(qn), _ptr(qp), _ptr(pl), pl.shape[0],
        _ptr(idx), inp.scale, inp.kv_scale,
        None if s is None else _ptr(s), 0 if s is None else len(s), _ptr(o), _ptr(lse)))
    if sel is None:
        return o.reshape(T, H, inp.d_v), lse.reshape(T, H)
    return o, lse


def dcp_shard(inp, cp_rank: int, cp_world: int):
    """Rank ``cp_rank``'s view of a ``DenseInputs`` under decode context
    parallelism (moonmath-ai/amd-kernels README, "Use / MLA decode": a rank holds
    the positions p with p % cp_world == cp_rank).  Returns a ``DenseInputs`` of
    the same queries whose request b lists only those positions' slots, in
    increasing position order, and the global lengths ``glen`` (int32 [B])."""
    lens = inp.seq_lens.tolist()
    indptr = inp.kv_indptr.tolist()
    idx = inp.kv_indices.tolist()
    local_lens, local_idx, local_ptr = [], [], [0]
    for b in range(inp.batch):
        mine = [idx[indptr[b] + p] for p in range(lens[b]) if p % cp_world == cp_rank]
        local_lens.append(len(mine))
        local_idx.extend(mine)
        local_ptr.append(len(local_idx))
    i32 = torch.int32
    shard = dataclasses.replace(inp, seq_lens=torch.tensor(local_lens, dtype=i32),
                                kv_indices=torch.tensor(local_idx, dtype=i32),
                                kv_indptr=torch.tensor(local_ptr, dtype=i32))
    return shard, torch.tensor(lens, dtype=i32)


def dcp_decode(inp, glen: torch.Tensor, cp_rank: int,
               cp_world: int) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 decode of one DCP rank's share: ``inp`` holds the rank's keys (local
    key j = global position j*cp_world + cp_rank), ``glen`` the global lengths.
    Returns o [B*q_len, H, d_v] and lse2 [B*q_len, H] of the share."""
    lib = _load()
    ql, qp = _u16(inp.q_lat), _u16(inp.q_pe)
    pl = _u8(inp.pool)
    R, H = inp.batch * inp.q_len, inp.num_heads
    o = np.zeros((R * H, inp.d_v), dtype=np.float64)
    lse = np.zeros(R * H, dtype=np.float64)
    lens = inp.seq_lens.to(torch.int32).contiguous()
    idx = inp.kv_indices.to(torch.int32).contiguous()
    if idx.numel() == 0:
        idx = torch.zeros(1, dtype=torch.int32)
    ptr = inp.kv_indptr.to(torch.int32).contiguous()
    gl = glen.to(torch.int32).contiguous()
    _check(lib.oracle_dcp_decode(
        inp.batch, inp.q_len, H, inp.d_v, inp.d_rope, _ptr(ql), _ptr(qp), _ptr(pl),
        pl.shape[0], _ptr(lens), _ptr(idx), _ptr(ptr), _ptr(gl), int(cp_rank),
        int(cp_world), inp.scale, inp.kv_scale, _ptr(o), _ptr(lse)))
    return o.reshape(R, H, inp.d_v), lse.reshape(R, H)


def dcp_merge_ranks(o_parts: np.ndarray, lse2_parts: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Merge of the ranks' shares: o_parts [W, ...rows, d_v], lse2_parts
    [W, ...rows] -> o [...rows, d_v], lse2 [...rows], row by row with ``merge``
    (out_scale 1; the ranks take the place of the splits)."""
    op = np.asarray(o_parts, dtype=np.float64)
    lp = np.asarray(lse2_parts, dtype=np.float64)
    W, d_v = op.shape[0], op.shape[-1]
    rows_shape = lp.shape[1:]
    op2 = op.reshape(W, -1, d_v)
    lp2 = lp.reshape(W, -1)
    o = np.zeros((op2.shape[1], d_v))
    lse = np.zeros(op2.shape[1])
    for r in range(op2.shape[1]):
        o[r], lse[r] = merge(op2[:, r, :], lp2[:, r])
    return o.reshape(rows_shape + (d_v,)), lse.reshape(rows_shape)


def sparse_extra_decode(inp) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 sparse decode over the main cache and a second (compressed) cache
    (flashinfer cake_sparse_mla_sm120_dsv4_nvfp4_plan_splits: ``extra_topk``
    candidate slots per token in the second cache).  Token t attends the union
    of its valid main candidates and its valid second-cache candidates in one
    softmax: the two caches are laid end to end as one pool, the second cache's
    slots shifted past the main pool's rows, and ``sparse_decode`` runs over the
    joined candidate rows."""
    n_main = inp.pool.shape[0]
    pool = torch.cat([_u8(inp.pool).reshape(n_main, -1),
                      _u8(inp.extra_pool).reshape(inp.extra_pool.shape[0], -1)], 0)
    extra = inp.extra_indices.to(torch.int64)
    shifted = torch.where(extra >= 0, extra + n_main, torch.full_like(extra, -1))
    joined = torch.cat([inp.indices.to(torch.int64), shifted], 1).to(torch.int32)
    one = dataclasses.replace(inp, pool=pool, indices=joined.contiguous(),
                              topk=joined.shape[1], extra_pool=None, extra_indices=None)
    return sparse_decode(one)


def split_partials(q_lat, q_pe, pool, slots, scale, kv_scale,
                   num_splits: int) -> Tuple[np.ndarray, np.ndarray]:
    """Partials of one row over ``num_splits`` contiguous key ranges of equal
    ceil-divided size (empty trailing ranges give o=0, lse2=-inf)."""
    sl = torch.as_tensor(slots, dtype=torch.int32).reshape(-1)
    n = sl.numel()
    chunk = -(-n // num_splits) if n else 0
    d_v = q_lat.numel()
    op = np.zeros((num_splits, d_v))
    lp = np.zeros(num_splits)
    for s in range(num_splits):
        lo, hi = min(s * chunk, n), min((s + 1) * chunk, n)
        op[s], lp[s] = attend(q_lat, q_pe, pool, sl[lo:hi], scale, kv_scale)
    return op, lp


# ---- independent pure-Python brute force (tiny inputs only) ----------------

def _torch_decode_rows(pool: torch.Tensor) -> list:
    return _u8(pool).reshape(pool.shape[0], -1).view(torch.float8_e4m3fn).to(
        torch.float64).tolist()


def brute_force_row(q: Sequence[float], rows: Sequence[Sequence[float]], d_v: int,
                    scale: float, kv_scale: float) -> Tuple[list, float]:
    """Softmax attention of one fp64 query over already-decoded key rows."""
    if not rows:
        return [0.0] * d_v, -math.inf
    logits = []
    for r in rows:
        acc = 0.0
        for a, b in zip(q, r):
            acc += a * (b * kv_scale)
        logits.append(scale * acc)
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    z = math.fsum(w)
    o = [math.fsum(wj * rows[j][c] * kv_scale for j, wj in enumerate(w)) / z
         for c in range(d_v)]
    return o, (m + math.log(z)) / math.log(2.0)


def brute_force_dense(inp) -> Tuple[np.ndarray, np.ndarray]:
    """Pure-Python dense decode for tiny ``DenseInputs`` (every row, every head)."""
    dec = _torch_decode_rows(inp.pool)
    ql = inp.q_lat.to(torch.float64).tolist()
    qp = inp.q_pe.to(torch.float64).tolist()
    R, H = inp.batch * inp.q_len, inp.num_heads
    o = np.zeros((R, H, inp.d_v))
    lse = np.zeros((R, H))
    indptr = inp.kv_indptr.tolist()
    idx = inp.kv_indices.tolist()
    lens = inp.seq_lens.tolist()
    for b in range(inp.batch):
        for t in range(inp.q_len):
            r = b * inp.q_len + t
            n = max(lens[b] - inp.q_len + t + 1, 0)
            rows = [dec[idx[indptr[b] + j]] for j in range(n)]
            for h in range(H):
                q = ql[r][h] + qp[r][h]
                ov, lv = brute_force_row(q, rows, inp.d_v, inp.scale, inp.kv_scale)
                o[r, h] = ov
                lse[r, h] = lv
    return o, lse


def brute_force_dcp(inp, cp_rank: int, cp_world: int) -> Tuple[np.ndarray, np.ndarray]:
    """Pure-Python decode of one DCP rank's share of a tiny unsharded
    ``DenseInputs``: row t of request b attends, in increasing order, the global
    positions p < S_b with p % cp_world == cp_rank and p <= S_b - q_len + t."""
    dec = _torch_decode_rows(inp.pool)
    ql = inp.q_lat.to(torch.float64).tolist()
    qp = inp.q_pe.to(torch.float64).tolist()
    R, H = inp.batch * inp.q_len, inp.num_heads
    o = np.zeros((R, H, inp.d_v))
    lse = np.zeros((R, H))
    indptr = inp.kv_indptr.tolist()
    idx = inp.kv_indices.tolist()
    lens = inp.seq_lens.tolist()
    for b in range(inp.batch):
        for t in range(inp.q_len):
            r = b * inp.q_len + t
            pos = [p for p in range(lens[b])
                   if p % cp_world == cp_rank and p <= lens[b] - inp.q_len + t]
            rows = [dec[idx[indptr[b] + p]] for p in pos]
            for h in range(H):
                ov, lv = brute_force_row(ql[r][h] + qp[r][h], rows, inp.d_v,
                                         inp.scale, inp.kv_scale)
                o[r, h] = ov
                lse[r, h] = lv
    return o, lse


def brute_force_sparse(inp) -> Tuple[np.ndarray, np.ndarray]:
    """Pure-Python sparse decode for tiny ``SparseInputs``."""
    dec = _torch_decode_rows(inp.pool)
    qn = inp.q_nope.to(torch.float64).tolist()
    qp = inp.q_pe.to(torch.float64).tolist()
    T, H = inp.num_tokens, inp.num_heads
    o = np.zeros((T, H, inp.d_v))
    lse = np.zeros((T, H))
    idx = inp.indices.tolist()
    for t in range(T):
        rows = [dec[s] for s in idx[t] if s >= 0]
        for h in range(H):
            ov, lv = brute_force_row(qn[t][h] + qp[t][h], rows, inp.d_v,
                                     inp.scale, inp.kv_scale)
            o[t, h] = ov
            lse[t, h] = lv
    return o, lse


def cpu_threads() -> int:
    """Threads the OpenMP oracle uses (OMP_NUM_THREADS, else all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return os.cpu_count() or 1

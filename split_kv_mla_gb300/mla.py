"""Thin Python binding of libmla (ctypes): argument marshalling only.

Every function has the name of the C entry point it calls (``mla_decode_plan``,
``mla_decode``, ``mla_sparse_decode``, ``mla_splitk_reduce`` ...).  Tensors are
PyTorch CUDA tensors: PyTorch owns device memory and streams, the library does
all of the work.  There is no fallback: if ``libmla.so`` is missing or a tensor
is not on a CUDA device the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

MLA_OK = 0
MLA_MAX_SPLITS = 256
MLA_WORKSPACE_HEADER_BYTES = 65536
MLA_DEVERR_BAD_SLOT = 1
MLA_DEVERR_TIMEOUT = 2
MLA_DEVERR_BAD_LENGTH = 4
MLA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
HEADER = os.path.join(_build.ROOT, "include", "mla_decode.h")


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} ({status})")


class mla_plan_t(ctypes.Structure):
    _fields_ = [
        ("num_splits", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32),
        ("block_n", ctypes.c_int32), ("head_blocks", ctypes.c_int32),
        ("grid_x", ctypes.c_int32), ("grid_y", ctypes.c_int32), ("grid_z", ctypes.c_int32),
        ("variant", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
        ("batch", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("d_v", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("sm_count", ctypes.c_int32),
        ("total_keys", ctypes.c_int64), ("kv_share", ctypes.c_int32),
        ("extra_topk", ctypes.c_int32), ("long_first", ctypes.c_int32),
        ("merge_cluster", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True, path: Optional[str] = None):
    """Load libmla.so (building it first if it is missing and nvcc exists), or
    the library at `path` (a variant build, e.g. the traced one) if given
    before the first load."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"libmla.so not built ({path})")
            _build.build()
        lib = ctypes.CDLL(path)
        i32, i64, f32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        P = ctypes.POINTER(mla_plan_t)
        sig = {
            "mla_decode_plan": (ctypes.c_int, [i32, i32, i32, i64, i32, i32, i32, P]),
            "mla_sparse_decode_plan": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32, i32,
                                                      P]),
            "mla_sparse_decode_extra": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, i64, vp, i32,
                                                       i32, i32, i32, f32, f32, vp, vp, vp, i64,
                                                       vp]),
            "mla_sparse_decode_extra_splits": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, i64, vp,
                                                              i32, i32, i32, i32, f32, f32, vp,
                                                              vp, vp, i64, vp]),
            "mla_decode": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, vp, i32, i32, i32, f32,
                                          f32, vp, vp, vp, i64, vp]),
            "mla_sparse_decode": (ctypes.c_int, [P, vp, vp, vp, i64, vp, i32, i32, i32, f32,
                                                 f32, vp, vp, vp, i64, vp]),
            "mla_decode_splits": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, vp, i32, i32, i32,
                                                 f32, f32, vp, vp, vp, i64, vp]),
            "mla_sparse_decode_splits": (ctypes.c_int, [P, vp, vp, vp, i64, vp, i32, i32, i32,
                                                        f32, f32, vp, vp, vp, i64, vp]),
            "mla_workspace_partials": (ctypes.c_int, [P, vp, ctypes.POINTER(vp),
                                                      ctypes.POINTER(vp)]),
            "mla_splitk_reduce": (ctypes.c_int, [vp, vp, i64, i32, i32, f32, vp, vp, vp]),
            "mla_decode_noalloc": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, vp, i32, i32, i32,
                                                  f32, f32, vp, vp, vp]),
            "mla_plan_force_splits": (ctypes.c_int, [P, i32]),
            "mla_workspace_reset": (ctypes.c_int, [vp, vp]),
            "mla_read_device_error": (ctypes.c_int, [vp, ctypes.POINTER(i32), vp]),
            "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "mla_wave_fill_splits": (i32, [i32, i64, i32, i32, i32, i32, i32, i32, i32]),
            "mla_debug_gather": (ctypes.c_int, [vp, i64, i32, vp, i64, vp, vp, vp]),
            "mla_debug_wait_limit": (i64, [i64]),
            "mla_decode_dcp": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, vp, i32, i32, i32,
                                              f32, f32, vp, i32, i32, i32, vp, vp, vp, i64,
                                              vp]),
            "mla_decode_dcp_splits": (ctypes.c_int, [P, vp, vp, vp, i64, vp, vp, vp, i32, i32,
                                                     i32, f32, f32, vp, i32, i32, i32, vp, vp,
                                                     vp, i64, vp]),
            "mla_dcp_lse_merge_ranks": (ctypes.c_int, [vp, i32, vp, i32, i64, i32, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def declared_symbols() -> list:
    """Function names declared in include/mla_decode.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().mla_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, where)


def _dev_ptr(t: Optional[torch.Tensor], name: str, dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def sm_count(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


# ---- planning ------------------------------------------------------------------

def mla_decode_plan(batch: int, q_len: int, num_heads: int, total_keys: int,
                    sm_count: int, d_v: int = 512, d_rope: int = 64) -> mla_plan_t:
    p = mla_plan_t()
    _check(load().mla_decode_plan(batch, q_len, num_heads, total_keys, d_v, d_rope, sm_count,
                                  ctypes.byref(p)), "mla_decode_plan")
    return p


def mla_sparse_decode_plan(num_tokens: int, num_heads: int, topk: int, sm_count: int,
                           max_splits: int = 0, d_v: int = 448, d_rope: int = 64,
                           extra_topk: int = 0) -> mla_plan_t:
    p = mla_plan_t()
    _check(load().mla_sparse_decode_plan(num_tokens, num_heads, topk, extra_topk, d_v, d_rope,
                                         sm_count, max_splits, ctypes.byref(p)),
           "mla_sparse_decode_plan")
    return p


def mla_plan_force_splits(plan: mla_plan_t, num_splits: int) -> mla_plan_t:
    """A copy of ``plan`` re-targeted to ``num_splits`` splits."""
    p = mla_plan_t.from_buffer_copy(plan)
    _check(load().mla_plan_force_splits(ctypes.byref(p), int(num_splits)), "mla_plan_force_splits")
    return p


def mla_wave_fill_splits(batch, keys_per_request, heads, sm_count, bm, page,
                         max_pages_per_split, max_splits, small_heads) -> int:
    return int(load().mla_wave_fill_splits(batch, keys_per_request, heads, sm_count, bm, page,
                                           max_pages_per_split, max_splits, small_heads))


def workspace(plan: mla_plan_t, device=None) -> torch.Tensor:
    """A zeroed workspace of plan.workspace_bytes (256-byte aligned by the allocator)."""
    n = max(int(plan.workspace_bytes), MLA_WORKSPACE_HEADER_BYTES)
    ws = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
    assert ws.data_ptr() % 256 == 0
    return ws


# ---- decode ----------------------------------------------------------------------

def mla_decode(plan: mla_plan_t, q_lat, q_pe, pool, seq_lens, kv_indices, kv_indptr,
               scale: float, kv_scale: float, o_lat=None, lse=None, workspace_t=None,
               stream=None, return_lse: bool = True, _entry: str = "mla_decode"):
    """Dense decode; returns (o_lat, lse).  Outputs are allocated when not given."""
    for name, t in (("q_lat", q_lat), ("q_pe", q_pe), ("pool", pool), ("seq_lens", seq_lens),
                    ("kv_indices", kv_indices), ("kv_indptr", kv_indptr)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    R, H = q_lat.shape[0], q_lat.shape[1]
    batch = seq_lens.shape[0]
    q_len = R // batch if batch else 1
    if o_lat is None:
        o_lat = torch.empty_like(q_lat)
    if lse is None and return_lse:
        lse = torch.empty(R, H, dtype=torch.float32, device=q_lat.device)
    if workspace_t is None:
        workspace_t = workspace(plan, q_lat.device)
    pool_u8 = pool.view(torch.uint8) if pool.dtype != torch.uint8 else pool
    rc = getattr(load(), _entry)(
        ctypes.byref(plan), _dev_ptr(q_lat, "q_lat", torch.bfloat16),
        _dev_ptr(q_pe, "q_pe", torch.bfloat16), _dev_ptr(pool_u8, "pool"), pool_u8.shape[0],
        _dev_ptr(seq_lens, "seq_lens", torch.int32), _dev_ptr(kv_indices, "kv_indices", torch.int32),
        _dev_ptr(kv_indptr, "kv_indptr", torch.int32), batch, q_len, H, float(scale),
        float(kv_scale), _dev_ptr(o_lat, "o_lat", torch.bfloat16), _dev_ptr(lse, "lse", torch.float32),
        _dev_ptr(workspace_t, "workspace"), workspace_t.numel(), _stream_ptr(stream))
    _check(rc, _entry)
    return o_lat, lse


def mla_decode_splits(*args, **kw):
    """Only the split kernel of mla_decode (see mla_workspace_partials)."""
    return mla_decode(*args, _entry="mla_decode_splits", **kw)


_DTYPE_CODE = {torch.bfloat16: 0, torch.float32: 1}   # MLA_DTYPE_BF16, MLA_DTYPE_F32


def mla_decode_dcp(plan: mla_plan_t, q_lat, q_pe, pool, seq_lens, kv_indices, kv_indptr,
                   scale: float, kv_scale: float, glen, cp_rank: int, cp_world: int,
                   o=None, lse=None, workspace_t=None, stream=None,
                   out_dtype=torch.bfloat16, _entry: str = "mla_decode_dcp"):
    """One decode-context-parallel rank's share; returns (o, lse).  The rank's
    page table lists its positions p % cp_world == cp_rank; ``glen`` int32 [B]
    holds the global lengths (may be None only when cp_world == 1).  The share
    is bf16 (``out_dtype``, or the dtype of a given ``o``) or fp32."""
    for name, t in (("q_lat", q_lat), ("q_pe", q_pe), ("pool", pool), ("seq_lens", seq_lens),
                    ("kv_indices", kv_indices), ("kv_indptr", kv_indptr)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    if glen is not None and not glen.is_cuda:
        raise ValueError("glen must be a CUDA tensor")
    R, H = q_lat.shape[0], q_lat.shape[1]
    batch = seq_lens.shape[0]
    q_len = R // batch if batch else 1
    if o is None:
        o = torch.empty(q_lat.shape, dtype=out_dtype, device=q_lat.device)
    if o.dtype not in _DTYPE_CODE:
        raise ValueError("o must be bf16 or fp32")
    if lse is None:
        lse = torch.empty(R, H, dtype=torch.float32, device=q_lat.device)
    if workspace_t is None:
        workspace_t = workspace(plan, q_lat.device)
    pool_u8 = pool.view(torch.uint8) if pool.dtype != torch.uint8 else pool
    rc = getattr(load(), _entry)(
        ctypes.byref(plan), _dev_ptr(q_lat, "q_lat", torch.bfloat16),
        _dev_ptr(q_pe, "q_pe", torch.bfloat16), _dev_ptr(pool_u8, "pool"), pool_u8.shape[0],
        _dev_ptr(seq_lens, "seq_lens", torch.int32), _dev_ptr(kv_indices, "kv_indices", torch.int32),
        _dev_ptr(kv_indptr, "kv_indptr", torch.int32), batch, q_len, H, float(scale),
        float(kv_scale), _dev_ptr(glen, "glen", torch.int32), int(cp_rank), int(cp_world),
        _DTYPE_CODE[o.dtype], _dev_ptr(o, "o"), _dev_ptr(lse, "lse", torch.float32),
        _dev_ptr(workspace_t, "workspace"), workspace_t.numel(), _stream_ptr(stream))
    _check(rc, _entry)
    return o, lse


def mla_decode_dcp_splits(*args, **kw):
    """Only the split kernel of mla_decode_dcp (see mla_workspace_partials)."""
    return mla_decode_dcp(*args, _entry="mla_decode_dcp_splits", **kw)


def mla_dcp_lse_merge_ranks(parts_in, lse_in, out=None, lse_out=None, stream=None,
                            return_lse: bool = True):
    """Merge the ranks' shares: parts_in bf16 or fp32 [W, ...rows, d_v]
    (rank-major), lse_in fp32 [W, ...rows]; returns (out bf16 [...rows, d_v],
    lse_out fp32 [...rows])."""
    if not parts_in.is_cuda or not lse_in.is_cuda:
        raise ValueError("parts_in and lse_in must be CUDA tensors")
    if parts_in.dtype not in _DTYPE_CODE:
        raise ValueError("parts_in must be bf16 or fp32")
    W, d_v = parts_in.shape[0], parts_in.shape[-1]
    rows_shape = tuple(lse_in.shape[1:])
    rows = lse_in[0].numel()
    if parts_in[0].numel() != rows * d_v:
        raise ValueError("parts_in and lse_in disagree on the rows")
    if out is None:
        out = torch.empty(rows_shape + (d_v,), dtype=torch.bfloat16, device=parts_in.device)
    if lse_out is None and return_lse:
        lse_out = torch.empty(rows_shape, dtype=torch.float32, device=parts_in.device)
    rc = load().mla_dcp_lse_merge_ranks(
        _dev_ptr(parts_in, "parts_in"), _DTYPE_CODE[parts_in.dtype],
        _dev_ptr(lse_in, "lse_in", torch.float32), W, rows, d_v, _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(lse_out, "lse_out", torch.float32),
        _stream_ptr(stream))
    _check(rc, "mla_dcp_lse_merge_ranks")
    return out, lse_out


def mla_sparse_decode(plan: mla_plan_t, q_nope, q_pe, pool, indices, scale: float,
                      kv_scale: float, o=None, lse=None, workspace_t=None, stream=None,
                      return_lse: bool = True, _entry: str = "mla_sparse_decode"):
    """Sparse top-k decode; returns (o, lse)."""
    for name, t in (("q_nope", q_nope), ("q_pe", q_pe), ("pool", pool), ("indices", indices)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    T, H = q_nope.shape[0], q_nope.shape[1]
    topk = indices.shape[1] if indices.dim() == 2 else 0
    if o is None:
        o = torch.empty_like(q_nope)
    if lse is None and return_lse:
        lse = torch.empty(T, H, dtype=torch.float32, device=q_nope.device)
    if workspace_t is None:
        workspace_t = workspace(plan, q_nope.device)
    pool_u8 = pool.view(torch.uint8) if pool.dtype != torch.uint8 else pool
    rc = getattr(load(), _entry)(
        ctypes.byref(plan), _dev_ptr(q_nope, "q_nope", torch.bfloat16),
        _dev_ptr(q_pe, "q_pe", torch.bfloat16), _dev_ptr(pool_u8, "pool"), pool_u8.shape[0],
        _dev_ptr(indices, "indices", torch.int32), T, H, topk, float(scale), float(kv_scale),
        _dev_ptr(o, "o", torch.bfloat16), _dev_ptr(lse, "lse", torch.float32),
        _dev_ptr(workspace_t, "workspace"), workspace_t.numel(), _stream_ptr(stream))
    _check(rc, _entry)
    return o, lse


def mla_sparse_decode_extra(plan: mla_plan_t, q_nope, q_pe, pool, indices, extra_pool,
                            extra_indices, scale: float, kv_scale: float, o=None, lse=None,
                            workspace_t=None, stream=None, return_lse: bool = True,
                            _entry: str = "mla_sparse_decode_extra"):
    """Sparse top-k decode over the main cache and a second (compressed) cache
    in one softmax: indices int32 [T, topk] into pool, extra_indices int32
    [T, extra_topk] into extra_pool (both uint8 [N, 512]); returns (o, lse)."""
    for name, t in (("q_nope", q_nope), ("q_pe", q_pe), ("pool", pool), ("indices", indices),
                    ("extra_pool", extra_pool), ("extra_indices", extra_indices)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    T, H = q_nope.shape[0], q_nope.shape[1]
    topk = indices.shape[1] if indices.dim() == 2 else 0
    extra_topk = extra_indices.shape[1] if extra_indices.dim() == 2 else 0
    if o is None:
        o = torch.empty_like(q_nope)
    if lse is None and return_lse:
        lse = torch.empty(T, H, dtype=torch.float32, device=q_nope.device)
    if workspace_t is None:
        workspace_t = workspace(plan, q_nope.device)
    pool_u8 = pool.view(torch.uint8) if pool.dtype != torch.uint8 else pool
    xpool_u8 = extra_pool.view(torch.uint8) if extra_pool.dtype != torch.uint8 else extra_pool
    rc = getattr(load(), _entry)(
        ctypes.byref(plan), _dev_ptr(q_nope, "q_nope", torch.bfloat16),
        _dev_ptr(q_pe, "q_pe", torch.bfloat16), _dev_ptr(pool_u8, "pool"), pool_u8.shape[0],
        _dev_ptr(indices, "indices", torch.int32), _dev_ptr(xpool_u8, "extra_pool"),
        xpool_u8.shape[0], _dev_ptr(extra_indices, "extra_indices", torch.int32), T, H, topk,
        extra_topk, float(scale), float(kv_scale), _dev_ptr(o, "o", torch.bfloat16),
        _dev_ptr(lse, "lse", torch.float32), _dev_ptr(workspace_t, "workspace"),
        workspace_t.numel(), _stream_ptr(stream))
    _check(rc, _entry)
    return o, lse


def mla_sparse_decode_extra_splits(*args, **kw):
    """Only the split kernel of mla_sparse_decode_extra."""
    return mla_sparse_decode_extra(*args, _entry="mla_sparse_decode_extra_splits", **kw)


def mla_sparse_decode_splits(*args, **kw):
    """Only the split kernel of mla_sparse_decode."""
    return mla_sparse_decode(*args, _entry="mla_sparse_decode_splits", **kw)


def mla_workspace_partials(plan: mla_plan_t, workspace_t):
    """(o_part, lse_part) fp32 views into the workspace, or (None, None) for one split."""
    o_ptr, l_ptr = ctypes.c_void_p(), ctypes.c_void_p()
    base = _dev_ptr(workspace_t, "workspace")
    _check(load().mla_workspace_partials(ctypes.byref(plan), base, ctypes.byref(o_ptr),
                                         ctypes.byref(l_ptr)), "mla_workspace_partials")
    if not o_ptr.value:
        return None, None
    rows = plan.batch * plan.q_len * plan.num_heads
    ns, d_v = plan.num_splits, plan.d_v
    f32 = workspace_t.view(torch.uint8)
    o_off, l_off = o_ptr.value - base, l_ptr.value - base
    o_part = f32[o_off:o_off + rows * ns * d_v * 4].view(torch.float32).view(rows, ns, d_v)
    lse_part = f32[l_off:l_off + rows * ns * 4].view(torch.float32).view(rows, ns)
    return o_part, lse_part


def mla_splitk_reduce(o_part, lse_part, out_scale: float = 1.0, o=None, lse=None,
                      stream=None, return_lse: bool = True):
    """Merge o_part fp32 [rows, ns, d_v] with lse_part fp32 [rows, ns]; returns (o, lse)."""
    rows, ns, d_v = o_part.shape
    if o is None:
        o = torch.empty(rows, d_v, dtype=torch.bfloat16, device=o_part.device)
    if lse is None and return_lse:
        lse = torch.empty(rows, dtype=torch.float32, device=o_part.device)
    rc = load().mla_splitk_reduce(
        _dev_ptr(o_part, "o_part", torch.float32), _dev_ptr(lse_part, "lse_part", torch.float32),
        rows, ns, d_v, float(out_scale), _dev_ptr(o, "o", torch.bfloat16),
        _dev_ptr(lse, "lse", torch.float32), _stream_ptr(stream))
    _check(rc, "mla_splitk_reduce")
    return o, lse


def mla_workspace_reset(workspace_t, stream=None) -> None:
    _check(load().mla_workspace_reset(_dev_ptr(workspace_t, "workspace"), _stream_ptr(stream)),
           "mla_workspace_reset")


def mla_read_device_error(workspace_t, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().mla_read_device_error(_dev_ptr(workspace_t, "workspace"), ctypes.byref(code),
                                        _stream_ptr(stream)), "mla_read_device_error")
    return int(code.value)


def mla_debug_gather(pool, indices, workspace_t=None, stream=None):
    """Rows pool[indices] copied through the split kernel's gather path (TMA
    gather4 into the swizzled stage layout, read back de-swizzled); an
    out-of-range index gives a zero row.  pool: uint8 [N, 576] or [N, 512]
    (a [N, 1, 576] cache is accepted); indices: int32 [n].  Returns
    (rows uint8 [n, row_bytes], workspace)."""
    p = pool.reshape(pool.shape[0], -1)
    row_bytes = p.shape[1]
    n = indices.numel()
    out = torch.empty(n, row_bytes, dtype=torch.uint8, device=p.device)
    ws = workspace_t if workspace_t is not None else torch.zeros(
        MLA_WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=p.device)
    _check(load().mla_debug_gather(_dev_ptr(p, "pool", torch.uint8), p.shape[0], row_bytes,
                                   _dev_ptr(indices, "indices", torch.int32), n,
                                   _dev_ptr(out, "out"), _dev_ptr(ws, "workspace"),
                                   _stream_ptr(stream)), "mla_debug_gather")
    return out, ws


def mla_debug_wait_limit(cycles: int) -> int:
    """Set the bound (SM cycles) of the split kernel's pipeline waits for later
    launches; <= 0 restores the default.  Returns the previous bound.  For tests
    of the timeout path."""
    return int(load().mla_debug_wait_limit(int(cycles)))


def mla_decode_noalloc(plan: mla_plan_t, q_lat, q_pe, pool, seq_lens, kv_indices, kv_indptr,
                       scale: float, kv_scale: float, o_lat, lse=None, stream=None):
    """Dense decode through the entry point that allocates nothing: the library's
    static scratch array stands in for the workspace.  For callers that cannot
    allocate device memory; the caller passes preallocated outputs.  Calls that
    overlap on the GPU share that scratch and race."""
    for name, t in (("q_lat", q_lat), ("q_pe", q_pe), ("pool", pool), ("seq_lens", seq_lens),
                    ("kv_indices", kv_indices), ("kv_indptr", kv_indptr), ("o_lat", o_lat)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    R, H = q_lat.shape[0], q_lat.shape[1]
    batch = seq_lens.shape[0]
    q_len = R // batch if batch else 1
    pool_u8 = pool.view(torch.uint8) if pool.dtype != torch.uint8 else pool
    rc = load().mla_decode_noalloc(
        ctypes.byref(plan), _dev_ptr(q_lat, "q_lat", torch.bfloat16),
        _dev_ptr(q_pe, "q_pe", torch.bfloat16), _dev_ptr(pool_u8, "pool"), pool_u8.shape[0],
        _dev_ptr(seq_lens, "seq_lens", torch.int32), _dev_ptr(kv_indices, "kv_indices", torch.int32),
        _dev_ptr(kv_indptr, "kv_indptr", torch.int32), batch, q_len, H, float(scale),
        float(kv_scale), _dev_ptr(o_lat, "o_lat", torch.bfloat16), _dev_ptr(lse, "lse", torch.float32),
        _stream_ptr(stream))
    _check(rc, "mla_decode_noalloc")
    return o_lat, lse

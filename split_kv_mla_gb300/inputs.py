"""Seeded synthetic inputs for absorbed-MLA decode.

This module only draws random numbers and lays them out; it performs none of the
attention arithmetic.  Both the fp64 oracle tests and the CUDA path take their
inputs from here, so the two sides always see identical bytes.

Recipe (moonmath-ai/amd-kernels README, "MLA decode" usage block and the MI300X
results table; the synthetic workloads of this library follow it):

* queries ``q_lat`` / ``q_pe`` are bf16 draws of N(0, 1), shaped
  ``[B*q_len, H, d_v]`` and ``[B*q_len, H, d_rope]`` (row ``b*q_len + t``);
* the pool holds one fused fp8 e4m3fn row per token, the cast of
  ``N(0, 1) / kv_scale`` with ``kv_scale = 1/32``; columns ``[0, d_v)`` are the
  latent part (also V) and ``[d_v, d_v + d_rope)`` the RoPE part;
* page size is 1: ``kv_indices`` is a seeded random permutation of the pool's
  slots, ``kv_indptr`` the prefix sums of the per-request lengths;
* ``scale = (d_v + d_rope) ** -0.5``.

Everything is generated on the CPU with ``torch.Generator`` so the oracle can read
exactly the bytes the GPU gets.  Large pools are drawn in fixed-size chunks from
one generator, which keeps the sequence identical whatever the chunk size.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

D_LATENT = 512
D_ROPE = 64
SPARSE_D_NOPE = 448
KV_SCALE = 1.0 / 32.0
_CHUNK = 1 << 22  # floats drawn per step when filling a pool


@dataclasses.dataclass
class DenseInputs:
    """One dense decode call's inputs (CPU tensors)."""

    batch: int
    q_len: int
    num_heads: int
    q_lat: torch.Tensor      # bf16 [B*q_len, H, d_v]
    q_pe: torch.Tensor       # bf16 [B*q_len, H, d_rope]
    pool: torch.Tensor       # uint8 [N, 1, d_v + d_rope]  (fp8 e4m3fn bytes)
    seq_lens: torch.Tensor   # int32 [B]
    kv_indices: torch.Tensor  # int32 [sum(seq_lens)]
    kv_indptr: torch.Tensor  # int32 [B + 1]
    scale: float
    kv_scale: float

    @property
    def d_v(self) -> int:
        return self.q_lat.shape[-1]

    @property
    def d_rope(self) -> int:
        return self.q_pe.shape[-1]

    @property
    def total_keys(self) -> int:
        return int(self.kv_indices.numel())


@dataclasses.dataclass
class SparseInputs:
    """One sparse top-k decode call's inputs (CPU tensors)."""

    num_tokens: int
    num_heads: int
    topk: int
    q_nope: torch.Tensor     # bf16 [T, H, d_v]
    q_pe: torch.Tensor       # bf16 [T, H, d_rope]
    pool: torch.Tensor       # uint8 [N, d_v + d_rope]
    indices: torch.Tensor    # int32 [T, topk]; negative = invalid entry
    scale: float
    kv_scale: float
    # optional second (compressed) cache: same row format, own slot space
    extra_pool: Optional[torch.Tensor] = None     # uint8 [N2, d_v + d_rope]
    extra_indices: Optional[torch.Tensor] = None  # int32 [T, extra_topk]; negative = invalid

    @property
    def extra_topk(self) -> int:
        return 0 if self.extra_indices is None else int(self.extra_indices.shape[1])

    @property
    def d_v(self) -> int:
        return self.q_nope.shape[-1]

    @property
    def d_rope(self) -> int:
        return self.q_pe.shape[-1]


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _bf16_normal(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def fp8_pool(rows: int, width: int, g: torch.Generator,
             kv_scale: float = KV_SCALE) -> torch.Tensor:
    """uint8 [rows, width]: e4m3fn bytes of N(0,1)/kv_scale, drawn chunk by chunk."""
    out = torch.empty(rows * width, dtype=torch.uint8)
    total = rows * width
    pos = 0
    while pos < total:
        n = min(_CHUNK, total - pos)
        x = torch.randn(n, generator=g) / kv_scale
        out[pos:pos + n] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        pos += n
    return out.view(rows, width)


def dense_inputs(batch: int, q_len: int, num_heads: int,
                 seq_lens: Sequence[int] | torch.Tensor,
                 seed: int = 0, *, d_v: int = D_LATENT, d_rope: int = D_ROPE,
                 kv_scale: float = KV_SCALE, scale: Optional[float] = None,
                 extra_slots: int = 0) -> DenseInputs:
    """Dense decode inputs with a shuffled page_size-1 pool.

    ``extra_slots`` adds unused pool rows, so slots are a random subset of the
    pool rather than all of it.
    """
    g = _gen(seed)
    lens = torch.as_tensor(list(seq_lens) if not torch.is_tensor(seq_lens)
                           else seq_lens, dtype=torch.int64).reshape(-1)
    assert lens.numel() == batch
    total = int(lens.sum())
    rows = batch * q_len
    q_lat = _bf16_normal((rows, num_heads, d_v), g)
    q_pe = _bf16_normal((rows, num_heads, d_rope), g)
    n_slots = total + int(extra_slots)
    pool = fp8_pool(max(n_slots, 1), d_v + d_rope, g, kv_scale).view(
        max(n_slots, 1), 1, d_v + d_rope)
    perm = torch.randperm(max(n_slots, 1), generator=g)[:total].to(torch.int32)
    indptr = torch.zeros(batch + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(lens, 0)
    return DenseInputs(
        batch=batch, q_len=q_len, num_heads=num_heads,
        q_lat=q_lat, q_pe=q_pe, pool=pool,
        seq_lens=lens.to(torch.int32), kv_indices=perm.contiguous(),
        kv_indptr=indptr.to(torch.int32),
        scale=float((d_v + d_rope) ** -0.5 if scale is None else scale),
        kv_scale=float(kv_scale))


def variable_lengths(batch: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Per-request lengths drawn uniformly from [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (batch,), generator=_gen(seed),
                         dtype=torch.int64)


def sparse_inputs(num_tokens: int, num_heads: int, topk: int, pool_rows: int,
                  seed: int = 0, *, d_v: int = SPARSE_D_NOPE, d_rope: int = D_ROPE,
                  kv_scale: float = KV_SCALE, scale: Optional[float] = None,
                  invalid_frac: float = 0.0) -> SparseInputs:
    """Sparse top-k inputs: per token ``topk`` distinct slots drawn without
    replacement; with ``invalid_frac`` > 0 that fraction of entries is set to -1."""
    g = _gen(seed)
    q_nope = _bf16_normal((num_tokens, num_heads, d_v), g)
    q_pe = _bf16_normal((num_tokens, num_heads, d_rope), g)
    pool = fp8_pool(pool_rows, d_v + d_rope, g, kv_scale)
    idx = torch.empty(num_tokens, topk, dtype=torch.int32)
    for t in range(num_tokens):
        idx[t] = torch.randperm(pool_rows, generator=g)[:topk].to(torch.int32)
    if invalid_frac > 0:
        mask = torch.rand(num_tokens, topk, generator=g) < invalid_frac
        idx[mask] = -1
    return SparseInputs(
        num_tokens=num_tokens, num_heads=num_heads, topk=topk,
        q_nope=q_nope, q_pe=q_pe, pool=pool, indices=idx,
        scale=float((d_v + d_rope) ** -0.5 if scale is None else scale),
        kv_scale=float(kv_scale))


def sparse_extra_inputs(num_tokens: int, num_heads: int, topk: int, extra_topk: int,
                        pool_rows: int, extra_rows: int, seed: int = 0, *,
                        invalid_frac: float = 0.0, **kw) -> SparseInputs:
    """``sparse_inputs(..., seed)`` plus a second cache of ``extra_rows`` rows
    and per token ``extra_topk`` distinct slots of it, drawn from a second
    generator (so the main part equals ``sparse_inputs`` with the same seed)."""
    inp = sparse_inputs(num_tokens, num_heads, topk, pool_rows, seed,
                        invalid_frac=invalid_frac, **kw)
    g = _gen(seed + 7919)
    inp.extra_pool = fp8_pool(extra_rows, inp.d_v + inp.d_rope, g, inp.kv_scale)
    idx = torch.empty(num_tokens, extra_topk, dtype=torch.int32)
    for t in range(num_tokens):
        idx[t] = torch.randperm(extra_rows, generator=g)[:extra_topk].to(torch.int32)
    if invalid_frac > 0:
        idx[torch.rand(num_tokens, extra_topk, generator=g) < invalid_frac] = -1
    inp.extra_indices = idx
    return inp


# --- the five synthetic workloads -------------------------------------------

def workload_c0(seed: int = 0) -> DenseInputs:
    """B=1, H=16, q_len=1, S=256."""
    return dense_inputs(1, 1, 16, [256], seed)


def workload_c1(q_len: int = 1, seed: int = 0, seq: int = 8192,
                batch: int = 8) -> DenseInputs:
    """B=8, H=16, S=8192 per request, q_len 1 or 4."""
    return dense_inputs(batch, q_len, 16, [seq] * batch, seed)


def workload_c2(batch: int, seq: int, seed: int = 0) -> DenseInputs:
    """H=64, q_len=1, split-heavy (B, S) points."""
    return dense_inputs(batch, 1, 64, [seq] * batch, seed)


def workload_c3(seed: int = 0, batch: int = 64, lo: int = 1024,
                hi: int = 32768) -> DenseInputs:
    """B=64, H=128, q_len=1, lengths uniform in [1024, 32768]."""
    lens = variable_lengths(batch, lo, hi, seed + 1000)
    return dense_inputs(batch, 1, 128, lens, seed)


def workload_c4(num_tokens: int, seed: int = 0, pool_rows: int = 131072,
                topk: int = 2048) -> SparseInputs:
    """Sparse top-k: T tokens, 64 heads, 448+64 dims, top-k 2048 of 131072."""
    return sparse_inputs(num_tokens, 64, topk, pool_rows, seed)


def workload_c4x(num_tokens: int, seed: int = 0, pool_rows: int = 131072, topk: int = 2048,
                 extra_rows: int = 32768, extra_topk: int = 512) -> SparseInputs:
    """Sparse top-k with a second (compressed) cache: the c4 shape plus, per
    token, ``extra_topk`` candidates of a ``extra_rows``-row second cache."""
    return sparse_extra_inputs(num_tokens, 64, topk, extra_topk, pool_rows, extra_rows, seed)


# --- structured variants for precision-edge tests -----------------------------
#
# These reshape a workload's draws (scale parts of the queries, plant outliers,
# copy rows) to build inputs whose numbers sit at the edges of the kernel's
# number formats: wide dynamic range inside one query row, logits that are
# nearly tied, logits far apart.  They only move and cast values; none of the
# attention arithmetic happens here.

def _queries(inp):
    """(latent/NoPE part, RoPE part) of dense or sparse inputs."""
    return (inp.q_lat, inp.q_pe) if isinstance(inp, DenseInputs) else (inp.q_nope, inp.q_pe)


def _set_queries(inp, lat, pe):
    if isinstance(inp, DenseInputs):
        inp.q_lat = lat.to(torch.bfloat16).contiguous()
    else:
        inp.q_nope = lat.to(torch.bfloat16).contiguous()
    inp.q_pe = pe.to(torch.bfloat16).contiguous()
    return inp


def scale_query_parts(inp, lat: float = 1.0, pe: float = 1.0):
    """Multiply the latent (NoPE) and RoPE query parts by separate factors."""
    ql, qp = _queries(inp)
    return _set_queries(inp, ql.float() * lat, qp.float() * pe)


def plant_query_outliers(inp, ratio: float, seed: int, part: str = "lat"):
    """In every (row, head) query, one seeded column of the given part becomes
    +-ratio while the other columns keep their N(0,1) draws."""
    g = _gen(seed)
    ql, qp = (t.float().clone() for t in _queries(inp))
    tgt = ql if part == "lat" else qp
    rows, heads, width = tgt.shape
    col = torch.randint(0, width, (rows, heads), generator=g)
    sign = torch.where(torch.rand(rows, heads, generator=g) < 0.5, -1.0, 1.0)
    tgt.view(-1, width)[torch.arange(rows * heads), col.reshape(-1)] = (sign * ratio).reshape(-1)
    return _set_queries(inp, ql, qp)


def share_query_across_heads(inp):
    """Every head of a query row gets head 0's query (all heads then rank the
    keys alike)."""
    ql, qp = _queries(inp)
    return _set_queries(inp, ql[:, :1].expand_as(ql), qp[:, :1].expand_as(qp))


def plant_dominant_key(inp: DenseInputs, strength: float, seed: int) -> DenseInputs:
    """For each request, one seeded key's pool row becomes the e4m3fn cast of
    strength * (that request's first query row, head 0) / kv_scale, so with
    queries shared across heads its logit exceeds the others' by about
    strength * |q|^2 * scale.  The other keys keep their draws."""
    g = _gen(seed)
    pool = inp.pool.clone()
    width = pool.shape[-1]
    for b in range(inp.batch):
        n = int(inp.seq_lens[b])
        if n == 0:
            continue
        j = int(torch.randint(0, n, (1,), generator=g))
        slot = int(inp.kv_indices[int(inp.kv_indptr[b]) + j])
        q = torch.cat([inp.q_lat[b * inp.q_len, 0].float(), inp.q_pe[b * inp.q_len, 0].float()])
        row = (q * strength / inp.kv_scale).to(torch.float8_e4m3fn).view(torch.uint8)
        pool.view(-1, width)[slot] = row
    inp.pool = pool
    return inp


def near_tied_pool(inp: DenseInputs, seed: int, flips: int = 4) -> DenseInputs:
    """Every slot holds one base row (the pool's slot 0) with `flips` seeded
    bytes moved to a neighbouring e4m3fn code, so all logits of a query are
    tied up to a few tiny terms."""
    g = _gen(seed)
    width = inp.pool.shape[-1]
    flat = inp.pool.view(-1, width)
    base = flat[0].clone()
    pool = base.unsqueeze(0).repeat(flat.shape[0], 1)
    cols = torch.randint(0, width, (flat.shape[0], flips), generator=g)
    rows = torch.arange(flat.shape[0]).unsqueeze(1).expand_as(cols)
    mag = pool[rows, cols] & 0x7F
    # step the magnitude code by one, staying inside finite non-NaN codes
    stepped = torch.where(mag >= 0x7E, mag - 1, mag + 1)
    pool[rows, cols] = (pool[rows, cols] & 0x80) | stepped
    inp.pool = pool.view(inp.pool.shape).contiguous()
    return inp

"""GPU: the page-table gather (step a2) byte for byte.  mla_debug_gather copies
rows through the split kernel's own TMA gather4 path and swizzled stage layout
and reads them back de-swizzled; the result must equal pool[indices] exactly,
for dense 576-byte and sparse 512-byte rows, ragged counts (not multiples of
the 128-row stage), repeated slots, and out-of-range slots (zero rows, never
read)."""
import pytest
import torch

from split_kv_mla_gb300 import mla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    mla.load()


@pytest.mark.parametrize("row_bytes,rows,n", [(576, 5000, 1), (576, 5000, 129), (576, 70000, 4096),
                                              (512, 131072, 2048), (512, 3000, 300)])
def test_gather_probe_matches_pool_indexing(row_bytes, rows, n):
    g = torch.Generator().manual_seed(row_bytes + n)
    pool = torch.randint(0, 256, (rows, row_bytes), dtype=torch.uint8, generator=g)
    idx = torch.randint(0, rows, (n,), dtype=torch.int32, generator=g)
    out, ws = mla.mla_debug_gather(pool.cuda(), idx.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), pool[idx.long()])
    assert mla.mla_read_device_error(ws) == 0


def test_gather_probe_dense_cache_layout_and_repeats():
    g = torch.Generator().manual_seed(7)
    pool = torch.randint(0, 256, (1000, 1, 576), dtype=torch.uint8, generator=g)
    idx = torch.tensor([5, 5, 999, 0, 0, 0, 512, 5] * 20, dtype=torch.int32)
    out, _ = mla.mla_debug_gather(pool.cuda(), idx.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), pool.reshape(1000, 576)[idx.long()])


def test_gather_probe_out_of_range_rows_are_zero():
    g = torch.Generator().manual_seed(8)
    pool = torch.randint(1, 256, (800, 576), dtype=torch.uint8, generator=g)
    idx = torch.randint(0, 800, (300,), dtype=torch.int32, generator=g)
    bad = torch.tensor([3, 77, 200, 299])
    idx[bad[:2]] = -1
    idx[bad[2:]] = 800 + 5
    out, _ = mla.mla_debug_gather(pool.cuda(), idx.cuda())
    torch.cuda.synchronize()
    ref = pool[idx.clamp(0, 799).long()].clone()
    ref[bad] = 0
    assert torch.equal(out.cpu(), ref)

"""idx_page_table_transform against the oracle, entry for entry ("[sglang]
logits를 쓰지 않는 top-k", section 3: row-relative positions to physical KV
slots of a page-size-64 cache, -1 kept, one flat grid over rows x topk)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


def positions(rows, topk, max_pos, seed, pad_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    p = torch.randint(0, max_pos, (rows, topk), generator=g, dtype=torch.int32)
    pad = torch.rand(rows, topk, generator=g) < pad_frac
    p[pad] = -1
    return p


def run(idx, pos, table, page_size, row_map=None, stats=None, dev_idx=None):
    d = dev_idx if dev_idx is not None else pos.to(DEV)
    idx.idx_page_table_transform(d, table.to(DEV), page_size,
                                 row_map=None if row_map is None else row_map.to(DEV),
                                 stats=stats)
    torch.cuda.synchronize()
    return d.cpu().numpy()


def test_fused_prefill_shape_vector_path(idx):
    """4096 rows x topk 2048 of one 65536-key request, 1024 pages of 64."""
    table, row_map = synth.paged_layout(1, 1024, 4096, seed=61)
    pos = positions(4096, 2048, 65536, seed=62)
    stats = idx.Stats(torch.device(DEV))
    got = run(idx, pos, table, 64, row_map, stats)
    ref, bad = oracle.page_transform(pos, table, 64, row_map)
    assert bad == 0 and np.array_equal(got, ref)
    assert stats.read()["status"] == 0


@pytest.mark.parametrize("topk,page_size", [(7, 64), (1, 64), (12, 16), (2048, 48), (5, 1)])
def test_sizes_and_page_sizes(idx, topk, page_size):
    pages = 300
    table, row_map = synth.paged_layout(5, pages, 9, seed=63 + topk)
    pos = positions(45, topk, pages * page_size, seed=64 + page_size)
    got = run(idx, pos, table, page_size, row_map)
    ref, bad = oracle.page_transform(pos, table, page_size, row_map)
    assert bad == 0 and np.array_equal(got, ref)


def test_unaligned_array_takes_scalar_path(idx):
    """An index array that starts 4 bytes past a 16-byte boundary."""
    table, row_map = synth.paged_layout(3, 64, 20, seed=65)
    pos = positions(60, 16, 64 * 64, seed=66)
    buf = torch.empty(60 * 16 + 1, dtype=torch.int32, device=DEV)
    view = buf[1:].view(60, 16)
    view.copy_(pos.to(DEV))
    assert view.data_ptr() % 16 != 0
    got = run(idx, pos, table, 64, row_map, dev_idx=view)
    ref, _ = oracle.page_transform(pos, table, 64, row_map)
    assert np.array_equal(got, ref)


def test_more_rows_than_one_grid_dimension(idx):
    """70000 rows: the flat grid needs no second dimension (65535 limit)."""
    table, row_map = synth.paged_layout(70, 32, 1000, seed=67)
    pos = positions(70000, 8, 32 * 64, seed=68)
    got = run(idx, pos, table, 64, row_map)
    ref, _ = oracle.page_transform(pos, table, 64, row_map)
    assert np.array_equal(got, ref)


def test_identity_table_without_row_map(idx):
    table = torch.arange(128, dtype=torch.int32).repeat(10, 1)
    pos = positions(10, 64, 128 * 64, seed=69, pad_frac=0.3)
    got = run(idx, pos, table, 64)
    assert np.array_equal(got, pos.numpy())


def test_out_of_range_pages_and_rows_raise(idx):
    """Pages past the table row and table rows outside the table give -1 and
    the range bit; everything else is transformed."""
    table, _ = synth.paged_layout(2, 8, 1, seed=70)
    pos = torch.tensor([[0, 63, 64 * 8, -1], [5, 64 * 7 + 1, 64 * 9, 3],
                        [1, 2, 3, 4]], dtype=torch.int32)
    row_map = torch.tensor([0, 1, 5], dtype=torch.int32)  # row 2 names a missing table row
    stats = idx.Stats(torch.device(DEV))
    got = run(idx, pos, table, 64, row_map, stats)
    t = table.numpy()
    assert got[0].tolist() == [t[0, 0] * 64, t[0, 0] * 64 + 63, -1, -1]
    assert got[1].tolist() == [t[1, 0] * 64 + 5, t[1, 7] * 64 + 1, -1, t[1, 0] * 64 + 3]
    assert got[2].tolist() == [-1, -1, -1, -1]
    assert stats.read()["status"] & 0x2  # IDX_DEV_RANGE
    # the oracle, given the table's row bound, agrees entry for entry
    ref, bad = oracle.page_transform(pos, table, 64, row_map)
    assert np.array_equal(got, ref) and bad == 6


def test_after_the_fused_top_k(idx):
    """The transform applied to idx_score_topk's output (tiny workload)."""
    inp = synth.workload("tiny")
    g = {n: getattr(inp, n).to(DEV) for n in ("q", "k", "k_scale", "w", "ks", "ke")}
    out = idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk)
    torch.cuda.synchronize()
    before = out.cpu()
    table, row_map = synth.paged_layout(1, inp.keys // 64, inp.rows, seed=71)
    got = run(idx, before, table, 64, row_map, dev_idx=out)
    ref, bad = oracle.page_transform(before, table, 64, row_map)
    assert bad == 0 and np.array_equal(got, ref)

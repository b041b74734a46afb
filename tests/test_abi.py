"""The C ABI without a GPU: the library loads, exports every function that
include/idx.h declares, and its host-only logic (workspace sizes, status text,
argument checks that precede any CUDA call) behaves as documented."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_tiles_gb300 import build
    build.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "idx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(idx_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"idx_score_topk", "idx_topk_from_scores", "idx_score_materialise"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libidx.so"


def test_status_strings(lib):
    import sparse_attention_indexer_tiles_gb300 as pkg
    texts = [pkg.idx_status_string(c) for c in range(7)]
    assert texts[0] == "ok" and len(set(texts)) == 7
    assert pkg.idx_status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    import sparse_attention_indexer_tiles_gb300 as pkg
    ws = pkg.idx_score_topk_workspace
    # short rows: slab + plan only; long rows add the sample and the rescan histograms
    small = ws(4096, 4096, 0, 64, 128, 2048, 2)
    big = ws(4096, 65536, 0, 64, 128, 2048, 2)
    assert 0 < small < big
    cap = 4608
    assert small >= 4096 * cap * 8
    # max_len bounds the sample scratch
    assert ws(4096, 1 << 20, 65536, 32, 128, 2048, 2) < ws(4096, 1 << 20, 0, 32, 128, 2048, 2)
    assert ws(0, 100, 0, 64, 128, 16, 2) == 0
    assert pkg.idx_topk_workspace(8, 1 << 20, 2048) >= 0


def test_argument_checks_before_cuda(lib):
    i64 = ctypes.c_longlong
    P = ctypes.c_void_p(16)  # never dereferenced: the checks below fail first
    # topk < 1
    assert lib.idx_score_topk(P, P, P, P, P, P, 4, 100, 0, 64, 128, 0, 2, P, P, 0, None, None) == 1
    # unsupported H
    assert lib.idx_score_topk(P, P, P, P, P, P, 4, 100, 0, 12, 128, 8, 2, P, P, 0, None, None) == 4
    # unsupported dtype
    assert lib.idx_score_materialise(P, P, P, P, P, P, 4, 100, 64, 128, 7, P, 100, None, None) == 4
    # a missing pointer
    assert lib.idx_score_materialise(None, P, P, P, P, P, 4, 100, 64, 128, 2, P, 100, None,
                                     None) == 1
    # misaligned q (needs 16 bytes for TMA)
    Q = ctypes.c_void_p(16 + 8)
    assert lib.idx_score_materialise(Q, P, P, P, P, P, 4, 100, 64, 128, 2, P, 100, None, None) == 2
    # rows == 0 is a no-op
    assert lib.idx_score_materialise(None, None, None, None, None, None, 0, 100, 64, 128, 2, None,
                                     100, None, None) == 0
    assert lib.idx_topk_from_scores(P, i64(10), P, P, 4, 0, P, None, 0, None, None) == 1
    assert lib.idx_topk_from_scores(P, i64(10), P, P, 4, 5000, P, None, 0, None, None) == 4
    # MXFP4 expansion: D a multiple of 32, 16-byte aligned arrays, n = 0 a no-op
    lib.idx_mxfp4_to_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.idx_mxfp4_to_e4m3(P, P, i64(4), 48, P, None, None) == 1
    assert lib.idx_mxfp4_to_e4m3(ctypes.c_void_p(24), P, i64(4), 64, P, None, None) == 2
    assert lib.idx_mxfp4_to_e4m3(None, None, i64(0), 64, None, None, None) == 0


def test_options_struct_layout():
    import sparse_attention_indexer_tiles_gb300 as pkg
    assert ctypes.sizeof(pkg.Options) == 48
    assert pkg.Options.d_status.offset == 16 and pkg.Options.relative_rows.offset == 32
    assert pkg.Options.stage_events.offset == 40


def test_product_path_has_no_oracle_import():
    """The library and its binding never load the oracle (test infrastructure)."""
    pkg_dir = os.path.join(ROOT, "sparse_attention_indexer_tiles_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle." not in text, f


def test_routing_gate_rule(lib):
    """The gate is host logic: fused from 24576 keys in the longest row on,
    two-pass for few rows (rows <= SMs / 4, rows x max_len <= 2^25; no device
    answers here: 148 SMs)."""
    import sparse_attention_indexer_tiles_gb300 as pkg
    assert pkg.idx_route_fused(4096, 4608, 2048)       # fits the slab: every key emitted
    assert pkg.idx_route_fused(8, 4608, 2048)
    assert not pkg.idx_route_fused(4096, 4609, 2048)
    assert not pkg.idx_route_fused(4096, 24575, 2048)
    assert not pkg.idx_route_fused(4096, 12288, 2048)
    assert not pkg.idx_route_fused(4096, 6144, 512)
    assert pkg.idx_route_fused(4096, 24576, 2048)
    assert pkg.idx_route_fused(4096, 1 << 20, 512)
    assert not pkg.idx_route_fused(16, 1 << 20, 2048)  # few rows over long keys
    assert not pkg.idx_route_fused(32, 1 << 20, 2048)
    assert pkg.idx_route_fused(33, 1 << 20, 2048)      # 33 x 2^20 > 2^25
    assert not pkg.idx_route_fused(37, 1 << 18, 2048)
    assert pkg.idx_route_fused(38, 1 << 18, 2048)      # 4 x 38 > 148
    # the dense route's workspace holds the logits; the fused one its slab
    dense = pkg.idx_score_topk_routed_workspace(64, 8192, 0, 64, 128, 2048, 2)
    assert dense >= 64 * 8192 * 4
    assert pkg.idx_score_topk_routed_workspace(64, 65536, 0, 64, 128, 256, 2) == \
        pkg.idx_score_topk_workspace(64, 65536, 0, 64, 128, 256, 2)


def _documented_workspace(rows, max_len, topk, nruns):
    """The fused workspace as the layout is documented: 256-byte aligned
    regions for the row plans (32 B each), the run counts [rows, nruns] int32,
    the slab [rows, nruns, cap_q] of (fp32 score, int32 index) pairs with
    cap_q = ceil(cap / 8) + 64 rounded up to even, the sample scratch [rows, max_len // S + 2
    rounded up to a multiple of 8] of 16-bit keys, the rescan histograms [rows, 4096] and the rescan's list and flags
    of row blocks [blocks] int32 (these only when rows can see more than cap
    keys), the emit pass's order of the row blocks [blocks] int32 (also only
    then), and sixteen counters (the rescan's and the scoring launches' unit
    counters)."""
    def up(x):
        return (x + 255) // 256 * 256
    cap = min(max(math.ceil(3.5 * topk), 4096), 12288)
    cap_q = (-(-cap // 8) + 64 + 1) // 2 * 2
    target = math.sqrt(cap / topk)
    t = max(32.0, (4.5 / math.log(max(target, 1.0001))) ** 2)
    S = max(s for s in (1, 3, 5, 7, 11, 15, 23, 31, 45, 63) if s <= target * topk / t)
    sampled = max_len > cap
    nblk = -(-rows // 4)  # row blocks of 256 / H rows at H = 64
    regions = [rows * 32, rows * nruns * 4, rows * nruns * cap_q * 8,
               rows * ((max_len // S + 2 + 7) // 8 * 8) * 2 if sampled else 0,
               rows * 4096 * 4 if sampled else 0,
               nblk * 4 if sampled else 0, nblk * 4 if sampled else 0,
               nblk * 4 if sampled else 0, 16 * 4]
    return sum(up(r) for r in regions), S


def test_fused_workspace_follows_the_documented_layout(lib):
    """Eight runs per row and key split.  With no device answering, the
    library takes 148 SMs.  Full waves keep whole row blocks; the blocks of the
    last wave are cut into the k parts that minimise ceil(tail k / SMs) (1 / k
    + 8 / tiles), every part keeping >= 32 key tiles: 4096 rows (1024 blocks
    of H = 64, a 136-block tail) are not split; 1024 rows (256 blocks: one
    whole wave and a 108-block tail) cut the tail in 4; calls with fewer blocks
    than SMs cut every block into up to one wave's worth."""
    import sparse_attention_indexer_tiles_gb300 as pkg
    ws = pkg.idx_score_topk_workspace
    cases = [  # rows, keys, topk, expected key splits (148 SMs: no device answers here)
        (4096, 65536, 2048, 1), (8, 65536, 2048, 16), (8, 16384, 2048, 4), (64, 65536, 512, 9),
        (8, 4096, 2048, 1), (1024, 65536, 2048, 4), (16, 1 << 20, 2048, 37)]
    for rows, keys, topk, k in cases:
        expect, S = _documented_workspace(rows, keys, topk, 8 * k)
        assert ws(rows, keys, 0, 64, 128, topk, 2) == expect, (rows, keys, topk, k)
    assert _documented_workspace(1, 1, 2048, 8)[1] == 63  # the stride for topk 2048
    assert _documented_workspace(1, 1, 512, 8)[1] == 45


def test_bindings_refuse_host_tensors(lib):
    """There is no CPU path: every compute entry point of the binding raises
    before any library call when handed host tensors."""
    import pytest
    import torch
    import sparse_attention_indexer_tiles_gb300 as pkg
    q = torch.zeros(4, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(100, 64, dtype=torch.bfloat16)
    sc, w = torch.ones(100), torch.ones(4, 8)
    ks, ke = torch.zeros(4, dtype=torch.int32), torch.full((4,), 100, dtype=torch.int32)
    calls = [
        lambda: pkg.idx_score_topk(q, k, sc, w, ks, ke, 16),
        lambda: pkg.idx_score_topk_routed(q, k, sc, w, ks, ke, 16),
        lambda: pkg.idx_score_topk_noalloc(q, k, sc, w, ks, ke, 16),
        lambda: pkg.idx_score_materialise(q, k, sc, w, ks, ke),
        lambda: pkg.idx_topk_from_scores(torch.zeros(4, 100), ks, ke, 16),
        lambda: pkg.idx_page_table_transform(torch.zeros(4, 16, dtype=torch.int32),
                                             torch.zeros(4, 2, dtype=torch.int32)),
        lambda: pkg.idx_mxfp4_to_e4m3(torch.zeros(4, 32, dtype=torch.uint8),
                                      torch.zeros(4, 2, dtype=torch.uint8)),
        lambda: pkg.idx_score_topk_mxfp4(torch.zeros(4, 8, 32, dtype=torch.uint8),
                                         torch.zeros(4, 8, 2, dtype=torch.uint8),
                                         torch.zeros(100, 32, dtype=torch.uint8),
                                         torch.zeros(100, 2, dtype=torch.uint8), sc, w, ks, ke, 16),
    ]
    before = pkg.idx_launch_count()
    for call in calls:
        with pytest.raises(ValueError, match="CUDA device"):
            call()
    assert pkg.idx_launch_count() == before


def test_bindings_refuse_tensors_on_two_devices():
    """Every tensor of a call must live on one device: the call runs with that
    device current (its stream, its copy of the library's state)."""
    import types
    import pytest
    import sparse_attention_indexer_tiles_gb300 as pkg

    def fake(dev):
        return types.SimpleNamespace(is_cuda=True, is_contiguous=lambda: True, device=dev)
    assert pkg._dev(fake("cuda:1"), None, fake("cuda:1")) == "cuda:1"
    with pytest.raises(ValueError, match="different devices"):
        pkg._dev(fake("cuda:0"), fake("cuda:1"))


def test_host_entry_checks_arguments_before_any_copy(lib):
    """idx_score_topk_host (host-memory inputs and output) validates on the
    host: bad sizes and missing pointers come back before anything is copied
    or launched, and its workspace holds the device copies of the inputs and
    of the indices plus the fused workspace of one row chunk."""
    import torch
    import sparse_attention_indexer_tiles_gb300 as pkg
    before = pkg.idx_launch_count()
    args = [None] * 6 + [4, 100, 0, 8, 64]
    assert lib.idx_score_topk_host(*args, 0, 1, None, None, 0, None, None) == 1   # topk < 1
    assert lib.idx_score_topk_host(*args, 16, 3, None, None, 0, None, None) == 4  # MXFP4 here
    assert lib.idx_score_topk_host(*args, 16, 1, None, None, 0, None, None) == 1  # no pointers
    assert lib.idx_score_topk_host(*([None] * 6), 0, 100, 0, 8, 64, 16, 1, None, None, 0,
                                   None, None) == 0                                # no rows
    assert pkg.idx_launch_count() == before
    rows, keys, H, D, topk = 4096, 65536, 64, 128, 2048
    ws = pkg.idx_score_topk_host_workspace(rows, keys, 0, H, D, topk, 2)
    copies = rows * H * D + keys * D + keys * 4 + rows * H * 4 + 2 * rows * 4 + rows * topk * 4
    chunk = pkg.idx_score_topk_workspace(rows // 2, keys, 0, H, D, topk, 2)
    assert copies + chunk <= ws <= copies + chunk + 8 * 256
    with pytest.raises(ValueError):
        pkg.idx_score_topk_host(torch.zeros(8, 4, 64, dtype=torch.bfloat16)[::2], None, None,
                                None, None, None, 16)

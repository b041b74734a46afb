"""The C ABI without a GPU: the library loads, exports every function that
include/idx.h declares, and its host-only logic (workspace sizes, status text,
argument checks that precede any CUDA call) behaves as documented."""
import ctypes
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
    """The gate is host logic: fused from 24576 keys in the longest row on."""
    import sparse_attention_indexer_tiles_gb300 as pkg
    assert pkg.idx_route_fused(4608, 2048)       # fits the slab: every key emitted
    assert not pkg.idx_route_fused(4609, 2048)
    assert not pkg.idx_route_fused(24575, 2048)
    assert not pkg.idx_route_fused(12288, 2048)
    assert not pkg.idx_route_fused(6144, 512)
    assert pkg.idx_route_fused(24576, 2048)
    assert pkg.idx_route_fused(1 << 20, 512)
    # the dense route's workspace holds the logits; the fused one its slab
    dense = pkg.idx_score_topk_routed_workspace(64, 8192, 0, 64, 128, 2048, 2)
    assert dense >= 64 * 8192 * 4
    assert pkg.idx_score_topk_routed_workspace(64, 65536, 0, 64, 128, 256, 2) == \
        pkg.idx_score_topk_workspace(64, 65536, 0, 64, 128, 256, 2)

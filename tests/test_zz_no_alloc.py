"""idx_score_topk_noalloc through the C ABI.

For callers that cannot allocate device memory (a plugin whose host framework
owns all memory and hands it no allocator, a serving loop that must not call
cudaMalloc): the call runs the fused path on the library's built-in scratch
array.  Two calls in a row, with different shapes, must return exactly what
idx_score_topk returns with a caller workspace; a problem larger than the array
is refused with IDX_EWORKSPACE.  This file sorts last so that a run that stops
at the first failure has run every other test first."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    L = pkg.load()
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    L.idx_score_topk_noalloc.argtypes = [P, P, P, P, P, P, I, LL, LL, I, I, I, I, P, P, P]
    L.idx_score_topk_noalloc.restype = I
    return L


def _inputs(seed, rows, keys, H, D, topk):
    inp = synth.indexer_inputs(rows, keys, H, D, topk, "fp8", seed=seed)
    return inp, {n: getattr(inp, n).to(DEV) for n in ("q", "k", "k_scale", "w", "ks", "ke")}


def _noalloc(lib, inp, g, opts=None):
    out = torch.full((inp.rows, inp.topk), -7, dtype=torch.int32, device=DEV)
    st = lib.idx_score_topk_noalloc(
        g["q"].data_ptr(), g["k"].data_ptr(), g["k_scale"].data_ptr(), g["w"].data_ptr(),
        g["ks"].data_ptr(), g["ke"].data_ptr(), inp.rows, inp.keys, 0, inp.H, inp.D, inp.topk,
        2, out.data_ptr(), None if opts is None else ctypes.byref(opts),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, out.cpu().numpy()


def _with_workspace(inp, g, opts=None):
    import sparse_attention_indexer_tiles_gb300 as pkg
    out = pkg.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk,
                             options=opts)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_noalloc_matches_workspace_path_twice(lib):
    # two calls in a row with different shapes; both long enough to sample,
    # the second with a small slab so that some rows take the exact rescan
    import sparse_attention_indexer_tiles_gb300 as pkg
    inp1, g1 = _inputs(90, 64, 20000, 64, 128, 512)
    st, got1 = _noalloc(lib, inp1, g1)
    assert st == 0
    assert np.array_equal(got1, _with_workspace(inp1, g1))

    inp2, g2 = _inputs(91, 40, 30000, 32, 128, 300)
    stats = pkg.Stats(torch.device(DEV))
    opts = pkg.make_options(pkg.Options(cap_factor=2.0, target_factor=0.5), stats)
    st, got2 = _noalloc(lib, inp2, g2, opts)
    assert st == 0
    rec = stats.read()
    # the rescan really ran, on the plan, histograms and counters the first
    # call left in the shared array
    assert rec["fallback_rows"] > 0 and rec["status"] == 0
    assert np.array_equal(got2, _with_workspace(inp2, g2, pkg.Options(cap_factor=2.0,
                                                                      target_factor=0.5)))


def test_noalloc_sampling_call_after_a_short_rows_call(lib):
    # a call whose rows all fit the slab (no sample, no rescan counters reset)
    # followed by one that samples and rescans: the second must not read
    # anything the first left behind
    import sparse_attention_indexer_tiles_gb300 as pkg
    inp1, g1 = _inputs(93, 48, 3000, 64, 128, 256)
    st, got1 = _noalloc(lib, inp1, g1)
    assert st == 0
    assert np.array_equal(got1, _with_workspace(inp1, g1))

    inp2, g2 = _inputs(94, 24, 40000, 64, 128, 300)
    stats = pkg.Stats(torch.device(DEV))
    opts = pkg.make_options(pkg.Options(cap_factor=2.0, target_factor=0.5), stats)
    st, got2 = _noalloc(lib, inp2, g2, opts)
    assert st == 0
    rec = stats.read()
    assert rec["fallback_rows"] > 0 and rec["status"] == 0
    assert np.array_equal(got2, _with_workspace(inp2, g2, pkg.Options(cap_factor=2.0,
                                                                      target_factor=0.5)))


def test_noalloc_without_rows_still_checks_its_arguments(lib):
    # no rows launches nothing, but an invalid topk is refused as by idx_score_topk
    null = None
    assert lib.idx_score_topk_noalloc(null, null, null, null, null, null, 0, 100, 0, 64, 128, 16,
                                      2, null, null, null) == 0
    assert lib.idx_score_topk_noalloc(null, null, null, null, null, null, 0, 100, 0, 64, 128, 0,
                                      2, null, null, null) == 1  # IDX_EINVAL


def test_noalloc_refuses_problems_beyond_the_array(lib):
    inp, g = _inputs(92, 4096, 65536, 64, 128, 2048)
    st, got = _noalloc(lib, inp, g)
    assert st == 3  # IDX_EWORKSPACE
    assert (got == -7).all()  # nothing was launched

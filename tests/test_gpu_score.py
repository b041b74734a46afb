"""Scoring and fused top-k on the GPU against the oracle.

idx_score_materialise: every score within 1e-3 * max(1, |s|) of the fp64 oracle.
idx_score_topk: the selected sets satisfy the tolerance rule of tests/_checks.py
(recall 1.0), are identical to the two-pass path on the same GPU scores, and
stay exact when the sampled threshold misses (forced short and overflowing
slabs, rows of pure ties)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _checks import check_fused_row, check_row_shape, check_scores

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


def to_dev(inp):
    return {n: getattr(inp, n).to(DEV) for n in ("q", "k", "k_scale", "w", "ks", "ke")}


def materialise(idx, inp, stride=None):
    g = to_dev(inp)
    n_max = int((inp.ke - inp.ks).max())
    stride = stride or max(n_max, 1)
    out = torch.full((inp.rows, stride), float("nan"), device=DEV)
    idx.idx_score_materialise(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def fused(idx, inp, stats=None, **opts):
    g = to_dev(inp)
    out = idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk,
                             options=opts or None, stats=stats)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def two_pass(idx, inp):
    g = to_dev(inp)
    n_max = int((inp.ke - inp.ks).max())
    S = idx.idx_score_materialise(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"],
                                  row_stride=max(n_max, 1))
    out = idx.idx_topk_from_scores(S, g["ks"], g["ke"], inp.topk, options={"relative_rows": 1})
    torch.cuda.synchronize()
    return out.cpu().numpy()


# ------------------------------------------------------------ materialise

@pytest.mark.parametrize("dtype,H,D", [("bf16", 8, 64), ("bf16", 64, 128), ("bf16", 32, 64),
                                       ("fp8", 64, 128), ("fp8", 32, 128), ("fp8", 16, 64),
                                       ("fp8", 8, 128)])
def test_materialise_matches_oracle(idx, dtype, H, D):
    """Several key tiles, a ragged last tile (keys % 128 != 0), row blocks
    with a ragged tail (rows % (256 / H) != 0), causal ranges."""
    rows = 256 // H * 3 + 1
    inp = synth.indexer_inputs(rows, 1000, H, D, 16, dtype, seed=31 + H + D)
    got = materialise(idx, inp)
    _, sc = oracle.score_topk(inp, want_scores=True)
    for r in range(rows):
        n = int(inp.ke[r] - inp.ks[r])
        check_scores(got[r, :n], sc[r, :n])
        assert np.isnan(got[r, n:]).all(), "entries past the visible range must stay untouched"


def test_materialise_tiny_workload(idx):
    inp = synth.workload("tiny")
    got = materialise(idx, inp)
    _, sc = oracle.score_topk(inp, want_scores=True)
    for r in range(inp.rows):
        n = int(inp.ke[r] - inp.ks[r])
        check_scores(got[r, :n], sc[r, :n])


def test_materialise_offsets_and_empty_rows(idx):
    ks = torch.tensor([0, 5, 129, 700, 300, 0, 1000, 999], dtype=torch.int32)
    ke = torch.tensor([0, 900, 130, 1000, 300, 1000, 1000, 1000], dtype=torch.int32)
    inp = synth.indexer_inputs(8, 1000, 32, 128, 16, "fp8", seed=33, ranges="given", ks=ks, ke=ke)
    got = materialise(idx, inp, stride=1000)
    _, sc = oracle.score_topk(inp, want_scores=True)
    for r in range(8):
        n = int(ke[r] - ks[r])
        check_scores(got[r, :n], sc[r, :n])
        assert np.isnan(got[r, n:]).all()


# ------------------------------------------------------------ fused

def check_fused(inp, got, rows=None):
    rows = list(range(inp.rows)) if rows is None else rows
    _, sc = oracle.score_topk(inp, rows=rows, want_scores=True)
    recall = []
    for i, r in enumerate(rows):
        n = int(inp.ke[r] - inp.ks[r])
        recall.append(check_fused_row(got[r], sc[i, :n], inp.topk))
    assert min(recall) == 1.0
    return recall


def test_fused_tiny_workload(idx):
    inp = synth.workload("tiny")
    got = fused(idx, inp)
    check_fused(inp, got)
    assert np.array_equal(got, two_pass(idx, inp))


@pytest.mark.parametrize("dtype,H,D,topk", [("fp8", 64, 128, 64), ("fp8", 32, 128, 100),
                                            ("bf16", 8, 64, 32), ("bf16", 16, 128, 50),
                                            ("fp8", 16, 64, 7)])
def test_fused_sampled_path(idx, dtype, H, D, topk):
    """Rows far longer than the slab: sample, threshold, filter, small top-k."""
    inp = synth.indexer_inputs(256 // H * 2 + 3, 9000, H, D, topk, dtype, seed=40 + H + topk)
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats, cap_factor=4.0)
    check_fused(inp, got)
    assert np.array_equal(got, two_pass(idx, inp)), "fused and two-pass disagree"
    st = stats.read()
    assert st["status"] == 0


def test_fused_equals_two_pass_bitwise(idx):
    """The fused path compares exactly the scores the two-pass path writes, so
    both select the same keys even at ties."""
    inp = synth.indexer_inputs(24, 20000, 64, 128, 256, "fp8", seed=41)
    got = fused(idx, inp, cap_factor=3.0)
    assert np.array_equal(got, two_pass(idx, inp))


def test_tail_blocks_split_into_key_parts(idx):
    """SMs + 3 row blocks (H = 64: 4 rows each): the full wave keeps whole
    blocks and the last three are cut into key parts, each emitting runs of
    its own while whole blocks leave those runs empty.  Every row equals the
    two-pass result bitwise; rows of whole and of split blocks match the
    oracle."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    rows = (sm + 3) * 4
    inp = synth.indexer_inputs(rows, 16384, 64, 128, 512, "fp8", seed=44)
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats)
    assert np.array_equal(got, two_pass(idx, inp))
    assert stats.read()["status"] == 0
    check_fused(inp, got, rows=[0, 1, 5, rows // 2, rows - 13, rows - 12, rows - 7, rows - 1])


@pytest.mark.parametrize("knob,stat", [({"target_factor": 0.3}, "short_rows"),
                                       ({"target_factor": 30.0}, "overflow_rows"),
                                       ({"sample_stride": 997}, None)])
def test_fused_forced_rescan_is_exact(idx, knob, stat):
    inp = synth.indexer_inputs(17, 12000, 32, 128, 200, "fp8", seed=42)
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats, cap_factor=2.0, **knob)
    check_fused(inp, got)
    assert np.array_equal(got, two_pass(idx, inp))
    st = stats.read()
    assert st["status"] == 0
    if stat:
        assert st[stat] > 0 and st["fallback_rows"] >= st[stat], st


def test_fused_all_ties(idx):
    """q = 0: every score is 0, so every row returns its first topk keys; the
    slab overflows and the rescan has to walk all three digits and then take
    the ties in index order."""
    inp = synth.indexer_inputs(9, 10000, 32, 128, 300, "fp8", seed=43)
    inp.q.zero_()
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats, cap_factor=2.0)
    for r in range(inp.rows):
        n = int(inp.ke[r] - inp.ks[r])
        assert got[r].tolist() == list(range(min(300, n))) + [-1] * (300 - min(300, n))
    st = stats.read()
    assert st["fallback_rows"] == 9 and st["status"] == 0


def test_fused_ties_below_positive_keys(idx):
    """Only a few keys score above 0 and every other key ties at exactly 0: the
    rescan keeps all positive keys plus the lowest-index zeros (index digits)."""
    inp = synth.indexer_inputs(6, 12000, 32, 128, 400, "fp8", seed=46)
    inp.q.zero_()
    inp.q[:, 0, 0] = 1.0
    k = inp.k.float()
    k[:, 0] = -1.0
    g = torch.Generator().manual_seed(47)
    pos = torch.randperm(12000, generator=g)[:150]
    k[pos, 0] = torch.rand(150, generator=g) * 4 + 0.5
    inp.k = k.to(torch.float8_e4m3fn)
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats, cap_factor=2.0)
    ref = oracle.score_topk(inp)
    assert np.array_equal(got, ref)
    st = stats.read()
    assert st["fallback_rows"] == 6 and st["status"] == 0


def _two_level_ties(rows, keys, n_top, n_tied, seed):
    """Scores 2.0 on n_top keys, 1.0 on n_tied keys and 0 elsewhere (head 0 and
    dimension 0 only, unit weight and key scale): the sampled threshold falls
    on 1.0, the slab holds every candidate, and the threshold value is a tie of
    n_tied keys that the slab top-k resolves by index."""
    inp = synth.indexer_inputs(rows, keys, 32, 128, 400, "fp8", seed=seed, ranges="full")
    inp.q.zero_()
    inp.q[:, 0, 0] = 1.0
    inp.w[:, 0] = 1.0
    inp.k_scale.fill_(1.0)
    g = torch.Generator().manual_seed(seed + 1)
    k = inp.k.float()
    k[:, 0] = -1.0
    pos = torch.randperm(keys, generator=g)[:n_top + n_tied]
    k[pos[:n_top], 0] = 2.0
    k[pos[n_top:], 0] = 1.0
    inp.k = k.to(torch.float8_e4m3fn)
    return inp


@pytest.mark.parametrize("rows,keys,n_tied,check_rows", [
    (8, 12000, 2500, None),          # one launch of few runs: the streamed slab top-k
    (8, 150000, 3000, [0, 7])])      # key splits into many short runs: the staged one
def test_fused_slab_resolves_a_tied_threshold_bin(idx, rows, keys, n_tied, check_rows):
    """More than 256 candidates in the threshold bin (exact ties at 1.0), no
    rescan: the slab top-k's radix selection over keys, then over the tied
    indices, against the oracle.  (topk 400: cap 4096, stride 31, the sample's
    42nd largest key sets the threshold; (150 + n_tied) / 31 sampled keys reach
    1.0, at least 4.8 standard deviations above 42.)"""
    inp = _two_level_ties(rows, keys, 150, n_tied, seed=60 + keys % 7)
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats)
    st = stats.read()
    assert st["fallback_rows"] == 0 and st["status"] == 0, st
    assert st["max_count"] == 150 + n_tied
    ref = oracle.score_topk(inp, rows=check_rows)
    sel = got if check_rows is None else got[check_rows]
    assert np.array_equal(sel, ref)


def test_fused_mixed_ranges(idx):
    """Rows of one CTA with different visible ranges, empty rows, rows shorter
    than topk (padded with -1) and rows longer than the slab."""
    ks = torch.tensor([0, 0, 5000, 5000, 100, 9000, 0, 7777, 3, 4], dtype=torch.int32)
    ke = torch.tensor([9000, 50, 9000, 5000, 8000, 9100, 9100, 9100, 300, 9100], dtype=torch.int32)
    inp = synth.indexer_inputs(10, 9100, 64, 128, 128, "fp8", seed=44, ranges="given", ks=ks, ke=ke)
    got = fused(idx, inp, cap_factor=3.0)
    check_fused(inp, got)
    assert (got[3] == -1).all()
    assert np.array_equal(got, two_pass(idx, inp))


# --------------------------------------------------- full-size workloads

def _sampled_workload(idx, name, nrows):
    inp = synth.workload(name)
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats)
    rows = synth.sample_rows(inp.ks, inp.ke, nrows, seed=inp.meta["seed"])
    check_fused(inp, got, rows)
    # every row: well formed
    n = (inp.ke - inp.ks).numpy()
    for r in range(inp.rows):
        check_row_shape(got[r], int(n[r]), inp.topk)
    st = stats.read()
    assert st["status"] == 0
    return inp, got, st


def test_fused_prefill_workload(idx):
    _sampled_workload(idx, "fused_prefill", 64)


def test_long_context_workload(idx):
    inp, got, st = _sampled_workload(idx, "long_context", 64)
    print("long-context stats", st)


def test_mixed_batch_workload(idx):
    inp, got, st = _sampled_workload(idx, "mixed_batch", 64)
    n = (inp.ke - inp.ks).numpy()
    short = np.flatnonzero(n < inp.topk)
    assert short.size > 0
    for r in short:
        assert got[r].tolist() == list(range(n[r])) + [-1] * (inp.topk - n[r])


# ------------------------------------------------------ decode-like shapes

@pytest.mark.parametrize("knob", [{}, {"target_factor": 30.0}, {"target_factor": 0.3}])
def test_few_rows_long_keys_key_split(idx, knob):
    """12 rows over 150000 keys (three row blocks): the scoring launches split
    every block's keys over up to eight CTAs, each with runs of its own; the
    rescan (forced by the knobs) re-emits over whole rows."""
    inp = synth.indexer_inputs(12, 150000, 64, 128, 512, "fp8", seed=48, ranges="full")
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats, **knob)
    assert np.array_equal(got, two_pass(idx, inp))
    check_fused(inp, got, rows=[0, 5, 11])
    st = stats.read()
    assert st["status"] == 0
    if knob:
        assert st["fallback_rows"] == 12


def test_materialise_few_rows_long_keys(idx):
    ks = torch.tensor([0, 1000, 0, 77], dtype=torch.int32)
    ke = torch.tensor([90000, 90000, 45000, 89999], dtype=torch.int32)
    inp = synth.indexer_inputs(4, 90000, 32, 128, 16, "fp8", seed=49, ranges="given", ks=ks, ke=ke)
    got = materialise(idx, inp)
    _, sc = oracle.score_topk(inp, rows=[0, 2], want_scores=True)
    for i, r in enumerate([0, 2]):
        n = int(ke[r] - ks[r])
        check_scores(got[r, :n], sc[i, :n])


def test_rows_beyond_max_len_are_reported(idx):
    """A call sized for max_len <= cap takes no sample.  A row longer than that
    bound is reported (IDX_DEV_RANGE, -1 output) and never selected from a
    threshold an earlier call left in the workspace; rows within the bound are
    exact."""
    ks = torch.zeros(8, dtype=torch.int32)
    ke = torch.tensor([3000, 20000, 2500, 20000, 4000, 20000, 100, 20000], dtype=torch.int32)
    inp = synth.indexer_inputs(8, 20000, 64, 128, 256, "fp8", seed=51, ranges="given", ks=ks,
                               ke=ke)
    g = to_dev(inp)
    need = idx.idx_score_topk_workspace(8, 20000, 0, 64, 128, 256, inp.q.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    # a sampled call first: it leaves row plans in the workspace
    first = idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], 256,
                               ws=ws)
    check_fused(inp, first.cpu().numpy())
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], 256,
                             max_len=4096, ws=ws, stats=stats)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    st = stats.read()
    assert st["status"] & 2  # IDX_DEV_RANGE
    long_rows = [1, 3, 5, 7]
    assert (got[long_rows] == -1).all()
    short = [r for r in range(8) if r not in long_rows]
    check_fused(inp, got, rows=short)
    assert np.array_equal(got[short], first.cpu().numpy()[short])


@pytest.mark.parametrize("name", ["fused_prefill", "long_context"])
def test_full_size_scores_on_sampled_rows(idx, name):
    """Every score of 64 seeded rows of a full-size workload, computed by the
    launch configuration of the whole workload (all row blocks, the key split
    the full grid takes, key indices far beyond 2^16), within
    1e-3 * max(1, |s|) of the oracle's fp64 scores."""
    inp = synth.workload(name)
    g = to_dev(inp)
    n = (inp.ke - inp.ks).numpy()
    S = torch.empty(inp.rows, int(n.max()), dtype=torch.float32, device=DEV)
    idx.idx_score_materialise(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], out=S)
    rows = synth.sample_rows(inp.ks, inp.ke, 64, seed=inp.meta["seed"] + 7)
    got = S[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    del S, g
    torch.cuda.empty_cache()
    _, sc = oracle.score_topk(inp, rows=rows, want_scores=True)
    for i, r in enumerate(rows):
        check_scores(got[i, :n[r]], sc[i, :n[r]])


@pytest.mark.parametrize("rows,keys", [(8, 40000), (4, 300000)])
def test_fused_largest_topk(idx, rows, keys):
    """topk 4096, the largest: the default slab clamps to 12288 candidates, and
    the slab top-k writes the output from its bitmap (40000-key rows) or from
    its ordered index list (300000-key rows: beyond the bitmap's 131072)."""
    inp = synth.indexer_inputs(rows, keys, 32, 128, 4096, "fp8", seed=70 + rows, ranges="full")
    stats = idx.Stats(torch.device(DEV))
    got = fused(idx, inp, stats=stats)
    assert np.array_equal(got, two_pass(idx, inp))
    check_fused(inp, got, rows=[0, rows - 1])
    st = stats.read()
    assert st["status"] == 0 and st["fallback_rows"] == 0, st

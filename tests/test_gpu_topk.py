"""idx_topk_from_scores against the oracle, byte for byte (the exact fp32
top-k of "[sglang] ROCm DSA Indexer Top-K 최적화": 12-bit histogram, tie
refinement, full-row rescan when the threshold bin overflows)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


DEV = "cuda:0"


def gpu_topk(idx, scores, ks, ke, topk, **kw):
    out = idx.idx_topk_from_scores(scores.to(DEV), None if ks is None else ks.to(DEV),
                                   ke.to(DEV), topk, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_small_rows_with_ties_and_short_rows(idx):
    si = synth.score_inputs(48, 5000, 300, seed=21, short_frac=0.25)
    got = gpu_topk(idx, si.scores, si.ks, si.ke, 300)
    ref = oracle.topk_from_scores(si.scores, si.ks, si.ke, 300)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("topk", [1, 2, 7, 64, 1000, 2048, 4096])
def test_topk_sizes(idx, topk):
    si = synth.score_inputs(12, 6001, topk, seed=22 + topk, short_frac=0.0)
    got = gpu_topk(idx, si.scores, si.ks, si.ke, topk)
    ref = oracle.topk_from_scores(si.scores, si.ks, si.ke, topk)
    assert np.array_equal(got, ref)


def test_edge_lengths_offsets_and_odd_stride(idx):
    """Rows of length 0, 1, topk-1, topk, topk+1 and longer, starting at odd
    columns of an odd row stride (every alignment of the first element)."""
    topk, stride = 257, 3001
    g = torch.Generator().manual_seed(23)
    S = (torch.randn(16, stride, generator=g) * 0.05).to(torch.bfloat16).float()
    lens = [0, 1, topk - 1, topk, topk + 1, 2 * topk, 1000, 2999, 5, 300, 258, 3000, 17, 1234, 600, 2]
    ks = torch.tensor([(3 * i + 1) % 7 for i in range(16)], dtype=torch.int32)
    ke = torch.tensor([min(int(ks[i]) + lens[i], stride) for i in range(16)], dtype=torch.int32)
    got = gpu_topk(idx, S, ks, ke, topk)
    ref = oracle.topk_from_scores(S, ks, ke, topk)
    assert np.array_equal(got, ref)
    # ks = NULL means every row starts at column 0
    got0 = gpu_topk(idx, S, None, ke - ks, topk)
    ref0 = oracle.topk_from_scores(S, torch.zeros_like(ks), ke - ks, topk)
    assert np.array_equal(got0, ref0)


def test_relative_rows(idx):
    """options.relative_rows: row r's data starts at column 0 although ks > 0."""
    g = torch.Generator().manual_seed(24)
    S = torch.randn(6, 4000, generator=g)
    ks = torch.tensor([0, 10, 100, 1000, 3, 7], dtype=torch.int32)
    ke = ks + torch.tensor([4000, 3990, 2000, 2500, 3997, 100], dtype=torch.int32)
    got = gpu_topk(idx, S, ks, ke, 128, options={"relative_rows": 1})
    ref = oracle.topk_from_scores(S, torch.zeros_like(ks), ke - ks, 128)
    assert np.array_equal(got, ref)


def test_massive_ties_take_the_rescan(idx):
    """Rows whose threshold bin holds far more than the 4096-entry tie buffer:
    all-equal rows, a two-valued row, and +0/-0 mixtures."""
    n, topk = 20000, 1500
    rows = []
    rows.append(np.full(n, 0.25, np.float32))
    two = np.full(n, 1.0, np.float32)
    two[::3] = 2.0  # 6667 keys at 2.0 > topk: the result is the first 1500 of them
    rows.append(two)
    z = np.zeros(n, np.float32)
    z[1::2] = -0.0
    z[5] = 1.0
    rows.append(z)
    near = np.full(n, 1.0, np.float32)
    near[np.arange(0, n, 2)] = np.nextafter(np.float32(1.0), np.float32(2.0))
    rows.append(near)
    S = torch.from_numpy(np.stack(rows))
    ks = torch.zeros(4, dtype=torch.int32)
    ke = torch.full((4,), n, dtype=torch.int32)
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, S, ks, ke, topk, stats=stats)
    ref = oracle.topk_from_scores(S, ks, ke, topk)
    assert np.array_equal(got, ref)
    assert got[0].tolist() == list(range(topk))
    st = stats.read()
    assert st["tie_rescan_rows"] >= 3 and st["status"] == 0


def test_one_pass_refinement_paths(idx):
    """Rows long enough for the sampled lower bound (more than 512 values per
    warp), one per branch of the refinement over the collected candidates:
    fp32 scores (the threshold bin holds several keys: a second histogram),
    bf16-grid scores (one key per bin), k planted values far above the rest
    (the boundary lands in the open last bin: the three-level refinement), a
    threshold among +0 and -0 (the float bound +0 admits -0), and an ascending
    row (the sample misses: the exact multi-pass path)."""
    n, topk = 40000, 1500
    g = torch.Generator().manual_seed(27)
    rows = [torch.randn(n, generator=g),
            (torch.randn(n, generator=g) * 0.05).to(torch.bfloat16).float()]
    planted = torch.randn(n, generator=g)
    pos = torch.randperm(n, generator=g)[:topk]
    planted[pos] = 100.0 + torch.arange(topk, dtype=torch.float32) * 1e-3
    rows.append(planted)
    z = -torch.rand(n, generator=g) - 0.5  # negative bulk
    perm = torch.randperm(n, generator=g)
    z[perm[:1000]] = torch.rand(1000, generator=g) + 0.5  # 1000 positives
    z[perm[1000:2000]] = 0.0
    z[perm[2000:3000]] = -0.0
    rows.append(z)
    rows.append(torch.arange(n, dtype=torch.float32))
    S = torch.stack(rows)
    R = S.shape[0]
    ks = torch.zeros(R, dtype=torch.int32)
    ke = torch.full((R,), n, dtype=torch.int32)
    got = gpu_topk(idx, S, ks, ke, topk)
    ref = oracle.topk_from_scores(S, ks, ke, topk)
    assert np.array_equal(got, ref)


def test_extreme_values(idx):
    g = torch.Generator().manual_seed(25)
    S = torch.randn(4, 7000, generator=g) * 1e30
    S[0, :100] = -3.4e38
    S[1, 50:60] = 3.4e38
    S[2] = -torch.rand(7000, generator=g)  # all negative
    S[3, ::2] = 1e-40  # subnormals
    ks = torch.zeros(4, dtype=torch.int32)
    ke = torch.full((4,), 7000, dtype=torch.int32)
    got = gpu_topk(idx, S, ks, ke, 999)
    ref = oracle.topk_from_scores(S, ks, ke, 999)
    assert np.array_equal(got, ref)


def test_standalone_workload_full(idx):
    """1024 rows x 131072 keys, topk 2048, bf16-grid N(0, 0.05), 5% short rows:
    every row against the oracle."""
    si = synth.workload("standalone_topk")
    got = gpu_topk(idx, si.scores, si.ks, si.ke, 2048)
    ref = oracle.topk_from_scores(si.scores, si.ks, si.ke, 2048)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------ row split

def test_row_split_workload(idx):
    """8 rows x 1M keys: the automatic rule splits every row over g blocks
    (g = min(SMs / rows, 32)); bit-exact on every row."""
    si = synth.workload("split_topk")
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, si.scores, si.ks, si.ke, 2048, stats=stats)
    ref = oracle.topk_from_scores(si.scores, si.ks, si.ke, 2048)
    assert np.array_equal(got, ref)
    st = stats.read()
    assert st["split_rows"] == 8 and st["status"] == 0


@pytest.mark.parametrize("g", [2, 5, 9])
def test_forced_row_split(idx, g):
    si = synth.score_inputs(12, 70000, 700, seed=26 + g, short_frac=0.2)
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, si.scores, si.ks, si.ke, 700, options={"row_split": g}, stats=stats)
    ref = oracle.topk_from_scores(si.scores, si.ks, si.ke, 700)
    assert np.array_equal(got, ref)
    assert stats.read()["split_rows"] > 0


@pytest.mark.parametrize("row_split", [-1, 0])
def test_long_rows_small_topk_keep_the_one_pass_bound(idx, row_split):
    """512K keys per row, topk 512: the sample holds only a few keys above a
    row's 512th largest (m = k P / n ~ 8 of 8192, ~4 per split slice), so the
    sample rank carries a margin of spreads above m rather than a fixed
    multiple of it; no row falls back to the exact multi-pass path, unsplit or
    split, and the result is exact."""
    si = synth.score_inputs(16, 1 << 19, 512, seed=31, short_frac=0.0, bf16_grid=False)
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, si.scores, si.ks, si.ke, 512, options={"row_split": row_split},
                   stats=stats)
    ref = oracle.topk_from_scores(si.scores, si.ks, si.ke, 512)
    assert np.array_equal(got, ref)
    st = stats.read()
    assert st["tie_rescan_rows"] == 0 and st["status"] == 0, st
    assert st["split_rows"] == (0 if row_split == -1 else 16)


def test_row_split_merge_refinement_paths(idx):
    """The merge block's refinement over the slices' candidates, one row per
    branch: fp32 scores (several keys in the threshold bin: a second
    histogram), bf16-grid scores (one key per bin), k planted values far above
    the rest (the open last bin: refinement by absolute digits) and a
    threshold among +0 and -0."""
    n, topk = 120000, 1500
    g = torch.Generator().manual_seed(44)
    rows = [torch.randn(n, generator=g),
            (torch.randn(n, generator=g) * 0.05).to(torch.bfloat16).float()]
    planted = torch.randn(n, generator=g)
    planted[torch.randperm(n, generator=g)[:topk]] = 100.0 + torch.arange(topk) * 1e-3
    rows.append(planted)
    z = -torch.rand(n, generator=g) - 0.5
    perm = torch.randperm(n, generator=g)
    z[perm[:1000]] = torch.rand(1000, generator=g) + 0.5
    z[perm[1000:2500]] = 0.0
    z[perm[2500:4000]] = -0.0
    rows.append(z)
    S = torch.stack(rows)
    R = S.shape[0]
    ks = torch.zeros(R, dtype=torch.int32)
    ke = torch.full((R,), n, dtype=torch.int32)
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, S, ks, ke, topk, options={"row_split": 4}, stats=stats)
    ref = oracle.topk_from_scores(S, ks, ke, topk)
    assert np.array_equal(got, ref)
    assert stats.read()["split_rows"] == R


def test_row_split_with_empty_slices_and_a_reused_workspace(idx):
    """64 blocks per row (the most a split takes), rows from just above topk
    (most blocks get an empty slice) to 70000 keys, ragged starts; two calls
    on the same workspace (the per-row tickets start at 0 every launch)."""
    rows, n, topk = 10, 70000, 100
    si = synth.score_inputs(rows, n, topk, seed=41, short_frac=0.0)
    ks = torch.tensor([0, 5, 0, 3, 0, 17, 1, 0, 2, 9], dtype=torch.int32)
    ke = ks + torch.tensor([101, 150, 257, 1000, 4099, 65536, 69999 - 1, 300, 8191, 50000],
                           dtype=torch.int32)
    ke = torch.minimum(ke, torch.full_like(ke, n))
    opts = {"row_split": 64}
    S = si.scores.to(DEV)
    need = idx.idx_topk_workspace(rows, n, topk, opts)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)  # stale bytes
    ref = oracle.topk_from_scores(si.scores, ks, ke, topk)
    for _ in range(2):
        stats = idx.Stats(torch.device(DEV))
        got = idx.idx_topk_from_scores(S, ks.to(DEV), ke.to(DEV), topk, ws=ws, options=opts,
                                       stats=stats)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), ref)
        assert stats.read()["split_rows"] == rows and stats.read()["status"] == 0


def test_row_split_bound_above_the_kth_falls_back(idx):
    """A block takes its lower bound from the first two float4 slots of every
    lane of each warp's part of its slice (512 threads, 16 warps).  Row 0's
    first slice holds 10.0 exactly there (96 values, enough to set its bound
    above 5.0) and 5.0 at 500 other places: values of the top k that this
    block leaves out.  The selected threshold then lies below the block's
    bound, and the row must be re-selected exactly."""
    n, topk, g = 90000, 1000, 6
    gen = torch.Generator().manual_seed(43)
    S = torch.rand(2, n, generator=gen)
    nvec = n // 4
    per = -(-nvec // g)                  # float4 slots per block
    seg = -(-per // 16)                  # per warp of block 0
    S[0, :4 * per] = 0.0
    for w in range(16):
        S[0, 4 * seg * w: 4 * seg * w + 6] = 10.0
    outside = [p for p in range(4 * per) if p % (4 * seg) >= 256]  # not sampled
    S[0, outside[::20][:500]] = 5.0
    ks = torch.zeros(2, dtype=torch.int32)
    ke = torch.full((2,), n, dtype=torch.int32)
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, S, ks, ke, topk, options={"row_split": g}, stats=stats)
    ref = oracle.topk_from_scores(S, ks, ke, topk)
    assert np.array_equal(got, ref)
    st = stats.read()
    assert st["split_rows"] == 2 and st["tie_rescan_rows"] >= 1 and st["status"] == 0


def test_row_split_ties_fall_back(idx):
    """All-equal and two-valued rows overflow the split candidate runs; the
    merge block re-selects them exactly."""
    n, topk = 90000, 1000
    S = torch.full((3, n), 0.5)
    S[1, ::7] = 2.0
    S[2] = torch.arange(n, dtype=torch.float32) % 3
    ks = torch.zeros(3, dtype=torch.int32)
    ke = torch.full((3,), n, dtype=torch.int32)
    stats = idx.Stats(torch.device(DEV))
    got = gpu_topk(idx, S, ks, ke, topk, options={"row_split": 6}, stats=stats)
    ref = oracle.topk_from_scores(S, ks, ke, topk)
    assert np.array_equal(got, ref)
    st = stats.read()
    assert st["split_rows"] == 3 and st["tie_rescan_rows"] >= 2

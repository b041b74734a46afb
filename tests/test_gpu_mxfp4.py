"""MXFP4 inputs (page "[sglang] logits를 쓰지 않는 top-k", section 1: an fp4
indexer over 64-byte keys) on the GPU.

idx_mxfp4_to_e4m3 expands e2m1 elements with e8m0 block scales to e4m3 exactly
(every such value with a block exponent in [-8, 6] is an e4m3 value): checked
byte for byte against torch's rounding of the decoded values, which is exact
for them, and out-of-range scales raise IDX_DEV_RANGE.  The MXFP4 entry points
score through that expansion: scores against the oracle's MXFP4 scores within
1e-3 * max(1, |s|), selections by the tolerance rule, and bit-identical to the
e4m3 path on the expanded values."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _checks import check_fused_row, check_scores

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
IDX_DEV_RANGE = 0x2
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


def decode(x, sf):
    """fp64 values of MXFP4 rows x [n, D/2], sf [n, D/32] (the format's definition)."""
    x, sf = x.numpy(), sf.numpy()
    lo, hi = x & 15, x >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(x.shape[0], -1)
    mag = np.array(E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
    return mag * np.repeat(scale, 32, axis=1)


def test_expansion_is_exact_in_range(idx):
    g = torch.Generator().manual_seed(81)
    n, D = 300, 128
    x = torch.randint(0, 256, (n, D // 2), generator=g, dtype=torch.uint8)
    sf = torch.randint(127 - 8, 127 + 7, (n, D // 32), generator=g, dtype=torch.uint8)
    sf[0, :] = torch.tensor([127 - 8, 127 - 7, 127 + 5, 127 + 6], dtype=torch.uint8)
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_mxfp4_to_e4m3(x.to(DEV), sf.to(DEV), stats=stats)
    torch.cuda.synchronize()
    want = torch.from_numpy(decode(x, sf)).to(torch.float32).to(torch.float8_e4m3fn)
    assert torch.equal(got.cpu().view(torch.uint8), want.view(torch.uint8))
    assert stats.read()["status"] == 0


def test_expansion_every_scale_code(idx):
    """All 256 e8m0 codes in one launch, in-range and out-of-range blocks side
    by side within a warp: an element exact in e4m3 is that value, one above
    448 saturates to ±448, one below the subnormals (or between two of them)
    flushes to ±0, signs kept (the NaN code 255 reads as 2^128: everything
    nonzero saturates), and the launch raises IDX_DEV_RANGE."""
    g = torch.Generator().manual_seed(83)
    n, D = 256, 128
    x = torch.randint(0, 256, (n, D // 2), generator=g, dtype=torch.uint8)
    sf = (torch.randperm(n * D // 32, generator=g) % 256).to(torch.uint8).reshape(n, D // 32)
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_mxfp4_to_e4m3(x.to(DEV), sf.to(DEV), stats=stats)
    torch.cuda.synchronize()
    v = decode(x, sf)
    f8 = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn)
    exact = f8.to(torch.float64).numpy() == v
    sign = np.where(np.signbit(v), 0x80, 0x00)
    want = np.where(exact, f8.view(torch.uint8).numpy(),
                    np.where(np.abs(v) > 448.0, sign | 0x7E, sign)).astype(np.uint8)
    assert (~exact).any() and exact.any()
    assert np.array_equal(got.cpu().view(torch.uint8).numpy(), want)
    assert stats.read()["status"] & IDX_DEV_RANGE


@pytest.mark.parametrize("code,what", [(127 + 7, "saturates"), (127 - 12, "flushes")])
def test_expansion_out_of_range_raises(idx, code, what):
    x = torch.full((4, 32), 0x77, dtype=torch.uint8)  # every element 6.0
    sf = torch.full((4, 2), 127, dtype=torch.uint8)
    sf[2, 1] = code
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_mxfp4_to_e4m3(x.to(DEV), sf.to(DEV), stats=stats)
    torch.cuda.synchronize()
    assert stats.read()["status"] & IDX_DEV_RANGE
    v = got.cpu().to(torch.float32)  # [4, 64]: row 2's second block has the odd scale
    assert (v[:2] == 6.0).all() and (v[3] == 6.0).all() and (v[2, :32] == 6.0).all()
    assert (v[2, 32:] == (448.0 if what == "saturates" else 0.0)).all()


@pytest.mark.parametrize("H,D", [(64, 128), (32, 128), (16, 64)])
def test_materialise_matches_oracle(idx, H, D):
    rows = 256 // H * 2 + 3
    inp = synth.indexer_inputs(rows, 900, H, D, 16, "mxfp4", seed=82 + H)
    g = {n: getattr(inp, n).to(DEV) for n in ("q", "q_sf", "k", "k_sf", "k_scale", "w", "ks",
                                              "ke")}
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_score_materialise_mxfp4(g["q"], g["q_sf"], g["k"], g["k_sf"], g["k_scale"],
                                          g["w"], g["ks"], g["ke"], stats=stats)
    torch.cuda.synchronize()
    assert stats.read()["status"] == 0
    got = got.cpu().numpy()
    _, sc = oracle.score_topk(inp, want_scores=True)
    for r in range(rows):
        n = int(inp.ke[r] - inp.ks[r])
        check_scores(got[r, :n], sc[r, :n])


def test_fused_selection_and_e4m3_equality(idx):
    """Rows longer than the slab (sampled thresholds) and shorter ones; the
    result equals the e4m3 path on the expanded values, bit for bit."""
    inp = synth.indexer_inputs(24, 20000, 64, 128, 512, "mxfp4", seed=85)
    g = {n: getattr(inp, n).to(DEV) for n in ("q", "q_sf", "k", "k_sf", "k_scale", "w", "ks",
                                              "ke")}
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_score_topk_mxfp4(g["q"], g["q_sf"], g["k"], g["k_sf"], g["k_scale"], g["w"],
                                   g["ks"], g["ke"], inp.topk, options={"cap_factor": 3.0},
                                   stats=stats)
    q8 = idx.idx_mxfp4_to_e4m3(g["q"], g["q_sf"])
    k8 = idx.idx_mxfp4_to_e4m3(g["k"], g["k_sf"])
    ref8 = idx.idx_score_topk(q8, k8, g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk,
                              options={"cap_factor": 3.0})
    torch.cuda.synchronize()
    assert stats.read()["status"] == 0
    got = got.cpu().numpy()
    assert np.array_equal(got, ref8.cpu().numpy())
    _, sc = oracle.score_topk(inp, want_scores=True)
    for r in range(inp.rows):
        n = int(inp.ke[r] - inp.ks[r])
        assert check_fused_row(got[r], sc[r, :n], inp.topk) == 1.0

"""idx_score_topk_routed: the same indices as the fused path on both sides of
the gate ("[sglang] logits를 쓰지 않는 top-k", section 4: fused only when the
longest row sees enough keys), and within the oracle's tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _checks import check_fused_row

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


def call(idx, fn, inp, **kw):
    g = {n: getattr(inp, n).to(DEV) for n in ("q", "k", "k_scale", "w", "ks", "ke")}
    out = fn(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("keys,H,topk,few,dense", [
    (6144, 64, 512, False, True), (9000, 32, 300, False, True), (20000, 16, 128, False, True),
    (24576, 64, 256, False, False), (30000, 16, 128, False, False), (3000, 64, 512, False, False),
    (65536, 32, 512, True, True)])      # few rows over long keys: the two-pass route
def test_routed_equals_fused(idx, keys, H, topk, few, dense):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    rows = 12 if few else max(256 // H * 4 + 3, sm // 4 + 1)
    assert idx.idx_route_fused(rows, keys, topk) == (not dense)
    inp = synth.indexer_inputs(rows, keys, H, 128, topk, "fp8", seed=80 + H)
    stats = idx.Stats(torch.device(DEV))
    got = call(idx, idx.idx_score_topk_routed, inp, stats=stats)
    ref = call(idx, idx.idx_score_topk, inp)
    assert np.array_equal(got, ref)
    assert stats.read()["status"] == 0
    rows = synth.sample_rows(inp.ks, inp.ke, 6, seed=81)
    _, sc = oracle.score_topk(inp, rows=rows, want_scores=True)
    for i, r in enumerate(rows):
        n = int(inp.ke[r] - inp.ks[r])
        assert check_fused_row(got[r], sc[i, :n], topk) == 1.0


def test_dense_route_mixed_ranges(idx):
    """Short-context batch with empty rows and rows shorter than topk."""
    ks = torch.tensor([0, 0, 3000, 3000, 100, 4000, 0, 10], dtype=torch.int32)
    ke = torch.tensor([5000, 40, 5000, 3000, 4000, 5100, 5100, 5100], dtype=torch.int32)
    inp = synth.indexer_inputs(8, 5100, 64, 128, 128, "fp8", seed=82, ranges="given", ks=ks,
                               ke=ke)
    got = call(idx, idx.idx_score_topk_routed, inp)
    ref = call(idx, idx.idx_score_topk, inp)
    assert np.array_equal(got, ref)
    assert (got[3] == -1).all() and got[1].tolist() == list(range(40)) + [-1] * 88

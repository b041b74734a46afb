"""The scoring kernel's bounded waits, run out on purpose.

Every wait of the scoring pipeline (producer on a free stage, MMA issuer on a
loaded stage or a free TMEM buffer, epilogue on a finished accumulator) gives
up after a limit, raises IDX_DEV_TIMEOUT and releases every other wait of the
CTA, which then drains what it already started and returns.  The test option
`test_stall_us` withholds the copy of key tile 1 of every scoring pass and
shortens the limit, so the MMA issuer's wait on that tile runs out.  Nothing
faults and nothing hangs: the call returns, the status word carries the
timeout bit, and the same context then computes a normal call exactly."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from _checks import check_fused_row, check_scores

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
IDX_DEV_TIMEOUT = 0x1


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


def test_withheld_tile_times_out_and_the_context_stays_usable(idx):
    # 8 rows of H = 64: two row blocks (two CTAs), 16 key tiles each
    inp = synth.indexer_inputs(8, 2048, 64, 128, 256, "fp8", seed=77)
    g = {n: getattr(inp, n).to(DEV) for n in ("q", "k", "k_scale", "w", "ks", "ke")}
    args = (g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"])
    stats = idx.Stats(DEV)

    # the materialising pass: one launch
    out = torch.full((8, 2048), float("nan"), device=DEV)
    t0 = time.time()
    idx.idx_score_materialise(*args, out=out, options={"test_stall_us": 200}, stats=stats)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30
    assert stats.read()["status"] & IDX_DEV_TIMEOUT

    # the fused call (sample, emit and the rescan all stall) returns as well
    stats.reset()
    idx.idx_score_topk(*args, inp.topk, options={"test_stall_us": 200, "cap_factor": 4.0},
                       stats=stats)
    torch.cuda.synchronize()
    assert stats.read()["status"] & IDX_DEV_TIMEOUT

    # the context is intact: normal calls match the oracle
    stats.reset()
    out.fill_(float("nan"))
    idx.idx_score_materialise(*args, out=out, stats=stats)
    sel = idx.idx_score_topk(*args, inp.topk, stats=stats)
    torch.cuda.synchronize()
    assert stats.read()["status"] == 0
    got, sel = out.cpu().numpy(), sel.cpu().numpy()
    _, sc = oracle.score_topk(inp, want_scores=True)
    for r in range(8):
        n = int(inp.ke[r] - inp.ks[r])
        check_scores(got[r, :n], sc[r, :n])
        assert np.isnan(got[r, n:]).all()
        assert check_fused_row(sel[r], sc[r, :n], inp.topk) == 1.0

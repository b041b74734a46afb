"""idx_score_topk_host: the fused call on inputs and output in host memory
(the rows in chunks whose copies overlap the compute) against idx_score_topk on
the same inputs on the device: identical indices, in every chunking, on the
caller's stream, and for calls queued back to back on one workspace."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NAMES = ("q", "k", "k_scale", "w", "ks", "ke")


@pytest.fixture(scope="module")
def idx():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_tiles_gb300 as pkg
    return pkg


def host_inputs(inp, pinned=True):
    host = {n: getattr(inp, n).contiguous() for n in NAMES}
    return {n: t.pin_memory() for n, t in host.items()} if pinned else host


def device_result(idx, inp):
    g = {n: getattr(inp, n).to(DEV) for n in NAMES}
    out = idx.idx_score_topk(*[g[n] for n in NAMES], inp.topk)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("rows,keys,H,D,topk,dtype,pinned", [
    (600, 20000, 64, 128, 256, "fp8", True),   # two chunks of 75 row blocks
    (77, 9000, 32, 128, 100, "bf16", False),   # pageable memory; chunks of 40 and 37 rows
    (3, 5000, 16, 64, 64, "fp8", True)])       # less than one row block: a single chunk
def test_host_entry_matches_device_entry(idx, rows, keys, H, D, topk, dtype, pinned):
    inp = synth.indexer_inputs(rows, keys, H, D, topk, dtype, seed=90 + rows)
    host = host_inputs(inp, pinned)
    stats = idx.Stats(torch.device(DEV))
    got = idx.idx_score_topk_host(*[host[n] for n in NAMES], topk, stats=stats)
    torch.cuda.synchronize()
    assert torch.equal(got, device_result(idx, inp))
    assert stats.read()["status"] == 0


def test_result_is_complete_when_the_callers_stream_is(idx):
    """Synchronising only the stream passed to the call is enough."""
    inp = synth.indexer_inputs(300, 30000, 64, 128, 512, "fp8", seed=95)
    host = host_inputs(inp)
    s = torch.cuda.Stream()
    out = torch.full((inp.rows, inp.topk), -7, dtype=torch.int32).pin_memory()
    idx.idx_score_topk_host(*[host[n] for n in NAMES], inp.topk, out=out, stream=s)
    s.synchronize()
    assert torch.equal(out, device_result(idx, inp))


def test_back_to_back_calls_on_one_workspace(idx):
    """The second call's copies into the shared workspace wait for the first
    call's compute and copies back."""
    a = synth.indexer_inputs(400, 25000, 64, 128, 256, "fp8", seed=96)
    b = synth.indexer_inputs(400, 25000, 64, 128, 256, "fp8", seed=97)
    ha, hb = host_inputs(a), host_inputs(b)
    need = idx.idx_score_topk_host_workspace(a.rows, a.keys, 0, a.H, a.D, a.topk, a.q.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out_a = idx.idx_score_topk_host(*[ha[n] for n in NAMES], a.topk, ws=ws)
    out_b = idx.idx_score_topk_host(*[hb[n] for n in NAMES], b.topk, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_a, device_result(idx, a))
    assert torch.equal(out_b, device_result(idx, b))
    assert not torch.equal(out_a, out_b)

"""The seeded input generators: determinism, shapes and the stated recipes."""
import math

import numpy as np
import torch

import synth


def test_generators_are_deterministic():
    a = synth.indexer_inputs(8, 500, 8, 64, 16, "fp8", seed=3)
    b = synth.indexer_inputs(8, 500, 8, 64, 16, "fp8", seed=3)
    for x, y in [(a.q, b.q), (a.k, b.k), (a.w, b.w), (a.k_scale, b.k_scale)]:
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    c = synth.indexer_inputs(8, 500, 8, 64, 16, "fp8", seed=4)
    assert not torch.equal(a.k.view(torch.uint8), c.k.view(torch.uint8))


def test_causal_ranges():
    ks, ke = synth.causal_ranges(4, 10)
    assert ks.tolist() == [0, 0, 0, 0] and ke.tolist() == [7, 8, 9, 10]


def test_tiny_workload_recipe():
    t = synth.workload("tiny")
    assert (t.rows, t.keys, t.H, t.D, t.topk) == (64, 4096, 8, 64, 256)
    assert t.q.dtype == torch.bfloat16 and t.k.dtype == torch.bfloat16
    assert torch.all(t.k_scale == 1.0)
    assert float(t.w.min()) >= 0 and float(t.w.max()) <= 1.0 / 8
    assert int(t.ke[0]) == 4096 - 64 + 1 and int(t.ke[-1]) == 4096


def test_planted_runs_and_factor():
    f = synth.planted_scale_factor(32, 128)
    assert 1.8 < f < 2.0
    inp = synth.indexer_inputs(16, 20000, 32, 128, 64, "fp8", seed=5, planted_runs=8)
    starts = inp.meta["planted_starts"]
    assert len(starts) == 8 and all(s % 64 for s in starts)
    assert all(b - a >= 64 for a, b in zip(starts, starts[1:]))
    assert max(starts) + 64 <= 20000 - 16


def test_score_inputs_short_rows_and_ties():
    s = synth.score_inputs(100, 4096, 256, seed=1)
    short = s.meta["short_rows"]
    assert len(short) == 5
    assert all(int(s.ke[r]) < 256 for r in short)
    x = s.scores[0].numpy()
    assert np.array_equal(x, torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    assert len(np.unique(x)) < x.size // 2  # dense clustering on the bf16 grid


def test_mixed_batch_lengths_are_log_uniform():
    g = torch.Generator().manual_seed(0)
    L = synth.mixed_batch_lengths(20000, 256, 262144, g).numpy()
    assert L.min() >= 256 and L.max() <= 262144
    logs = np.log(L)
    assert abs(np.median(logs) - 0.5 * (math.log(256) + math.log(262144))) < 0.1


def test_sample_rows_keeps_extremes():
    ks = torch.zeros(500, dtype=torch.int32)
    ke = torch.arange(1, 501, dtype=torch.int32)
    rows = synth.sample_rows(ks, ke, 64, seed=2)
    assert len(rows) == 64 and 0 in rows and 499 in rows
    assert rows == synth.sample_rows(ks, ke, 64, seed=2)


def test_mxfp4_encoding_recipe():
    """quantise_mxfp4: each block's scale puts its largest magnitude in [4, 8)
    (e = floor(log2 max|x|) - 2), every element is the nearest e2m1 value of
    x / 2^e with ties to even and saturation at 6 (checked against ml_dtypes'
    own rounding), two codes per byte with element 2i in the low nibble, and
    the generator draws q and k from the same random stream as fp8/bf16."""
    import pytest
    mld = pytest.importorskip("ml_dtypes")
    g = torch.Generator().manual_seed(1)
    x = torch.randn(5, 3, 128, generator=g)
    x[0, 0, :32] = 0.0                       # an all-zero block
    x[0, 1, :32] = torch.linspace(-6, 6, 32)  # exact grid points and halves
    codes, sf = synth.quantise_mxfp4(x)
    assert codes.shape == (5, 3, 64) and sf.shape == (5, 3, 4)
    assert codes.dtype == torch.uint8 and sf.dtype == torch.uint8
    scale = np.ldexp(1.0, sf.numpy().astype(np.int64) - 127)
    xb = x.double().numpy().reshape(5, 3, 4, 32)
    amax = np.abs(xb).max(-1)
    nz = amax > 0
    assert np.all((amax[nz] / scale[nz] >= 4) & (amax[nz] / scale[nz] < 8))
    el = np.stack([codes.numpy() & 0xF, codes.numpy() >> 4], -1).reshape(5, 3, 128)
    got = np.frombuffer(el.astype(np.uint8).tobytes(), dtype=mld.float4_e2m1fn)
    got = got.astype(np.float64).reshape(5, 3, 4, 32)
    ref = np.clip(xb / scale[..., None], -6, 6).astype(mld.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(got, ref)
    mx = synth.indexer_inputs(4, 100, 2, 64, 8, "mxfp4", seed=5)
    e4 = synth.indexer_inputs(4, 100, 2, 64, 8, "fp8", seed=5)
    assert torch.equal(mx.w, e4.w) and torch.equal(mx.k_scale, e4.k_scale)
    assert mx.q.shape == (4, 2, 32) and mx.k_sf.shape == (100, 2) and mx.D == 64

"""Pins of the CPU oracle against facts that do not come from the oracle itself:
the bit formats (checked against torch's own casts), a hand-worked example, closed
forms of the score, identities of ReLU, brute-force subset enumeration of the
selection rule, and invariants of every returned index set."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- decoders

def test_e4m3_decoder_exhaustive_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    # format landmarks: max normal, smallest subnormal, one, sign
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    assert got[0xB8] == -1.0 and got[0x08] == 2.0 ** -6


def test_bf16_decoder_exhaustive_matches_torch(orc):
    codes = np.arange(65536, dtype=np.uint32)
    ref = torch.from_numpy(codes.astype(np.int32).astype(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()
    got = orc.bf16_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x3F80] == 1.0 and got[0x7F80] == math.inf and got[0x0001] == 2.0 ** -133


# ------------------------------------------------------- hand-worked example

def _golden_inputs(g, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float8_e4m3fn
    q = torch.tensor(g["q"], dtype=torch.float32).to(tdt)
    k = torch.tensor(g["k"], dtype=torch.float32).to(tdt)
    # every value of the fixture is exact in both formats
    assert torch.equal(q.float(), torch.tensor(g["q"])) and torch.equal(k.float(), torch.tensor(g["k"]))
    return q, k


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_hand_worked_example(orc, dtype):
    g = json.load(open(os.path.join(GOLDEN, "hand_scores.json")))
    q, k = _golden_inputs(g, dtype)
    w = torch.tensor(g["w"], dtype=torch.float32)
    sc = torch.tensor(g["k_scale"], dtype=torch.float32)
    full = synth.indexer_inputs  # noqa: F841  (shapes only come from the fixture)
    for case in g["cases"]:
        inp = synth.IndexerInputs(q=q, k=k, k_scale=sc, w=w,
                                  ks=torch.tensor([case["ks"]], dtype=torch.int32),
                                  ke=torch.tensor([case["ke"]], dtype=torch.int32),
                                  topk=case["topk"])
        s = orc.scores_row(inp, 0)
        assert s.tolist() == g["scores_full"][case["ks"]:case["ke"]]
        got = orc.score_topk(inp, nthreads=1)[0].tolist()
        assert got == case["expect"], case["why"]


# ---------------------------------------------------------- score closed forms

@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_unit_query_reads_first_coordinate(orc, dtype):
    """H=1, w=1, scale=1, q=e_0  =>  s_j = ReLU(k[j,0])."""
    inp = synth.indexer_inputs(1, 300, 1, 64, 8, dtype, seed=11, ranges="full", scale="one")
    inp.q.zero_()
    inp.q[0, 0, 0] = 1.0
    inp.w.fill_(1.0)
    s = orc.scores_row(inp, 0)
    k0 = inp.k[:, 0].to(torch.float64).numpy()
    assert np.array_equal(s, np.maximum(k0, 0.0))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_relu_identity_gives_the_dot_product(orc, dtype):
    """ReLU(x) - ReLU(-x) = x: for H=1, w=1, scale=1 the difference of the
    scores of q and -q is q.k_j, here compared with a numpy matmul of the
    torch-decoded inputs.  A dropped ReLU, a wrong d index or a transposed
    operand breaks it."""
    inp = synth.indexer_inputs(1, 257, 1, 128, 8, dtype, seed=12, ranges="full", scale="one")
    inp.w.fill_(1.0)
    pos = orc.scores_row(inp, 0)
    neg_inp = synth.IndexerInputs(q=(-inp.q.float()).to(inp.q.dtype), k=inp.k, k_scale=inp.k_scale,
                                  w=inp.w, ks=inp.ks, ke=inp.ke, topk=8)
    neg = orc.scores_row(neg_inp, 0)
    dots = inp.k.to(torch.float64).numpy() @ inp.q[0, 0].to(torch.float64).numpy()
    np.testing.assert_allclose(pos - neg, dots, rtol=1e-12, atol=1e-12)
    assert (pos >= 0).all() and (neg >= 0).all()
    assert np.all((pos == 0) | (neg == 0))  # only one side of ReLU is open


def test_heads_weights_and_scale_are_linear(orc):
    """Doubling w doubles s; k_scale multiplies s per key; swapping two heads
    (q and w together) leaves s unchanged; a head with w=0 contributes
    nothing; every row uses its own q and w."""
    inp = synth.indexer_inputs(3, 200, 4, 64, 8, "bf16", seed=13, ranges="full", scale="one")
    base = np.stack([orc.scores_row(inp, r) for r in range(3)])
    inp2 = synth.IndexerInputs(q=inp.q, k=inp.k, k_scale=inp.k_scale, w=inp.w * 2, ks=inp.ks,
                               ke=inp.ke, topk=8)
    assert np.array_equal(np.stack([orc.scores_row(inp2, r) for r in range(3)]), 2 * base)
    sc = torch.arange(1, 201, dtype=torch.float32)
    inp3 = synth.IndexerInputs(q=inp.q, k=inp.k, k_scale=sc, w=inp.w, ks=inp.ks, ke=inp.ke, topk=8)
    np.testing.assert_allclose(np.stack([orc.scores_row(inp3, r) for r in range(3)]),
                               base * sc.numpy()[None, :], rtol=1e-15)
    perm = [2, 0, 3, 1]
    inp4 = synth.IndexerInputs(q=inp.q[:, perm].contiguous(), k=inp.k, k_scale=inp.k_scale,
                               w=inp.w[:, perm].contiguous(), ks=inp.ks, ke=inp.ke, topk=8)
    np.testing.assert_allclose(np.stack([orc.scores_row(inp4, r) for r in range(3)]), base,
                               rtol=1e-14)
    # single head kept: equals w_h * ReLU(q_h . k) from the decoded inputs
    w1 = torch.zeros_like(inp.w)
    w1[1, 2] = 0.75
    inp5 = synth.IndexerInputs(q=inp.q, k=inp.k, k_scale=inp.k_scale, w=w1, ks=inp.ks, ke=inp.ke,
                               topk=8)
    s5 = np.stack([orc.scores_row(inp5, r) for r in range(3)])
    dots = inp.k.to(torch.float64).numpy() @ inp.q[1, 2].to(torch.float64).numpy()
    assert np.array_equal(s5[0], np.zeros(200)) and np.array_equal(s5[2], np.zeros(200))
    np.testing.assert_allclose(s5[1], 0.75 * np.maximum(dots, 0), rtol=1e-14)


def test_zero_query_selects_the_first_keys(orc):
    """q = 0  =>  every score is 0  =>  the first topk visible keys."""
    inp = synth.indexer_inputs(4, 500, 8, 64, 37, "fp8", seed=14)
    inp.q.zero_()
    out = orc.score_topk(inp, nthreads=2)
    for r in range(4):
        n = int(inp.ke[r] - inp.ks[r])
        assert out[r].tolist() == list(range(min(37, n))) + [-1] * (37 - min(37, n))


def test_visible_range_is_relative(orc):
    """Row scores over [ks, ke) equal the slice of the full-range scores."""
    inp = synth.indexer_inputs(2, 400, 2, 64, 16, "bf16", seed=15, ranges="full")
    full = orc.scores_row(inp, 1)
    inp.ks[1], inp.ke[1] = 123, 345
    part = orc.scores_row(inp, 1)
    assert np.array_equal(part, full[123:345])
    top = orc.score_topk(inp, rows=[1], nthreads=1)[0]
    assert top.max() < 222 and top.min() >= 0


# ------------------------------------------------------------------ selection

def _brute_force_topk(s, topk):
    """Enumerate every subset of size min(topk, n); the rule's answer is the
    unique subset whose sorted (score desc, index asc) sequence is
    lexicographically best."""
    n = len(s)
    m = min(topk, n)
    best, best_key = None, None
    for sub in itertools.combinations(range(n), m):
        key = sorted(((-s[j], j) for j in sub))
        if best_key is None or key < best_key:
            best, best_key = sub, key
    return list(best) + [-1] * (topk - m)


def test_selection_matches_subset_enumeration(orc):
    rng = np.random.default_rng(0)
    for trial in range(60):
        n = int(rng.integers(0, 9))
        topk = int(rng.integers(1, 8))
        s = rng.integers(-3, 4, size=n).astype(np.float64) / 2  # many exact ties
        assert orc.select_row(s, topk).tolist() == _brute_force_topk(s, topk)


def test_selection_matches_lexsort(orc):
    rng = np.random.default_rng(1)
    for trial in range(40):
        n = int(rng.integers(1, 65))
        topk = int(rng.integers(1, 70))
        s = np.round(rng.normal(size=n), 1)
        order = np.lexsort((np.arange(n), -s))[:topk]
        expect = sorted(order.tolist()) + [-1] * (topk - min(topk, n))
        assert orc.select_row(s, topk).tolist() == expect


def test_selection_closed_forms(orc):
    n, topk = 1000, 64
    assert orc.select_row(np.arange(n, dtype=np.float64), topk).tolist() == list(range(n - topk, n))
    assert orc.select_row(np.full(n, 0.5), topk).tolist() == list(range(topk))
    s = np.zeros(n)
    planted = [5, 77, 300, 301, 999]
    s[planted] = 1.0
    assert orc.select_row(s, 5).tolist() == planted
    assert orc.select_row(s, 7).tolist() == [0, 1, 5, 77, 300, 301, 999]
    assert orc.select_row(np.zeros(0), 3).tolist() == [-1, -1, -1]


def test_signed_zero_ties_by_index(orc):
    s = np.array([-0.0, 0.0, -0.0, 1.0, 0.0])
    assert orc.select_row(s, 3).tolist() == [0, 1, 3]


def _check_invariants(s, out, topk):
    n = len(s)
    m = min(topk, n)
    sel = out[:m]
    assert (out[m:] == -1).all()
    assert (sel >= 0).all() and (sel < n).all()
    assert len(set(sel.tolist())) == m
    assert (np.diff(sel) > 0).all()
    if m < n:
        mask = np.zeros(n, bool)
        mask[sel] = True
        lo = s[mask].min()
        assert lo >= s[~mask].max()
        tied_out = np.flatnonzero(~mask & (s == lo))
        tied_in = np.flatnonzero(mask & (s == lo))
        if tied_out.size:
            assert tied_in.max() < tied_out.min()


def test_invariants_on_indexer_rows(orc):
    inp = synth.indexer_inputs(16, 3000, 8, 64, 200, "fp8", seed=16)
    out, sc = orc.score_topk(inp, want_scores=True, nthreads=4)
    for i in range(16):
        n = int(inp.ke[i] - inp.ks[i])
        _check_invariants(sc[i, :n], out[i], 200)


# ------------------------------------------------------ top-k on given scores

def test_topk_from_scores_matches_lexsort_with_ties(orc):
    inp = synth.score_inputs(24, 5000, 300, seed=17, short_frac=0.25)
    out = orc.topk_from_scores(inp.scores, inp.ks, inp.ke, 300, nthreads=4)
    S = inp.scores.numpy()
    for r in range(24):
        n = int(inp.ke[r])
        s = S[r, :n].astype(np.float64)
        order = np.lexsort((np.arange(n), -s))[:300]
        expect = sorted(order.tolist()) + [-1] * (300 - min(300, n))
        assert out[r].tolist() == expect
        _check_invariants(s, out[r], 300)
    # the bf16 grid leaves exact ties at the k-th value on the long rows
    long_rows = [r for r in range(24) if int(inp.ke[r]) == 5000]
    r = long_rows[0]
    s = S[r].astype(np.float64)
    kth = np.sort(s)[::-1][299]
    assert (s == kth).sum() > 1


def test_topk_from_scores_row_subset_and_stride(orc):
    S = torch.arange(40, dtype=torch.float32).reshape(4, 10)
    ks = torch.tensor([0, 2, 5, 9], dtype=torch.int32)
    ke = torch.tensor([10, 7, 5, 10], dtype=torch.int32)
    out = orc.topk_from_scores(S, ks, ke, 3, rows=[3, 1, 2])
    assert out.tolist() == [[0, -1, -1], [2, 3, 4], [-1, -1, -1]]


# ------------------------------------------------------------ page transform

def test_page_transform_hand_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "page_transform.json")))
    idx = np.array([r["idx"] for r in g["rows"]], dtype=np.int32)
    rmap = np.array([r["table_row"] for r in g["rows"]], dtype=np.int32)
    table = np.array(g["table"], np.int32)
    # first with a third row present in memory but outside the declared table:
    # the row bound, not the array's end, decides
    padded = np.vstack([table, np.ones((1, table.shape[1]), np.int32)])
    got, bad = orc.page_transform(idx, padded, g["page_size"], rmap, table_rows=len(table))
    assert got.tolist() == [r["expect"] for r in g["rows"]]
    assert bad == g["out_of_range"]
    got, bad = orc.page_transform(idx, table, g["page_size"], rmap)
    assert got.tolist() == [r["expect"] for r in g["rows"]]
    assert bad == g["out_of_range"]


def test_page_transform_identity_table_is_identity(orc):
    rng = np.random.default_rng(5)
    idx = rng.integers(-1, 4096, size=(7, 33)).astype(np.int32)
    table = np.tile(np.arange(64, dtype=np.int32), (7, 1))  # page j is physical page j
    got, bad = orc.page_transform(idx, table, 64)
    assert bad == 0 and np.array_equal(got, idx)


def test_page_transform_permuted_table_inverts(orc):
    """A table row that permutes the pages is undone by the inverse permutation,
    and distinct positions stay distinct; the -1 padding passes through."""
    rng = np.random.default_rng(6)
    P, pages = 64, 40
    table = np.stack([rng.permutation(pages).astype(np.int32) + 100 * t for t in range(3)])
    idx = np.stack([rng.choice(P * pages, 50, replace=False) for _ in range(5)]).astype(np.int32)
    idx[:, -3:] = -1
    rmap = np.array([2, 0, 1, 2, 0], np.int32)
    got, bad = orc.page_transform(idx, table, P, rmap)
    assert bad == 0
    for r in range(5):
        t = rmap[r]
        inv = {int(v): j for j, v in enumerate(table[t])}
        back = [inv[int(x) // P] * P + int(x) % P for x in got[r, :-3]]
        assert back == idx[r, :-3].tolist()
        assert (got[r, -3:] == -1).all()
        assert len(set(got[r, :-3].tolist())) == 47


# ------------------------------------------------------------- MXFP4 inputs

# OCP Microscaling Formats (MX) v1.0, FP4 E2M1: the magnitudes of codes 0..7.
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decoder_exhaustive(orc):
    got = orc.e2m1_to_f64(np.arange(16))
    assert got[:8].tolist() == E2M1_VALUES
    assert np.array_equal(got[8:], -got[:8]) and np.signbit(got[8])  # code 8 is -0
    mld = pytest.importorskip("ml_dtypes")
    ref = np.frombuffer(np.arange(16, dtype=np.uint8).tobytes(),
                        dtype=mld.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(got, ref) and np.array_equal(np.signbit(got), np.signbit(ref))


def test_e8m0_decoder_exhaustive_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = orc.e8m0_to_f64(codes)
    nan = np.isnan(ref)
    assert np.flatnonzero(nan).tolist() == [255]
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def _mx_inputs(q, q_sf, k, k_sf, topk=4, w=None, k_scale=None):
    """An MXFP4 input set from raw bytes: w = 1 and k_scale = 1 unless given,
    every row sees every key."""
    rows, H = q.shape[0], q.shape[1]
    keys = k.shape[0]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8))  # noqa: E731
    return synth.IndexerInputs(
        q=t(q), k=t(k), q_sf=t(q_sf), k_sf=t(k_sf),
        k_scale=torch.ones(keys) if k_scale is None else k_scale,
        w=torch.ones(rows, H) if w is None else w,
        ks=torch.zeros(rows, dtype=torch.int32), ke=torch.full((rows,), keys, dtype=torch.int32),
        topk=topk)


def test_mxfp4_nibble_order_and_block_scales(orc):
    """Closed forms with D = 128 (four scale blocks).  q holds 1.0 in every
    even element and 0 in every odd one; k rows hold 1.0 in the even, the odd
    and all elements: the scores 64, 0, 64 fix the nibble order.  Then all
    elements 1.0, q's block b scaled by 2^b and k's blocks by 1, 1/2, 1, 2:
    32 (1 + 2 + 4 + 8) = 480 and 32 (1 + 1 + 4 + 16) = 704 fix which scale
    byte covers which element."""
    D, one = 128, 0x2  # 0x2: the e2m1 code of 1.0
    q = np.full((1, 1, D // 2), one, np.uint8)
    k = np.array([[one] * (D // 2), [one << 4] * (D // 2), [one | one << 4] * (D // 2)])
    unit = lambda *shape: np.full(shape, 127, np.uint8)  # noqa: E731  e8m0 of 1.0
    s = orc.scores_row(_mx_inputs(q, unit(1, 1, D // 32), k, unit(3, D // 32)), 0)
    assert s.tolist() == [64.0, 0.0, 64.0]
    q2 = np.full((1, 1, D // 2), one | one << 4, np.uint8)
    q2_sf = (127 + np.arange(D // 32)).reshape(1, 1, -1)
    k2 = np.full((2, D // 2), one | one << 4, np.uint8)
    k2_sf = np.array([[127, 127, 127, 127], [127, 126, 127, 128]])
    s2 = orc.scores_row(_mx_inputs(q2, q2_sf, k2, k2_sf), 0)
    assert s2.tolist() == [480.0, 704.0]


def _decode_mx_independently(codes, sf):
    """MXFP4 bytes -> fp64 values through ml_dtypes (e2m1) and torch (e8m0),
    not through the oracle."""
    mld = pytest.importorskip("ml_dtypes")
    el = np.stack([codes & 0xF, codes >> 4], -1).reshape(*codes.shape[:-1], -1)
    v = np.frombuffer(el.astype(np.uint8).tobytes(), dtype=mld.float4_e2m1fn)
    v = v.astype(np.float64).reshape(el.shape)
    sc = torch.from_numpy(np.ascontiguousarray(sf, np.uint8)).view(torch.float8_e8m0fnu)
    return v * np.repeat(sc.to(torch.float64).numpy(), 32, axis=-1)


def test_mxfp4_scores_equal_the_e4m3_scores_of_the_same_values(orc):
    """Random MXFP4 bytes with block scales in 2^-3 .. 2^3: every value (an
    e2m1 magnitude times its block scale, |v| <= 48, nonzero |v| >= 2^-4) is
    exact in e4m3, so the oracle's MXFP4 scores equal, bit for bit, its e4m3
    scores of the same values, which are decoded here by ml_dtypes and torch.
    A swapped nibble, a misplaced scale block or a wrong bias breaks it."""
    rng = np.random.default_rng(7)
    rows, keys, H, D = 3, 50, 4, 64
    q = rng.integers(0, 256, (rows, H, D // 2), dtype=np.uint8)
    k = rng.integers(0, 256, (keys, D // 2), dtype=np.uint8)
    q_sf = rng.integers(124, 131, (rows, H, D // 32), dtype=np.uint8)
    k_sf = rng.integers(124, 131, (keys, D // 32), dtype=np.uint8)
    qv = torch.from_numpy(_decode_mx_independently(q, q_sf))
    kv = torch.from_numpy(_decode_mx_independently(k, k_sf))
    q8, k8 = qv.to(torch.float8_e4m3fn), kv.to(torch.float8_e4m3fn)
    assert torch.equal(q8.to(torch.float64), qv) and torch.equal(k8.to(torch.float64), kv)
    g = torch.Generator().manual_seed(8)
    w = torch.rand(rows, H, generator=g)
    sc = 0.5 + torch.rand(keys, generator=g)
    mx = _mx_inputs(q, q_sf, k, k_sf, topk=9, w=w, k_scale=sc)
    e4 = synth.IndexerInputs(q=q8, k=k8, k_scale=sc, w=w, ks=mx.ks, ke=mx.ke, topk=9)
    for r in range(rows):
        assert np.array_equal(orc.scores_row(mx, r), orc.scores_row(e4, r))
    assert np.array_equal(orc.score_topk(mx, nthreads=2), orc.score_topk(e4, nthreads=2))


def test_mxfp4_generated_inputs_score_like_their_decoded_values(orc):
    """synth's MXFP4 workload inputs: the oracle's scores equal a numpy
    evaluation of the definition on the independently decoded values."""
    inp = synth.indexer_inputs(2, 40, 3, 64, 5, "mxfp4", seed=9, ranges="full")
    assert inp.D == 64 and inp.dtype == "mxfp4"
    qv = _decode_mx_independently(inp.q.numpy(), inp.q_sf.numpy())
    kv = _decode_mx_independently(inp.k.numpy(), inp.k_sf.numpy())
    for r in range(2):
        dots = kv @ qv[r].T  # [keys, H]
        ref = inp.k_scale.double().numpy() * (np.maximum(dots, 0) @ inp.w[r].double().numpy())
        np.testing.assert_allclose(orc.scores_row(inp, r), ref, rtol=1e-12, atol=1e-12)

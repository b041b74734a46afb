"""Seeded synthetic inputs for the prefill indexer.

This module draws inputs only.  It holds none of the indexer's arithmetic (no
scoring, no selection), so both the CPU oracle and the CUDA library can consume
the very same bytes: every tensor is made on the CPU with a seeded
``torch.Generator`` and copied to the device by the caller.

Workloads follow the problem statement of the sparse-attention prefill indexer
("[sglang] logits를 쓰지 않는 top-k ... LiteTopK prefill indexer", introduction:
per query row, an indexer score over every visible key, then the top 512-2048
keys) and the standalone exact top-k of "[sglang] ROCm DSA Indexer Top-K 최적화"
(fp32 scores, dense clustering, topk 2048).

Layouts (row-major, contiguous):
  q        [rows, H, D]  bfloat16 or float8_e4m3fn; MXFP4: uint8 [rows, H, D/2]
                         (two e2m1 codes per byte, element 2i in the low
                         nibble) with q_sf uint8 [rows, H, D/32] (e8m0 scales)
  k        [keys, D]     same format as q; MXFP4: uint8 [keys, D/2], k_sf
                         uint8 [keys, D/32]
  k_scale  [keys]        float32, > 0
  w        [rows, H]     float32, >= 0
  ks, ke   [rows]        int32, visible keys of row r are ks[r] <= j < ke[r]
  scores   [rows, keys]  float32 (standalone top-k only)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "IndexerInputs", "ScoreInputs", "indexer_inputs", "score_inputs", "quantise_mxfp4",
    "causal_ranges", "mixed_batch_lengths", "planted_scale_factor",
    "workload", "WORKLOADS", "sample_rows",
]


@dataclass
class IndexerInputs:
    q: torch.Tensor
    k: torch.Tensor
    k_scale: torch.Tensor
    w: torch.Tensor
    ks: torch.Tensor
    ke: torch.Tensor
    topk: int
    meta: dict = field(default_factory=dict)
    q_sf: torch.Tensor | None = None  # MXFP4 block scales of q
    k_sf: torch.Tensor | None = None  # MXFP4 block scales of k

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def keys(self) -> int:
        return int(self.k.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def D(self) -> int:
        return int(self.q.shape[2]) * (2 if self.q_sf is not None else 1)

    @property
    def dtype(self) -> str:
        if self.q_sf is not None:
            return "mxfp4"
        return "bf16" if self.q.dtype == torch.bfloat16 else "fp8_e4m3"

    def pairs(self) -> int:
        return int((self.ke.long() - self.ks.long()).clamp_min(0).sum())


@dataclass
class ScoreInputs:
    scores: torch.Tensor
    ks: torch.Tensor
    ke: torch.Tensor
    topk: int
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return int(self.scores.shape[0])

    @property
    def stride(self) -> int:
        return int(self.scores.shape[1])


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def causal_ranges(rows: int, keys: int):
    """ks = 0, ke_r = keys - rows + r + 1 (the last `rows` query tokens of a
    prefill over `keys` tokens)."""
    r = torch.arange(rows, dtype=torch.int64)
    ke = (keys - rows + r + 1).clamp(0, keys)
    ks = torch.zeros(rows, dtype=torch.int64)
    return ks.to(torch.int32), ke.to(torch.int32)


def mixed_batch_lengths(requests: int, lo: int, hi: int, g: torch.Generator):
    """Per-request lengths L = floor(exp(U(ln lo, ln hi)))."""
    u = torch.rand(requests, generator=g, dtype=torch.float64)
    L = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return L.to(torch.int64).clamp(lo, hi)


def planted_scale_factor(H: int, D: int) -> float:
    """Per-key scale multiplier that lifts a key's expected score by three
    within-row standard deviations.

    With q, k entries ~ N(0,1) each head logit x_h = q_h . k is ~ N(0, D);
    E[ReLU(x)] = sqrt(D / 2pi), Var[ReLU(x)] = D (1/2 - 1/(2 pi)).  With
    w_h ~ U(0,1)/H (E[w] = 1/(2H), E[w^2] = 1/(3H^2)) and heads treated as
    independent, the unscaled score u = sum_h w_h ReLU(x_h) has
    mean mu = sqrt(D/(2 pi))/2 and within-row variance
    sigma^2 = (D/H)(1/3)(1/2 - 1/(2 pi)).  Multiplying the scale by
    1 + 3 sigma/mu shifts the key's expected score by +3 sigma.
    This is a property of the input distribution, not of the indexer.
    """
    mu = 0.5 * math.sqrt(D / (2.0 * math.pi))
    var = (D / H) * (1.0 / 3.0) * (0.5 - 1.0 / (2.0 * math.pi))
    return 1.0 + 3.0 * math.sqrt(var) / mu


def _quantise(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype in ("fp8", "fp8_e4m3", "e4m3"):
        return x.to(torch.float8_e4m3fn)
    raise ValueError(f"unknown dtype {dtype!r}")


# magnitudes of the e2m1 codes 0..7 (code 8 + c is the negative of code c)
_E2M1_MAG = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)


def quantise_mxfp4(x: torch.Tensor):
    """Encode fp32 x [..., D] (D a multiple of 32) as MXFP4: per block of 32
    consecutive values the shared scale 2^e with e = floor(log2 max|x|) - 2
    (the largest e2m1 magnitude is 1.5 * 2^2; the OCP recipe), clamped to
    [-127, 127], stored as the e8m0 byte e + 127; each value divided by 2^e,
    rounded to the nearest e2m1 magnitude (ties to the even code, i.e. the
    mantissa bit 0), saturated at 6, and packed two per byte, element 2i in
    the low nibble.  Returns (codes uint8 [..., D/2], scales uint8 [..., D/32]).
    This is input encoding only; the indexer consumes the bytes."""
    *lead, D = x.shape
    if D % 32:
        raise ValueError("MXFP4 needs D % 32 == 0")
    xb = x.to(torch.float64).reshape(*lead, D // 32, 32)
    amax = xb.abs().amax(-1)
    _, ex = torch.frexp(amax)  # amax = m * 2^ex, 0.5 <= m < 1, so floor(log2 amax) = ex - 1
    e = torch.where(amax > 0, ex.to(torch.int64) - 1 - 2, torch.zeros_like(ex, dtype=torch.int64))
    e = e.clamp(-127, 127)
    scaled = xb / torch.ldexp(torch.ones_like(amax), e)[..., None]
    mag = scaled.abs().clamp(max=6.0)
    lo = (torch.searchsorted(_E2M1_MAG, mag.contiguous(), right=True) - 1).clamp(0, 7)
    hi = (lo + 1).clamp(max=7)
    dl = mag - _E2M1_MAG[lo]
    dh = _E2M1_MAG[hi] - mag
    up = (dh < dl) | ((dh == dl) & (hi % 2 == 0) & (hi != lo))
    code = torch.where(up, hi, lo) | ((scaled < 0).to(torch.int64) << 3)
    code = code.reshape(*lead, D).to(torch.uint8)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).contiguous()
    return packed, (e + 127).to(torch.uint8).contiguous()


def indexer_inputs(rows: int, keys: int, H: int, D: int, topk: int, dtype: str,
                   seed: int, *, ranges: str = "causal", scale: str = "uniform",
                   planted_runs: int = 0, planted_len: int = 64,
                   ks=None, ke=None) -> IndexerInputs:
    """q, k ~ N(0,1) rounded to `dtype`; w ~ U(0,1)/H; k_scale ~ U(0.5, 2) or 1.

    ranges: "causal" (ks = 0, ke_r = keys - rows + r + 1), "full" (0, keys),
    or "given" (ks/ke passed in).
    planted_runs: that many non-overlapping runs of `planted_len` keys whose
    scale is multiplied by planted_scale_factor(H, D); run starts are seeded,
    uniform, not aligned to 64, and placed where every causal row sees them.
    """
    g = _gen(seed)
    qf = torch.randn(rows, H, D, generator=g, dtype=torch.float32)
    kf = torch.randn(keys, D, generator=g, dtype=torch.float32)
    if dtype == "mxfp4":
        (q, q_sf), (k, k_sf) = quantise_mxfp4(qf), quantise_mxfp4(kf)
    else:
        q, k, q_sf, k_sf = _quantise(qf, dtype), _quantise(kf, dtype), None, None
    del qf, kf
    w = torch.rand(rows, H, generator=g, dtype=torch.float32) / H
    if scale == "uniform":
        k_scale = 0.5 + 1.5 * torch.rand(keys, generator=g, dtype=torch.float32)
    elif scale == "one":
        k_scale = torch.ones(keys, dtype=torch.float32)
    else:
        raise ValueError(scale)
    meta = {"seed": seed, "ranges": ranges, "scale": scale}
    if planted_runs:
        factor = planted_scale_factor(H, D)
        span = max(keys - rows - planted_len, planted_runs * planted_len)
        starts = []
        # rejection sampling of non-overlapping, non-64-aligned starts
        while len(starts) < planted_runs:
            s = int(torch.randint(0, span, (1,), generator=g))
            if s % 64 == 0:
                continue
            if any(abs(s - t) < planted_len for t in starts):
                continue
            starts.append(s)
        starts.sort()
        for s in starts:
            k_scale[s:s + planted_len] *= factor
        meta.update(planted_starts=starts, planted_len=planted_len,
                    planted_factor=factor)
    if ranges == "causal":
        ks_t, ke_t = causal_ranges(rows, keys)
    elif ranges == "full":
        ks_t = torch.zeros(rows, dtype=torch.int32)
        ke_t = torch.full((rows,), keys, dtype=torch.int32)
    elif ranges == "given":
        ks_t = torch.as_tensor(ks, dtype=torch.int32).clone()
        ke_t = torch.as_tensor(ke, dtype=torch.int32).clone()
    else:
        raise ValueError(ranges)
    return IndexerInputs(q=q, k=k, k_scale=k_scale, w=w, ks=ks_t, ke=ke_t,
                         topk=topk, meta=meta, q_sf=q_sf, k_sf=k_sf)


def score_inputs(rows: int, keys: int, topk: int, seed: int, *,
                 sigma: float = 0.05, short_frac: float = 0.05,
                 bf16_grid: bool = True) -> ScoreInputs:
    """fp32 scores ~ N(0, sigma) rounded to the bf16 grid (dense clustering and
    many exact ties); round(short_frac * rows) seeded rows get ke ~ U[0, topk),
    every other row sees all keys."""
    g = _gen(seed)
    s = torch.randn(rows, keys, generator=g, dtype=torch.float32) * sigma
    if bf16_grid:
        s = s.to(torch.bfloat16).to(torch.float32)
    ks = torch.zeros(rows, dtype=torch.int32)
    ke = torch.full((rows,), keys, dtype=torch.int32)
    n_short = int(round(short_frac * rows))
    if n_short:
        short_rows = torch.randperm(rows, generator=g)[:n_short]
        ke[short_rows] = torch.randint(0, min(topk, keys), (n_short,), generator=g,
                                       dtype=torch.int64).to(torch.int32)
    else:
        short_rows = torch.zeros(0, dtype=torch.int64)
    return ScoreInputs(scores=s, ks=ks, ke=ke, topk=topk,
                       meta={"seed": seed, "sigma": sigma,
                             "short_rows": sorted(int(x) for x in short_rows)})


def _mixed_batch(seed: int, requests: int = 64, rows_per_request: int = 128,
                 lo: int = 256, hi: int = 262144, H: int = 64, D: int = 128,
                 topk: int = 512, dtype: str = "fp8") -> IndexerInputs:
    """Requests of log-uniform length L_i; K is the concatenation of every
    request's keys.  Row j of request i is one of its last `rows_per_request`
    tokens: ks = off_i, ke = off_i + L_i - rows_per_request + j + 1."""
    g = _gen(seed + 7919)
    L = mixed_batch_lengths(requests, lo, hi, g)
    off = torch.zeros(requests, dtype=torch.int64)
    off[1:] = torch.cumsum(L, 0)[:-1]
    keys = int(L.sum())
    j = torch.arange(rows_per_request, dtype=torch.int64)
    ks = off.repeat_interleave(rows_per_request)
    ke = (off + L - rows_per_request)[:, None] + j[None, :] + 1
    ke = ke.reshape(-1)
    inp = indexer_inputs(requests * rows_per_request, keys, H, D, topk, dtype,
                         seed, ranges="given", ks=ks, ke=ke)
    inp.meta.update(requests=requests, lengths=[int(x) for x in L])
    return inp


def paged_layout(requests: int, pages_per_request: int, rows_per_request: int, seed: int,
                 pool_pages: int | None = None):
    """A paged KV cache: each request owns pages_per_request distinct physical
    pages drawn at random (seeded) from a pool shared by all requests, and its
    query rows use its table row.  Returns (table [requests, pages] int32,
    row_map [requests * rows_per_request] int32)."""
    g = _gen(seed)
    pool = pool_pages or 2 * requests * pages_per_request
    perm = torch.randperm(pool, generator=g)[: requests * pages_per_request]
    table = perm.view(requests, pages_per_request).to(torch.int32).contiguous()
    row_map = torch.arange(requests, dtype=torch.int32).repeat_interleave(rows_per_request)
    return table, row_map


# The named workloads: small case first, then the standalone top-k, the fused
# prefill, the long-context stress and the mixed batch, plus the low-batch
# long-row top-k that exercises the multi-block row split.
WORKLOADS = {
    "tiny": dict(kind="indexer", rows=64, keys=4096, H=8, D=64, topk=256,
                 dtype="bf16", seed=0, scale="one"),
    "standalone_topk": dict(kind="scores", rows=1024, keys=131072, topk=2048, seed=1),
    "fused_prefill": dict(kind="indexer", rows=4096, keys=65536, H=64, D=128,
                          topk=2048, dtype="fp8", seed=2, scale="uniform"),
    "long_context": dict(kind="indexer", rows=4096, keys=1048576, H=32, D=128,
                         topk=2048, dtype="fp8", seed=3, scale="uniform",
                         planted_runs=32),
    "mixed_batch": dict(kind="mixed", seed=4),
    "split_topk": dict(kind="scores", rows=8, keys=1048576, topk=2048, seed=5,
                       short_frac=0.0),
}


def workload(name: str):
    cfg = dict(WORKLOADS[name])
    kind = cfg.pop("kind")
    if kind == "indexer":
        return indexer_inputs(cfg.pop("rows"), cfg.pop("keys"), cfg.pop("H"),
                              cfg.pop("D"), cfg.pop("topk"), cfg.pop("dtype"),
                              cfg.pop("seed"), **cfg)
    if kind == "scores":
        return score_inputs(cfg.pop("rows"), cfg.pop("keys"), cfg.pop("topk"),
                            cfg.pop("seed"), **cfg)
    if kind == "mixed":
        return _mixed_batch(cfg.pop("seed"))
    raise ValueError(kind)


def sample_rows(ks: torch.Tensor, ke: torch.Tensor, count: int, seed: int):
    """A seeded subset of `count` rows that always holds the shortest and the
    longest visible row (numpy default_rng(seed + 1000))."""
    import numpy as np
    n = (ke.long() - ks.long()).clamp_min(0).numpy()
    rows = n.shape[0]
    if rows <= count:
        return list(range(rows))
    rng = np.random.default_rng(seed + 1000)
    pick = {int(np.argmin(n)), int(np.argmax(n))}
    for r in rng.permutation(rows):
        if len(pick) >= count:
            break
        pick.add(int(r))
    return sorted(pick)

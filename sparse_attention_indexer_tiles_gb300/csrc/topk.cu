// Exact radix top-k kernels of libidx.
//
//  * topk_rows_kernel   one CTA per row of fp32 scores in global memory:
//                       12-bit histogram pass, a collection pass of the
//                       threshold bin into a shared tie buffer (or, when that
//                       bin holds more than kTieCap keys, another histogram
//                       pass over the row: the full-row rescan), then an
//                       ordered compaction pass that writes ascending indices.
//                       Page "[sglang] ROCm DSA Indexer Top-K 최적화": fp32
//                       coarse histogram, radix tie refinement, overflow
//                       rescan, single-block kernel per row.
//  * the same kernel in threshold mode returns only the exact t-th largest
//    key of each row; the fused path uses it on the strided score sample
//    (page "[sglang] logits를 쓰지 않는 top-k", section 2).
//  * cand_topk_kernel   one CTA per row of the candidate slab held in shared
//                       memory (page 1: the small top-k over ~2.25 x topk
//                       candidates); flags rows whose slab is short or
//                       overflowed for the exact rescan.
#include "plan.cuh"
#include "radix.cuh"
#include "topk.cuh"

namespace idx {

void count_launches(unsigned n);  // api.cu

constexpr int kTieCap = 4096;
constexpr int kCandScratch = 96;  // scan words + row state of cand_topk_kernel

// A row of fp32 values addressed through an aligned float4 view: element p
// (0 <= p < n) sits in slot p + off of the 16-byte aligned base.  Reads may
// touch the up-to-12 bytes that share a 16-byte block with the row's first or
// last element; such a block never straddles a page.
struct RowView {
    const float4* base;
    int off;
    long long n;
    long long nvec;
};

IDX_DEVI RowView make_view(const float* p, long long n) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    RowView v;
    v.off = static_cast<int>((a & 15u) >> 2);
    v.base = reinterpret_cast<const float4*>(a - (a & 15u));
    v.n = n;
    v.nvec = (n + v.off + 3) >> 2;
    return v;
}

IDX_DEVI float4 ldg4(const float4* p) { return __ldg(p); }

// Histogram of `level`'s digit over the row's keys that carry `prefix`.
template <int THREADS, int UNROLL>
IDX_DEVI void hist_pass(const RowView& v, int level, uint32_t prefix, uint32_t* hist) {
    for (long long base = threadIdx.x; base < v.nvec; base += (long long)THREADS * UNROLL) {
        float4 f[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            f[u] = s < v.nvec ? ldg4(v.base + s) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const long long p = 4 * s + c - v.off;
                if (s < v.nvec && p >= 0 && p < v.n) {
                    const uint32_t key = fkey(e[c]);
                    if (has_prefix(key, level, prefix)) atomicAdd(&hist[digit_of(key, level)], 1u);
                }
            }
        }
    }
}

// Append (key, position) of every key carrying `prefix` at `level`.
template <int THREADS, int UNROLL>
IDX_DEVI void collect_pass(const RowView& v, int level, uint32_t prefix, uint32_t* tkey,
                           uint32_t* tpos, uint32_t* tcount) {
    for (long long base = threadIdx.x; base < v.nvec; base += (long long)THREADS * UNROLL) {
        float4 f[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            f[u] = s < v.nvec ? ldg4(v.base + s) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const long long p = 4 * s + c - v.off;
                if (s < v.nvec && p >= 0 && p < v.n) {
                    const uint32_t key = fkey(e[c]);
                    if (has_prefix(key, level, prefix)) {
                        const uint32_t slot = atomicAdd(tcount, 1u);
                        if (slot < (uint32_t)kTieCap) {
                            tkey[slot] = key;
                            tpos[slot] = static_cast<uint32_t>(p);
                        }
                    }
                }
            }
        }
    }
}

struct Threshold {
    uint32_t key;   // exact threshold key T
    uint32_t need;  // keys equal to T that belong to the result (lowest indices first)
};

// Digit refinement over the shared tie buffer, from `level` down to the exact key.
template <int THREADS>
IDX_DEVI Threshold refine_in_smem(const uint32_t* tkey, uint32_t cnt, int level, uint32_t prefix,
                                  uint32_t need, uint32_t* hist, uint32_t* scratch) {
    for (int lev = level; lev <= 2; ++lev) {
        zero_shared<THREADS>(hist, kHistBins);
        __syncthreads();
        for (uint32_t e = threadIdx.x; e < cnt; e += THREADS) {
            const uint32_t key = tkey[e];
            if (has_prefix(key, lev, prefix)) atomicAdd(&hist[digit_of(key, lev)], 1u);
        }
        __syncthreads();
        const DigitPick pk = pick_digit<THREADS>(hist, 1 << digit_bits(lev), need, scratch);
        need -= pk.above;
        prefix = (prefix << digit_bits(lev)) | pk.digit;
    }
    return {prefix, need};
}

// Exact threshold of the k largest keys of a global row (k <= n).  Uses the
// tie buffer when the threshold bin fits, otherwise rescans the row digit by
// digit.  `rescans` counts the extra full-row histogram passes.
template <int THREADS, int UNROLL>
IDX_DEVI Threshold find_threshold(const RowView& v, uint32_t k, uint32_t* hist, uint32_t* tkey,
                                  uint32_t* tpos, uint32_t* scratch, int* rescans) {
    uint32_t prefix = 0, need = k;
    *rescans = 0;
    for (int level = 0; level <= 2; ++level) {
        zero_shared<THREADS>(hist, kHistBins);
        __syncthreads();
        hist_pass<THREADS, UNROLL>(v, level, prefix, hist);
        __syncthreads();
        const DigitPick pk = pick_digit<THREADS>(hist, 1 << digit_bits(level), need, scratch);
        need -= pk.above;
        prefix = (prefix << digit_bits(level)) | pk.digit;
        if (level == 2) return {prefix, need};
        if (pk.count <= (uint32_t)kTieCap) {
            uint32_t* tcount = scratch + 40;
            if (threadIdx.x == 0) *tcount = 0u;
            __syncthreads();
            collect_pass<THREADS, UNROLL>(v, level + 1, prefix, tkey, tpos, tcount);
            __syncthreads();
            const uint32_t cnt = min(*tcount, (uint32_t)kTieCap);
            __syncthreads();
            return refine_in_smem<THREADS>(tkey, cnt, level + 1, prefix, need, hist, scratch);
        }
        ++*rescans;
    }
    return {prefix, need};  // not reached
}

// Ordered compaction of the selected keys of a global row into out[0..k):
// key > T, plus the first `need` keys equal to T in index order.
template <int THREADS>
IDX_DEVI void ordered_output(const RowView& v, Threshold th, uint32_t k, int* out,
                             uint32_t* scratch) {
    uint32_t a_run = 0, e_run = 0;
    for (long long base = 0; base < v.nvec; base += THREADS) {
        const long long s = base + threadIdx.x;
        float4 f = s < v.nvec ? ldg4(v.base + s) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float e[4] = {f.x, f.y, f.z, f.w};
        uint32_t ab = 0, tb = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const long long p = 4 * s + c - v.off;
            if (s < v.nvec && p >= 0 && p < v.n) {
                const uint32_t key = fkey(e[c]);
                ab |= (key > th.key ? 1u : 0u) << c;
                tb |= (key == th.key ? 1u : 0u) << c;
            }
        }
        const uint32_t mine = (__popc(ab) << 16) | __popc(tb);
        uint32_t tot;
        const uint32_t incl = block_incl_scan<THREADS>(mine, scratch, &tot);
        const uint32_t excl = incl - mine;
        uint32_t a_b = a_run + (excl >> 16), e_b = e_run + (excl & 0xFFFFu);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int p = static_cast<int>(4 * s + c - v.off);
            if ((ab >> c) & 1u) {
                const uint32_t pos = a_b + min(e_b, th.need);
                if (pos < k) out[pos] = p;
                ++a_b;
            } else if ((tb >> c) & 1u) {
                if (e_b < th.need && a_b + e_b < k) out[a_b + e_b] = p;
                ++e_b;
            }
        }
        a_run += tot >> 16;
        e_run += tot & 0xFFFFu;
    }
}

// ------------------------------------------------------- one-pass path
//
// A row is streamed from HBM once.  A lower bound L on the threshold is
// estimated from the 12-bit histogram of a 4096-value sample (aiming at about
// 2 k keys >= L): the first 256 values of each warp's slice, which the filter
// loads first anyway.  Every key >= L is then appended to its warp's run in
// shared memory, and the top digits of the appended keys are counted on the
// way (level 0 of the refinement).  Warp w owns the contiguous slice w of the row and appends in index
// order, so the runs, taken in warp order, list the candidates in ascending
// index order.  The exact threshold is then refined over the candidates and an
// ordered compaction writes the result.  When L was too high (fewer than k
// candidates) or a run overflowed, the row falls back to the multi-pass path
// above, which is exact for any input.

constexpr int kRunCap = 512;       // candidates per warp run
constexpr int kPrefix = 4096;      // values that estimate L

template <int THREADS>
struct StreamSmem {
    static constexpr int W = THREADS / 32;
    static constexpr int RUN_WORDS = W * kRunCap;          // per array
    static_assert(2 * RUN_WORDS >= 2 * kTieCap, "tie buffer aliases the runs");
    // hist | scratch(64) | rcnt(W) | wsum(2W) | run keys | run idx
    static constexpr size_t BYTES =
        (kHistBins + 64 + 3 * W + 2 * (size_t)RUN_WORDS) * sizeof(uint32_t);
};

// One step of a warp's filter: lane `lane` holds the four values of float4
// slot sl; every value >= L (key order; Lf is the float of L) is appended to
// the warp's run in index order.  With HIST the 12-bit top digit of every hit
// is counted in hist as well (level 0 of the refinement over the runs).
template <bool HIST>
IDX_DEVI void filter_step(const float4 f, int sl, bool interior, int s1, int n, int off,
                          uint32_t L, float Lf, uint32_t lt, uint32_t& cnt, uint32_t* mk,
                          uint32_t* mi, uint32_t* hist) {
    const float e[4] = {f.x, f.y, f.z, f.w};
    bool h[4];
    if (interior) {
#pragma unroll
        for (int c = 0; c < 4; ++c) h[c] = e[c] >= Lf;
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int p = 4 * sl + c - off;
            h[c] = sl < s1 && p >= 0 && p < n && (L == 0u || e[c] >= Lf);
        }
    }
    const uint32_t hits = (h[0] ? 1u : 0u) | (h[1] ? 2u : 0u) | (h[2] ? 4u : 0u) |
                          (h[3] ? 8u : 0u);
    const uint32_t any = __ballot_sync(0xffffffffu, hits != 0u);
    if (any == 0u) return;
    if (!__any_sync(0xffffffffu, (hits & (hits - 1u)) != 0u)) {
        // at most one hit per lane: its place is the number of lower lanes with a hit
        if (hits) {
            const uint32_t pos = cnt + __popc(any & lt);
            const int c = __ffs(hits) - 1;
            const uint32_t key = fkey(c == 0 ? e[0] : c == 1 ? e[1] : c == 2 ? e[2] : e[3]);
            if (pos < (uint32_t)kRunCap) {
                mk[pos] = key;
                mi[pos] = static_cast<uint32_t>(4 * sl + c - off);
            }
            if (HIST) atomicAdd(&hist[key >> 20], 1u);
        }
        cnt += __popc(any);
        return;
    }
    // some lane holds several hits: one ballot per lane component; a hit's
    // place is the number of hits in lower lanes plus those of lower
    // components in its own lane
    const uint32_t b0 = __ballot_sync(0xffffffffu, h[0]);
    const uint32_t b1 = __ballot_sync(0xffffffffu, h[1]);
    const uint32_t b2 = __ballot_sync(0xffffffffu, h[2]);
    const uint32_t b3 = __ballot_sync(0xffffffffu, h[3]);
    uint32_t pos = cnt + __popc(b0 & lt) + __popc(b1 & lt) + __popc(b2 & lt) + __popc(b3 & lt);
    cnt += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
    uint32_t rest = hits;
    while (rest) {
        const int c = __ffs(rest) - 1;
        const uint32_t key = fkey(c == 0 ? e[0] : c == 1 ? e[1] : c == 2 ? e[2] : e[3]);
        if (pos < (uint32_t)kRunCap) {
            mk[pos] = key;
            mi[pos] = static_cast<uint32_t>(4 * sl + c - off);
        }
        if (HIST) atomicAdd(&hist[key >> 20], 1u);
        ++pos;
        rest &= rest - 1u;
    }
}

// Warp w's contiguous slice [s0, s1) of the row's float4 slots.
template <int THREADS>
IDX_DEVI void warp_slice(const RowView& v, int w, int* s0, int* s1) {
    constexpr int W = THREADS / 32;
    const int nvec = (int)v.nvec;
    const int seg = (nvec + W - 1) / W;
    *s0 = w * seg;
    *s1 = *s0 + seg < nvec ? *s0 + seg : nvec;
}

// Append every key >= L of warp w's slice to its run; returns through rcnt[w].
// The hot loop compares floats; order keys are formed for the few hits only,
// and element bounds are checked only in the row's first and last 16 bytes.
template <int THREADS, int UNROLL, bool HIST>
IDX_DEVI void stream_collect(const RowView& v, uint32_t L, uint32_t* rkey, uint32_t* ridx,
                             uint32_t* rcnt, uint32_t* hist) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nvec = (int)v.nvec, n = (int)v.n, off = v.off;
    int s0, s1;
    warp_slice<THREADS>(v, w, &s0, &s1);
    const float Lf = key_floor_float(L);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t* mk = rkey + w * kRunCap;
    uint32_t* mi = ridx + w * kRunCap;
    uint32_t cnt = 0;
    for (int base = s0; base < s1; base += 32 * UNROLL) {
        float4 f[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int sl = base + u * 32 + lane;
            f[u] = sl < s1 ? ldg4(v.base + sl) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // every slot of this step holds 4 visible values (warp-uniform)
        const bool interior = base >= 1 && base + 32 * UNROLL <= s1 && base + 32 * UNROLL < nvec;
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            filter_step<HIST>(f[u], base + u * 32 + lane, interior, s1, n, off, L, Lf, lt, cnt,
                              mk, mi, hist);
    }
    if (lane == 0) rcnt[w] = cnt;
}

// The one-pass collection of a whole row by one CTA, lower bound included.
// L is the lower edge of the 12-bit bin that holds about the 2 k P / n-th
// largest of a sample of P values: the first two float4 slots of every lane
// in the first step of every warp's slice (P = 4096 for 512 threads), values
// the filter loads anyway.  hist leaves holding the top digits of the hits.
template <int THREADS, int UNROLL>
IDX_DEVI void stream_collect_estimate(const RowView& v, uint32_t k, uint32_t* hist,
                                      uint32_t* scratch, uint32_t* rkey, uint32_t* ridx,
                                      uint32_t* rcnt) {
    constexpr int SAMPLE = 2;  // float4 slots per lane in the sample
    static_assert(UNROLL >= SAMPLE, "the sample comes from the first step");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nvec = (int)v.nvec, n = (int)v.n, off = v.off;
    int s0, s1;
    warp_slice<THREADS>(v, w, &s0, &s1);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t* mk = rkey + w * kRunCap;
    uint32_t* mi = ridx + w * kRunCap;
    float4 f[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int sl = s0 + u * 32 + lane;
        f[u] = sl < s1 ? ldg4(v.base + sl) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    zero_shared<THREADS>(hist, kHistBins);
    if (threadIdx.x == 0) scratch[44] = 0u;
    __syncthreads();
    uint32_t ns = 0;
#pragma unroll
    for (int u = 0; u < SAMPLE; ++u) {
        const int sl = s0 + u * 32 + lane;
        const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int p = 4 * sl + c - off;
            if (sl < s1 && p >= 0 && p < n) {
                atomicAdd(&hist[fkey(e[c]) >> 20], 1u);
                ++ns;
            }
        }
    }
    ns = __reduce_add_sync(0xffffffffu, ns);
    if (lane == 0) atomicAdd(&scratch[44], ns);
    __syncthreads();
    const uint32_t P = scratch[44];
    // ceil(2 k P / n) in integers: 2 k P < 2^25 and n < 2^31, so nothing wraps
    uint32_t tg = (2u * k * P + (uint32_t)n - 1u) / (uint32_t)n;
    tg = tg < 1u ? 1u : tg > P ? P : tg;
    const uint32_t L = pick_digit<THREADS>(hist, kHistBins, tg, scratch).digit << 20;
    zero_shared<THREADS>(hist, kHistBins);
    __syncthreads();
    const float Lf = key_floor_float(L);
    uint32_t cnt = 0;
    for (int base = s0; base < s1; base += 32 * UNROLL) {
        if (base != s0) {
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int sl = base + u * 32 + lane;
                f[u] = sl < s1 ? ldg4(v.base + sl) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        const bool interior = base >= 1 && base + 32 * UNROLL <= s1 && base + 32 * UNROLL < nvec;
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            filter_step<true>(f[u], base + u * 32 + lane, interior, s1, n, off, L, Lf, lt, cnt,
                              mk, mi, hist);
    }
    if (lane == 0) rcnt[w] = cnt;
}

// Exact threshold of the k largest keys held in the warp runs.
// hist holds the level-0 histogram of the runs on entry (built while they
// were collected).
template <int THREADS>
IDX_DEVI Threshold refine_runs(const uint32_t* rkey, const uint32_t* rcnt, uint32_t k,
                               uint32_t* hist, uint32_t* scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t cnt = rcnt[w];
    const uint32_t* mk = rkey + w * kRunCap;
    uint32_t prefix = 0, need = k;
    for (int lev = 0; lev <= 2; ++lev) {
        if (lev > 0) {
            zero_shared<THREADS>(hist, kHistBins);
            __syncthreads();
            for (uint32_t i = lane; i < cnt; i += 32) {
                const uint32_t key = mk[i];
                if (has_prefix(key, lev, prefix)) atomicAdd(&hist[digit_of(key, lev)], 1u);
            }
        }
        __syncthreads();
        const DigitPick pk = pick_digit<THREADS>(hist, 1 << digit_bits(lev), need, scratch);
        need -= pk.above;
        prefix = (prefix << digit_bits(lev)) | pk.digit;
    }
    return {prefix, need};
}

// Ordered output from the runs: key > T, plus the first `need` keys == T.
template <int THREADS>
IDX_DEVI void ordered_output_runs(const uint32_t* rkey, const uint32_t* ridx,
                                  const uint32_t* rcnt, uint32_t* wsum, Threshold th,
                                  uint32_t k, int* out) {
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t cnt = rcnt[w];
    const uint32_t* mk = rkey + w * kRunCap;
    const uint32_t* mi = ridx + w * kRunCap;
    uint32_t na = 0, nt = 0;
    for (uint32_t i = lane; i < cnt; i += 32) {
        na += mk[i] > th.key;
        nt += mk[i] == th.key;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        na += __shfl_xor_sync(0xffffffffu, na, o);
        nt += __shfl_xor_sync(0xffffffffu, nt, o);
    }
    if (lane == 0) {
        wsum[w] = na;
        wsum[W + w] = nt;
    }
    __syncthreads();
    uint32_t a_run = 0, t_run = 0;
    for (int j = 0; j < w; ++j) {
        a_run += wsum[j];
        t_run += wsum[W + j];
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (uint32_t base = 0; base < cnt; base += 32) {
        const uint32_t i = base + lane;
        const uint32_t key = i < cnt ? mk[i] : 0u;
        const bool ab = i < cnt && key > th.key;
        const bool tb = i < cnt && key == th.key;
        const uint32_t A = __ballot_sync(0xffffffffu, ab), T = __ballot_sync(0xffffffffu, tb);
        const uint32_t a_b = a_run + __popc(A & lt), t_b = t_run + __popc(T & lt);
        if (ab) {
            const uint32_t pos = a_b + min(t_b, th.need);
            if (pos < k) out[pos] = static_cast<int>(mi[i]);
        } else if (tb && t_b < th.need && a_b + t_b < k) {
            out[a_b + t_b] = static_cast<int>(mi[i]);
        }
        a_run += __popc(A);
        t_run += __popc(T);
    }
}

// Visible length of row r and its first column; -1 marks a range that does
// not fit the row.
IDX_DEVI long long output_row(const TopkRowsArgs& a, int r, long long* col0) {
    const long long ks = a.ks ? a.ks[r] : 0, ke = a.ke[r];
    long long n = ke - ks;
    *col0 = a.relative ? 0 : ks;
    if (ks < 0 || n < 0 || *col0 + n > a.row_len || n > 0x7fffffffll) return ke > ks ? -1 : 0;
    return n;
}

// Lower bound L of the threshold of the k largest of a row: the lower edge of
// the 12-bit bin that holds about the 2 k * P / n-th largest of the row's
// first P = 4096 values, so that about 2 k keys of the row reach it.  The
// blocks of a split row all take this same L.
template <int THREADS>
IDX_DEVI uint32_t estimate_lower_bound(const RowView& v, uint32_t k, uint32_t* hist,
                                       uint32_t* scratch) {
    const long long n = v.n;
    const long long P = n < kPrefix ? n : kPrefix;
    const float* row = reinterpret_cast<const float*>(v.base) + v.off;
    // all loads of the prefix are issued before the first atomic
    constexpr int PER = (kPrefix + THREADS - 1) / THREADS;
    float x[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const long long p = threadIdx.x + (long long)i * THREADS;
        x[i] = p < P ? __ldg(row + p) : 0.f;
    }
    zero_shared<THREADS>(hist, kHistBins);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (threadIdx.x + (long long)i * THREADS < P) atomicAdd(&hist[fkey(x[i]) >> 20], 1u);
    __syncthreads();
    // ceil(2 k P / n) in integers: 2 k P < 2^25 and n < 2^31, so nothing wraps
    uint32_t tg = (2u * k * (uint32_t)P + (uint32_t)n - 1u) / (uint32_t)n;
    tg = tg < 1u ? 1u : tg > (uint32_t)P ? (uint32_t)P : tg;
    return pick_digit<THREADS>(hist, kHistBins, tg, scratch).digit << 20;
}

template <int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS)
topk_rows_kernel(TopkRowsArgs a) {
    using SM = StreamSmem<THREADS>;
    constexpr int W = SM::W;
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t* hist = smem;
    uint32_t* scratch = hist + kHistBins;
    uint32_t* rcnt = scratch + 64;
    uint32_t* wsum = rcnt + W;
    uint32_t* rkey = wsum + 2 * W;
    uint32_t* ridx = rkey + SM::RUN_WORDS;

    const int r = blockIdx.x;
    long long n, col0;
    {
        const long long ks = a.ks ? a.ks[r] : 0, ke = a.ke[r];
        n = ke - ks;
        col0 = a.relative ? 0 : ks;
        if (ks < 0 || n < 0 || col0 + n > a.row_len || n > 0x7fffffffll) {
            if (threadIdx.x == 0 && ke > ks) raise_status(a.d_status, IDX_DEV_RANGE);
            n = 0;
        }
        int* out = a.out + (long long)r * a.topk;
        if (n <= a.topk) {
            for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
            return;
        }
    }
    const uint32_t k = static_cast<uint32_t>(a.topk);

    const RowView v = make_view(a.scores + (long long)r * a.row_stride + col0, n);

    // a lower bound L of the threshold, or L = 0 (every key) when the runs hold the row
    const long long per_warp = 4 * ((v.nvec + W - 1) / W);
    if (per_warp > kRunCap) {
        stream_collect_estimate<THREADS, UNROLL>(v, k, hist, scratch, rkey, ridx, rcnt);
    } else {
        zero_shared<THREADS>(hist, kHistBins);
        __syncthreads();
        stream_collect<THREADS, UNROLL, true>(v, 0u, rkey, ridx, rcnt, hist);
    }
    __syncthreads();
    uint32_t total = 0;
    bool fits = true;
    for (int j = 0; j < W; ++j) {
        total += rcnt[j];
        fits = fits && rcnt[j] <= (uint32_t)kRunCap;
    }
    Threshold th;
    bool runs_ok = fits && total >= k;
    if (runs_ok) {
        th = refine_runs<THREADS>(rkey, rcnt, k, hist, scratch);
    } else {
        // the estimate missed: exact multi-pass path over the row
        __syncthreads();
        int rescans = 0;
        th = find_threshold<THREADS, 4>(v, k, hist, rkey, ridx, scratch, &rescans);
        if (threadIdx.x == 0 && a.d_stats) atomicAdd(&a.d_stats->tie_rescan_rows, 1);
    }

    int* out = a.out + (long long)r * a.topk;
    if (runs_ok)
        ordered_output_runs<THREADS>(rkey, ridx, rcnt, wsum, th, k, out);
    else
        ordered_output<THREADS>(v, th, k, out, scratch);
}

// ------------------------------------------------------ sample threshold
//
// Page 1, "Sampled Threshold": T_r is the t-th largest of the m scores of row
// r's strided sample, t = ceil(m * target * topk / len) with len the row's
// visible length, so that about target * topk keys of the row reach it.  One
// warp per row finds the exact t-th largest order key with four 8-bit radix
// passes over the sample (a warp-private 256-bin histogram each), reading the
// sample from L2; no block-wide synchronisation.
// Samples longer than this go to sample_threshold_cta_kernel.
constexpr long long kThrCtaMin = 8192;

template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
sample_threshold_kernel(TopkRowsArgs a) {
    __shared__ uint32_t hist_all[WARPS][256];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int r = blockIdx.x * WARPS + w;
    if (r >= a.rows) return;  // whole warps only: nothing below syncs the block
    uint32_t* hist = hist_all[w];
    RowPlan* plan = a.plan + r;
    const long long vks = a.vis_ks[r], vke = a.vis_ke[r];
    const long long len = vke - vks;
    const long long phase = hash32((uint32_t)(r / a.rows_per_block) ^ a.phase_seed) % a.S;
    const SampleSpan sp = sample_span(vks, vke, phase, a.S, a.nsamp);
    const long long n = sp.b - sp.a;
    if (len <= a.cap || n <= 0 || n > a.row_len) {
        if (lane == 0) {
            plan->thr = 0u;  // every visible key becomes a candidate
            plan->idx_cut = kAllIdx;
            plan->state = ST_MAIN;
            if (a.d_stats && len > 0 && len <= a.cap) atomicAdd(&a.d_stats->emit_all_rows, 1);
        }
        return;
    }
    if (a.split > 1 && n > kThrCtaMin) return;  // a whole CTA takes this row
    double t = ceil((double)n * (double)a.target * (double)a.topk / (double)len);
    if (t < 1.0) t = 1.0;
    if (t > (double)n) t = (double)n;
    const float* row = a.scores + (long long)r * a.row_stride;
    uint32_t prefix = 0u, need = (uint32_t)t;
    bool ok = true;
    for (int lev = 0; lev < 4; ++lev) {
        const int shift = 24 - 8 * lev;
#pragma unroll
        for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
        __syncwarp();
        for (long long e = lane; e < n; e += 32) {
            const uint32_t key = fkey(__ldg(row + e));
            if (lev == 0 || (key >> (shift + 8)) == prefix)
                atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncwarp();
        // lane l holds bins 255 - 8l ... 248 - 8l (from the largest keys down)
        uint32_t c[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = hist[255 - 8 * lane - j];
            local += c[j];
        }
        uint32_t incl = local;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t excl = incl - local;
        const uint32_t owner = __ballot_sync(0xffffffffu, excl < need && need <= incl);
        if (owner == 0u) {  // cannot happen: need never exceeds the keys left
            ok = false;
            break;
        }
        const int src = __ffs(owner) - 1;
        uint32_t digit = 0u, above = 0u;
        if (lane == src) {
            uint32_t cum = excl;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (cum + c[j] >= need) {
                    digit = 255u - 8u * (uint32_t)lane - (uint32_t)j;
                    above = cum;
                    break;
                }
                cum += c[j];
            }
        }
        digit = __shfl_sync(0xffffffffu, digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        need -= above;
        prefix = (prefix << 8) | digit;
        __syncwarp();
    }
    if (lane == 0) {
        // a failed pick leaves thr = 0: every key a candidate, the slab
        // overflows and the exact rescan takes the row
        plan->thr = ok ? prefix : 0u;
        plan->idx_cut = kAllIdx;
        plan->state = ST_MAIN;
    }
}

// The same threshold for long samples (tens of thousands of scores per row):
// one 256-thread CTA per row, a 12-bit histogram pass over the sample, then
// the values of the threshold bin gathered into shared memory and refined
// there (further passes over the sample only if that bin holds more than
// 4096), i.e. two passes over the sample instead of four.
constexpr int kThrCtaThreads = 256;
constexpr size_t kThrCtaSmem = (kHistBins + 64 + 2 * (size_t)kTieCap) * sizeof(uint32_t);

__global__ void __launch_bounds__(kThrCtaThreads) sample_threshold_cta_kernel(TopkRowsArgs a) {
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t* hist = smem;
    uint32_t* scratch = hist + kHistBins;
    uint32_t* tkey = scratch + 64;
    uint32_t* tpos = tkey + kTieCap;
    const int r = blockIdx.x;
    RowPlan* plan = a.plan + r;
    const long long vks = a.vis_ks[r], vke = a.vis_ke[r];
    const long long len = vke - vks;
    const long long phase = hash32((uint32_t)(r / a.rows_per_block) ^ a.phase_seed) % a.S;
    const SampleSpan sp = sample_span(vks, vke, phase, a.S, a.nsamp);
    const long long n = sp.b - sp.a;
    // rows the warp kernel handled (short samples, or no sampling at all)
    if (len <= a.cap || n <= kThrCtaMin || n > a.row_len) return;
    double t = ceil((double)n * (double)a.target * (double)a.topk / (double)len);
    if (t < 1.0) t = 1.0;
    if (t > (double)n) t = (double)n;
    const RowView v = make_view(a.scores + (long long)r * a.row_stride, n);
    int rescans = 0;
    const Threshold th =
        find_threshold<kThrCtaThreads, 4>(v, (uint32_t)t, hist, tkey, tpos, scratch, &rescans);
    if (threadIdx.x == 0) {
        plan->thr = th.key;
        plan->idx_cut = kAllIdx;
        plan->state = ST_MAIN;
    }
}

// ------------------------------------------------------- row split
//
// Page "[sglang] ROCm DSA Indexer Top-K 최적화", row_split / launch: at low
// batch a long row is split over g blocks.  Here block (c, r) streams the c-th
// contiguous slice of row r once, appends the values at or above the row's
// lower bound L (the same estimate in every block of the row) to its warps'
// runs and copies them, in index order, to the workspace; one block per row
// then selects from the concatenation (already in index order), or takes the
// exact multi-pass path over the row when a slice overflowed or L was too high.

static_assert(kSplitCap == 16 * kRunCap, "a split block hands over its 16 warp runs");

template <int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS)
topk_split_collect_kernel(TopkRowsArgs a) {
    using SM = StreamSmem<THREADS>;
    constexpr int W = SM::W;
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t* hist = smem;
    uint32_t* scratch = hist + kHistBins;
    uint32_t* rcnt = scratch + 64;
    uint32_t* wsum = rcnt + W;
    uint32_t* rkey = wsum + 2 * W;
    uint32_t* ridx = rkey + SM::RUN_WORDS;
    (void)wsum;

    const int c = blockIdx.x, r = blockIdx.y, g = gridDim.x;
    long long col0;
    const long long n = output_row(a, r, &col0);
    if (n <= a.topk) return;  // the merge block writes such rows
    const RowView v = make_view(a.scores + (long long)r * a.row_stride + col0, n);
    const uint32_t L = estimate_lower_bound<THREADS>(v, (uint32_t)a.topk, hist, scratch);
    // the slice as a view whose element indices stay row-relative
    const long long per = (v.nvec + g - 1) / g;
    const long long s0 = (long long)c * per;
    const long long s1 = s0 + per < v.nvec ? s0 + per : v.nvec;
    RowView sv;
    sv.base = v.base + s0;
    sv.off = v.off - (int)(4 * s0);
    sv.n = v.n;
    sv.nvec = s1 > s0 ? s1 - s0 : 0;
    stream_collect<THREADS, UNROLL, false>(sv, L, rkey, ridx, rcnt, nullptr);
    __syncthreads();
    // hand the runs over in warp (= index) order
    const long long slot = (long long)r * g + c;
    uint32_t* gk = a.split_keys + slot * kSplitCap;
    uint32_t* gi = a.split_idx + slot * kSplitCap;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t before = 0, total = 0;
    bool over = false;
    for (int j = 0; j < W; ++j) {
        const uint32_t cj = rcnt[j];
        over = over || cj > (uint32_t)kRunCap;
        if (j < w) before += cj;
        total += cj;
    }
    if (!over) {
        for (uint32_t i = lane; i < rcnt[w]; i += 32) {
            gk[before + i] = rkey[w * kRunCap + i];
            gi[before + i] = ridx[w * kRunCap + i];
        }
    }
    if (threadIdx.x == 0) a.split_cnt[slot] = over ? -1 : (int)total;
}

// Ordered compaction of cnt keys held in index order in shared memory.
template <int THREADS>
IDX_DEVI void ordered_output_smem(const uint32_t* keys, const uint32_t* idxs, uint32_t cnt,
                                  Threshold th, uint32_t k, int* out, uint32_t* scratch) {
    uint32_t a_run = 0, e_run = 0;
    for (uint32_t base = 0; base < cnt; base += THREADS * 4) {
        uint32_t ab = 0, tb = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t e = base + threadIdx.x * 4 + c;
            if (e < cnt) {
                ab |= (keys[e] > th.key ? 1u : 0u) << c;
                tb |= (keys[e] == th.key ? 1u : 0u) << c;
            }
        }
        const uint32_t mine = (__popc(ab) << 16) | __popc(tb);
        uint32_t tot;
        const uint32_t incl = block_incl_scan<THREADS>(mine, scratch, &tot);
        const uint32_t excl = incl - mine;
        uint32_t a_b = a_run + (excl >> 16), e_b = e_run + (excl & 0xFFFFu);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t e = base + threadIdx.x * 4 + c;
            if ((ab >> c) & 1u) {
                const uint32_t pos = a_b + min(e_b, th.need);
                if (pos < k) out[pos] = (int)idxs[e];
                ++a_b;
            } else if ((tb >> c) & 1u) {
                if (e_b < th.need && a_b + e_b < k) out[a_b + e_b] = (int)idxs[e];
                ++e_b;
            }
        }
        a_run += tot >> 16;
        e_run += tot & 0xFFFFu;
    }
}

constexpr int kMergeCap = 16384;  // candidates of a split row selected in shared memory
constexpr size_t kMergeSmem = (kHistBins + 64 + 2 * (size_t)kMergeCap) * sizeof(uint32_t);

template <int THREADS>
__global__ void __launch_bounds__(THREADS)
topk_split_merge_kernel(TopkRowsArgs a, int g) {
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t* hist = smem;
    uint32_t* scratch = hist + kHistBins;
    uint32_t* keys = scratch + 64;
    uint32_t* idxs = keys + kMergeCap;
    const int r = blockIdx.x;
    long long col0;
    long long n = output_row(a, r, &col0);
    int* out = a.out + (long long)r * a.topk;
    if (n < 0) {
        if (threadIdx.x == 0) raise_status(a.d_status, IDX_DEV_RANGE);
        n = 0;
    }
    if (n <= a.topk) {
        for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
        return;
    }
    const uint32_t k = (uint32_t)a.topk;
    if (threadIdx.x == 0) {
        uint32_t total = 0, bad = 0;
        for (int c = 0; c < g; ++c) {
            const int cc = a.split_cnt[(long long)r * g + c];
            bad |= cc < 0;
            total += cc < 0 ? 0u : (uint32_t)cc;
        }
        scratch[48] = total;
        scratch[49] = bad || total < k || total > (uint32_t)kMergeCap;
        if (a.d_stats) atomicAdd(&a.d_stats->split_rows, 1);
    }
    __syncthreads();
    const uint32_t total = scratch[48];
    const RowView v = make_view(a.scores + (long long)r * a.row_stride + col0, n);
    if (scratch[49]) {
        // a slice overflowed or L was too high: exact multi-pass path
        int rescans = 0;
        const Threshold th = find_threshold<THREADS, 4>(v, k, hist, keys, idxs, scratch, &rescans);
        if (threadIdx.x == 0 && a.d_stats) atomicAdd(&a.d_stats->tie_rescan_rows, 1);
        ordered_output<THREADS>(v, th, k, out, scratch);
        return;
    }
    uint32_t off = 0;
    for (int c = 0; c < g; ++c) {
        const long long slot = (long long)r * g + c;
        const uint32_t cc = (uint32_t)a.split_cnt[slot];
        for (uint32_t i = threadIdx.x; i < cc; i += THREADS) {
            keys[off + i] = a.split_keys[slot * kSplitCap + i];
            idxs[off + i] = a.split_idx[slot * kSplitCap + i];
        }
        off += cc;
    }
    __syncthreads();
    const Threshold th = refine_in_smem<THREADS>(keys, total, 0, 0u, k, hist, scratch);
    ordered_output_smem<THREADS>(keys, idxs, total, th, k, out, scratch);
}

// ---------------------------------------------------------------- slab
//
// Page 1, "Sampled Threshold": the small exact top-k over the ~2.25 x topk
// candidates of a row.  The scoring pass leaves each row's candidates in
// eight runs, each in ascending key order; the rescan re-emission leaves a
// single ordered run.  One CTA of 256 threads per row loads the runs into
// shared memory as (order key, index), finds the exact threshold key T with
// four 8-bit radix passes (per-warp histograms), keeps the lowest indices
// among the keys equal to T, and writes the selected indices in ascending order through a bitmap of
// the index range (65536 indices per pass): each thread owns eight bitmap
// words, and a block scan of their popcounts gives every set bit its output
// position.

constexpr int kCandThreads = 256;
constexpr int kCandWarps = kCandThreads / 32;
constexpr int kBitmapWords = kCandWarps * 256;  // the histograms' words, 65536 bits

// Exact need-th largest value among the elements e < cnt with valid(e), of
// the 32-bit values val(e), by four 8-bit digits from the top.  Returns the
// value and, through *need_at, how many elements equal to it are taken.
template <class Valid, class Val>
IDX_DEVI uint32_t cand_select(uint32_t cnt, uint32_t need, Valid valid, Val val, uint32_t* hist,
                              uint32_t* scratch, uint32_t* need_at) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t* hw = hist + w * 256;
    uint32_t prefix = 0u;
    for (int lev = 0; lev < 4; ++lev) {
        const int shift = 24 - 8 * lev;
#pragma unroll
        for (int j = 0; j < 8; ++j) hw[lane * 8 + j] = 0u;
        __syncwarp();
        for (uint32_t base = 0; base < cnt; base += 4 * kCandThreads) {
            uint32_t v[4];
            bool in[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t e = base + u * kCandThreads + threadIdx.x;
                in[u] = e < cnt && valid(e);
                v[u] = in[u] ? val(e) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (in[u] && (lev == 0 || (v[u] >> (shift + 8)) == prefix))
                    atomicAdd(&hw[(v[u] >> shift) & 255u], 1u);
        }
        __syncthreads();
        // thread t owns digit 255 - t: a scan from the top digit down
        uint32_t c = 0;
#pragma unroll
        for (int ww = 0; ww < kCandWarps; ++ww) c += hist[ww * 256 + 255 - threadIdx.x];
        const uint32_t incl = block_incl_scan<kCandThreads>(c, scratch, nullptr);
        const uint32_t excl = incl - c;
        if (excl < need && need <= incl) {
            scratch[40] = 255u - threadIdx.x;
            scratch[41] = excl;
        }
        __syncthreads();
        need -= scratch[41];
        prefix = (prefix << 8) | scratch[40];
        __syncthreads();
    }
    *need_at = need;
    return prefix;
}

__global__ void __launch_bounds__(kCandThreads)
cand_topk_kernel(CandArgs a) {
    constexpr int THREADS = kCandThreads;
    extern __shared__ __align__(16) uint32_t smem[];
    const int CR = a.nruns * a.cap_q;          // slab row (all key splits)
    const int CS = kRuns * a.cap_q;            // candidates held in shared memory
    uint32_t* hist = smem;                     // [kCandWarps][256], later the bitmap
    uint32_t* scratch = hist + kBitmapWords;   // [0,35) scans; row state from 48 on
    uint32_t* keys = scratch + kCandScratch;
    uint32_t* idxs = keys + CS;
    uint32_t* run_off = idxs + CS;             // [nruns + 1] run starts in keys[]

    if (a.fallback && *(volatile int*)(a.fb_cnt + 6) == 0) return;  // no row was re-emitted
    for (int r = blockIdx.x; r < a.rows; r += gridDim.x) {
        __syncthreads();  // the previous row's shared state is no longer read
        RowPlan* plan = a.plan + r;
        const long long n = (long long)a.ke[r] - (long long)a.ks[r];
        int* out = a.out + (long long)r * a.topk;
        if (threadIdx.x == 0) {
            scratch[48] = (uint32_t)plan->state;
            uint32_t off = 0, total = 0, trunc = 0;
            for (int q = 0; q < a.nruns; ++q) {
                const uint32_t c = (uint32_t)a.run_cnt[(long long)r * a.nruns + q];
                trunc |= c > (uint32_t)a.cap_q;
                total += c;
                run_off[q] = off;
                off += c < (uint32_t)a.cap_q ? c : (uint32_t)a.cap_q;
            }
            // more candidates than shared memory holds (possible with key
            // splits): the exact rescan takes the row
            trunc |= off > (uint32_t)CS;
            run_off[a.nruns] = off;
            scratch[49] = trunc;
            scratch[60] = total;
        }
        __syncthreads();
        const int state = (int)scratch[48];
        if (a.fallback) {
            if (state != ST_EMIT) continue;
        } else if (n <= a.topk) {
            for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
            if (threadIdx.x == 0) plan->state = ST_DONE;
            continue;
        }
        const uint32_t total = scratch[60];
        const bool trunc = scratch[49] != 0;
        if (threadIdx.x == 0 && a.d_stats && !a.fallback) atomicMax(&a.d_stats->max_count, (int)total);
        if (trunc || total < (uint32_t)a.topk) {
            if (!a.fallback && !a.fb_hist) {
                // no rescan storage: the row was longer than the max_len the
                // workspace was sized for
                for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = -1;
                if (threadIdx.x == 0) {
                    raise_status(a.d_status, IDX_DEV_RANGE);
                    plan->state = ST_DONE;
                }
            } else if (!a.fallback) {
                // the sampled threshold missed: exact full-row rescan
                for (int i = threadIdx.x; i < kHistBins; i += THREADS)
                    a.fb_hist[(long long)r * kHistBins + i] = 0u;
                if (threadIdx.x == 0) {
                    plan->state = ST_HIST;
                    plan->level = 0;
                    plan->prefix = 0u;
                    plan->above = 0;
                    atomicAdd(&a.fb_cnt[0], 1);
                    // list the row's block once for the rescan launch
                    const int blk = r / a.rows_per_block;
                    if (atomicExch(&a.fb_bflag[blk], 1) == 0)
                        a.fb_blocks[atomicAdd(&a.fb_cnt[7], 1)] = blk;
                    if (a.d_stats) {
                        atomicAdd(trunc ? &a.d_stats->overflow_rows : &a.d_stats->short_rows, 1);
                        atomicAdd(&a.d_stats->fallback_rows, 1);
                    }
                }
            } else if (threadIdx.x == 0) {
                raise_status(a.d_status, IDX_DEV_STATE);
                plan->state = ST_DONE;
            }
            continue;
        }

        // load the runs back to back, four independent loads per thread in flight
        const int2* sl = a.slab + (long long)r * CR;
        const uint32_t cnt = run_off[a.nruns];
        for (uint32_t base = 0; base < cnt; base += 4 * THREADS) {
            float sv[4];
            int iv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t e = base + u * THREADS + threadIdx.x;
                if (e < cnt) {
                    // the run holding entry e: the last q with run_off[q] <= e
                    int q = 0;
                    if (a.nruns == kRuns) {
#pragma unroll
                        for (int j = 1; j < kRuns; ++j) q += e >= run_off[j];
                    } else {
                        int hi = a.nruns;
                        while (hi - q > 1) {
                            const int mid = (q + hi) >> 1;
                            if (run_off[mid] <= e) q = mid;
                            else hi = mid;
                        }
                    }
                    const uint32_t src = (uint32_t)q * (uint32_t)a.cap_q + (e - run_off[q]);
                    const int2 c = sl[src];
                    sv[u] = __int_as_float(c.x);
                    iv[u] = c.y;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t e = base + u * THREADS + threadIdx.x;
                if (e < cnt) {
                    keys[e] = fkey(sv[u]);
                    idxs[e] = (uint32_t)iv[u];
                }
            }
        }
        __syncthreads();

        // exact threshold key T and how many keys equal to T are taken
        uint32_t need;
        const uint32_t T = cand_select(
            cnt, (uint32_t)a.topk, [](uint32_t) { return true; },
            [&](uint32_t e) { return keys[e]; }, hist, scratch, &need);
        // the lowest `need` indices among the keys equal to T
        uint32_t nt = 0;
        for (uint32_t e = threadIdx.x; e < cnt; e += THREADS) nt += keys[e] == T;
        uint32_t ntie;
        block_incl_scan<THREADS>(nt, scratch, &ntie);
        uint32_t idx_cut = 0xffffffffu;
        if (ntie > need) {
            uint32_t unused;
            idx_cut = ~cand_select(
                cnt, need, [&](uint32_t e) { return keys[e] == T; },
                [&](uint32_t e) { return ~idxs[e]; }, hist, scratch, &unused);
        }

        // ascending output through the index bitmap, 65536 indices per pass
        uint32_t* bm = hist;
        constexpr int WPT = kBitmapWords / THREADS;  // bitmap words per thread
        uint32_t written = 0;
        for (long long c0 = 0; c0 < n && written < (uint32_t)a.topk; c0 += 32ll * kBitmapWords) {
#pragma unroll
            for (int j = 0; j < WPT; ++j) bm[threadIdx.x * WPT + j] = 0u;
            __syncthreads();
            for (uint32_t base = 0; base < cnt; base += 4 * THREADS) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t e = base + u * THREADS + threadIdx.x;
                    if (e < cnt) {
                        const uint32_t ky = keys[e], ix = idxs[e];
                        const long long rel = (long long)ix - c0;
                        if ((ky > T || (ky == T && ix <= idx_cut)) && rel >= 0 &&
                            rel < 32ll * kBitmapWords)
                            atomicOr(&bm[rel >> 5], 1u << (rel & 31));
                    }
                }
            }
            __syncthreads();
            uint32_t wv[WPT], local = 0;
#pragma unroll
            for (int j = 0; j < WPT; ++j) {
                wv[j] = bm[threadIdx.x * WPT + j];
                local += __popc(wv[j]);
            }
            uint32_t tot;
            const uint32_t incl = block_incl_scan<THREADS>(local, scratch, &tot);
            uint32_t pos = written + incl - local;
#pragma unroll
            for (int j = 0; j < WPT; ++j) {
                uint32_t x = wv[j];
                const long long wbase = c0 + 32ll * (threadIdx.x * WPT + j);
                while (x) {
                    const int bit = __ffs(x) - 1;
                    if (pos < (uint32_t)a.topk) out[pos] = (int)(wbase + bit);
                    ++pos;
                    x &= x - 1u;
                }
            }
            written += tot;
        }
        if (threadIdx.x == 0) plan->state = ST_DONE;
    }
}

// ------------------------------------------------------------ launchers

cudaError_t launch_topk_rows(const TopkRowsArgs& a, cudaStream_t s) {
    constexpr int T = 512, U = 8;
    constexpr size_t SMEM = StreamSmem<T>::BYTES;
    if (a.rows == 0) return cudaSuccess;
    if (a.mode == TOPK_THRESHOLD) {
        // one warp per row; when some row's sample may exceed kThrCtaMin
        // scores, those rows are left to one CTA each (two passes over the
        // sample instead of four), flagged to the warp kernel by split = 2
        constexpr int WARPS = 8;
        TopkRowsArgs b = a;
        b.split = a.row_len > kThrCtaMin ? 2 : 0;
        sample_threshold_kernel<WARPS><<<(a.rows + WARPS - 1) / WARPS, WARPS * 32, 0, s>>>(b);
        if (b.split) {
            static cudaError_t attr = cudaFuncSetAttribute(
                sample_threshold_cta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                (int)kThrCtaSmem);
            if (attr != cudaSuccess) return attr;
            sample_threshold_cta_kernel<<<a.rows, kThrCtaThreads, kThrCtaSmem, s>>>(b);
            count_launches(1);
        }
        return cudaGetLastError();
    }
    if (a.split > 1) {
        auto coll = topk_split_collect_kernel<T, U>;
        auto merge = topk_split_merge_kernel<T>;
        static cudaError_t attr = [&] {
            cudaError_t e = cudaFuncSetAttribute(coll, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kMergeSmem);
            return e;
        }();
        if (attr != cudaSuccess) return attr;
        coll<<<dim3((unsigned)a.split, (unsigned)a.rows), T, SMEM, s>>>(a);
        merge<<<a.rows, T, kMergeSmem, s>>>(a, a.split);
        return cudaGetLastError();
    }
    auto kern = topk_rows_kernel<T, U>;
    static cudaError_t attr = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (attr != cudaSuccess) return attr;
    kern<<<a.rows, T, SMEM, s>>>(a);
    return cudaGetLastError();
}

size_t split_workspace_bytes(int rows, int g) {
    if (g < 2) return 0;
    const size_t slots = (size_t)rows * g;
    return slots * (size_t)kSplitCap * 2 * sizeof(uint32_t) + slots * sizeof(int) + 256;
}

size_t cand_smem_bytes(int cap_q, int nruns) {
    return (kBitmapWords + kCandScratch + (size_t)nruns + 1) * sizeof(uint32_t) +
           (size_t)cap_q * kRuns * 2 * sizeof(uint32_t);
}

cudaError_t launch_cand_topk(const CandArgs& a, cudaStream_t s) {
    const size_t sm = cand_smem_bytes(a.cap_q, a.nruns);
    cudaError_t e =
        cudaFuncSetAttribute(cand_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (a.rows == 0) return cudaSuccess;
    // the rescan's pass usually has no row to select: a short grid that strides
    // over the rows exits at once
    const int grid = a.fallback ? (a.rows < a.grid_limit ? a.rows : a.grid_limit) : a.rows;
    cand_topk_kernel<<<grid, kCandThreads, sm, s>>>(a);
    return cudaGetLastError();
}

}  // namespace idx

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
//  * cand_topk_kernel   one CTA per row of the candidate slab (page 1: the
//                       small top-k over ~2.25 x topk candidates), read from
//                       global memory by every pass or, with key splits,
//                       copied into shared memory first; flags rows whose
//                       slab is short or overflowed for the exact rescan.
#include "plan.cuh"
#include "radix.cuh"
#include "threshold.cuh"
#include "topk.cuh"

namespace idx {

void count_launches(unsigned n);  // api.cu

constexpr int kTieCap = 4096;

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
// estimated from a sample of up to 8192 values (aiming at about 1.5 k keys >=
// L): the first 512 values of each warp's slice, which the filter loads first
// anyway.  Every key >= L is then appended to its warp's run in
// shared memory, and the top digits of the appended keys are counted on the
// way (level 0 of the refinement).  Warp w owns the contiguous slice w of the row and appends in index
// order, so the runs, taken in warp order, list the candidates in ascending
// index order.  The exact threshold is then refined over the candidates and an
// ordered compaction writes the result.  When L was too high (fewer than k
// candidates) or a run overflowed, the row falls back to the multi-pass path
// above, which is exact for any input.

constexpr int kRunCap = 512;       // candidates per warp run

template <int THREADS>
struct StreamSmem {
    static constexpr int W = THREADS / 32;
    static constexpr int RUN_WORDS = W * kRunCap;          // per array
    static_assert(2 * RUN_WORDS >= 2 * kTieCap, "tie buffer aliases the runs");
    // hist | scratch(64) | rcnt(W) | wsum(2W) | run keys | run idx
    static constexpr size_t BYTES =
        (kHistBins + 64 + 3 * W + 2 * (size_t)RUN_WORDS) * sizeof(uint32_t);
};

// One step of a warp's filter over the 32 · UNROLL float4 slots [base, base +
// 32 · UNROLL) of its slice, lane l holding slots base + 32 u + l (u < UNROLL:
// coalesced loads), so the step's index order is slot row u, then lane, then
// component: every value >= L (key order; Lf is the float of L; L = 0 takes
// every value) is appended to the warp's run in index order.  The step has two
// halves.  hit_mask forms the lane's 32-bit hit mask (bit 4 u + c) from the
// values in registers; after it the registers are free, so the caller issues
// the next step's loads before append_hits, which packs the lane's eight
// per-row hit counts into two words of 8-bit fields; two warp scans of those
// words give every lane its place in every row at once.  Each lane then
// appends only its own hits, re-reading their values (L1 hits, two loads in
// flight at a time): the cross-lane work is paid once per 32 · UNROLL · 4
// values.  With HIST every hit is counted in hist as well: rel = false, by its
// 12-bit top digit (level 0 of the refinement over the runs); rel = true, in
// bin min((key - hb) >> 12, 4095) of a histogram relative to hb, a key at or
// below every hit.
template <int UNROLL>
IDX_DEVI uint32_t hit_mask(const float4 (&f)[UNROLL], int base, bool interior, int s1, int n,
                           int off, uint32_t L, float Lf, int lane) {
    static_assert(UNROLL == 8, "eight rows of 4 values: one 32-bit mask, two count words");
    uint32_t m = 0u;
    if (interior) {
        // each compare gives 1.0 or 0.0 (one ALU instruction, the busiest pipe
        // here); the bits are summed as exact powers of two on the FMA pipe,
        // 16 per accumulator
        auto ge = [](float x, float y) {
            float r;
            asm("set.ge.f32.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "f"(y));
            return r;
        };
        float acc[2] = {0.f, 0.f};
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int h = u >> 2, b = 4 * (u & 3);
            acc[h] = fmaf(ge(f[u].x, Lf), (float)(1u << b), acc[h]);
            acc[h] = fmaf(ge(f[u].y, Lf), (float)(1u << (b + 1)), acc[h]);
            acc[h] = fmaf(ge(f[u].z, Lf), (float)(1u << (b + 2)), acc[h]);
            acc[h] = fmaf(ge(f[u].w, Lf), (float)(1u << (b + 3)), acc[h]);
        }
        m = (uint32_t)acc[0] | ((uint32_t)acc[1] << 16);
    } else {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int sl = base + 32 * u + lane;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int p = 4 * sl + c - off;
                const bool h = sl < s1 && p >= 0 && p < n && (L == 0u || e[c] >= Lf);
                m |= (h ? 1u : 0u) << (4 * u + c);
            }
        }
    }
    return m;
}

template <int UNROLL, bool HIST>
IDX_DEVI void append_hits(const RowView& v, uint32_t m, int base, int off, int lane,
                          uint32_t& cnt, uint32_t* mk, uint32_t* mi, uint32_t* hist,
                          uint32_t hb = 0u, bool rel = false) {
    if (!__any_sync(0xffffffffu, m != 0u)) return;
    // per-row hit counts, four 8-bit fields per word (a row's warp total <=
    // 128): the eight nibble counts of m side by side (two SWAR steps), then
    // rows 0-3 and 4-7 gathered into the bytes of w0 and w1
    uint32_t x = m - ((m >> 1) & 0x55555555u);
    x = (x & 0x33333333u) + ((x >> 2) & 0x33333333u);  // nibble u: hits of row u
    const uint32_t ev = x & 0x0f0f0f0fu, od = (x >> 4) & 0x0f0f0f0fu;
    const uint32_t w0 = __byte_perm(ev, od, 0x5140u), w1 = __byte_perm(ev, od, 0x7362u);
    uint32_t i0 = w0, i1 = w1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t0 = __shfl_up_sync(0xffffffffu, i0, o);
        const uint32_t t1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
            i0 += t0;
            i1 += t1;
        }
    }
    const uint32_t t0 = __shfl_sync(0xffffffffu, i0, 31), t1 = __shfl_sync(0xffffffffu, i1, 31);
    const uint32_t e0 = i0 - w0, e1 = i1 - w1;  // lanes below, per row
    // where row u starts in the run: cnt + the totals of rows 0 .. u - 1
    const uint32_t r1 = t0 & 0xffu, r2 = r1 + ((t0 >> 8) & 0xffu), r3 = r2 + ((t0 >> 16) & 0xffu),
                   r4 = r3 + (t0 >> 24);
    const uint32_t r5 = r4 + (t1 & 0xffu), r6 = r5 + ((t1 >> 8) & 0xffu),
                   r7 = r6 + ((t1 >> 16) & 0xffu), r8 = r7 + (t1 >> 24);
    const uint32_t rs[UNROLL] = {0u, r1, r2, r3, r4, r5, r6, r7};
    const float* vals = reinterpret_cast<const float*>(v.base);
    const uint32_t m0 = m;  // the lane's hits (m loses them one by one below)
    // run position and value address of hit bit i
    auto place = [&](int i, uint32_t* pos) {
        const int u = i >> 2, c = i & 3;
        const uint32_t below = __byte_perm(e0, e1, (uint32_t)u) & 0xffu;  // byte u of (e1:e0)
        uint32_t start = 0u;
#pragma unroll
        for (int j = 1; j < UNROLL; ++j) start = u == j ? rs[j] : start;
        *pos = cnt + start + below + (uint32_t)__popc((m0 >> (4 * u)) & ((1u << c) - 1u));
        return 4 * (base + 32 * u + lane) + c;  // float offset from v.base
    };
    auto put = [&](uint32_t pos, int e, float x) {
        const uint32_t key = fkey(x);
        if (pos < (uint32_t)kRunCap) {
            mk[pos] = key;
            mi[pos] = static_cast<uint32_t>(e - off);
        }
        if (HIST) {
            const uint32_t d = (key - hb) >> 12;
            atomicAdd(&hist[rel ? (d < (uint32_t)kHistBins ? d : (uint32_t)kHistBins - 1u)
                                : key >> 20],
                      1u);
        }
    };
    while (m) {
        // two hits per round, both loads in flight before either value is used
        const int i0 = __ffs(m) - 1;
        m &= m - 1u;
        const bool two = m != 0u;
        const int i1 = two ? __ffs(m) - 1 : i0;
        if (two) m &= m - 1u;
        uint32_t p0, p1;
        const int a0 = place(i0, &p0), a1 = place(i1, &p1);
        const float x0 = __ldg(vals + a0), x1 = __ldg(vals + a1);
        put(p0, a0, x0);
        if (two) put(p1, a1, x1);
    }
    cnt += r8;
}

// Both halves of a step on values already in registers.
template <int UNROLL, bool HIST>
IDX_DEVI void filter_block(const RowView& v, const float4 (&f)[UNROLL], int base, bool interior,
                           int s1, int n, int off, uint32_t L, float Lf, int lane, uint32_t& cnt,
                           uint32_t* mk, uint32_t* mi, uint32_t* hist) {
    const uint32_t m = hit_mask<UNROLL>(f, base, interior, s1, n, off, L, Lf, lane);
    append_hits<UNROLL, HIST>(v, m, base, off, lane, cnt, mk, mi, hist);
}

// The UNROLL float4 slots of lane `lane` in one step of a warp's part: slots
// base + 32 u + lane (coalesced; see filter_block).
template <int UNROLL>
IDX_DEVI void load_step(const RowView& v, int base, int s1, int lane, float4 (&f)[UNROLL]) {
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int sl = base + 32 * u + lane;
        f[u] = sl < s1 ? ldg4(v.base + sl) : make_float4(0.f, 0.f, 0.f, 0.f);
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
    uint32_t* mk = rkey + w * kRunCap;
    uint32_t* mi = ridx + w * kRunCap;
    uint32_t cnt = 0;
    float4 f[UNROLL];
    load_step<UNROLL>(v, s0, s1, lane, f);
    for (int base = s0; base < s1; base += 32 * UNROLL) {
        const int nb = base + 32 * UNROLL;
        // every slot of this step holds 4 visible values (warp-uniform)
        const bool interior = base >= 1 && nb <= s1 && nb < nvec;
        const uint32_t m = hit_mask<UNROLL>(f, base, interior, s1, n, off, L, Lf, lane);
        if (nb < s1) load_step<UNROLL>(v, nb, s1, lane, f);  // in flight during the append
        append_hits<UNROLL, HIST>(v, m, base, off, lane, cnt, mk, mi, hist);
    }
    if (lane == 0) rcnt[w] = cnt;
}

// The one-pass collection of a whole row by one CTA, lower bound included.
// The sample is the first SAMPLE float4 slots of every lane in the first step
// of every warp's slice (P <= 8192 values for 512 threads), values the filter
// loads anyway.  L is the 20-bit floor of the sample's tg-th largest order
// key: the 12-bit digit that holds it, then the next 8 bits among the sample
// keys of that digit.  The row has fewer than k keys >= L only when tg or more
// sample keys exceed the row's k-th largest, a binomial count of mean
// m = k P / n.  tg = max(1.5 m, min(m + 5.7 sqrt(m) + 1, c)), c being the rank
// at which the expected count of keys >= L (tg n / P) fills 70 % of the runs:
// a miss is a 5.7-spread event whatever n / k is (about 1.5 k keys reach L for
// n = 131072 and k = 2048, m = 128; for a long row and a small k, m is a few
// and the margin above m decides, not 1.5 m), while the runs keep room.  A
// miss costs time only (the row takes the exact multi-pass path).  hist leaves
// holding the histogram of the hits relative to the returned key B (bins of
// 4096 keys from B up, the last bin open), B being the order key of the float
// bound (every hit has key >= B: fkey folds -0 onto +0, so a bound of zero
// holds both zeros at B).
template <int THREADS, int UNROLL>
IDX_DEVI uint32_t stream_collect_estimate(const RowView& v, uint32_t k, uint32_t* hist,
                                      uint32_t* scratch, uint32_t* rkey, uint32_t* ridx,
                                      uint32_t* rcnt) {
    constexpr int SAMPLE = 4;  // float4 slots per lane in the sample
    static_assert(UNROLL >= SAMPLE, "the sample comes from the first step");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nvec = (int)v.nvec, n = (int)v.n, off = v.off;
    int s0, s1;
    warp_slice<THREADS>(v, w, &s0, &s1);
    uint32_t* mk = rkey + w * kRunCap;
    uint32_t* mi = ridx + w * kRunCap;
    float4 f[UNROLL];
    load_step<UNROLL>(v, s0, s1, lane, f);
    zero_shared<THREADS>(hist, kHistBins);
    if (threadIdx.x == 0) scratch[44] = 0u;
    __syncthreads();
    // in_sample(u, c): slot s0 + 32 u + lane holds visible value c
    auto in_sample = [&](int u, int c) {
        const int sl = s0 + 32 * u + lane;
        const int p = 4 * sl + c - off;
        return sl < s1 && p >= 0 && p < n;
    };
    uint32_t ns = 0;
#pragma unroll
    for (int u = 0; u < SAMPLE; ++u) {
        const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (in_sample(u, c)) {
                atomicAdd(&hist[fkey(e[c]) >> 20], 1u);
                ++ns;
            }
        }
    }
    ns = __reduce_add_sync(0xffffffffu, ns);
    if (lane == 0) atomicAdd(&scratch[44], ns);
    __syncthreads();
    const uint32_t P = scratch[44];
    // m = the sample keys expected above the row's k-th largest; a miss needs
    // tg of them, so tg = m + 5.7 sqrt(m) + 1 keeps it a 5.7-spread event at
    // any n / k (1.5 m alone, the floor, is that only for m >= ~130), as long
    // as the expected candidates (tg n / P) fill at most 70 % of the runs
    const float m = (float)k * (float)P / (float)n;
    const float t_safe = m + 5.7f * sqrtf(m) + 1.0f;
    const float t_cap = 0.7f * (float)((THREADS / 32) * kRunCap) * (float)P / (float)n;
    const float t = fmaxf(ceilf(1.5f * m), fminf(t_safe, t_cap));
    const uint32_t tg = t < 1.0f ? 1u : t >= (float)P ? P : (uint32_t)ceilf(t);
    const DigitPick d0 = pick_digit<THREADS>(hist, kHistBins, tg, scratch);
    // the next 8 bits of the sample keys in digit d0 (pick_digit ends on a barrier)
    zero_shared<THREADS>(hist, 256);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < SAMPLE; ++u) {
        const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t key = fkey(e[c]);
            if (in_sample(u, c) && (key >> 20) == d0.digit) atomicAdd(&hist[(key >> 12) & 0xffu], 1u);
        }
    }
    __syncthreads();
    const DigitPick d1 = pick_digit<THREADS>(hist, 256, tg - d0.above, scratch);
    const uint32_t L = (d0.digit << 20) | (d1.digit << 12);
    zero_shared<THREADS>(hist, kHistBins);
    __syncthreads();
    const float Lf = key_floor_float(L);
    const uint32_t B = fkey(Lf);
    uint32_t cnt = 0;
    for (int base = s0; base < s1; base += 32 * UNROLL) {
        const int nb = base + 32 * UNROLL;
        const bool interior = base >= 1 && nb <= s1 && nb < nvec;
        const uint32_t m = hit_mask<UNROLL>(f, base, interior, s1, n, off, L, Lf, lane);
        if (nb < s1) load_step<UNROLL>(v, nb, s1, lane, f);  // in flight during the append
        append_hits<UNROLL, true>(v, m, base, off, lane, cnt, mk, mi, hist, B, true);
    }
    if (lane == 0) rcnt[w] = cnt;
    return B;
}

// Exact threshold of the k largest keys held in the warp runs, by the three
// key levels.  With lev0_ready hist holds the level-0 histogram of the runs on
// entry (built while they were collected); otherwise it is built here.
template <int THREADS>
IDX_DEVI Threshold refine_runs(const uint32_t* rkey, const uint32_t* rcnt, uint32_t k,
                               uint32_t* hist, uint32_t* scratch, bool lev0_ready) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t cnt = rcnt[w];
    const uint32_t* mk = rkey + w * kRunCap;
    uint32_t prefix = 0, need = k;
    for (int lev = 0; lev <= 2; ++lev) {
        if (lev > 0 || !lev0_ready) {
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

// Exact threshold of the k largest of the keys held in shared memory, warp w
// holding those in [lo, hi) (its run, or its chunk), from hist, the histogram
// of all of them relative to B (bin min((key - B) >> 12, 4095), every key >=
// B).  The bin that holds the k-th largest key gives T's top bits; one pass
// then takes the least and the largest key of that bin and counts, per warp,
// the keys above the bin and in it.  When the bin holds a single key value
// (always for scores on the bf16 grid, whose low 16 bits are constant) that
// value is T and the per-warp counts are those of keys > T and == T, left in
// wsum for the output (*counted); otherwise the bin's low 12 bits are
// resolved by one more histogram.  Returns false when the k-th largest key
// lies in the open last bin (the caller then refines by absolute digits).
// wsum may alias scratch (the counts take its first 2 W words).
template <int THREADS>
IDX_DEVI bool refine_rel(const uint32_t* keys, uint32_t lo, uint32_t hi, uint32_t k, uint32_t B,
                         uint32_t* hist, uint32_t* scratch, uint32_t* wsum, Threshold* th,
                         bool* counted) {
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        scratch[48] = 0xffffffffu;  // least in-bin offset
        scratch[49] = 0u;           // largest in-bin offset
    }
    __syncthreads();
    const DigitPick pk = pick_digit<THREADS>(hist, kHistBins, k, scratch);
    if (pk.digit == (uint32_t)kHistBins - 1u) return false;
    const uint32_t bl = B + (pk.digit << 12);  // the bin holds keys bl .. bl + 4095
    uint32_t mn = 0xffffffffu, mx = 0u, na = 0u, nt = 0u;
    for (uint32_t i = lo + lane; i < hi; i += 32) {
        const uint32_t key = keys[i], d = key - bl;
        if (d < 4096u) {
            mn = min(mn, d);
            mx = max(mx, d);
            ++nt;
        } else {
            na += key > bl;
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    na = __reduce_add_sync(0xffffffffu, na);
    nt = __reduce_add_sync(0xffffffffu, nt);
    if (lane == 0) {
        wsum[w] = na;
        wsum[W + w] = nt;
        if (nt) {
            atomicMin(&scratch[48], mn);
            atomicMax(&scratch[49], mx);
        }
    }
    __syncthreads();
    const uint32_t need = k - pk.above;
    if (scratch[48] == scratch[49]) {
        *th = {bl + scratch[48], need};
        *counted = true;
        return true;
    }
    zero_shared<THREADS>(hist, kHistBins);
    __syncthreads();
    for (uint32_t i = lo + lane; i < hi; i += 32) {
        const uint32_t d = keys[i] - bl;
        if (d < 4096u) atomicAdd(&hist[d], 1u);
    }
    __syncthreads();
    const DigitPick p2 = pick_digit<THREADS>(hist, kHistBins, need, scratch);
    *th = {bl + p2.digit, need - p2.above};
    *counted = false;
    return true;
}

// Ordered output from keys held in index order in shared memory, warp w
// holding [lo, hi) and the warps following each other: key > T, plus the
// first `need` keys == T.  One count pass (skipped with counted: wsum already
// holds every warp's counts of keys > T and == T), one synchronisation for
// the warp offsets, then each warp writes its range with ballot ranks (32 keys
// per step).
template <int THREADS>
IDX_DEVI void ordered_output_range(const uint32_t* keys, const uint32_t* idxs, uint32_t lo,
                                   uint32_t hi, uint32_t* wsum, Threshold th, uint32_t k,
                                   int* out, bool counted) {
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (!counted) {
        uint32_t na = 0, nt = 0;
        for (uint32_t i = lo + lane; i < hi; i += 32) {
            na += keys[i] > th.key;
            nt += keys[i] == th.key;
        }
        na = __reduce_add_sync(0xffffffffu, na);
        nt = __reduce_add_sync(0xffffffffu, nt);
        if (lane == 0) {
            wsum[w] = na;
            wsum[W + w] = nt;
        }
        __syncthreads();
    }
    uint32_t a_run = 0, t_run = 0;
    for (int j = 0; j < w; ++j) {
        a_run += wsum[j];
        t_run += wsum[W + j];
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (uint32_t base = lo; base < hi; base += 32) {
        const uint32_t i = base + lane;
        const uint32_t key = i < hi ? keys[i] : 0u;
        const bool ab = i < hi && key > th.key;
        const bool tb = i < hi && key == th.key;
        const uint32_t A = __ballot_sync(0xffffffffu, ab), T = __ballot_sync(0xffffffffu, tb);
        const uint32_t a_b = a_run + __popc(A & lt), t_b = t_run + __popc(T & lt);
        if (ab) {
            const uint32_t pos = a_b + min(t_b, th.need);
            if (pos < k) out[pos] = static_cast<int>(idxs[i]);
        } else if (tb && t_b < th.need && a_b + t_b < k) {
            out[a_b + t_b] = static_cast<int>(idxs[i]);
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
    const bool rel = per_warp > kRunCap;  // hist relative to B (else level 0 by absolute digit)
    uint32_t B = 0u;
    if (rel) {
        B = stream_collect_estimate<THREADS, UNROLL>(v, k, hist, scratch, rkey, ridx, rcnt);
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
    bool counted = false;
    const bool runs_ok = fits && total >= k;
    const int w = threadIdx.x >> 5;
    if (runs_ok) {
        const uint32_t lo = w * kRunCap;
        if (!rel || !refine_rel<THREADS>(rkey, lo, lo + rcnt[w], k, B, hist, scratch, wsum, &th,
                                         &counted))
            th = refine_runs<THREADS>(rkey, rcnt, k, hist, scratch, !rel);
    } else {
        // the estimate missed: exact multi-pass path over the row
        __syncthreads();
        int rescans = 0;
        th = find_threshold<THREADS, 4>(v, k, hist, rkey, ridx, scratch, &rescans);
        if (threadIdx.x == 0 && a.d_stats) atomicAdd(&a.d_stats->tie_rescan_rows, 1);
    }

    int* out = a.out + (long long)r * a.topk;
    if (runs_ok)
        ordered_output_range<THREADS>(rkey, ridx, w * kRunCap, w * kRunCap + rcnt[w], wsum, th,
                                      k, out, counted);
    else
        ordered_output<THREADS>(v, th, k, out, scratch);
}

// ------------------------------------------------------ sample threshold
//
// T_r of every sampled row (threshold.cuh): one warp per row; rows whose
// sample holds more than kThrCtaMin keys go to sample_threshold_cta_kernel.
constexpr long long kThrCtaMin = 8192;

IDX_DEVI ThrParams thr_params(const TopkRowsArgs& a) {
    ThrParams p;
    p.ks = a.vis_ks;
    p.ke = a.vis_ke;
    p.samp = a.samp;
    p.samp_stride = a.row_stride;
    p.nsamp = a.nsamp;
    p.S = a.S;
    p.cap = a.cap;
    p.topk = a.topk;
    p.target = a.target;
    p.rows_per_block = a.rows_per_block;
    p.phase_seed = a.phase_seed;
    p.plan = a.plan;
    p.d_stats = a.d_stats;
    return p;
}

// The emit pass's block order (TopkRowsArgs::order): row blocks by the number
// of 128-key tiles their rows' visible ranges span, longest first, so that the
// persistent launch hands out the long units before the short ones (a long
// unit taken last leaves the other SMs idle while it runs).  A counting sort
// over 1024 buckets, 32 per octave of the tile count (bucket 0: nothing to
// score); the order within a bucket is arbitrary.
template <int THREADS>
IDX_DEVI void block_order(const TopkRowsArgs& a, uint32_t* bins /* 1024 + 32 */) {
    constexpr int NB = 1024, BPT = NB / THREADS;
    static_assert(NB % THREADS == 0 && THREADS % 32 == 0, "bins per thread");
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nblk = a.order_nblk, R = a.order_rpb;
    auto bucket = [&](int b) -> uint32_t {
        long long lo = 0x7fffffffffffffffll, hi = -1;
        for (int j = 0; j < R; ++j) {
            const long long r = (long long)b * R + j;
            if (r >= a.rows) break;
            const long long s0 = a.vis_ks[r], s1 = a.vis_ke[r];
            if (s1 > s0) {
                lo = s0 < lo ? s0 : lo;
                hi = s1 > hi ? s1 : hi;
            }
        }
        if (hi <= lo) return 0u;
        const long long tl = (hi - lo + 127) / 128;
        const uint32_t t = tl < (1ll << 30) ? (uint32_t)tl : (1u << 30);
        const int e = 31 - __clz(t);
        const uint32_t m = e >= 5 ? (t >> (e - 5)) & 31u : (t << (5 - e)) & 31u;
        return 1u + 32u * (uint32_t)e + m;  // < 1 + 32 * 31 + 32 = 1025: <= 1023 for e <= 30
    };
    for (int i = tid; i < NB; i += THREADS) bins[i] = 0u;
    __syncthreads();
    for (int b = tid; b < nblk; b += THREADS) atomicAdd(&bins[min(bucket(b), (uint32_t)NB - 1u)], 1u);
    __syncthreads();
    // bucket starts, the largest bucket first: thread t owns buckets
    // NB - 1 - BPT t ... NB - BPT (t + 1)
    uint32_t c[BPT], loc = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        c[j] = bins[NB - 1 - (BPT * tid + j)];
        loc += c[j];
    }
    uint32_t incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    uint32_t* wsum = bins + NB;
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    uint32_t st = incl - loc;
    for (int j = 0; j < w; ++j) st += wsum[j];
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        bins[NB - 1 - (BPT * tid + j)] = st;
        st += c[j];
    }
    __syncthreads();
    for (int b = tid; b < nblk; b += THREADS)
        a.order[atomicAdd(&bins[min(bucket(b), (uint32_t)NB - 1u)], 1u)] = b;
}

template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
sample_threshold_kernel(TopkRowsArgs a) {
    __shared__ uint32_t hist_all[WARPS][256];
    __shared__ uint4 stage_all[WARPS][kThrStage];
    static_assert(sizeof(stage_all) >= (1024 + 32) * sizeof(uint32_t), "order bins");
    pdl_wait();
    if (a.order && blockIdx.x == gridDim.x - 1) {
        // the last CTA: the emit pass's block order
        block_order<WARPS * 32>(a, reinterpret_cast<uint32_t*>(&stage_all[0][0]));
        return;
    }
    const int w = threadIdx.x >> 5;
    const int r = blockIdx.x * WARPS + w;
    if (r >= a.rows) return;  // whole warps only: nothing below syncs the block
    warp_row_threshold(thr_params(a), r, hist_all[w], a.split > 1 ? (uint32_t)kThrCtaMin : 0u,
                       stage_all[w]);
}

// The same threshold for long samples (tens of thousands of keys per row):
// one 256-thread CTA per row, the two 8-bit passes over per-warp histograms.
constexpr int kThrCtaThreads = 256;

__global__ void __launch_bounds__(kThrCtaThreads) sample_threshold_cta_kernel(TopkRowsArgs a) {
    constexpr int THREADS = kThrCtaThreads, W = THREADS / 32;
    __shared__ uint32_t hist[W * 256];
    __shared__ uint32_t scratch[64];
    pdl_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int r = blockIdx.x;
    SampleRow sr;
    // rows the warp kernel handled (short samples, or no sampling at all)
    if (!sample_row(thr_params(a), r, &sr) || sr.n <= kThrCtaMin) return;
    uint32_t* hw = hist + w * 256;
    uint32_t prefix = 0u, need = sr.t;
    for (int lev = 0; lev < 2; ++lev) {
        const int shift = 8 - 8 * lev;
#pragma unroll
        for (int j = 0; j < 8; ++j) hw[lane * 8 + j] = 0u;
        __syncthreads();
        // four independent 16-byte loads of 8 keys each per thread in flight
        const uint4* v4 = reinterpret_cast<const uint4*>(sr.keys);
        const uint32_t n8 = sr.n / 8;
        for (uint32_t base = threadIdx.x; base < n8; base += 4 * THREADS) {
            uint4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                x[u] = base + u * THREADS < n8 ? __ldcg(v4 + base + u * THREADS) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (base + u * THREADS >= n8) continue;
                const uint32_t wd[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = (wd[h >> 1] >> (16 * (h & 1))) & 0xffffu;
                    if (lev == 0 || (key >> 8) == prefix) atomicAdd(&hw[(key >> shift) & 255u], 1u);
                }
            }
        }
        for (uint32_t e = n8 * 8 + threadIdx.x; e < sr.n; e += THREADS) {
            const uint32_t key = sr.keys[e];
            if (lev == 0 || (key >> 8) == prefix) atomicAdd(&hw[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        // thread t owns digit 255 - t: a scan from the top digit down
        uint32_t c = 0;
#pragma unroll
        for (int ww = 0; ww < W; ++ww) c += hist[ww * 256 + 255 - threadIdx.x];
        const uint32_t incl = block_incl_scan<THREADS>(c, scratch, nullptr);
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
    if (threadIdx.x == 0) set_plan_threshold(a.plan + r, prefix << 16);
}

// ------------------------------------------------------- row split
//
// Page "[sglang] ROCm DSA Indexer Top-K 최적화", row_split / launch: at low
// batch a long row is split over g blocks.  Here block (c, r) streams the c-th
// contiguous slice of row r once, appends the values at or above a lower
// bound L_c to its warps' runs and copies them, in index order, to the
// workspace together with L_c.  L_c comes from the values the block loads
// first (the lower edge of the 12-bit bin of about the 2 k P / n-th largest of
// its P sampled values: about 2 k n_c / n of its n_c values reach it), so no
// block waits for another read.  The block of the row that finishes last (it
// draws the last ticket of a per-row counter whose word carries the call's
// epoch in its high half, so that a word left by another call, or never
// written, counts as no ticket drawn: no clearing before the launch) then
// selects from the concatenation, already in index order.  The result is
// exact when the k-th largest candidate T' is >= every L_c: a value a block
// left out is below its L_c <= T', hence below the row's k-th largest, and
// every value >= T' is a candidate.  Otherwise (or when a slice overflowed or
// fewer than k values reached their bounds) the block takes the exact
// multi-pass path over the row.  Selection thus starts as soon as a row's
// slices are in, in the same launch.
static_assert(kSplitCap == 16 * kRunCap, "a split block hands over its 16 warp runs");

constexpr int kMergeCap = 16384;  // candidates of a split row selected in shared memory
constexpr int kMaxSplit = 64;

template <int THREADS>
struct SplitSmem {
    // collection: the StreamSmem layout; selection, over the same memory:
    // hist | scratch (64) | slice offsets and row words (kMaxSplit + 8) | keys | idxs
    static constexpr size_t COLLECT = StreamSmem<THREADS>::BYTES;
    static constexpr int OFFS = kHistBins + 64;
    static constexpr int KEYS = OFFS + kMaxSplit + 8;
    static constexpr size_t MERGE = (KEYS + 2 * (size_t)kMergeCap) * sizeof(uint32_t);
    static constexpr size_t BYTES = COLLECT > MERGE ? COLLECT : MERGE;
};

template <int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS, 1)
topk_split_kernel(TopkRowsArgs a) {
    using SM = StreamSmem<THREADS>;
    using SS = SplitSmem<THREADS>;
    constexpr int W = SM::W;
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ int s_last;
    uint32_t* hist = smem;
    uint32_t* scratch = hist + kHistBins;
    uint32_t* rcnt = scratch + 64;
    uint32_t* rkey = rcnt + 3 * W;
    uint32_t* ridx = rkey + SM::RUN_WORDS;

    const int c = blockIdx.x, r = blockIdx.y, g = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    long long col0;
    long long n = output_row(a, r, &col0);
    if (n <= a.topk) {
        // the same decision in every block of the row: the first writes it
        if (c != 0) return;
        if (n < 0) {
            if (tid == 0) raise_status(a.d_status, IDX_DEV_RANGE);
            n = 0;
        }
        int* out = a.out + (long long)r * a.topk;
        for (int i = tid; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
        return;
    }
    const uint32_t k = (uint32_t)a.topk;
    const RowView v = make_view(a.scores + (long long)r * a.row_stride + col0, n);
    // the slice as a view whose element indices stay row-relative
    const long long per = (v.nvec + g - 1) / g;
    const long long c0 = (long long)c * per;
    const long long c1 = c0 + per < v.nvec ? c0 + per : v.nvec;
    RowView sv;
    sv.base = v.base + c0;
    sv.off = v.off - (int)(4 * c0);
    sv.n = v.n;
    sv.nvec = c1 > c0 ? c1 - c0 : 0;

    // ---- collection: the loads of the first two steps are in flight while L
    // is estimated from the first two slots of every lane; after that the
    // loads of step i + 2 go out before step i is filtered
    int s0, s1;
    warp_slice<THREADS>(sv, w, &s0, &s1);
    constexpr int STEP = 32 * UNROLL, SAMPLE = 2;
    static_assert(UNROLL >= SAMPLE, "the sample comes from the first step");
    float4 f[UNROLL], nf[UNROLL];
    load_step<UNROLL>(sv, s0, s1, lane, f);
    load_step<UNROLL>(sv, s0 + STEP, s1, lane, nf);
    uint32_t L;
    {
        const int nn = (int)sv.n, off = sv.off;
        zero_shared<THREADS>(hist, kHistBins);
        if (tid == 0) scratch[44] = 0u;
        __syncthreads();
        uint32_t ns = 0;
#pragma unroll
        for (int u = 0; u < SAMPLE; ++u) {
            const int sl = s0 + 32 * u + lane;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int p = 4 * sl + q - off;
                if (sl < s1 && p >= 0 && p < nn) {
                    atomicAdd(&hist[fkey(e[q]) >> 20], 1u);
                    ++ns;
                }
            }
        }
        ns = __reduce_add_sync(0xffffffffu, ns);
        if (lane == 0 && ns) atomicAdd(&scratch[44], ns);
        __syncthreads();
        const uint32_t P = scratch[44];
        // m = this slice's sample keys expected above the row's k-th largest
        // (k / g of those in P of its n / g values); the slice's bound lies
        // above the row's threshold (the row then takes the exact path) only
        // when tg of them do, so tg = max(2 m, min(m + 4 sqrt(m) + 1, c)), c
        // the rank at which the row's expected kept count (tg n / P over the
        // slices) fills 70 % of the merge buffer (4 spreads: the bound is the
        // 12-bit floor of the tg-th sample key, well below it)
        const float m = (float)k * (float)P / (float)n;
        const float t = fmaxf(ceilf(2.0f * m),
                              fminf(m + 4.0f * sqrtf(m) + 1.0f,
                                    0.7f * (float)kMergeCap * (float)P / (float)n));
        const uint32_t tg = t < 1.0f ? 1u : t >= (float)P ? P : (uint32_t)ceilf(t);
        const uint32_t d = pick_digit<THREADS>(hist, kHistBins, tg, scratch).digit;
        L = P ? d << 20 : 0u;  // an empty slice takes nothing and bounds nothing
    }
    {
        const int nvec = (int)sv.nvec, nn = (int)sv.n, off = sv.off;
        const float Lf = key_floor_float(L);
        uint32_t* mk = rkey + w * kRunCap;
        uint32_t* mi = ridx + w * kRunCap;
        uint32_t cnt = 0;
        for (int base = s0; base < s1; base += STEP) {
            const int nb = base + STEP;
            const bool interior = base >= 1 && nb <= s1 && nb < nvec;
            filter_block<UNROLL, false>(sv, f, base, interior, s1, nn, off, L, Lf, lane, cnt, mk,
                                        mi, nullptr);
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) f[u] = nf[u];
            if (nb + STEP < s1) load_step<UNROLL>(sv, nb + STEP, s1, lane, nf);
        }
        if (lane == 0) rcnt[w] = cnt;
    }
    __syncthreads();
    // hand the runs over in warp (= index) order
    const long long slot = (long long)r * g + c;
    {
        uint32_t* gk = a.split_keys + slot * kSplitCap;
        uint32_t* gi = a.split_idx + slot * kSplitCap;
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
        if (tid == 0) {
            a.split_cnt[slot] = over ? -1 : (int)total;
            a.split_lb[slot] = L;
        }
    }
    // publish, then draw a ticket: the row's last block goes on
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        // draw a ticket: a word of another epoch is first restarted at this
        // call's first ticket by a compare-and-swap (one block wins, the others
        // see the new epoch); a word of this epoch takes an add
        unsigned long long* tk = a.split_ticket + r;
        const unsigned long long ep = (unsigned long long)a.epoch << 32;
        unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(tk);
        int last = 0;
        for (int it = 0; it < 64; ++it) {
            if ((cur & 0xffffffff00000000ull) == ep) {
                const unsigned long long old = atomicAdd(tk, 1ull);
                last = (old & 0xffffffffull) + 1ull == (unsigned long long)g;
                break;
            }
            const unsigned long long seen = atomicCAS(tk, cur, ep | 1ull);
            if (seen == cur) {
                last = g == 1;
                break;
            }
            cur = seen;
            if (it == 63) raise_status(a.d_status, IDX_DEV_STATE);
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- selection by the row's last block (reads bypass L1: other SMs wrote)
    // [g + 1] slice offsets; [kMaxSplit + 1] the largest bound, +2 total, +3 bad,
    // +4 the least bound of a slice with candidates
    uint32_t* soff = smem + SS::OFFS;
    uint32_t* keys = smem + SS::KEYS;
    uint32_t* idxs = keys + kMergeCap;
    int* out = a.out + (long long)r * a.topk;
    if (w == 0) {
        const int j0 = lane, j1 = lane + 32;
        const int n0 = j0 < g ? __ldcg(a.split_cnt + (long long)r * g + j0) : 0;
        const int n1 = j1 < g ? __ldcg(a.split_cnt + (long long)r * g + j1) : 0;
        const uint32_t l0 = j0 < g ? __ldcg(a.split_lb + (long long)r * g + j0) : 0u;
        const uint32_t l1 = j1 < g ? __ldcg(a.split_lb + (long long)r * g + j1) : 0u;
        const uint32_t lmax = __reduce_max_sync(0xffffffffu, l0 > l1 ? l0 : l1);
        const uint32_t m0 = n0 > 0 ? l0 : 0xffffffffu, m1 = n1 > 0 ? l1 : 0xffffffffu;
        const uint32_t lmin = __reduce_min_sync(0xffffffffu, m0 < m1 ? m0 : m1);
        const bool bad = __any_sync(0xffffffffu, n0 < 0 || n1 < 0);
        uint32_t i0 = n0 > 0 ? (uint32_t)n0 : 0u, i1 = n1 > 0 ? (uint32_t)n1 : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u0 = __shfl_up_sync(0xffffffffu, i0, o);
            const uint32_t u1 = __shfl_up_sync(0xffffffffu, i1, o);
            if (lane >= o) {
                i0 += u0;
                i1 += u1;
            }
        }
        const uint32_t t0 = __shfl_sync(0xffffffffu, i0, 31);
        const uint32_t total = t0 + __shfl_sync(0xffffffffu, i1, 31);
        if (lane == 0) soff[0] = 0u;
        if (j0 < g) soff[j0 + 1] = i0;
        if (j1 < g) soff[j1 + 1] = t0 + i1;
        if (lane == 0) {
            soff[kMaxSplit + 1] = lmax;
            soff[kMaxSplit + 2] = total;
            soff[kMaxSplit + 3] = bad || total < k || total > (uint32_t)kMergeCap;
            soff[kMaxSplit + 4] = lmin;
            if (a.d_stats) atomicAdd(&a.d_stats->split_rows, 1);
        }
    }
    __syncthreads();
    const uint32_t total = soff[kMaxSplit + 2];
    const uint32_t lmax = soff[kMaxSplit + 1];
    auto exact_path = [&]() {
        int rescans = 0;
        const Threshold th = find_threshold<THREADS, 4>(v, k, hist, keys, idxs, scratch, &rescans);
        if (tid == 0 && a.d_stats) atomicAdd(&a.d_stats->tie_rescan_rows, 1);
        ordered_output<THREADS>(v, th, k, out, scratch);
    };
    if (soff[kMaxSplit + 3]) {
        // a slice overflowed or too few values reached their bounds
        exact_path();
        return;
    }
    // one warp per slice: 16-byte loads (a slot's arrays start 16-byte
    // aligned; words past the count are loaded but not kept), four of each
    // array per lane in flight
    for (int cs = w; cs < g; cs += W) {
        const uint32_t o = soff[cs], cnt = soff[cs + 1] - o;
        const long long at = ((long long)r * g + cs) * kSplitCap;
        const uint4* sk = reinterpret_cast<const uint4*>(a.split_keys + at);
        const uint4* si = reinterpret_cast<const uint4*>(a.split_idx + at);
        for (uint32_t b = 0; b < cnt; b += 4 * 128) {
            uint4 kk[4], ii[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t e = b + j * 128 + 4 * lane;
                if (e < cnt) {
                    kk[j] = __ldcg(sk + e / 4);
                    ii[j] = __ldcg(si + e / 4);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t e = b + j * 128 + 4 * lane;
                const uint32_t kv[4] = {kk[j].x, kk[j].y, kk[j].z, kk[j].w};
                const uint32_t iv[4] = {ii[j].x, ii[j].y, ii[j].z, ii[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (e + q < cnt) {
                        keys[o + e + q] = kv[q];
                        idxs[o + e + q] = iv[q];
                    }
            }
        }
    }
    // every candidate's key is at least B, the key of the least slice bound
    // as a float: histogram relative to B, then the one-bin refinement over
    // the warps' chunks
    const uint32_t B = fkey(key_floor_float(soff[kMaxSplit + 4]));
    zero_shared<THREADS>(hist, kHistBins);
    __syncthreads();
    for (uint32_t e = tid; e < total; e += THREADS) {
        const uint32_t d = (keys[e] - B) >> 12;
        atomicAdd(&hist[d < (uint32_t)kHistBins ? d : (uint32_t)kHistBins - 1u], 1u);
    }
    __syncthreads();
    const uint32_t cper = (total + W * 32 - 1) / (W * 32) * 32;
    const uint32_t m0 = min(total, w * cper), m1 = min(total, m0 + cper);  // this warp's chunk
    Threshold th;
    bool counted = false;
    if (!refine_rel<THREADS>(keys, m0, m1, k, B, hist, scratch, scratch, &th, &counted))
        th = refine_in_smem<THREADS>(keys, total, 0, 0u, k, hist, scratch);
    if (th.key < lmax) {
        // a slice's bound lies above the k-th candidate: it may have left
        // out values of the top k
        exact_path();
        return;
    }
    ordered_output_range<THREADS>(keys, idxs, m0, m1, scratch, th, k, out, counted);
}

// ---------------------------------------------------------------- slab
//
// Page 1, "Sampled Threshold": the small exact top-k over the ~2.25 x topk
// candidates of a row.  The scoring pass leaves each row's candidates in runs
// of (score, row-relative index) pairs (eight runs per key split; the
// rescan's re-emission uses the first eight).  One CTA of 256 threads per row.
// A launch of many rows reads the runs from global memory in every pass (warp
// w the runs w, w + 8, ...; a row's ~26 KB stay in L1/L2 between its passes)
// and keeps no copy, so that six rows share an SM.  A launch of fewer rows
// than three per SM over more than 64 runs (decode-like: a few rows whose
// keys were split over many CTAs, so many short runs) first copies each row's
// runs into shared memory, one bulk copy each (run lengths rounded up to an
// even count, the extra slot marked empty), and the passes read that copy.
// Then:
//   1. a histogram of 1024 bins of the candidates' order keys above a base B.
//      A row with a sampled threshold has every candidate at or above it, so
//      B is that threshold and a bin is 2^14 keys wide (the bins span two
//      octaves of the score above B; larger keys share the top bin); another
//      row takes B = its smallest key and bins just wide enough for its
//      largest (one more pass);
//   2. the bin b that holds the topk-th largest key, scanned from the top:
//      every candidate of a higher bin is selected, and when b holds at most
//      kCandGather candidates they are gathered and the `need` of them ranked
//      first by (key descending, index ascending) are selected; a fuller bin
//      is resolved by radix selection over its keys (8-bit digits), then over
//      the indices of the keys tied at the threshold;
//   3. the selected indices in ascending order: from a bitmap over the row's
//      indices (rows of up to 32 x kCandBitmapWords keys), else from a list
//      bucketed by index (1024 buckets of a power-of-two width), the buckets
//      placed by a scan and each index placed by its rank within its bucket.
// Rows whose candidate count fell below topk, or that held more than a whole
// row's slab (eight runs) or lost candidates to a full run, are flagged for
// the exact rescan instead.

constexpr int kCandThreads = 256;
constexpr int kCandWarps = kCandThreads / 32;
constexpr int kCandBins = 1024;
constexpr int kCandGather = 256;        // candidates of the threshold bin ranked directly
constexpr int kCandBitmapWords = 4096;  // the bitmap output covers rows of up to 131072 keys
constexpr int kCandRelShift = 14;       // bin width above a sampled threshold: 2^14 keys
constexpr int kCandU = 4;               // pairs per lane in flight (streamed rows)
constexpr uint32_t kEmptyKey = 0u;      // a padding slot of a copied run (no finite score)
constexpr int kCandStreamRuns = 8 * kRuns;  // launches of few rows and more runs copy them

// Block-wide maximum and minimum of one value per thread (scratch >= 16 words).
IDX_DEVI void block_max_min(uint32_t& mx, uint32_t& mn, uint32_t* scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
        scratch[w] = mx;
        scratch[8 + w] = mn;
    }
    __syncthreads();
    mx = scratch[0];
    mn = scratch[8];
#pragma unroll
    for (int j = 1; j < kCandWarps; ++j) {
        mx = max(mx, scratch[j]);
        mn = min(mn, scratch[8 + j]);
    }
    __syncthreads();
}

// A row's candidates.  Streamed: run q holds cnt[q] pairs from srow + q * cap_q
// in global memory.  Staged: `pairs` holds n pairs (padding slots included)
// in shared memory.
struct CandRow {
    const int2* srow;
    const uint32_t* cnt;
    int nruns, cap_q;
    const int2* pairs;
    uint32_t n;
};

// f(key, index) for every candidate of a row.  Streamed: warp w reads runs w,
// w + 8, ..., kCandU pairs per lane in flight.
template <bool STAGED, class F>
IDX_DEVI void cand_each(const CandRow& R, F&& f) {
    if (STAGED) {
        for (uint32_t e = threadIdx.x; e < R.n; e += kCandThreads) {
            const int2 v = R.pairs[e];
            const uint32_t key = fkey(__int_as_float(v.x));
            if (key != kEmptyKey) f(key, (uint32_t)v.y);
        }
        return;
    }
    const int lane = threadIdx.x & 31;
    for (int q = threadIdx.x >> 5; q < R.nruns; q += kCandWarps) {
        const int c = (int)R.cnt[q];
        const int2* src = R.srow + (long long)q * R.cap_q;
        for (int j0 = 0; j0 < c; j0 += 32 * kCandU) {
            int2 v[kCandU];
#pragma unroll
            for (int u = 0; u < kCandU; ++u) {
                const int j = j0 + 32 * u + lane;
                v[u] = j < c ? __ldg(src + j) : make_int2(0, 0);
            }
#pragma unroll
            for (int u = 0; u < kCandU; ++u)
                if (j0 + 32 * u + lane < c) f(fkey(__int_as_float(v[u].x)), (uint32_t)v[u].y);
        }
    }
}

// The bin of a histogram of nb <= 1024 bins that holds the need-th largest
// element (count(> b) < need <= count(>= b), 1 <= need <= the total); every
// thread gets it.  scratch: [0, 8) the scan, [40, 43) the result.
IDX_DEVI DigitPick cand_pick(const uint32_t* hist, int nb, uint32_t need, uint32_t* scratch) {
    constexpr int BPT = kCandBins / kCandThreads;
    const int t = threadIdx.x;
    uint32_t c[BPT], loc = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        const int b = nb - 1 - (BPT * t + j);
        c[j] = b >= 0 ? hist[b] : 0u;
        loc += c[j];
    }
    const uint32_t incl = block_incl_scan<kCandThreads>(loc, scratch, nullptr);
    uint32_t cum = incl - loc;
    if (cum < need && need <= incl) {
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            if (cum + c[j] >= need) {
                scratch[40] = (uint32_t)(nb - 1 - (BPT * t + j));
                scratch[41] = cum;
                scratch[42] = c[j];
                break;
            }
            cum += c[j];
        }
    }
    __syncthreads();
    const DigitPick p{scratch[40], scratch[41], scratch[42]};
    __syncthreads();
    return p;
}

// The need-th largest v = val(key, index) among the candidates with
// in(key, index), by 8-bit digits from the top (four passes);
// *need_at = how many of the elements equal to it are taken.
template <bool STAGED, class In, class Val>
IDX_DEVI uint32_t cand_radix_select(const CandRow& R, uint32_t need, In in, Val val,
                                    uint32_t* hist, uint32_t* scratch, uint32_t* need_at) {
    uint32_t pre = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kCandThreads) hist[i] = 0u;
        __syncthreads();
        const uint32_t above_mask = shift == 24 ? 0u : ~0u << (shift + 8);
        cand_each<STAGED>(R, [&](uint32_t key, uint32_t ix) {
            if (!in(key, ix)) return;
            const uint32_t v = val(key, ix);
            if ((v & above_mask) == pre) atomicAdd(&hist[(v >> shift) & 255u], 1u);
        });
        __syncthreads();
        const DigitPick p = cand_pick(hist, 256, need, scratch);
        need -= p.above;
        pre |= p.digit << shift;
    }
    *need_at = need;
    return pre;
}

// Shared memory of cand_topk_kernel, in 32-bit words.
struct CandSmem {
    int nruns, topk, cap_q;
    bool staged;
    __host__ __device__ CandSmem(int nruns_, int topk_, int cap_q_, bool staged_)
        : nruns(nruns_), topk(topk_), cap_q(cap_q_), staged(staged_) {}
    // the bitmap, or the selected indices and their ordered copy (2 x topk)
    __host__ __device__ int region_words() const {
        return 2 * topk > kCandBitmapWords ? 2 * topk : kCandBitmapWords;
    }
    // staged pairs: a whole row's slab (eight runs) plus a padding slot per run
    __host__ __device__ int cap() const { return staged ? kRuns * cap_q + nruns : 0; }
    __host__ __device__ int hist() const { return 0; }                         // [1024]
    __host__ __device__ int region() const { return kCandBins; }
    __host__ __device__ int gather() const { return region() + region_words(); }  // [256] x 2
    __host__ __device__ int scratch() const { return gather() + 2 * kCandGather; }  // [64]
    __host__ __device__ int bar() const { return scratch() + 64; }             // 2 (8-byte aligned)
    __host__ __device__ int runs() const { return bar() + 2; }                 // [nruns]
    __host__ __device__ int offs() const { return runs() + nruns; }            // [nruns + 1] staged
    __host__ __device__ int pairs() const {
        return (offs() + (staged ? nruns + 1 : 0) + 3) / 4 * 4;  // 16-byte aligned
    }
    __host__ __device__ int words() const { return pairs() + 2 * cap(); }
};

template <bool STAGED>
__global__ void __launch_bounds__(kCandThreads, STAGED ? 1 : 6)  // streamed: six rows per SM
cand_topk_kernel(CandArgs a) {
    constexpr int THREADS = kCandThreads;
    extern __shared__ __align__(16) uint32_t smem[];
    pdl_wait();
    const CandSmem L(a.nruns, a.topk, a.cap_q, STAGED);
    uint32_t* hist = smem + L.hist();
    uint32_t* reg = smem + L.region();
    uint2* gat = reinterpret_cast<uint2*>(smem + L.gather());  // (key, index)
    uint32_t* scratch = smem + L.scratch();  // [0,16) scans, [40,43) picks, [48,53) row state
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar());
    uint32_t* cnt = smem + L.runs();         // run lengths (capped)
    uint32_t* offs = smem + L.offs();        // staged: where each run's copy starts
    int2* pairs = reinterpret_cast<int2*>(smem + L.pairs());
    const int tid = threadIdx.x;
    const long long CR = (long long)a.nruns * a.cap_q;  // slab row (all key splits)
    const uint32_t k = (uint32_t)a.topk;

    if (a.fallback && *(volatile int*)(a.fb_cnt + 6) == 0) return;  // no row was re-emitted
    if (STAGED && tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    uint32_t phase = 0;
    // runs of this thread: a contiguous range, so that offsets follow run order
    const int per = (a.nruns + THREADS - 1) / THREADS;
    const int q0 = min(a.nruns, tid * per), q1 = min(a.nruns, q0 + per);
    for (int r = blockIdx.x; r < a.rows; r += gridDim.x) {
        __syncthreads();  // the previous row's shared state is no longer read
        RowPlan* plan = a.plan + r;
        const long long n = (long long)a.ke[r] - (long long)a.ks[r];
        int* out = a.out + (long long)r * a.topk;
        if (tid == 0) {
            scratch[48] = (uint32_t)plan->state;
            scratch[49] = 0u;  // candidates (uncapped)
            scratch[50] = plan->thr;
            scratch[51] = 0u;  // gathered
            scratch[52] = 0u;  // listed
        }
        __syncthreads();
        const int state = (int)scratch[48];
        if (a.fallback) {
            if (state != ST_EMIT) continue;
        } else if (n <= a.topk) {
            for (int i = tid; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
            if (tid == 0) plan->state = ST_DONE;
            continue;
        }

        // ---- run lengths
        const int* rc = a.run_cnt + (long long)r * a.nruns;
        const int2* srow = a.slab + (long long)r * CR;
        uint32_t lcnt = 0, lpad = 0;
        bool ltr = false;
        for (int q = STAGED ? q0 : tid; q < (STAGED ? q1 : a.nruns); q += STAGED ? 1 : THREADS) {
            const uint32_t c = (uint32_t)rc[q];
            const uint32_t cl = c < (uint32_t)a.cap_q ? c : (uint32_t)a.cap_q;
            ltr |= c > (uint32_t)a.cap_q;
            lcnt += c;
            lpad += (cl + 1u) & ~1u;
            cnt[q] = cl;
        }
        if (lcnt) atomicAdd(&scratch[49], lcnt);
        // a run that overflowed lost candidates, and a row of key splits may
        // hold more than the slab of a whole row (eight runs): either way the
        // exact rescan takes the row
        const bool lost = __syncthreads_or(ltr);
        const uint32_t total = scratch[49];
        const bool trunc = lost || total > (uint32_t)(kRuns * a.cap_q);
        if (tid == 0 && a.d_stats && !a.fallback) atomicMax(&a.d_stats->max_count, (int)total);
        if (trunc || total < k) {
            if (!a.fallback && !a.fb_hist) {
                // no rescan storage: the row was longer than the max_len the
                // workspace was sized for
                for (int i = tid; i < a.topk; i += THREADS) out[i] = -1;
                if (tid == 0) {
                    raise_status(a.d_status, IDX_DEV_RANGE);
                    plan->state = ST_DONE;
                }
            } else if (!a.fallback) {
                // the sampled threshold missed: exact full-row rescan
                for (int i = tid; i < kHistBins; i += THREADS)
                    a.fb_hist[(long long)r * kHistBins + i] = 0u;
                if (tid == 0) {
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
            } else if (tid == 0) {
                raise_status(a.d_status, IDX_DEV_STATE);
                plan->state = ST_DONE;
            }
            continue;
        }

        CandRow R{srow, cnt, a.nruns, a.cap_q, pairs, 0u};
        if (STAGED) {
            // ---- the runs into shared memory, one bulk copy each (even
            // lengths: 16-byte multiples; the runs hold them, cap_q is even)
            uint32_t ptot;
            uint32_t off = block_incl_scan<THREADS>(lpad, scratch, &ptot) - lpad;
            for (int q = q0; q < q1; ++q) {
                offs[q] = off;
                off += (cnt[q] + 1u) & ~1u;
            }
            if (tid == 0) mbar_arrive_expect_tx(bar, ptot * (uint32_t)sizeof(int2));
            __syncthreads();
            for (int q = q0; q < q1; ++q) {
                const uint32_t len = (cnt[q] + 1u) & ~1u;
                if (len) bulk_g2s(pairs + offs[q], srow + (long long)q * a.cap_q, len * 8u, bar);
            }
            if (!mbar_wait(bar, phase, nullptr, 1ll << 30)) {
                // copies that never completed: report and leave (bounded wait for them)
                if (tid == 0) raise_status(a.d_status, IDX_DEV_TIMEOUT);
                mbar_wait(bar, phase, nullptr, 1ll << 30);
                return;
            }
            phase ^= 1u;
            // the slot that rounded a run up to an even length holds no candidate
            for (int q = q0; q < q1; ++q)
                if (cnt[q] & 1u) pairs[offs[q] + cnt[q]].x = -1;  // order key kEmptyKey
            __syncthreads();
            R.n = ptot;
        }

        // ---- the bins: base B, width 2^sh
        const uint32_t thr = scratch[50];
        uint32_t B, sh;
        if (!a.fallback && thr != 0u) {
            B = thr;
            sh = (uint32_t)kCandRelShift;
        } else {
            uint32_t mx = 0u, mn = 0xffffffffu;
            cand_each<STAGED>(R, [&](uint32_t key, uint32_t) {
                mx = max(mx, key);
                mn = min(mn, key);
            });
            block_max_min(mx, mn, scratch);
            B = mn;
            const uint32_t span = mx - mn;
            sh = span < (uint32_t)kCandBins ? 0u : (uint32_t)(32 - __clz(span)) - 10u;
        }
        auto bin = [&](uint32_t key) -> uint32_t {
            if (key < B) return 0u;
            const uint32_t d = (key - B) >> sh;
            return d < (uint32_t)kCandBins ? d : (uint32_t)kCandBins - 1u;
        };
        const bool use_bm = n <= 32ll * L.region_words();
        const uint32_t bm_words = use_bm ? (uint32_t)((n + 31) / 32) : 0u;
        for (int i = tid; i < kCandBins; i += THREADS) hist[i] = 0u;
        for (uint32_t i = tid; i < bm_words; i += THREADS) reg[i] = 0u;
        __syncthreads();
        cand_each<STAGED>(R, [&](uint32_t key, uint32_t) { atomicAdd(&hist[bin(key)], 1u); });
        __syncthreads();
        const DigitPick pk = cand_pick(hist, kCandBins, k, scratch);
        const uint32_t bs = pk.digit, need = k - pk.above;
        const bool direct = pk.count <= (uint32_t)kCandGather;
        // a selected index: its bit, or an entry of the (unordered) list
        auto mark = [&](uint32_t ix) {
            if (use_bm) {
                atomicOr(&reg[ix >> 5], 1u << (ix & 31u));
            } else {
                const uint32_t p = atomicAdd(&scratch[52], 1u);
                if (p < k) reg[p] = ix;
            }
        };

        // ---- the higher bins, and the threshold bin's candidates
        cand_each<STAGED>(R, [&](uint32_t key, uint32_t ix) {
            const uint32_t d = bin(key);
            if (d > bs)
                mark(ix);
            else if (d == bs && direct)
                gat[atomicAdd(&scratch[51], 1u)] = make_uint2(key, ix);
        });
        __syncthreads();
        if (direct) {
            const uint32_t ng = scratch[51];
            for (uint32_t i = tid; i < ng; i += THREADS) {
                const uint2 gi = gat[i];
                uint32_t rank = 0;
                for (uint32_t j = 0; j < ng; ++j) {
                    const uint2 gj = gat[j];
                    rank += gj.x > gi.x || (gj.x == gi.x && gj.y < gi.y);
                }
                if (rank < need) mark(gi.y);
            }
        } else {
            // T = the need-th largest key of the bin, then the lowest indices
            // among the keys equal to T
            uint32_t need_t;
            const uint32_t T = cand_radix_select<STAGED>(
                R, need, [&](uint32_t key, uint32_t) { return bin(key) == bs; },
                [](uint32_t key, uint32_t) { return key; }, hist, scratch, &need_t);
            uint32_t nt = 0;
            cand_each<STAGED>(R, [&](uint32_t key, uint32_t) { nt += key == T; });
            uint32_t ntie;
            block_incl_scan<THREADS>(nt, scratch, &ntie);
            uint32_t cut = 0xffffffffu;
            if (ntie > need_t) {
                uint32_t unused;
                cut = ~cand_radix_select<STAGED>(
                    R, need_t, [&](uint32_t key, uint32_t) { return key == T; },
                    [](uint32_t, uint32_t ix) { return ~ix; }, hist, scratch, &unused);
            }
            cand_each<STAGED>(R, [&](uint32_t key, uint32_t ix) {
                if (bin(key) == bs && (key > T || (key == T && ix <= cut))) mark(ix);
            });
        }
        __syncthreads();
        if (use_bm) {
            // ---- ascending output from the bitmap: each thread owns a
            // contiguous range of words and writes the indices of their set
            // bits from its offset in a block scan of the bit counts
            const uint32_t per = (bm_words + THREADS - 1) / THREADS;
            const uint32_t w0 = min(bm_words, tid * per), w1 = min(bm_words, w0 + per);
            uint32_t c = 0;
            for (uint32_t i = w0; i < w1; ++i) c += __popc(reg[i]);
            uint32_t nsel;
            uint32_t pos = block_incl_scan<THREADS>(c, scratch, &nsel) - c;
            if (nsel != k) {
                // cannot happen for finite scores: report it rather than write past
                // the row's output
                for (int i = tid; i < a.topk; i += THREADS) out[i] = -1;
                if (tid == 0) {
                    raise_status(a.d_status, IDX_DEV_STATE);
                    plan->state = ST_DONE;
                }
                continue;
            }
            for (uint32_t i = w0; i < w1; ++i) {
                uint32_t m = reg[i];
                while (m) {
                    const int b = __ffs(m) - 1;
                    m &= m - 1u;
                    out[pos++] = (int)(32u * i + (uint32_t)b);
                }
            }
            if (tid == 0) plan->state = ST_DONE;
            continue;
        }
        // ---- ascending output, longer rows: the listed indices bucketed by
        // index (1024 buckets of width 2^bsh >= n / 1024), the buckets placed
        // by a scan, and each index placed by its rank among its bucket's
        if (scratch[52] != k) {
            for (int i = tid; i < a.topk; i += THREADS) out[i] = -1;
            if (tid == 0) {
                raise_status(a.d_status, IDX_DEV_STATE);
                plan->state = ST_DONE;
            }
            continue;
        }
        uint32_t* ord = reg + k;
        int bsh = 0;
        while (((long long)kCandBins << bsh) < n) ++bsh;
        for (int i = tid; i < kCandBins; i += THREADS) hist[i] = 0u;
        __syncthreads();
        for (uint32_t p = tid; p < k; p += THREADS) atomicAdd(&hist[reg[p] >> bsh], 1u);
        __syncthreads();
        {
            // bucket starts: thread t owns buckets BPT t .. BPT t + BPT - 1
            constexpr int BPT = kCandBins / THREADS;
            uint32_t cb[BPT], loc = 0;
#pragma unroll
            for (int j = 0; j < BPT; ++j) {
                cb[j] = hist[BPT * tid + j];
                loc += cb[j];
            }
            uint32_t st = block_incl_scan<THREADS>(loc, scratch, nullptr) - loc;
#pragma unroll
            for (int j = 0; j < BPT; ++j) {
                hist[BPT * tid + j] = st;
                st += cb[j];
            }
        }
        __syncthreads();
        for (uint32_t p = tid; p < k; p += THREADS) {
            const uint32_t x = reg[p];
            ord[atomicAdd(&hist[x >> bsh], 1u)] = x;
        }
        __syncthreads();
        // hist[b] is now the end of bucket b (the start of b + 1)
        for (uint32_t p = tid; p < k; p += THREADS) {
            const uint32_t x = ord[p];
            const uint32_t b = x >> bsh;
            const uint32_t lo = b ? hist[b - 1] : 0u, hi = hist[b];
            uint32_t rank = 0;
            for (uint32_t j = lo; j < hi; ++j) rank += ord[j] < x;
            out[lo + rank] = (int)x;
        }
        if (tid == 0) plan->state = ST_DONE;
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
        constexpr int WARPS = 4;
        TopkRowsArgs b = a;
        b.split = a.row_len > kThrCtaMin ? 2 : 0;
        // (one more CTA for the block order)
        cudaError_t e = launch_k(sample_threshold_kernel<WARPS>,
                                 dim3((unsigned)((a.rows + WARPS - 1) / WARPS + (a.order ? 1 : 0))),
                                 dim3(WARPS * 32), 0, s, a.pdl != 0, b);
        if (e == cudaSuccess && b.split) {
            e = launch_k(sample_threshold_cta_kernel, dim3((unsigned)a.rows), dim3(kThrCtaThreads),
                         0, s, a.pdl != 0, b);
            count_launches(1);
        }
        return e;
    }
    if (a.split > 1) {
        if (a.split > kMaxSplit) return cudaErrorInvalidValue;
        auto kern = topk_split_kernel<T, U>;
        constexpr size_t SPLIT_SMEM = SplitSmem<T>::BYTES;
        static cudaError_t attr = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPLIT_SMEM);
        if (attr != cudaSuccess) return attr;
        if (a.epoch == 0u) return cudaErrorInvalidValue;
        kern<<<dim3((unsigned)a.split, (unsigned)a.rows), T, SPLIT_SMEM, s>>>(a);
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
    return slots * (size_t)kSplitCap * 2 * sizeof(uint32_t) + 2 * slots * sizeof(int) +
           (size_t)rows * sizeof(unsigned long long) + 256;
}

size_t cand_smem_bytes(int cap_q, int nruns, int topk, bool staged) {
    return (size_t)CandSmem(nruns, topk, cap_q, staged).words() * sizeof(uint32_t);
}

cudaError_t launch_cand_topk(const CandArgs& a, cudaStream_t s) {
    bool staged = a.nruns > kCandStreamRuns && a.rows < 3 * a.sm_count &&
                  cand_smem_bytes(a.cap_q, a.nruns, a.topk, true) <= 227u * 1024u;
    const CandSmem L(a.nruns, a.topk, a.cap_q, staged);
    // the gathered (key, index) pairs and the mbarrier are 8-byte aligned; the
    // staged runs' bulk copies want 16-byte aligned runs
    if (L.gather() % 2 != 0 || L.bar() % 2 != 0 || a.cap_q % 2 != 0)
        return cudaErrorInvalidValue;
    const size_t sm = cand_smem_bytes(a.cap_q, a.nruns, a.topk, staged);
    auto kern = staged ? cand_topk_kernel<true> : cand_topk_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (a.rows == 0) return cudaSuccess;
    // the rescan's pass usually has no row to select: a short grid that strides
    // over the rows exits at once
    const int grid = a.fallback ? (a.rows < a.grid_limit ? a.rows : a.grid_limit) : a.rows;
    return launch_k(kern, dim3((unsigned)grid), dim3(kCandThreads), sm, s, a.pdl != 0, a);
}

}  // namespace idx

// Block-wide building blocks of the exact radix selection.
//
// Keys are the order-preserving uint32 images of fp32 scores (fkey).  The
// selection walks the key from the top in three digits, 12 + 12 + 8 bits
// (page "[sglang] ROCm DSA Indexer Top-K 최적화": fp32 keys, a 12-bit coarse
// histogram, radix tie refinement).  After the third digit the threshold key T
// is exact; ties at T are then taken in ascending index order by an ordered
// compaction pass, which is what makes the result bit-exact.
#pragma once

#include "common.cuh"
#include "plan.cuh"

namespace idx {

// digit geometry: level 0 = key bits 31..20, level 1 = 19..8, level 2 = 7..0
IDX_DEVI int digit_bits(int level) { return level < 2 ? 12 : 8; }
IDX_DEVI int digit_shift(int level) { return level == 0 ? 20 : (level == 1 ? 8 : 0); }
IDX_DEVI uint32_t digit_of(uint32_t key, int level) {
    return (key >> digit_shift(level)) & ((1u << digit_bits(level)) - 1u);
}
// Bits of the key above this level's digit, and whether `key` carries `prefix`.
IDX_DEVI bool has_prefix(uint32_t key, int level, uint32_t prefix) {
    if (level == 0) return true;
    const int sh = digit_shift(level) + digit_bits(level);
    return (key >> sh) == prefix;
}

// Index digits of the rescan levels 3..5: bits 30..20, 19..10, 9..0.
IDX_DEVI int idx_digit_bits(int level) { return level == 3 ? 11 : 10; }
IDX_DEVI int idx_digit_shift(int level) { return level == 3 ? 20 : (level == 4 ? 10 : 0); }
IDX_DEVI uint32_t idx_digit_of(uint32_t idx, int level) {
    return (idx >> idx_digit_shift(level)) & ((1u << idx_digit_bits(level)) - 1u);
}
IDX_DEVI bool idx_has_prefix(uint32_t idx, int level, uint32_t prefix) {
    if (level == 3) return true;
    return (idx >> (idx_digit_shift(level) + idx_digit_bits(level))) == prefix;
}

constexpr int kHistBins = 4096;

// Inclusive block-wide sum scan of one uint32 per thread.  `warp_tot` is a
// shared array of >= 32 entries.  Every thread of the block must call it.
template <int THREADS>
IDX_DEVI uint32_t block_incl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
    static_assert(THREADS % 32 == 0 && THREADS <= 1024, "block size");
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[wid] = v;
    __syncthreads();
    if (wid == 0) {
        uint32_t t = lane < W ? warp_tot[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += u;
        }
        if (lane < W) warp_tot[lane] = t;  // inclusive totals per warp
    }
    __syncthreads();
    const uint32_t before = wid ? warp_tot[wid - 1] : 0u;
    if (total) *total = warp_tot[W - 1];
    const uint32_t r = v + before;
    __syncthreads();  // warp_tot may be reused right away
    return r;
}

struct DigitPick {
    uint32_t digit;  // chosen digit value
    uint32_t above;  // elements of the prefix set with a larger digit
    uint32_t count;  // elements with exactly this digit
};

// Given the histogram of one digit over the elements that carry the current
// prefix, find the digit d with count(> d) < need <= count(>= d), need >= 1.
// Bins are scanned from the top.  Every thread gets the result.
template <int THREADS>
IDX_DEVI DigitPick pick_digit(const uint32_t* hist, int nbins, uint32_t need,
                              uint32_t* scratch /* >= 32 + 3 words */) {
    constexpr int BPT = kHistBins / THREADS > 0 ? kHistBins / THREADS : 1;
    const int t = threadIdx.x;
    uint32_t local = 0;
    uint32_t c[BPT];
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        const int b = nbins - 1 - (t * BPT + j);
        c[j] = b >= 0 ? hist[b] : 0u;
        local += c[j];
    }
    uint32_t* res = scratch + 32;
    if (t == 0) { res[0] = 0u; res[1] = 0u; res[2] = 0u; }
    const uint32_t incl = block_incl_scan<THREADS>(local, scratch, nullptr);
    const uint32_t excl = incl - local;
    if (excl < need && need <= incl) {
        uint32_t cum = excl;
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            if (cum + c[j] >= need) {
                res[0] = static_cast<uint32_t>(nbins - 1 - (t * BPT + j));
                res[1] = cum;
                res[2] = c[j];
                break;
            }
            cum += c[j];
        }
    }
    __syncthreads();
    DigitPick p{res[0], res[1], res[2]};
    __syncthreads();
    return p;
}

// ------------------------------------------------------ rescan digit step
//
// One warp, one row: given the histogram of this level's digit (global
// memory, written by this CTA), pick the digit that holds the boundary of the
// top-k and advance the row's plan.  Key levels 0..2 count from the top (the
// largest keys), index levels 3..5 from the bottom (the lowest indices among
// the keys equal to T).  The histogram row is cleared for the next level.
// fb_cnt[l] counts the rows waiting for level l, fb_cnt[6] those ready to emit.
IDX_DEVI void rescan_pick_warp(RowPlan* plan, uint32_t* hist, int level, int topk, int cap,
                               int* fb_cnt) {
    const int lane = threadIdx.x & 31;
    const bool by_key = level <= 2;
    const int bits = by_key ? digit_bits(level) : idx_digit_bits(level);
    const int nb = 1 << bits;
    const int per = nb / 32;
    const uint32_t above = (uint32_t)plan->above;
    const uint32_t need = by_key ? (uint32_t)topk - above : (uint32_t)plan->quota - above;
    // lane l owns the l-th chunk of bins in scan order
    auto bin_at = [&](int k) { return by_key ? nb - 1 - k : k; };
    uint32_t local = 0;
    for (int k = lane * per; k < (lane + 1) * per; ++k) local += __ldcg(hist + bin_at(k));
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - local;
    const bool mine = excl < need && need <= incl;
    uint32_t digit = 0, before = 0, count = 0;
    if (mine) {
        uint32_t cum = excl;
        for (int k = lane * per; k < (lane + 1) * per; ++k) {
            const uint32_t c = __ldcg(hist + bin_at(k));
            if (cum + c >= need) {
                digit = (uint32_t)bin_at(k);
                before = cum;
                count = c;
                break;
            }
            cum += c;
        }
    }
    const uint32_t who = __ballot_sync(0xffffffffu, mine);
    const int src = who ? __ffs(who) - 1 : 0;
    digit = __shfl_sync(0xffffffffu, digit, src);
    before = __shfl_sync(0xffffffffu, before, src);
    count = __shfl_sync(0xffffffffu, count, src);
    for (int k = lane; k < nb; k += 32) hist[k] = 0u;  // ready for the next level
    if (lane != 0) return;
    if (!who) {  // inconsistent histogram: give up on the row
        plan->state = ST_DONE;
        return;
    }
    if (by_key) {
        const uint32_t above_new = above + before;
        const uint32_t prefix = (plan->prefix << bits) | digit;
        if (above_new + count <= (uint32_t)cap) {
            plan->thr = prefix << digit_shift(level);
            plan->idx_cut = kAllIdx;
            plan->state = ST_EMIT;
            atomicAdd(&fb_cnt[6], 1);
        } else if (level < 2) {
            plan->prefix = prefix;
            plan->above = (int32_t)above_new;
            plan->level = level + 1;
            atomicAdd(&fb_cnt[level + 1], 1);
        } else {
            // T exact; its ties overflow the slab: keep the lowest indices
            plan->thr = prefix;
            plan->above_thr = (int32_t)above_new;
            plan->quota = topk - (int32_t)above_new;
            plan->prefix = 0u;
            plan->above = 0;
            plan->level = 3;
            atomicAdd(&fb_cnt[3], 1);
        }
    } else {
        const uint32_t below_new = above + before;  // ties with a smaller index
        const uint32_t prefix = (plan->prefix << bits) | digit;
        const uint32_t keep = (uint32_t)plan->above_thr + below_new + count;
        const int sh = idx_digit_shift(level);
        if (keep <= (uint32_t)cap || level == 5) {
            plan->idx_cut = (int32_t)((prefix << sh) | ((1u << sh) - 1u));
            plan->state = ST_EMIT;
            atomicAdd(&fb_cnt[6], 1);
        } else {
            plan->prefix = prefix;
            plan->above = (int32_t)below_new;
            plan->level = level + 1;
            atomicAdd(&fb_cnt[level + 1], 1);
        }
    }
}

template <int THREADS>
IDX_DEVI void zero_shared(uint32_t* a, int n) {
    for (int i = threadIdx.x; i < n; i += THREADS) a[i] = 0u;
}

}  // namespace idx

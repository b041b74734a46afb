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

template <int THREADS>
IDX_DEVI void zero_shared(uint32_t* a, int n) {
    for (int i = threadIdx.x; i < n; i += THREADS) a[i] = 0u;
}

}  // namespace idx

// Per-row state shared by the kernels of the fused path and the layout of the
// caller's workspace.  Host and device code both include this file.
#pragma once

#include <cstddef>
#include <cstdint>

namespace idx {

// Row states of the fused path.
enum : int32_t {
    ST_MAIN = 0,      // candidates of the main scoring pass are being selected
    ST_HIST = 1,      // exact rescan: next pass histograms digit `level`
    ST_EMIT = 2,      // exact rescan: next pass re-emits with the refined rule
    ST_DONE = 3,      // out_idx row is final
};

constexpr int32_t kAllIdx = 0x7fffffff;

// Emit rule of a row: a key is a candidate when its order key is above thr,
// or equal to thr with a row-relative index <= idx_cut.
//
// Exact rescan levels: 0..2 walk the order key from the top (12, 12, 8 bits);
// once the threshold key T is exact and its ties still exceed the slab, 3..5
// walk the row-relative index of the ties from the bottom (11, 10, 10 bits),
// so that the lowest indices among the ties are the ones kept.
struct RowPlan {
    uint32_t thr;
    int32_t idx_cut;
    int32_t state;
    int32_t level;
    uint32_t prefix;     // key bits (levels 0..2) or index bits (3..5) above the digit
    int32_t above;       // keys above the prefix set (0..2) / ties below it (3..5)
    int32_t quota;       // levels 3..5: ties at T that belong to the result
    int32_t above_thr;   // levels 3..5: keys strictly above T
};
static_assert(sizeof(RowPlan) == 32, "RowPlan layout");

// Candidate runs per row: one per (TMEM lane quarter, epilogue team).
constexpr int kRuns = 8;

// Sample indices i of the strided threshold sample are keys phase + S*i
// (i < nsamp = floor(keys / S)).  Row r sees samples [a, b).
struct SampleSpan { long long a, b; };

__host__ __device__ inline SampleSpan sample_span(long long ks, long long ke, long long phase,
                                                  long long S, long long nsamp) {
    auto first_at_or_after = [&](long long key) -> long long {
        if (key <= phase) return 0;
        return (key - phase + S - 1) / S;
    };
    long long a = first_at_or_after(ks), b = first_at_or_after(ke);
    if (b > nsamp) b = nsamp;
    if (a > b) a = b;
    return {a, b};
}

// Chris Wellons' "lowbias32" integer hash; picks the sample phase of a block
// of rows (page 1, section 2: odd stride with a hashed phase).
__host__ __device__ inline uint32_t hash32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace idx

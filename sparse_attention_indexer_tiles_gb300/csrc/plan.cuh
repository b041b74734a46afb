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

struct RowPlan {
    uint32_t thr;     // emit rule: key >= thr (quota == 0) ...
    int32_t quota;    // ... or key > thr plus the first `quota` keys == thr in index order
    int32_t state;
    int32_t level;    // digit level of the next histogram pass (ST_HIST)
    uint32_t prefix;  // key bits above that digit (ST_HIST)
    int32_t above;    // keys known to lie strictly above the prefix set
    int32_t count;    // candidates of the last emit pass (may exceed cap)
    int32_t pad;
};
static_assert(sizeof(RowPlan) == 32, "RowPlan layout");

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

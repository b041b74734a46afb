// Page-table transform of top-k indices (page "[sglang] logits를 쓰지 않는
// top-k", section 3): a consumer of a paged KV cache wants physical slots, so
// each row-relative position p >= 0 becomes table[t, p / P] * P + p % P, with
// t the page-table row of the query row and P the page size; negative
// positions (the -1 padding) are kept.  The indices are rewritten in place.
//
// The grid is flat over all rows x topk entries (a row count above 65535 needs
// no second grid dimension): each 256-thread block owns a contiguous chunk of
// 1024 units (a unit is four entries, one 16-byte load and store, when
// topk % 4 == 0 and the array is 16-byte aligned; else one entry).  A thread
// issues the loads of its four units before it uses any, then the page-table
// reads of all of them, so a thread has several independent HBM and L2 reads
// in flight instead of a chain per unit.  The block finds its first row with
// one 64-bit division; a unit's row is that row plus a 32-bit quotient (at
// most a few rows per chunk).  The page size is a template constant for the
// common 64 (shift and mask) and a runtime divisor otherwise.  HBM-bound: 8
// bytes per entry plus the page-table reads, which stay in L2 (a table row
// is a few KB).
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "page_table.cuh"

namespace idx {

namespace {

template <int PS>
IDX_DEVI int map_pos(int p, const int* trow, long long pages, int page_size, bool& bad) {
    if (p < 0) return p;
    const int P = PS > 0 ? PS : page_size;
    const int page = p / P;
    if ((long long)page >= pages) {
        bad = true;
        return -1;
    }
    return __ldg(trow + page) * P + (p - page * P);
}

constexpr int kUnitsPerThread = 4;
constexpr int kChunk = 256 * kUnitsPerThread;  // units per block

template <int PS, bool VEC>
__global__ void __launch_bounds__(256) page_transform_kernel(PageArgs a) {
    using Unit = typename std::conditional<VEC, int4, int>::type;
    const int per_row = VEC ? a.topk / 4 : a.topk;  // units per row
    const long long n = (long long)a.rows * per_row;
    const long long base = (long long)blockIdx.x * kChunk;
    const long long r0 = base / per_row;
    const int off0 = (int)(base - r0 * per_row);
    Unit* const p = reinterpret_cast<Unit*>(a.idx);
    Unit v[kUnitsPerThread];
    long long t[kUnitsPerThread];
#pragma unroll
    for (int i = 0; i < kUnitsPerThread; ++i) {
        const int j = (int)threadIdx.x + 256 * i;
        const long long row = r0 + (off0 + j) / per_row;
        t[i] = base + j < n ? (a.row_map ? (long long)a.row_map[row] : row) : -1;
        if constexpr (VEC)
            v[i] = make_int4(-1, -1, -1, -1);  // past the end: padding, left alone
        else
            v[i] = -1;
        if (base + j < n) v[i] = p[base + j];
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kUnitsPerThread; ++i) {
        const bool trow_ok = t[i] >= 0 && t[i] < a.table_rows;
        const int* trow = a.table + (trow_ok ? t[i] : 0) * a.table_stride;
        const long long pages = trow_ok ? a.table_stride : 0;
        if constexpr (VEC) {
            v[i].x = map_pos<PS>(v[i].x, trow, pages, a.page_size, bad);
            v[i].y = map_pos<PS>(v[i].y, trow, pages, a.page_size, bad);
            v[i].z = map_pos<PS>(v[i].z, trow, pages, a.page_size, bad);
            v[i].w = map_pos<PS>(v[i].w, trow, pages, a.page_size, bad);
        } else {
            v[i] = map_pos<PS>(v[i], trow, pages, a.page_size, bad);
        }
    }
#pragma unroll
    for (int i = 0; i < kUnitsPerThread; ++i) {
        const int j = (int)threadIdx.x + 256 * i;
        if (base + j < n) p[base + j] = v[i];
    }
    if (bad) raise_status(a.d_status, IDX_DEV_RANGE);
}

template <int PS>
cudaError_t launch_ps(const PageArgs& a, int grid, cudaStream_t s) {
    if (a.vec)
        page_transform_kernel<PS, true><<<grid, 256, 0, s>>>(a);
    else
        page_transform_kernel<PS, false><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_page_transform(const PageArgs& a, int sm_count, cudaStream_t s) {
    (void)sm_count;
    const long long units = (long long)a.rows * (a.vec ? a.topk / 4 : a.topk);
    if (units == 0) return cudaSuccess;
    const long long grid = (units + kChunk - 1) / kChunk;
    if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
    return a.page_size == 64 ? launch_ps<64>(a, (int)grid, s) : launch_ps<0>(a, (int)grid, s);
}

}  // namespace idx

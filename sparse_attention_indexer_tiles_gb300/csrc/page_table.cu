// Page-table transform of top-k indices (page "[sglang] logits를 쓰지 않는
// top-k", section 3): a consumer of a paged KV cache wants physical slots, so
// each row-relative position p >= 0 becomes table[t, p / P] * P + p % P, with
// t the page-table row of the query row and P the page size; negative
// positions (the -1 padding) are kept.  The indices are rewritten in place.
//
// The grid is flat over all rows x topk entries (a row count above 65535 needs
// no second grid dimension) and strides over them; with topk % 4 == 0 and a
// 16-byte aligned array every thread moves four entries with one 16-byte load
// and store.  The page size is a template constant for the common 64 (shift
// and mask) and a runtime divisor otherwise.  HBM-bound: 8 bytes per entry
// plus the page-table reads, which stay in L2 (a table row is a few KB).
#include <cstdint>

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

template <int PS, bool VEC>
__global__ void __launch_bounds__(256) page_transform_kernel(PageArgs a) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long per_row = VEC ? a.topk / 4 : a.topk;
    const long long n = (long long)a.rows * per_row;
    bool bad = false;
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += stride) {
        const long long row = q / per_row;
        const long long t = a.row_map ? (long long)a.row_map[row] : row;
        const bool trow_ok = t >= 0 && t < a.table_rows;
        const int* trow = a.table + (trow_ok ? t : 0) * a.table_stride;
        const long long pages = trow_ok ? a.table_stride : 0;
        if (VEC) {
            int4* p4 = reinterpret_cast<int4*>(a.idx) + q;
            int4 v = *p4;
            v.x = map_pos<PS>(v.x, trow, pages, a.page_size, bad);
            v.y = map_pos<PS>(v.y, trow, pages, a.page_size, bad);
            v.z = map_pos<PS>(v.z, trow, pages, a.page_size, bad);
            v.w = map_pos<PS>(v.w, trow, pages, a.page_size, bad);
            *p4 = v;
        } else {
            a.idx[q] = map_pos<PS>(a.idx[q], trow, pages, a.page_size, bad);
        }
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
    const long long units = (long long)a.rows * (a.vec ? a.topk / 4 : a.topk);
    if (units == 0) return cudaSuccess;
    const long long want = (units + 255) / 256;
    const long long cap = 8ll * sm_count;  // eight 256-thread blocks per SM, then stride
    const int grid = (int)(want < cap ? want : cap);
    return a.page_size == 64 ? launch_ps<64>(a, grid, s) : launch_ps<0>(a, grid, s);
}

}  // namespace idx

// Argument block and launcher of the page-table transform kernel.
#pragma once

#include <cuda_runtime.h>

namespace idx {

struct PageArgs {
    int* idx;                // [rows, topk] row-relative positions, rewritten in place
    int rows;
    int topk;
    const int* table;        // [table_rows, table_stride] physical page of each logical page
    int table_rows;
    long long table_stride;  // pages per table row
    const int* row_map;      // [rows] table row of each query row; null = row r uses row r
    int page_size;
    int vec;                 // 1: four entries per thread (topk % 4 == 0, idx 16-byte aligned)
    int* d_status;
};

cudaError_t launch_page_transform(const PageArgs& a, int sm_count, cudaStream_t s);

}  // namespace idx

// Host-visible argument blocks and launchers of the top-k kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/idx.h"
#include "plan.cuh"

namespace idx {

enum : int { TOPK_OUTPUT = 0, TOPK_THRESHOLD = 1 };

// Candidates one block of a split row can hand over (16 warps x 512).
constexpr int kSplitCap = 8192;

struct TopkRowsArgs {
    const float* scores;  // [rows, row_stride]
    long long row_stride;
    long long row_len;    // columns a row may address (bounds check)
    const int* ks;        // may be null (0)
    const int* ke;        // end of the visible range (or its length when ks is null)
    int rows;
    int topk;
    int relative;         // row r's data starts at column 0 instead of ks[r]
    int mode;             // TOPK_OUTPUT or TOPK_THRESHOLD
    int* out;             // [rows, topk] (TOPK_OUTPUT)
    // TOPK_THRESHOLD: per-row sample threshold written into plan[r], from the
    // samples' 16-bit order keys samp [rows, row_stride]
    const uint16_t* samp;
    RowPlan* plan;
    const int* vis_ks;    // the row's visible key range, for the rank t
    const int* vis_ke;
    int cap;
    float target;
    int S;                // sample stride
    long long nsamp;      // floor(keys / S)
    int rows_per_block;   // rows sharing one sample phase
    uint32_t phase_seed;
    // TOPK_OUTPUT row split: g blocks per row (0/1 = none) and their workspace
    int split;
    uint32_t* split_keys;  // [rows * g, kSplitCap]
    uint32_t* split_idx;   // [rows * g, kSplitCap]
    int* split_cnt;        // [rows * g] candidates handed over, -1 = a run overflowed
    uint32_t* split_lb;    // [rows * g] the lower bound (order key) each block used
    unsigned long long* split_ticket;  // [rows] (epoch << 32) | blocks of the row done so far
    uint32_t epoch;        // this call's epoch, never 0: the tickets need no clearing
    // TOPK_THRESHOLD, optional: one more CTA writes order[order_nblk], the
    // scoring row blocks (order_rpb rows each) by their key span in tiles,
    // longest first, for the emit pass's units
    int* order;
    int order_nblk;
    int order_rpb;
    int pdl;              // launch overlapping the kernel before it on the stream
    int* d_status;
    idx_stats* d_stats;
};

struct CandArgs {
    const int2* slab;     // [rows, nruns, cap_q] (score bits, row-relative index) pairs
    const int* run_cnt;   // [rows, nruns]
    int nruns;            // kRuns per key split of the emit pass
    int cap_q;
    RowPlan* plan;
    uint32_t* fb_hist;    // [rows, 4096]
    int* fb_cnt;          // [8] rescan counters (see ScoreArgs)
    int* fb_blocks;       // [row blocks] list of row blocks with a flagged row
    int* fb_bflag;        // [row blocks] listed-once flags
    int rows_per_block;   // rows of one scoring row block
    const int* ks;
    const int* ke;
    int rows, topk, cap;
    int fallback;         // 0: main pass (flags rows), 1: rows re-emitted by the rescan
    int grid_limit;       // CTAs of the rescan's pass (they stride over the rows)
    int sm_count;         // SMs of the device (the launch copies the runs of few rows)
    int* out;
    int pdl;              // launch overlapping the kernel before it on the stream
    int* d_status;
    idx_stats* d_stats;
};


cudaError_t launch_topk_rows(const TopkRowsArgs& a, cudaStream_t s);
cudaError_t launch_cand_topk(const CandArgs& a, cudaStream_t s);
size_t cand_smem_bytes(int cap_q, int nruns, int topk, bool staged);
size_t split_workspace_bytes(int rows, int g);

}  // namespace idx

// Host-visible interface of the tcgen05 scoring kernel.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/idx.h"
#include "plan.cuh"

namespace idx {

// What the epilogue does with the fp32 scores of a key tile.
enum : int {
    SM_MATERIALISE = 0,  // write s[r, j - ks[r]]
    SM_SAMPLE = 1,       // score the strided sample, write samp[r, i - a_r]
    SM_EMIT = 2,         // main pass: emit key >= T_r into the slab
    SM_FB_HIST = 3,      // exact rescan: histogram one digit of flagged rows
    SM_FB_EMIT = 4,      // exact rescan: re-emit flagged rows with the refined rule
    SM_RESCAN = 5,       // the exact rescan as one launch: per flagged row block, the
                         // SM_FB_HIST passes it needs, then SM_FB_EMIT
};

struct ScoreArgs {
    const float* k_scale;
    const float* w;
    const int* ks;
    const int* ke;
    int rows;
    int topk;
    long long keys;
    int mode;
    // SM_MATERIALISE
    float* out;
    long long out_stride;
    // SM_SAMPLE
    uint16_t* samp;       // [rows, samp_stride] the top 16 bits of each sample score's order key
    long long samp_stride;
    int S;
    long long nsamp;
    uint32_t phase_seed;
    // SM_EMIT / SM_FB_*
    int sampled;          // the call took thresholds from a sample (rows may exceed cap)
    RowPlan* plan;
    int2* slab;           // [rows, nruns, cap_q] (score bits, row-relative index) pairs
    int cap;              // nominal slab cap (rows seeing <= cap keys emit every key)
    int cap_q;            // capacity of one warp run: slab row = nruns runs of cap_q
    int* run_cnt;         // [rows, nruns] candidates appended per run (may exceed cap_q)
    int nruns;            // runs per row: kRuns per key split of the main emit pass
    int nwhole;           // CTAs 0 .. nwhole - 1 score row blocks 0 .. nwhole - 1 whole;
    int ksplit;           // every later row block is split into ksplit contiguous parts
                          // of its key tiles, one CTA each (CTA nwhole + ksplit * j + c
                          // scores part c of block nwhole + j)
    uint32_t* fb_hist;
    int* fb_cnt;          // [8] rows waiting per rescan level, [6] ready to emit,
                          // [7] row blocks listed in fb_blocks
    int* fb_blocks;       // [row blocks] the blocks with a row in the rescan
    int* fb_bflag;        // [row blocks] 1 once a block is listed
    int grid_x;           // at most this many CTAs (one per SM): a scoring launch's CTAs
                          // take units in turn, a rescan's stride over its list
    int* sched;           // optional launch counter, 0 before the launch: CTAs take
                          // units gridDim.x + atomicAdd(sched, 1) in turn (null: every
                          // gridDim.x-th unit)
    const int* order;     // optional [row blocks]: the i-th block the units take (whole
                          // blocks, then the split tail) is order[i] (null: block i)
    int level;
    // bounded waits: a wait on the pipeline gives up after wait_limit clock
    // cycles; withhold_tile >= 0 (a test of that path) makes the producer issue
    // no copy for that tile of every pass, so the waits on it run out
    long long wait_limit;
    int withhold_tile;
    int* d_status;
    idx_stats* d_stats;
};

struct ScoreLaunch {
    const void* q;
    const void* k;
    int H, D;
    idx_dtype dt;
    int pdl;  // launch overlapping the kernel before it on the stream
    ScoreArgs a;
};

// Rows handled by one CTA (the MMA's N = rows x H = 256).
inline int score_rows_per_block(int H) { return 256 / H; }

// How a scoring launch cuts row blocks into key parts: blocks 0 .. nwhole - 1
// whole, every later block in k parts (ScoreArgs::nwhole, ::ksplit).
struct SplitPlan {
    int nwhole;
    int k;
};

bool score_supported(idx_dtype dt, int H, int D);
cudaError_t launch_score(const ScoreLaunch& L, cudaStream_t s);

}  // namespace idx

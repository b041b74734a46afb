// C ABI of libidx: argument validation, workspace carving and the launch
// sequence of each entry point.  Everything that computes runs in the kernels
// of topk.cu and score_*.cu; this file only decides what to launch.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "mxfp4.cuh"
#include "page_table.cuh"
#include "plan.cuh"
#include "score.cuh"
#include "topk.cuh"

namespace idx {

cudaError_t launch_score_bf16(const ScoreLaunch& L, cudaStream_t s);
cudaError_t launch_score_fp8(const ScoreLaunch& L, cudaStream_t s);

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool score_supported(idx_dtype dt, int H, int D) {
    const bool h_ok = H == 8 || H == 16 || H == 32 || H == 64;
    const bool d_ok = D == 64 || D == 128;
    return h_ok && d_ok && (dt == IDX_BF16 || dt == IDX_FP8_E4M3);
}

std::atomic<unsigned long long> g_launches{0};

void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

cudaError_t launch_score(const ScoreLaunch& L, cudaStream_t s) {
    const cudaError_t e = L.dt == IDX_BF16 ? launch_score_bf16(L, s) : launch_score_fp8(L, s);
    if (e == cudaSuccess && L.a.rows > 0) count_launches(1);
    return e;
}

namespace {

constexpr int kMaxTopk = 4096;
constexpr int kMaxCap = 12288;
// Route to the fused path from this many keys in the longest row on (measured
// fused / two-pass crossover on GB300, see idx_score_topk_routed).
constexpr long long kRouteMinKeys = 24576;

size_t logits_bytes(int rows, long long stride) {
    return ((size_t)rows * (size_t)stride * sizeof(float) + 255) / 256 * 256;
}
constexpr uint32_t kPhaseSeed = 0x9E3779B9u;

// Is the current device an sm_103 part?  Cached per device.
bool arch_ok() {
    static std::mutex mu;
    static int cached[64];
    static bool init = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> g(mu);
    if (!init) {
        for (int& c : cached) c = -1;
        init = true;
    }
    if (cached[dev] < 0) {
        int maj = 0, min = 0;
        cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
        cached[dev] = (maj == 10 && min == 3) ? 1 : 0;
    }
    return cached[dev] == 1;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SM count of the current device (cached); 148 when no device answers (a
// host-only workspace query).
int sm_count() {
    static std::mutex mu;
    static int cached[64];
    static bool init = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 148;
    }
    std::lock_guard<std::mutex> g(mu);
    if (!init) {
        for (int& c : cached) c = 0;
        init = true;
    }
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

// A per-call epoch for the split rows' ticket words (never 0).
uint32_t next_epoch() {
    static std::atomic<uint32_t> ctr{
        0x9e3779b9u ^ (uint32_t)std::chrono::steady_clock::now().time_since_epoch().count()};
    uint32_t e;
    do e = ctr.fetch_add(1u, std::memory_order_relaxed) + 1u;
    while (e == 0u);
    return e;
}

// Blocks per row of the standalone top-k (page "[sglang] ROCm DSA Indexer
// Top-K 최적화", row_split): none below 65536 columns; otherwise
// g = min(SMs / rows, 32), and none when g < 4.  options->row_split: -1 or 1
// never splits, g >= 2 forces g blocks (at most 64).
int row_split_blocks(int rows, long long row_len_hint, const idx_options* opt) {
    const int force = opt ? opt->row_split : 0;
    if (force == -1 || force == 1 || rows > 65535) return 0;  // split grids keep rows in y
    if (force >= 2) return force < 64 ? force : 64;
    if (row_len_hint < 65536) return 0;
    const int g = std::min(sm_count() / std::max(rows, 1), 32);
    return g < 4 ? 0 : g;
}

struct FusedParams {
    int cap;    // nominal slab cap
    int cap_q;  // one warp run: ceil(cap / 8) + 64 (a contiguous range of n keys puts
                // at most n / 8 + 64 of them into the 32-key column of the even or of the odd
                // 128-key tiles that one run collects)
    float target;
    int S;
};

// Slab cap, threshold target and sample stride of the fused path.
//   cap    = ceil(cap_factor * topk) when cap_factor is given, else
//            min(max(ceil(3.5 * topk), 4096), kMaxCap): the page's slab holds
//            about 2.25 topk; at 3.5 topk the rule below reaches the widest
//            stride of the table for topk >= 1170, and the sample pass, which
//            scores keys / S of every row, costs less than the larger slab adds
//   target = expected candidates / topk the sampled threshold aims at; the
//            geometric middle sqrt(cap / topk) of [1, cap / topk] by default
//   S      = the largest odd stride from the table that still leaves about
//            t = max(32, (4.5 / ln target)^2) sample hits above the threshold
//            (the relative spread of the candidate count is ~ 1/sqrt(t), so
//            4.5 spreads fit between topk and cap)
FusedParams fused_params(int topk, const idx_options* opt) {
    FusedParams p;
    const double cf = opt && opt->cap_factor > 0.f ? (double)opt->cap_factor : 0.0;
    if (cf > 0.0)
        p.cap = (int)std::ceil(cf * topk);
    else
        p.cap = std::min(std::max((int)std::ceil(3.5 * topk), 4096), kMaxCap);
    if (p.cap < topk) p.cap = topk;
    p.cap_q = ((p.cap + kRuns - 1) / kRuns + 64 + 1) / 2 * 2;  // even: 16-byte run copies
    const double ratio = (double)p.cap / topk;
    double target = opt && opt->target_factor > 0.f ? (double)opt->target_factor : std::sqrt(ratio);
    p.target = (float)target;
    if (opt && opt->sample_stride > 0) {
        p.S = opt->sample_stride;
    } else {
        static const int table[] = {1, 3, 5, 7, 11, 15, 23, 31, 45, 63};
        const double lt = std::log(std::max(target, 1.0001));
        const double t = std::max(32.0, (4.5 / lt) * (4.5 / lt));
        const double smax = target * topk / t;
        p.S = 1;
        for (int s : table)
            if (s <= smax) p.S = s;
    }
    return p;
}

struct FusedLayout {
    size_t plan, run_cnt, slab, samp, fb_hist, fb_blocks, fb_bflag, order, fb_cnt, total;
    long long samp_stride;
};

FusedLayout fused_layout(int rows, long long max_len, int cap, int cap_q, int S, int nruns,
                         int H) {
    const size_t nblk = (size_t)((rows + score_rows_per_block(H) - 1) / score_rows_per_block(H));
    FusedLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.samp_stride = (max_len / S + 2 + 7) / 8 * 8;  // 16-byte aligned rows of 16-bit keys
    L.plan = take((size_t)rows * sizeof(RowPlan));
    L.run_cnt = take((size_t)rows * nruns * sizeof(int));
    L.slab = take((size_t)rows * nruns * cap_q * sizeof(int2));
    L.samp = take(max_len > cap ? (size_t)rows * L.samp_stride * sizeof(uint16_t) : 0);
    L.fb_hist = take(max_len > cap ? (size_t)rows * 4096 * sizeof(uint32_t) : 0);
    L.fb_blocks = take(max_len > cap ? nblk * sizeof(int) : 0);
    L.fb_bflag = take(max_len > cap ? nblk * sizeof(int) : 0);
    L.order = take(max_len > cap ? nblk * sizeof(int) : 0);  // the emit pass's block order
    // [0, 8) rescan counters, [8] [9] the sample and emit launches' unit counters
    L.fb_cnt = take(16 * sizeof(int));
    L.total = off;
    return L;
}

idx_status check_indexer_args(const void* q, const void* k, const float* k_scale, const float* w,
                              const int* ks, const int* ke, int rows, long long keys, int H, int D,
                              idx_dtype dt) {
    if (rows < 0 || keys < 0) return IDX_EINVAL;
    if (dt != IDX_BF16 && dt != IDX_FP8_E4M3) return IDX_EUNSUPPORTED;
    if (!score_supported(dt, H, D)) return IDX_EUNSUPPORTED;
    if (rows == 0) return IDX_OK;
    if (!q || !k || !k_scale || !w || !ks || !ke) return IDX_EINVAL;
    if (keys < 1 || keys > 0x7fffff00ll || (long long)rows * H > 0x7fffff00ll) return IDX_EUNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(k_scale, 4) || !aligned(w, 4) ||
        !aligned(ks, 4) || !aligned(ke, 4))
        return IDX_EALIGN;
    if (!arch_ok()) return IDX_EUNSUPPORTED;
    return IDX_OK;
}

ScoreLaunch make_score_launch(const void* q, const void* k, const float* k_scale, const float* w,
                              const int* ks, const int* ke, int rows, long long keys, int H, int D,
                              idx_dtype dt, int topk, const idx_options* opt) {
    ScoreLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.q = q;
    L.k = k;
    L.H = H;
    L.D = D;
    L.dt = dt;
    L.a.k_scale = k_scale;
    L.a.w = w;
    L.a.ks = ks;
    L.a.ke = ke;
    L.a.rows = rows;
    L.a.keys = keys;
    L.a.topk = topk;
    L.a.d_status = opt ? opt->d_status : nullptr;
    L.a.d_stats = opt ? opt->d_stats : nullptr;
    L.a.nwhole = (rows + score_rows_per_block(H) - 1) / score_rows_per_block(H);
    L.a.ksplit = 1;
    L.a.nruns = kRuns;
    L.a.grid_x = sm_count();
    // about 2 s at the GB300's clock; the test knob shortens it and withholds
    // key tile 1 of every scoring pass
    const int stall_us = opt ? opt->test_stall_us : 0;
    L.a.wait_limit = stall_us > 0 ? 2100LL * stall_us : (1LL << 32);
    L.a.withhold_tile = stall_us > 0 ? 1 : -1;
    return L;
}

// Key splits of a scoring launch.  One wave is SM-count many CTAs (one per
// SM), so a grid of nblk row blocks runs floor(nblk / SMs) full waves and a
// last one with only tail = nblk % SMs blocks, leaving the other SMs idle; a
// call with fewer blocks than SMs (few query rows over long rows, a decode
// shape) leaves most of the GPU idle.  So the full waves keep whole blocks,
// and each of the tail blocks is cut into k contiguous parts of its key
// tiles, one CTA each: the tail then takes ceil(tail k / SMs) rounds of 1 / k
// of a block's time, plus a per-part overhead o (the CTA prologue and the
// pipeline's fill and drain, about 8 tiles' worth: o = 8 / tiles of a block).
// The k in [1, 128] with the smallest ceil(tail k / SMs) (1 / k + o) is taken
// (a larger k only when it is 1 % cheaper), every part keeping >= 32 tiles.
// Each key split adds kRuns runs per row to the emit pass's slab.
SplitPlan score_split(int rows, int H, long long max_len) {
    const int nblk = (rows + score_rows_per_block(H) - 1) / score_rows_per_block(H);
    const long long tiles = (max_len + 127) / 128;
    const int sm = std::max(sm_count(), 1);
    const int tail = nblk % sm;
    SplitPlan p{nblk, 1};
    if (tail == 0 || tiles < 64) return p;
    const double o = 8.0 / (double)tiles;
    double best = 1.0 + o;
    for (int k = 2; k <= 128 && tiles / k >= 32; ++k) {
        const double rounds = std::ceil((double)tail * k / sm);
        const double cost = rounds * (1.0 / k + o);
        if (cost < best * 0.99) {
            best = cost;
            p.k = k;
        }
    }
    if (p.k > 1) p.nwhole = nblk - tail;
    return p;
}

// ------------------------------------------------------------ host entry

// Rows per chunk of idx_score_topk_host: two chunks of whole row blocks.  A
// chunk is one fused call with its fixed costs (the sample, threshold and slab
// launches, the emit pass's last wave: ~0.05 ms at 4096 x 65536, H 64), while
// the copies left exposed (k, the first chunk's inputs, the last chunk's
// indices) shrink only slowly with more chunks.  Measured at that shape: one
// call 2.082 ms of compute, two chunks 2.135, three 2.19, four 2.27.
constexpr int kHostChunks = 2;

struct HostChunks {
    int rows_per_chunk, n;
};

HostChunks host_chunks(int rows, int H) {
    const int rpb = score_rows_per_block(H);
    const int nblk = (rows + rpb - 1) / rpb;
    const int per = std::max((nblk + kHostChunks - 1) / kHostChunks, 1) * rpb;
    return {per, (rows + per - 1) / per};
}

// The device copies of an idx_score_topk_host call at the front of its
// workspace, then one chunk's fused workspace.
struct HostLayout {
    size_t q, k, k_scale, w, ks, ke, out, fused, total;
};

HostLayout host_layout(int rows, long long keys, int H, int D, int topk, idx_dtype dt,
                       size_t fused_bytes) {
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t es = dt == IDX_BF16 ? 2 : 1;
    HostLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += up(bytes);
        return o;
    };
    L.q = take((size_t)rows * H * D * es);
    L.k = take((size_t)keys * D * es);
    L.k_scale = take((size_t)keys * sizeof(float));
    L.w = take((size_t)rows * H * sizeof(float));
    L.ks = take((size_t)rows * sizeof(int));
    L.ke = take((size_t)rows * sizeof(int));
    L.out = take((size_t)rows * topk * sizeof(int));
    L.fused = take(fused_bytes);
    L.total = off;
    return L;
}

// One upload and one download stream per device, with the events that order
// them against the compute stream; a call holds the device's mutex while it
// enqueues.
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, fin = nullptr;
    cudaEvent_t in_ready[kHostChunks + 1] = {}, done[kHostChunks] = {};
};

constexpr int kMaxDevices = 64;
HostPipe g_host_pipes[kMaxDevices];

cudaError_t host_pipe_init(HostPipe& p) {
    if (p.ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.fin, cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i <= kHostChunks; ++i)
        e = cudaEventCreateWithFlags(&p.in_ready[i], cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i < kHostChunks; ++i)
        e = cudaEventCreateWithFlags(&p.done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) p.ready = true;
    return e;
}

void record(const idx_options* opt, int i, cudaStream_t s) {
    if (opt && opt->stage_events && opt->stage_events[i])
        cudaEventRecord(static_cast<cudaEvent_t>(opt->stage_events[i]), s);
}

// The CUDA error behind the calling thread's last failed call.
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

idx_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return IDX_OK;
    t_last_cuda_error = e;
    cudaGetLastError();  // clear a sticky launch error of ours
    return e == cudaErrorNotSupported ? IDX_EUNSUPPORTED : IDX_ECUDA;
}

}  // namespace
}  // namespace idx

using namespace idx;

extern "C" {

const char* idx_status_string(idx_status s) {
    switch (s) {
        case IDX_OK: return "ok";
        case IDX_EINVAL: return "invalid argument";
        case IDX_EALIGN: return "misaligned pointer";
        case IDX_EWORKSPACE: return "workspace too small";
        case IDX_EUNSUPPORTED: return "unsupported dtype, shape or GPU";
        case IDX_ECUDA: return "CUDA error";
        case IDX_ETIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int idx_version(void) { return (0 << 16) | 2; }

const char* idx_last_cuda_error(void) {
    return t_last_cuda_error == cudaSuccess ? "" : cudaGetErrorString(t_last_cuda_error);
}

unsigned long long idx_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t idx_score_topk_workspace(int rows, long long keys, long long max_len, int H, int D,
                                int topk, idx_dtype dt, const idx_options* opt) {
    (void)H;
    (void)D;
    (void)dt;
    if (rows <= 0 || topk < 1 || topk > kMaxTopk) return 0;
    if (max_len <= 0 || max_len > keys) max_len = keys;
    const FusedParams p = fused_params(topk, opt);
    const int nruns = kRuns * score_split(rows, H, max_len).k;
    return fused_layout(rows, max_len, p.cap, p.cap_q, p.S, nruns, H).total;
}

idx_status idx_score_topk(const void* q, const void* k, const float* k_scale, const float* w,
                          const int* ks, const int* ke, int rows, long long keys, long long max_len,
                          int H, int D, int topk, idx_dtype dt, int* out_idx, void* ws,
                          size_t ws_bytes, const idx_options* opt, void* stream) {
    if (topk < 1) return IDX_EINVAL;
    if (topk > kMaxTopk) return IDX_EUNSUPPORTED;
    idx_status st = check_indexer_args(q, k, k_scale, w, ks, ke, rows, keys, H, D, dt);
    if (st != IDX_OK || rows == 0) return st;
    if (!out_idx) return IDX_EINVAL;
    if (!aligned(out_idx, 4)) return IDX_EALIGN;
    if (max_len <= 0 || max_len > keys) max_len = keys;
    const FusedParams p = fused_params(topk, opt);
    if (p.cap > kMaxCap || p.S < 1) return IDX_EUNSUPPORTED;
    const SplitPlan split = score_split(rows, H, max_len);
    const int nruns = kRuns * split.k;
    const FusedLayout lay = fused_layout(rows, max_len, p.cap, p.cap_q, p.S, nruns, H);
    if (!ws || ws_bytes < lay.total) return IDX_EWORKSPACE;
    if (!aligned(ws, 256)) return IDX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    RowPlan* plan = reinterpret_cast<RowPlan*>(base + lay.plan);
    int* run_cnt = reinterpret_cast<int*>(base + lay.run_cnt);
    int2* slab = reinterpret_cast<int2*>(base + lay.slab);
    uint16_t* samp = reinterpret_cast<uint16_t*>(base + lay.samp);
    uint32_t* fb_hist = reinterpret_cast<uint32_t*>(base + lay.fb_hist);
    int* fb_cnt = reinterpret_cast<int*>(base + lay.fb_cnt);
    const bool sampling = max_len > p.cap;
    int* fb_blocks = sampling ? reinterpret_cast<int*>(base + lay.fb_blocks) : nullptr;
    int* fb_bflag = sampling ? reinterpret_cast<int*>(base + lay.fb_bflag) : nullptr;
    int* order = sampling ? reinterpret_cast<int*>(base + lay.order) : nullptr;
    int* d_status = opt ? opt->d_status : nullptr;
    idx_stats* d_stats = opt ? opt->d_stats : nullptr;

    ScoreLaunch L = make_score_launch(q, k, k_scale, w, ks, ke, rows, keys, H, D, dt, topk, opt);
    L.a.plan = plan;
    L.a.slab = slab;
    L.a.cap = p.cap;
    L.a.cap_q = p.cap_q;
    L.a.nruns = nruns;
    L.a.run_cnt = run_cnt;
    L.a.fb_hist = fb_hist;
    L.a.fb_cnt = fb_cnt;
    L.a.fb_blocks = fb_blocks;
    L.a.fb_bflag = fb_bflag;
    L.a.S = p.S;
    L.a.nsamp = keys / p.S;
    L.a.sampled = sampling ? 1 : 0;
    L.a.samp = samp;
    L.a.samp_stride = lay.samp_stride;
    L.a.phase_seed = kPhaseSeed;
    cudaError_t e;

    record(opt, 0, s);
    // the persistent scoring launches take units from counters that start at 0
    if ((e = cudaMemsetAsync(fb_cnt + 8, 0, 2 * sizeof(int), s)) != cudaSuccess)
        return cuda_status(e);
    if (sampling) {
        // 1. score the odd-stride sample of every long row (key splits over the
        //    sample index range, as for the emit pass)
        L.a.mode = SM_SAMPLE;
        L.a.sched = fb_cnt + 8;
        const SplitPlan sp = score_split(rows, H, max_len / p.S + 1);
        L.a.nwhole = sp.nwhole;
        L.a.ksplit = sp.k;
        if ((e = launch_score(L, s)) != cudaSuccess) return cuda_status(e);
        // 2. T_r = exact t-th largest sample score of each row
        TopkRowsArgs t;
        std::memset(&t, 0, sizeof(t));
        t.samp = samp;
        t.row_stride = lay.samp_stride;
        t.row_len = lay.samp_stride;
        t.rows = rows;
        t.topk = topk;
        t.relative = 1;
        t.mode = TOPK_THRESHOLD;
        t.plan = plan;
        t.vis_ks = ks;
        t.vis_ke = ke;
        t.cap = p.cap;
        t.target = p.target;
        t.S = p.S;
        t.nsamp = keys / p.S;
        t.rows_per_block = score_rows_per_block(H);
        t.phase_seed = kPhaseSeed;
        t.d_status = d_status;
        t.d_stats = d_stats;
        t.pdl = 1;  // after the sample pass
        // the same launch orders the row blocks for the emit pass, longest first
        t.order = order;
        t.order_nblk = (rows + score_rows_per_block(H) - 1) / score_rows_per_block(H);
        t.order_rpb = score_rows_per_block(H);
        if ((e = launch_topk_rows(t, s)) != cudaSuccess) return cuda_status(e);
        count_launches(1);
    }
    record(opt, 1, s);
    // 3. one scoring pass emits every key at or above T_r into the slab
    //    (key splits write runs of their own)
    L.a.mode = SM_EMIT;
    L.a.nwhole = split.nwhole;
    L.a.ksplit = split.k;
    L.a.sched = fb_cnt + 9;
    L.a.order = order;  // (null without a sample: block order)
    L.pdl = sampling ? 1 : 0;  // after the thresholds (else the memset: plain launch)
    if ((e = launch_score(L, s)) != cudaSuccess) return cuda_status(e);
    record(opt, 2, s);
    // 4. exact top-k of every slab; rows whose count missed [topk, cap] are flagged
    CandArgs c;
    std::memset(&c, 0, sizeof(c));
    c.slab = slab;
    c.run_cnt = run_cnt;
    c.cap_q = p.cap_q;
    c.nruns = nruns;
    c.plan = plan;
    c.fb_hist = sampling ? fb_hist : nullptr;
    c.fb_cnt = fb_cnt;
    c.fb_blocks = fb_blocks;
    c.fb_bflag = fb_bflag;
    c.rows_per_block = score_rows_per_block(H);
    c.ks = ks;
    c.ke = ke;
    c.rows = rows;
    c.topk = topk;
    c.cap = p.cap;
    c.out = out_idx;
    c.d_status = d_status;
    c.d_stats = d_stats;
    c.fallback = 0;
    c.grid_limit = 2 * sm_count();
    c.sm_count = sm_count();
    c.pdl = 1;  // after the emit pass
    if ((e = launch_cand_topk(c, s)) != cudaSuccess) return cuda_status(e);
    count_launches(1);
    record(opt, 3, s);
    if (sampling) {
        // 5. exact rescan of flagged rows, one launch: a grid of at most one CTA
        //    per SM strides over the device list of flagged row blocks; per block
        //    up to six digit passes (three over the score key, three over the
        //    index of exact ties), each finishing its digit step in the CTA, then
        //    one re-emission.  With no block listed every CTA ends at once.
        L.a.mode = SM_RESCAN;
        L.a.grid_x = sm_count();
        if ((e = launch_score(L, s)) != cudaSuccess) return cuda_status(e);
        c.fallback = 1;
        if ((e = launch_cand_topk(c, s)) != cudaSuccess) return cuda_status(e);
        count_launches(1);
    }
    record(opt, 4, s);
    return IDX_OK;
}

size_t idx_score_topk_host_workspace(int rows, long long keys, long long max_len, int H, int D,
                                     int topk, idx_dtype dt, const idx_options* opt) {
    if (rows <= 0 || keys <= 0 || topk < 1) return 0;
    if (max_len <= 0 || max_len > keys) max_len = keys;
    const HostChunks hc = host_chunks(rows, H);
    const size_t fused = idx_score_topk_workspace(std::min(rows, hc.rows_per_chunk), keys, max_len,
                                                  H, D, topk, dt, opt);
    return host_layout(rows, keys, H, D, topk, dt, fused).total;
}

idx_status idx_score_topk_host(const void* q, const void* k, const float* k_scale,
                               const float* w, const int* ks, const int* ke, int rows,
                               long long keys, long long max_len, int H, int D, int topk,
                               idx_dtype dt, int* out_idx, void* ws, size_t ws_bytes,
                               const idx_options* opt, void* stream) {
    if (topk < 1) return IDX_EINVAL;
    if (topk > kMaxTopk) return IDX_EUNSUPPORTED;
    if (rows < 0 || keys < 0) return IDX_EINVAL;
    if (dt != IDX_BF16 && dt != IDX_FP8_E4M3) return IDX_EUNSUPPORTED;
    if (!score_supported(dt, H, D)) return IDX_EUNSUPPORTED;
    if (rows == 0) return IDX_OK;
    if (!q || !k || !k_scale || !w || !ks || !ke || !out_idx || !ws) return IDX_EINVAL;
    if (keys < 1 || keys > 0x7fffff00ll || (long long)rows * H > 0x7fffff00ll) return IDX_EUNSUPPORTED;
    if (!aligned(ws, 256)) return IDX_EALIGN;
    if (max_len <= 0 || max_len > keys) max_len = keys;
    const FusedParams fp = fused_params(topk, opt);
    if (fp.cap > kMaxCap || fp.S < 1) return IDX_EUNSUPPORTED;
    if (!arch_ok()) return IDX_EUNSUPPORTED;
    const HostChunks hc = host_chunks(rows, H);
    const size_t fused_bytes = idx_score_topk_workspace(std::min(rows, hc.rows_per_chunk), keys,
                                                        max_len, H, D, topk, dt, opt);
    const HostLayout L = host_layout(rows, keys, H, D, topk, dt, fused_bytes);
    if (ws_bytes < L.total) return IDX_EWORKSPACE;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return IDX_EUNSUPPORTED;
    HostPipe& P = g_host_pipes[dev];
    std::lock_guard<std::mutex> lock(P.mu);
    if ((e = host_pipe_init(P)) != cudaSuccess) return cuda_status(e);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    record(opt, 0, s);
    idx_options o;
    if (opt) o = *opt;
    else std::memset(&o, 0, sizeof(o));
    o.stage_events = nullptr;

    uint8_t* base = static_cast<uint8_t*>(ws);
    const size_t es = dt == IDX_BF16 ? 2 : 1;
    const size_t q_row = (size_t)H * D * es, w_row = (size_t)H * sizeof(float);
    auto h2d = [&](size_t dst, const void* src, size_t bytes) {
        return cudaMemcpyAsync(base + dst, src, bytes, cudaMemcpyHostToDevice, P.up);
    };
    // the copies start after the work the caller queued before this call (the
    // workspace may still be in use there)
    if ((e = cudaEventRecord(P.start, s)) != cudaSuccess) return cuda_status(e);
    if ((e = cudaStreamWaitEvent(P.up, P.start, 0)) != cudaSuccess) return cuda_status(e);
    if ((e = cudaStreamWaitEvent(P.down, P.start, 0)) != cudaSuccess) return cuda_status(e);
    if ((e = h2d(L.k, k, (size_t)keys * D * es)) != cudaSuccess) return cuda_status(e);
    if ((e = h2d(L.k_scale, k_scale, (size_t)keys * sizeof(float))) != cudaSuccess)
        return cuda_status(e);
    for (int c = 0; c < hc.n; ++c) {
        const int r0 = c * hc.rows_per_chunk, nr = std::min(hc.rows_per_chunk, rows - r0);
        if ((e = h2d(L.q + r0 * q_row, static_cast<const uint8_t*>(q) + r0 * q_row, nr * q_row)) !=
                cudaSuccess ||
            (e = h2d(L.w + r0 * w_row, w + (size_t)r0 * H, nr * w_row)) != cudaSuccess ||
            (e = h2d(L.ks + r0 * sizeof(int), ks + r0, nr * sizeof(int))) != cudaSuccess ||
            (e = h2d(L.ke + r0 * sizeof(int), ke + r0, nr * sizeof(int))) != cudaSuccess ||
            (e = cudaEventRecord(P.in_ready[c], P.up)) != cudaSuccess)
            return cuda_status(e);
    }
    for (int c = 0; c < hc.n; ++c) {
        const int r0 = c * hc.rows_per_chunk, nr = std::min(hc.rows_per_chunk, rows - r0);
        if ((e = cudaStreamWaitEvent(s, P.in_ready[c], 0)) != cudaSuccess) return cuda_status(e);
        const idx_status st = idx_score_topk(
            base + L.q + r0 * q_row, base + L.k, reinterpret_cast<const float*>(base + L.k_scale),
            reinterpret_cast<const float*>(base + L.w + r0 * w_row),
            reinterpret_cast<const int*>(base + L.ks) + r0,
            reinterpret_cast<const int*>(base + L.ke) + r0, nr, keys, max_len, H, D, topk, dt,
            reinterpret_cast<int*>(base + L.out) + (size_t)r0 * topk, base + L.fused, fused_bytes,
            &o, stream);
        if (st != IDX_OK) return st;
        if ((e = cudaEventRecord(P.done[c], s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(P.down, P.done[c], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(out_idx + (size_t)r0 * topk,
                                 reinterpret_cast<int*>(base + L.out) + (size_t)r0 * topk,
                                 (size_t)nr * topk * sizeof(int), cudaMemcpyDeviceToHost,
                                 P.down)) != cudaSuccess)
            return cuda_status(e);
    }
    // the caller's stream (and the next call's copies) wait for the last copy back
    if ((e = cudaEventRecord(P.fin, P.down)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, P.fin, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(P.up, P.fin, 0)) != cudaSuccess)
        return cuda_status(e);
    record(opt, 1, s);
    return IDX_OK;
}

size_t idx_topk_workspace(int rows, long long row_stride, int topk, const idx_options* opt) {
    (void)topk;
    if (rows <= 0) return 0;
    return split_workspace_bytes(rows, row_split_blocks(rows, row_stride, opt));
}

idx_status idx_topk_from_scores(const float* scores, long long row_stride, const int* ks,
                                const int* ke, int rows, int topk, int* out_idx, void* ws,
                                size_t ws_bytes, const idx_options* opt, void* stream) {
    if (rows < 0 || topk < 1 || row_stride < 0) return IDX_EINVAL;
    if (topk > kMaxTopk) return IDX_EUNSUPPORTED;
    if (rows == 0) return IDX_OK;
    if (!scores || !ke || !out_idx) return IDX_EINVAL;
    if (!aligned(scores, 4) || !aligned(out_idx, 4) || !aligned(ke, 4) || (ks && !aligned(ks, 4)))
        return IDX_EALIGN;
    if (!arch_ok()) return IDX_EUNSUPPORTED;
    TopkRowsArgs t;
    std::memset(&t, 0, sizeof(t));
    t.scores = scores;
    t.row_stride = row_stride;
    t.row_len = row_stride;
    t.ks = ks;
    t.ke = ke;
    t.rows = rows;
    t.topk = topk;
    t.relative = opt ? opt->relative_rows : 0;
    t.mode = TOPK_OUTPUT;
    t.out = out_idx;
    t.d_status = opt ? opt->d_status : nullptr;
    t.d_stats = opt ? opt->d_stats : nullptr;
    const int g = row_split_blocks(rows, row_stride, opt);
    if (g >= 2) {
        const size_t need = split_workspace_bytes(rows, g);
        if (!ws || ws_bytes < need) return IDX_EWORKSPACE;
        if (!aligned(ws, 256)) return IDX_EALIGN;
        const size_t slots = (size_t)rows * g;
        uint8_t* base = static_cast<uint8_t*>(ws);
        t.split = g;
        t.split_keys = reinterpret_cast<uint32_t*>(base);
        t.split_idx = t.split_keys + slots * kSplitCap;
        t.split_cnt = reinterpret_cast<int*>(t.split_idx + slots * kSplitCap);
        t.split_lb = reinterpret_cast<uint32_t*>(t.split_cnt + slots);
        t.split_ticket = reinterpret_cast<unsigned long long*>(t.split_lb + slots);
        t.epoch = next_epoch();
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    record(opt, 0, s);
    const cudaError_t e = launch_topk_rows(t, s);
    if (e == cudaSuccess) count_launches(1);
    record(opt, 1, s);
    return cuda_status(e);
}

idx_status idx_score_materialise(const void* q, const void* k, const float* k_scale,
                                 const float* w, const int* ks, const int* ke, int rows,
                                 long long keys, int H, int D, idx_dtype dt, float* scores,
                                 long long row_stride, const idx_options* opt, void* stream) {
    idx_status st = check_indexer_args(q, k, k_scale, w, ks, ke, rows, keys, H, D, dt);
    if (st != IDX_OK || rows == 0) return st;
    if (!scores || row_stride < 1) return IDX_EINVAL;
    if (!aligned(scores, 4)) return IDX_EALIGN;
    ScoreLaunch L = make_score_launch(q, k, k_scale, w, ks, ke, rows, keys, H, D, dt, 1, opt);
    L.a.mode = SM_MATERIALISE;
    L.a.out = scores;
    L.a.out_stride = row_stride;
    const SplitPlan sp = score_split(rows, H, std::min<long long>(keys, row_stride));
    L.a.nwhole = sp.nwhole;
    L.a.ksplit = sp.k;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    record(opt, 0, s);
    const cudaError_t e = launch_score(L, s);
    record(opt, 1, s);
    return cuda_status(e);
}

int idx_route_fused(int rows, long long max_len, int topk) {
    // rows of at most max(2.25 topk, 4096) keys fit the default slab and are
    // emitted whole (no sampling): fused, as measured
    const long long cap = std::max<long long>((long long)std::ceil(2.25 * topk), 4096);
    if (max_len <= cap) return 1;
    // few rows: the logits (rows x max_len x 4 B) are cheap to write and read
    // back and the top-k splits every long row over >= 4 blocks, while the
    // fused path pays its sample, threshold and slab launches whatever the
    // rows (measured: 8 / 16 / 32 rows x 1M keys, H 32, topk 2048: two-pass
    // 1.36 / 1.19 / 1.02x faster, fused 3.6x faster at 64 rows where the
    // top-k no longer splits; 8-128 rows x 256K keys, H 64: two-pass 1.57-1.02x)
    if (rows > 0 && 4ll * rows <= sm_count() && (long long)rows * max_len <= (1ll << 25)) return 0;
    return max_len >= kRouteMinKeys ? 1 : 0;
}

size_t idx_score_topk_routed_workspace(int rows, long long keys, long long max_len, int H,
                                       int D, int topk, idx_dtype dt, const idx_options* opt) {
    if (rows <= 0 || topk < 1 || topk > kMaxTopk) return 0;
    if (max_len <= 0 || max_len > keys) max_len = keys;
    if (idx_route_fused(rows, max_len, topk))
        return idx_score_topk_workspace(rows, keys, max_len, H, D, topk, dt, opt);
    const long long stride = max_len > 0 ? max_len : 1;
    return logits_bytes(rows, stride) + idx_topk_workspace(rows, stride, topk, opt);
}

idx_status idx_score_topk_routed(const void* q, const void* k, const float* k_scale,
                                 const float* w, const int* ks, const int* ke, int rows,
                                 long long keys, long long max_len, int H, int D, int topk,
                                 idx_dtype dt, int* out_idx, void* ws, size_t ws_bytes,
                                 const idx_options* opt, void* stream) {
    if (topk < 1) return IDX_EINVAL;
    if (topk > kMaxTopk) return IDX_EUNSUPPORTED;
    const long long ml = (max_len <= 0 || max_len > keys) ? keys : max_len;
    if (idx_route_fused(rows, ml, topk))
        return idx_score_topk(q, k, k_scale, w, ks, ke, rows, keys, max_len, H, D, topk, dt,
                              out_idx, ws, ws_bytes, opt, stream);
    // dense route: the logits [rows, max_len] in the workspace, then their top-k
    idx_status st = check_indexer_args(q, k, k_scale, w, ks, ke, rows, keys, H, D, dt);
    if (st != IDX_OK || rows == 0) return st;
    if (!out_idx) return IDX_EINVAL;
    if (!aligned(out_idx, 4)) return IDX_EALIGN;
    const long long stride = ml > 0 ? ml : 1;
    const size_t lb = logits_bytes(rows, stride);
    const size_t need = lb + idx_topk_workspace(rows, stride, topk, opt);
    if (!ws || ws_bytes < need) return IDX_EWORKSPACE;
    if (!aligned(ws, 256)) return IDX_EALIGN;
    idx_options o;
    std::memset(&o, 0, sizeof(o));
    if (opt) o = *opt;
    o.stage_events = nullptr;  // the stage boundaries are recorded here
    o.relative_rows = 1;       // the logits start at column 0 of each row
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    record(opt, 0, s);
    record(opt, 1, s);
    st = idx_score_materialise(q, k, k_scale, w, ks, ke, rows, keys, H, D, dt,
                               reinterpret_cast<float*>(base), stride, &o, stream);
    if (st != IDX_OK) return st;
    record(opt, 2, s);
    st = idx_topk_from_scores(reinterpret_cast<const float*>(base), stride, ks, ke, rows, topk,
                              out_idx, base + lb, ws_bytes - lb, &o, stream);
    record(opt, 3, s);
    record(opt, 4, s);
    return st;
}

idx_status idx_page_table_transform(int* idx_out, int rows, int topk, const int* table,
                                    int table_rows, long long table_stride, const int* row_map,
                                    int page_size, const idx_options* opt, void* stream) {
    if (rows < 0 || topk < 0 || table_rows < 0 || table_stride < 0 || page_size < 1)
        return IDX_EINVAL;
    if (rows == 0 || topk == 0) return IDX_OK;
    if (!idx_out || (!table && table_rows > 0)) return IDX_EINVAL;
    if (!aligned(idx_out, 4) || (table && !aligned(table, 4)) || (row_map && !aligned(row_map, 4)))
        return IDX_EALIGN;
    if (!arch_ok()) return IDX_EUNSUPPORTED;
    PageArgs a;
    std::memset(&a, 0, sizeof(a));
    a.idx = idx_out;
    a.rows = rows;
    a.topk = topk;
    a.table = table;
    a.table_rows = table_rows;
    a.table_stride = table_stride;
    a.row_map = row_map;
    a.page_size = page_size;
    a.vec = (topk % 4 == 0 && aligned(idx_out, 16)) ? 1 : 0;
    a.d_status = opt ? opt->d_status : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    record(opt, 0, s);
    const cudaError_t e = launch_page_transform(a, sm_count(), s);
    if (e == cudaSuccess) count_launches(1);
    record(opt, 1, s);
    return cuda_status(e);
}


// ---------------------------------------------------------------- MXFP4

namespace {

// One expansion launch over one or two arrays (seg[1].n == 0: one).
idx_status mxfp4_launch(const Mxfp4Segment& s0, const Mxfp4Segment& s1, int D,
                        const idx_options* opt, void* stream) {
    if (D < 32 || D % 32 != 0) return IDX_EINVAL;
    const Mxfp4Segment* seg[2] = {&s0, &s1};
    for (const Mxfp4Segment* g : seg) {
        if (g->n < 0) return IDX_EINVAL;
        if (g->n == 0) continue;
        if (!g->x || !g->sf || !g->out) return IDX_EINVAL;
        if (!aligned(g->x, 16) || !aligned(g->out, 16)) return IDX_EALIGN;
    }
    if (s0.n + s1.n == 0) return IDX_OK;
    if (!arch_ok()) return IDX_EUNSUPPORTED;
    Mxfp4Args a;
    a.seg[0] = s0;
    a.seg[1] = s1;
    a.D = D;
    a.d_status = opt ? opt->d_status : nullptr;
    const cudaError_t e = launch_mxfp4_to_e4m3(a, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) count_launches(1);
    return cuda_status(e);
}

}  // namespace

idx_status idx_mxfp4_to_e4m3(const uint8_t* x, const uint8_t* sf, long long n, int D,
                             uint8_t* out, const idx_options* opt, void* stream) {
    return mxfp4_launch(Mxfp4Segment{x, sf, n, out}, Mxfp4Segment{nullptr, nullptr, 0, nullptr},
                        D, opt, stream);
}

namespace {

// The e4m3 copies of q and k at the front of an MXFP4 call's workspace, then
// the e4m3 path's own workspace.
struct Mxfp4Layout {
    size_t q8, k8, rest, total;
};

Mxfp4Layout mxfp4_layout(int rows, long long keys, int H, int D, size_t rest_bytes) {
    Mxfp4Layout L;
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    L.q8 = 0;
    L.k8 = up((size_t)rows * H * D);
    L.rest = L.k8 + up((size_t)keys * D);
    L.total = L.rest + rest_bytes;
    return L;
}

// Expand q and k into the workspace in one launch (after the checks every
// MXFP4 entry point makes).
idx_status mxfp4_expand_qk(const uint8_t* q, const uint8_t* q_sf, const uint8_t* k,
                           const uint8_t* k_sf, int rows, long long keys, int H, int D,
                           uint8_t* base, const Mxfp4Layout& L, const idx_options* opt,
                           void* stream) {
    if (!q || !q_sf || !k || !k_sf) return IDX_EINVAL;
    return mxfp4_launch(Mxfp4Segment{q, q_sf, (long long)rows * H, base + L.q8},
                        Mxfp4Segment{k, k_sf, keys, base + L.k8}, D, opt, stream);
}

}  // namespace

size_t idx_score_topk_mxfp4_workspace(int rows, long long keys, long long max_len, int H,
                                      int D, int topk, const idx_options* opt) {
    if (rows <= 0) return 0;
    const size_t rest = idx_score_topk_workspace(rows, keys, max_len, H, D, topk, IDX_FP8_E4M3, opt);
    return mxfp4_layout(rows, keys, H, D, rest).total;
}

idx_status idx_score_topk_mxfp4(const uint8_t* q, const uint8_t* q_sf, const uint8_t* k,
                                const uint8_t* k_sf, const float* k_scale, const float* w,
                                const int* ks, const int* ke, int rows, long long keys,
                                long long max_len, int H, int D, int topk, int* out_idx,
                                void* ws, size_t ws_bytes, const idx_options* opt,
                                void* stream) {
    if (topk < 1) return IDX_EINVAL;
    if (topk > kMaxTopk) return IDX_EUNSUPPORTED;
    // the e4m3 path's checks, on the packed arrays (same alignment rules)
    idx_status st = check_indexer_args(q, k, k_scale, w, ks, ke, rows, keys, H, D, IDX_FP8_E4M3);
    if (st != IDX_OK || rows == 0) return st;
    if (!out_idx) return IDX_EINVAL;
    const size_t rest = idx_score_topk_workspace(rows, keys, max_len, H, D, topk, IDX_FP8_E4M3, opt);
    const Mxfp4Layout L = mxfp4_layout(rows, keys, H, D, rest);
    if (!ws || ws_bytes < L.total) return IDX_EWORKSPACE;
    if (!aligned(ws, 256)) return IDX_EALIGN;
    uint8_t* base = static_cast<uint8_t*>(ws);
    st = mxfp4_expand_qk(q, q_sf, k, k_sf, rows, keys, H, D, base, L, opt, stream);
    if (st != IDX_OK) return st;
    return idx_score_topk(base + L.q8, base + L.k8, k_scale, w, ks, ke, rows, keys, max_len, H, D,
                          topk, IDX_FP8_E4M3, out_idx, base + L.rest, ws_bytes - L.rest, opt,
                          stream);
}

size_t idx_score_materialise_mxfp4_workspace(int rows, long long keys, int H, int D) {
    if (rows <= 0) return 0;
    return mxfp4_layout(rows, keys, H, D, 0).total;
}

idx_status idx_score_materialise_mxfp4(const uint8_t* q, const uint8_t* q_sf, const uint8_t* k,
                                       const uint8_t* k_sf, const float* k_scale,
                                       const float* w, const int* ks, const int* ke, int rows,
                                       long long keys, int H, int D, float* scores,
                                       long long row_stride, void* ws, size_t ws_bytes,
                                       const idx_options* opt, void* stream) {
    idx_status st = check_indexer_args(q, k, k_scale, w, ks, ke, rows, keys, H, D, IDX_FP8_E4M3);
    if (st != IDX_OK || rows == 0) return st;
    if (!scores || row_stride < 1) return IDX_EINVAL;
    const Mxfp4Layout L = mxfp4_layout(rows, keys, H, D, 0);
    if (!ws || ws_bytes < L.total) return IDX_EWORKSPACE;
    if (!aligned(ws, 256)) return IDX_EALIGN;
    uint8_t* base = static_cast<uint8_t*>(ws);
    st = mxfp4_expand_qk(q, q_sf, k, k_sf, rows, keys, H, D, base, L, opt, stream);
    if (st != IDX_OK) return st;
    return idx_score_materialise(base + L.q8, base + L.k8, k_scale, w, ks, ke, rows, keys, H, D,
                                 IDX_FP8_E4M3, scores, row_stride, opt, stream);
}

}  // extern "C"

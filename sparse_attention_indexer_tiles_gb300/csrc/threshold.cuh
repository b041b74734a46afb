// The sample threshold T_r of one row, computed by one warp (page 1,
// "Sampled Threshold": T_r is the t-th largest of the m scores of row r's
// strided sample, t = ceil(m * target * topk / len) with len the row's
// visible length, so that about target * topk keys of the row reach it).
// The scoring pass stores each sample as the top 16 bits of its order key;
// T_r is the exact t-th largest of those keys, by two 8-bit radix passes
// over a warp-private 256-bin histogram, and the emit pass takes every key at
// or above T_r << 16.  The threshold only steers how many candidates the slab
// receives (the slab top-k and the rescan make the result exact), so the
// 16-bit resolution costs nothing but a few extra candidates.
#pragma once

#include "common.cuh"
#include "plan.cuh"

namespace idx {

struct ThrParams {
    const int* ks;
    const int* ke;
    const uint16_t* samp;     // [rows, samp_stride] 16-bit sample keys
    long long samp_stride;
    long long nsamp;          // floor(keys / S)
    int S;
    int cap;
    int topk;
    float target;
    int rows_per_block;       // rows sharing one sample phase
    uint32_t phase_seed;
    RowPlan* plan;
    idx_stats* d_stats;
};

// The row's sample and its rank t, or false for rows without a sample
// threshold (every visible key a candidate).
struct SampleRow {
    const uint16_t* keys;
    uint32_t n, t;
};

IDX_DEVI bool sample_row(const ThrParams& p, int r, SampleRow* out) {
    const long long vks = p.ks[r], vke = p.ke[r];
    const long long len = vke - vks;
    const long long phase = hash32((uint32_t)(r / p.rows_per_block) ^ p.phase_seed) % p.S;
    const SampleSpan sp = sample_span(vks, vke, phase, p.S, p.nsamp);
    const long long n = sp.b - sp.a;
    if (len <= p.cap || n <= 0 || n > p.samp_stride) return false;
    double t = ceil((double)n * (double)p.target * (double)p.topk / (double)len);
    if (t < 1.0) t = 1.0;
    if (t > (double)n) t = (double)n;
    out->keys = p.samp + (long long)r * p.samp_stride;
    out->n = (uint32_t)n;
    out->t = (uint32_t)t;
    return true;
}

IDX_DEVI void set_plan_threshold(RowPlan* plan, uint32_t thr) {
    plan->thr = thr;
    plan->idx_cut = kAllIdx;
    plan->state = ST_MAIN;
}

// Sample keys one warp stages in shared memory (kThrStage x 16 bytes).
constexpr int kThrStage = 384;

// One warp: the threshold of row r into plan[r].  Rows with no sample
// threshold get thr = 0 (every visible key a candidate).  `max_n` > 0 leaves
// rows with longer samples alone (a CTA per row takes them) and returns false.
// `stage`, when given, is the warp's kThrStage-entry staging buffer.
IDX_DEVI bool warp_row_threshold(const ThrParams& p, int r, uint32_t* hist, uint32_t max_n = 0,
                                 uint4* stage = nullptr) {
    const int lane = threadIdx.x & 31;
    RowPlan* plan = p.plan + r;
    SampleRow sr;
    if (!sample_row(p, r, &sr)) {
        if (lane == 0) {
            set_plan_threshold(plan, 0u);
            const long long len = (long long)p.ke[r] - p.ks[r];
            if (p.d_stats && len > 0 && len <= p.cap) atomicAdd(&p.d_stats->emit_all_rows, 1);
        }
        return true;
    }
    if (max_n && sr.n > max_n) return false;
    // A sample of up to 8 * kThrStage keys is staged in shared memory once
    // (16-byte asynchronous copies of eight keys, all in flight at once; a
    // row's sample starts 16-byte aligned) and read there by every pass; a
    // longer one is read from global memory by each pass.
    const uint4* v4 = reinterpret_cast<const uint4*>(sr.keys);
    const uint32_t n8 = sr.n / 8;
    const bool staged = stage && n8 <= (uint32_t)kThrStage;
    if (staged) {
        for (uint32_t i = lane; i < n8; i += 32) cp_async16(stage + i, v4 + i);
        cp_async_wait_all();
        __syncwarp();
    }
    // fn(key) for every sample key this lane holds
    auto each_key = [&](auto fn) {
        auto do8 = [&](const uint4& x) {
            const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 8; ++h) fn((wd[h >> 1] >> (16 * (h & 1))) & 0xffffu);
        };
        if (staged) {
            for (uint32_t i = lane; i < n8; i += 32) do8(stage[i]);
        } else {
            // four loads per lane in flight, then the next four
            for (uint32_t base = lane; base < n8; base += 4 * 32) {
                uint4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    x[u] = base + u * 32 < n8 ? __ldcg(v4 + base + u * 32) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (base + u * 32 < n8) do8(x[u]);
            }
        }
        for (uint32_t e = n8 * 8 + lane; e < sr.n; e += 32) fn((uint32_t)sr.keys[e]);  // the odd tail
    };
    // The digit steps start below the bits every key shares (the sample's least
    // and largest key agree there): an 8-bit digit from the highest differing
    // bit down, then the bits below it among the keys of the chosen digit.  (A
    // fixed top byte would put nearly every key of a row, whose scores span a
    // few octaves, into one or two bins: serialised shared-memory atomics.)
    uint32_t mn = 0xffffu, mx = 0u;
    each_key([&](uint32_t k) {
        mn = k < mn ? k : mn;
        mx = k > mx ? k : mx;
    });
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    // the digit of bins [0, 256) that holds the need-th largest key
    uint32_t need = sr.t;
    auto pick = [&](uint32_t* digit) -> bool {
        __syncwarp();
        // lane l holds bins 255 - 8l ... 248 - 8l (from the largest keys down)
        uint32_t c[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = hist[255 - 8 * lane - j];
            local += c[j];
        }
        uint32_t incl = local;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t excl = incl - local;
        const uint32_t owner = __ballot_sync(0xffffffffu, excl < need && need <= incl);
        if (owner == 0u) return false;  // cannot happen: need never exceeds the keys left
        const int src = __ffs(owner) - 1;
        uint32_t dg = 0u, above = 0u;
        if (lane == src) {
            uint32_t cum = excl;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (cum + c[j] >= need) {
                    dg = 255u - 8u * (uint32_t)lane - (uint32_t)j;
                    above = cum;
                    break;
                }
                cum += c[j];
            }
        }
        *digit = __shfl_sync(0xffffffffu, dg, src);
        need -= __shfl_sync(0xffffffffu, above, src);
        __syncwarp();
        return true;
    };
    auto clear = [&] {
#pragma unroll
        for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
        __syncwarp();
    };
    bool ok = true;
    uint32_t T = mx;  // every key equal: the largest is the t-th largest
    if (mn != mx) {
        const int hb = 31 - __clz(mn ^ mx);
        const int w0 = hb + 1 < 8 ? hb + 1 : 8, s0 = hb + 1 - w0;
        const uint32_t m0 = (1u << w0) - 1u;
        clear();
        each_key([&](uint32_t k) { atomicAdd(&hist[(k >> s0) & m0], 1u); });
        uint32_t d0 = 0u, d1 = 0u;
        ok = pick(&d0);
        const uint32_t pre = ((mx >> (hb + 1)) << w0) | d0;  // the key's bits from s0 up
        T = pre << s0;
        if (ok && s0 > 0) {
            const uint32_t m1 = (1u << s0) - 1u;
            clear();
            each_key([&](uint32_t k) {
                if ((k >> s0) == pre) atomicAdd(&hist[k & m1], 1u);
            });
            ok = pick(&d1);
            T |= d1;
        }
    }
    // a failed pick leaves thr = 0: every key a candidate, the slab overflows
    // and the exact rescan takes the row
    if (lane == 0) set_plan_threshold(plan, ok ? T << 16 : 0u);
    return true;
}

}  // namespace idx

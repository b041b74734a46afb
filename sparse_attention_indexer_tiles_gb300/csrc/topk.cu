// Exact radix top-k kernels of libidx.
//
//  * topk_rows_kernel   one CTA per row of fp32 scores in global memory:
//                       12-bit histogram pass, a collection pass of the
//                       threshold bin into a shared tie buffer (or, when that
//                       bin holds more than kTieCap keys, another histogram
//                       pass over the row: the full-row rescan), then an
//                       ordered compaction pass that writes ascending indices.
//                       Page "[sglang] ROCm DSA Indexer Top-K 최적화": fp32
//                       coarse histogram, radix tie refinement, overflow
//                       rescan, single-block kernel per row.
//  * the same kernel in threshold mode returns only the exact t-th largest
//    key of each row; the fused path uses it on the strided score sample
//    (page "[sglang] logits를 쓰지 않는 top-k", section 2).
//  * cand_topk_kernel   one CTA per row of the candidate slab held in shared
//                       memory (page 1: the small top-k over ~2.25 x topk
//                       candidates); flags rows whose slab is short or
//                       overflowed for the exact rescan.
//  * fb_pick_kernel     one digit step of that rescan.
#include "plan.cuh"
#include "radix.cuh"
#include "topk.cuh"

namespace idx {

constexpr int kTieCap = 4096;

// A row of fp32 values addressed through an aligned float4 view: element p
// (0 <= p < n) sits in slot p + off of the 16-byte aligned base.  Reads may
// touch the up-to-12 bytes that share a 16-byte block with the row's first or
// last element; such a block never straddles a page.
struct RowView {
    const float4* base;
    int off;
    long long n;
    long long nvec;
};

IDX_DEVI RowView make_view(const float* p, long long n) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    RowView v;
    v.off = static_cast<int>((a & 15u) >> 2);
    v.base = reinterpret_cast<const float4*>(a - (a & 15u));
    v.n = n;
    v.nvec = (n + v.off + 3) >> 2;
    return v;
}

IDX_DEVI float4 ldg4(const float4* p) { return __ldg(p); }

// Histogram of `level`'s digit over the row's keys that carry `prefix`.
template <int THREADS, int UNROLL>
IDX_DEVI void hist_pass(const RowView& v, int level, uint32_t prefix, uint32_t* hist) {
    for (long long base = threadIdx.x; base < v.nvec; base += (long long)THREADS * UNROLL) {
        float4 f[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            f[u] = s < v.nvec ? ldg4(v.base + s) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const long long p = 4 * s + c - v.off;
                if (s < v.nvec && p >= 0 && p < v.n) {
                    const uint32_t key = fkey(e[c]);
                    if (has_prefix(key, level, prefix)) atomicAdd(&hist[digit_of(key, level)], 1u);
                }
            }
        }
    }
}

// Append (key, position) of every key carrying `prefix` at `level`.
template <int THREADS, int UNROLL>
IDX_DEVI void collect_pass(const RowView& v, int level, uint32_t prefix, uint32_t* tkey,
                           uint32_t* tpos, uint32_t* tcount) {
    for (long long base = threadIdx.x; base < v.nvec; base += (long long)THREADS * UNROLL) {
        float4 f[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            f[u] = s < v.nvec ? ldg4(v.base + s) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long s = base + (long long)u * THREADS;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const long long p = 4 * s + c - v.off;
                if (s < v.nvec && p >= 0 && p < v.n) {
                    const uint32_t key = fkey(e[c]);
                    if (has_prefix(key, level, prefix)) {
                        const uint32_t slot = atomicAdd(tcount, 1u);
                        if (slot < (uint32_t)kTieCap) {
                            tkey[slot] = key;
                            tpos[slot] = static_cast<uint32_t>(p);
                        }
                    }
                }
            }
        }
    }
}

struct Threshold {
    uint32_t key;   // exact threshold key T
    uint32_t need;  // keys equal to T that belong to the result (lowest indices first)
};

// Digit refinement over the shared tie buffer, from `level` down to the exact key.
template <int THREADS>
IDX_DEVI Threshold refine_in_smem(const uint32_t* tkey, uint32_t cnt, int level, uint32_t prefix,
                                  uint32_t need, uint32_t* hist, uint32_t* scratch) {
    for (int lev = level; lev <= 2; ++lev) {
        zero_shared<THREADS>(hist, kHistBins);
        __syncthreads();
        for (uint32_t e = threadIdx.x; e < cnt; e += THREADS) {
            const uint32_t key = tkey[e];
            if (has_prefix(key, lev, prefix)) atomicAdd(&hist[digit_of(key, lev)], 1u);
        }
        __syncthreads();
        const DigitPick pk = pick_digit<THREADS>(hist, 1 << digit_bits(lev), need, scratch);
        need -= pk.above;
        prefix = (prefix << digit_bits(lev)) | pk.digit;
    }
    return {prefix, need};
}

// Exact threshold of the k largest keys of a global row (k <= n).  Uses the
// tie buffer when the threshold bin fits, otherwise rescans the row digit by
// digit.  `rescans` counts the extra full-row histogram passes.
template <int THREADS, int UNROLL>
IDX_DEVI Threshold find_threshold(const RowView& v, uint32_t k, uint32_t* hist, uint32_t* tkey,
                                  uint32_t* tpos, uint32_t* scratch, int* rescans) {
    uint32_t prefix = 0, need = k;
    *rescans = 0;
    for (int level = 0; level <= 2; ++level) {
        zero_shared<THREADS>(hist, kHistBins);
        __syncthreads();
        hist_pass<THREADS, UNROLL>(v, level, prefix, hist);
        __syncthreads();
        const DigitPick pk = pick_digit<THREADS>(hist, 1 << digit_bits(level), need, scratch);
        need -= pk.above;
        prefix = (prefix << digit_bits(level)) | pk.digit;
        if (level == 2) return {prefix, need};
        if (pk.count <= (uint32_t)kTieCap) {
            uint32_t* tcount = scratch + 40;
            if (threadIdx.x == 0) *tcount = 0u;
            __syncthreads();
            collect_pass<THREADS, UNROLL>(v, level + 1, prefix, tkey, tpos, tcount);
            __syncthreads();
            const uint32_t cnt = min(*tcount, (uint32_t)kTieCap);
            __syncthreads();
            return refine_in_smem<THREADS>(tkey, cnt, level + 1, prefix, need, hist, scratch);
        }
        ++*rescans;
    }
    return {prefix, need};  // not reached
}

// Ordered compaction of the selected keys of a global row into out[0..k):
// key > T, plus the first `need` keys equal to T in index order.
template <int THREADS>
IDX_DEVI void ordered_output(const RowView& v, Threshold th, uint32_t k, int* out,
                             uint32_t* scratch) {
    uint32_t a_run = 0, e_run = 0;
    for (long long base = 0; base < v.nvec; base += THREADS) {
        const long long s = base + threadIdx.x;
        float4 f = s < v.nvec ? ldg4(v.base + s) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float e[4] = {f.x, f.y, f.z, f.w};
        uint32_t ab = 0, tb = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const long long p = 4 * s + c - v.off;
            if (s < v.nvec && p >= 0 && p < v.n) {
                const uint32_t key = fkey(e[c]);
                ab |= (key > th.key ? 1u : 0u) << c;
                tb |= (key == th.key ? 1u : 0u) << c;
            }
        }
        const uint32_t mine = (__popc(ab) << 16) | __popc(tb);
        uint32_t tot;
        const uint32_t incl = block_incl_scan<THREADS>(mine, scratch, &tot);
        const uint32_t excl = incl - mine;
        uint32_t a_b = a_run + (excl >> 16), e_b = e_run + (excl & 0xFFFFu);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int p = static_cast<int>(4 * s + c - v.off);
            if ((ab >> c) & 1u) {
                const uint32_t pos = a_b + min(e_b, th.need);
                if (pos < k) out[pos] = p;
                ++a_b;
            } else if ((tb >> c) & 1u) {
                if (e_b < th.need && a_b + e_b < k) out[a_b + e_b] = p;
                ++e_b;
            }
        }
        a_run += tot >> 16;
        e_run += tot & 0xFFFFu;
    }
}

// Shared memory of topk_rows_kernel: histogram, tie buffer (keys, positions),
// scan scratch.
constexpr size_t kRowsSmem = (kHistBins + 2 * kTieCap + 64) * sizeof(uint32_t);

template <int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS, 1)
topk_rows_kernel(TopkRowsArgs a) {
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t* hist = smem;
    uint32_t* tkey = hist + kHistBins;
    uint32_t* tpos = tkey + kTieCap;
    uint32_t* scratch = tpos + kTieCap;

    const int r = blockIdx.x;
    long long n, col0;
    uint32_t k;
    if (a.mode == TOPK_OUTPUT) {
        const long long ks = a.ks ? a.ks[r] : 0, ke = a.ke[r];
        n = ke - ks;
        col0 = a.relative ? 0 : ks;
        if (ks < 0 || n < 0 || col0 + n > a.row_len || n > 0x7fffffffll) {
            if (threadIdx.x == 0 && ke > ks) raise_status(a.d_status, IDX_DEV_RANGE);
            n = 0;
        }
        int* out = a.out + (long long)r * a.topk;
        if (n <= a.topk) {
            for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
            return;
        }
        k = static_cast<uint32_t>(a.topk);
    } else {
        // Threshold of the strided sample of row r: the t-th largest of its m
        // sample scores, t = ceil(m * target * topk / len) with len the row's
        // visible length, so that about target * topk keys reach it.
        RowPlan* plan = a.plan + r;
        const long long vks = a.vis_ks[r], vke = a.vis_ke[r];
        const long long len = vke - vks;
        const long long phase = hash32((uint32_t)(r / a.rows_per_block) ^ a.phase_seed) % a.S;
        const SampleSpan sp = sample_span(vks, vke, phase, a.S, a.nsamp);
        n = sp.b - sp.a;
        col0 = 0;
        if (len <= a.cap || n <= 0 || n > a.row_len) {
            if (threadIdx.x == 0) {
                plan->thr = 0u;  // every visible key becomes a candidate
                plan->quota = 0;
                plan->state = ST_MAIN;
                plan->count = 0;
                if (a.d_stats && len > 0 && len <= a.cap) atomicAdd(&a.d_stats->emit_all_rows, 1);
            }
            return;
        }
        double t = ceil((double)n * (double)a.target * (double)a.topk / (double)len);
        if (t < 1.0) t = 1.0;
        if (t > (double)n) t = (double)n;
        k = static_cast<uint32_t>(t);
    }

    const RowView v = make_view(a.scores + (long long)r * a.row_stride + col0, n);
    int rescans = 0;
    const Threshold th = find_threshold<THREADS, UNROLL>(v, k, hist, tkey, tpos, scratch, &rescans);
    if (rescans && threadIdx.x == 0 && a.d_stats) atomicAdd(&a.d_stats->tie_rescan_rows, 1);

    if (a.mode == TOPK_OUTPUT) {
        ordered_output<THREADS>(v, th, k, a.out + (long long)r * a.topk, scratch);
    } else if (threadIdx.x == 0) {
        RowPlan* plan = a.plan + r;
        plan->thr = th.key;
        plan->quota = 0;
        plan->state = ST_MAIN;
        plan->count = 0;
    }
}

// ---------------------------------------------------------------- slab

// Threshold of the k largest among `cnt` keys in shared memory.
template <int THREADS>
IDX_DEVI Threshold smem_threshold(const uint32_t* keys, uint32_t cnt, uint32_t k, uint32_t* hist,
                                  uint32_t* scratch) {
    return refine_in_smem<THREADS>(keys, cnt, 0, 0u, k, hist, scratch);
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS)
cand_topk_kernel(CandArgs a) {
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t* hist = smem;
    uint32_t* scratch = hist + kHistBins;
    uint32_t* keys = scratch + 64;
    int32_t* idxs = reinterpret_cast<int32_t*>(keys + a.cap);

    const int r = blockIdx.x;
    RowPlan* plan = a.plan + r;
    const long long n = (long long)a.ke[r] - (long long)a.ks[r];
    int* out = a.out + (long long)r * a.topk;
    // one read of the row's plan, shared by the block before anyone writes it
    if (threadIdx.x == 0) {
        scratch[48] = (uint32_t)plan->state;
        scratch[49] = (uint32_t)plan->count;
    }
    __syncthreads();
    const int state = (int)scratch[48];

    if (a.fallback) {
        if (state != ST_EMIT) return;
    } else {
        if (n <= a.topk) {
            for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = i < n ? i : -1;
            if (threadIdx.x == 0) plan->state = ST_DONE;
            return;
        }
    }
    const int count = (int)scratch[49];
    if (threadIdx.x == 0 && a.d_stats && !a.fallback) atomicMax(&a.d_stats->max_count, count);
    if (count < a.topk || count > a.cap) {
        if (!a.fallback && !a.fb_hist) {
            // no rescan storage: the row was longer than the max_len the
            // workspace was sized for
            for (int i = threadIdx.x; i < a.topk; i += THREADS) out[i] = -1;
            if (threadIdx.x == 0) {
                raise_status(a.d_status, IDX_DEV_RANGE);
                plan->state = ST_DONE;
            }
        } else if (!a.fallback) {
            // the sampled threshold missed: exact full-row rescan
            for (int i = threadIdx.x; i < kHistBins; i += THREADS)
                a.fb_hist[(long long)r * kHistBins + i] = 0u;
            if (threadIdx.x == 0) {
                plan->state = ST_HIST;
                plan->level = 0;
                plan->prefix = 0u;
                plan->above = 0;
                if (a.d_stats) {
                    atomicAdd(count > a.cap ? &a.d_stats->overflow_rows : &a.d_stats->short_rows, 1);
                    atomicAdd(&a.d_stats->fallback_rows, 1);
                }
            }
        } else if (threadIdx.x == 0) {
            raise_status(a.d_status, IDX_DEV_STATE);
            plan->state = ST_DONE;
        }
        return;
    }

    const float* ss = a.slab_s + (long long)r * a.cap;
    const int* si = a.slab_i + (long long)r * a.cap;
    for (int e = threadIdx.x; e < count; e += THREADS) {
        keys[e] = fkey(ss[e]);
        idxs[e] = si[e];
    }
    __syncthreads();
    const Threshold th = smem_threshold<THREADS>(keys, count, a.topk, hist, scratch);

    // ordered compaction over the slab, which is in ascending key order
    uint32_t a_run = 0, e_run = 0;
    for (int base = 0; base < count; base += THREADS * 4) {
        uint32_t ab = 0, tb = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int e = base + threadIdx.x * 4 + c;
            if (e < count) {
                ab |= (keys[e] > th.key ? 1u : 0u) << c;
                tb |= (keys[e] == th.key ? 1u : 0u) << c;
            }
        }
        const uint32_t mine = (__popc(ab) << 16) | __popc(tb);
        uint32_t tot;
        const uint32_t incl = block_incl_scan<THREADS>(mine, scratch, &tot);
        const uint32_t excl = incl - mine;
        uint32_t a_b = a_run + (excl >> 16), e_b = e_run + (excl & 0xFFFFu);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int e = base + threadIdx.x * 4 + c;
            if ((ab >> c) & 1u) {
                const uint32_t pos = a_b + min(e_b, th.need);
                if (pos < (uint32_t)a.topk) out[pos] = idxs[e];
                ++a_b;
            } else if ((tb >> c) & 1u) {
                if (e_b < th.need && a_b + e_b < (uint32_t)a.topk) out[a_b + e_b] = idxs[e];
                ++e_b;
            }
        }
        a_run += tot >> 16;
        e_run += tot & 0xFFFFu;
    }
    if (threadIdx.x == 0) plan->state = ST_DONE;
}

// One digit step of the exact rescan for rows in ST_HIST at `level`.
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
fb_pick_kernel(FbPickArgs a) {
    __shared__ uint32_t hist[kHistBins];
    __shared__ uint32_t scratch[64];
    const int r = blockIdx.x;
    RowPlan* plan = a.plan + r;
    if (plan->state != ST_HIST || plan->level != a.level) return;
    const int level = a.level;
    const int nb = 1 << digit_bits(level);
    uint32_t* gh = a.fb_hist + (long long)r * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += THREADS) hist[i] = i < nb ? gh[i] : 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < nb; i += THREADS) gh[i] = 0u;  // ready for the next level
    const uint32_t above = static_cast<uint32_t>(plan->above);
    const uint32_t need = static_cast<uint32_t>(a.topk) - above;
    const DigitPick pk = pick_digit<THREADS>(hist, nb, need, scratch);
    if (threadIdx.x == 0) {
        const uint32_t above_new = above + pk.above;
        const uint32_t prefix = (plan->prefix << digit_bits(level)) | pk.digit;
        if (above_new + pk.count <= (uint32_t)a.cap) {
            plan->thr = prefix << digit_shift(level);
            plan->quota = 0;
            plan->state = ST_EMIT;
        } else if (level < 2) {
            plan->prefix = prefix;
            plan->above = static_cast<int32_t>(above_new);
            plan->level = level + 1;
        } else {
            plan->thr = prefix;  // exact key; ties taken in index order
            plan->quota = a.topk - static_cast<int32_t>(above_new);
            plan->state = ST_EMIT;
        }
    }
}

// ------------------------------------------------------------ launchers

cudaError_t launch_topk_rows(const TopkRowsArgs& a, cudaStream_t s) {
    constexpr int T = 1024, U = 4;
    auto kern = topk_rows_kernel<T, U>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRowsSmem);
    if (e != cudaSuccess) return e;
    if (a.rows == 0) return cudaSuccess;
    kern<<<a.rows, T, kRowsSmem, s>>>(a);
    return cudaGetLastError();
}

size_t cand_smem_bytes(int cap) {
    return (kHistBins + 64) * sizeof(uint32_t) + (size_t)cap * 2 * sizeof(uint32_t);
}

cudaError_t launch_cand_topk(const CandArgs& a, cudaStream_t s) {
    constexpr int T = 512;
    auto kern = cand_topk_kernel<T>;
    const size_t sm = cand_smem_bytes(a.cap);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (a.rows == 0) return cudaSuccess;
    kern<<<a.rows, T, sm, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fb_pick(const FbPickArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    fb_pick_kernel<256><<<a.rows, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace idx

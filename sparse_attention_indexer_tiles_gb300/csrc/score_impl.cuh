// The tcgen05 scoring kernel of libidx (sm_103a).
//
// Page "[sglang] logits를 쓰지 않는 top-k", section 1: a KV tile is the A
// operand (M = keys) of the tensor-core MMA, the accumulator lives in TMEM,
// every epilogue thread owns one key of the tile and reduces the heads in
// registers.  Here:
//   A = 128 keys x D        (TMA, 128/64-byte swizzle, a ring of stages)
//   B = 256 (row, head) x D (TMA, loaded once: rows_per_block = 256 / H rows)
//   D = 128 x 256 fp32 in TMEM, double buffered (2 x 256 columns), so the
//       epilogue of tile t overlaps the MMA of tile t + 1.
// Warp roles (12 warps): 0 = TMA producer, 1 = TMEM owner + MMA issuer,
// 4..11 = epilogue (two warpgroups, each owning half of the block's rows; a
// warp reads the TMEM lane quarter 32 * (warp % 4)).
//
// Score of (row, key), summed over heads in ascending order in fp32:
//   s = k_scale[key] * sum_h fma(w[row,h], max(acc[h], 0), .)
// Every mode runs the same arithmetic, so the fused path compares exactly the
// scores that the materialising baseline writes.
#pragma once

#include "plan.cuh"
#include "radix.cuh"
#include "score.cuh"

namespace idx {

template <int DT, int H, int RB>
struct ScoreCfg {
    static constexpr int R = 256 / H;                       // rows per CTA
    static constexpr int N = 256;                           // MMA N
    static constexpr int M = 128;                           // keys per tile
    static constexpr int CHUNK_B = RB >= 128 ? 128 : RB;    // swizzle width
    static constexpr int NCHUNK = RB / CHUNK_B;             // 128-byte slices of a row
    static constexpr int ELEM = DT == IDX_BF16 ? 2 : 1;
    static constexpr int CHUNK_ELEMS = CHUNK_B / ELEM;
    static constexpr int KSTEP_B = 32;                      // bytes of K per MMA
    static constexpr int KSTEPS = CHUNK_B / KSTEP_B;
    static constexpr int A_BYTES = M * RB;
    static constexpr int A_CHUNK = M * CHUNK_B;
    static constexpr int B_BYTES = N * RB;
    static constexpr int B_CHUNK = N * CHUNK_B;
    static constexpr int NS = RB >= 256 ? 4 : (RB == 128 ? 8 : 12);
    static constexpr int EPI_WARPS = 16;                    // 4 per SM sub-partition
    static constexpr int NGROUPS = EPI_WARPS / 4;           // warps sharing a lane quarter
    static constexpr int RG = R / NGROUPS;                  // rows per epilogue warp
    static constexpr int THREADS = 32 * (4 + EPI_WARPS);
    static constexpr uint32_t IDESC = instr_desc(DT == IDX_BF16 ? 1u : 0u, M, N);
    // shared memory carve (offsets from a 1024-byte aligned base)
    static constexpr int OFF_B = 0;
    static constexpr int OFF_A = B_BYTES;
    static constexpr int OFF_BAR = OFF_A + NS * A_BYTES;
    static constexpr int NBAR = 2 * NS + 5 + NGROUPS;
    static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
    static constexpr int OFF_W = (OFF_TSLOT + 16 + 15) / 16 * 16;
    static constexpr int OFF_META = OFF_W + R * H * 4;
    static constexpr int META_WORDS = 12;                   // per row
    static constexpr int OFF_BAL = OFF_META + R * META_WORDS * 4;
    static constexpr int BAL_WORDS = 2 * NGROUPS * RG * 4 * 2;  // parity x group x row x warp x {above, tie}
    static constexpr int OFF_MISC = OFF_BAL + BAL_WORDS * 4;
    static constexpr int SMEM_USED = OFF_MISC + 64;
    // at least ~120 KB so that one CTA owns an SM (and its 512 TMEM columns)
    static constexpr int SMEM_ALLOC = (SMEM_USED + 1024 > 122880 ? SMEM_USED + 1024 : 122880);
};

// per-row metadata words in shared memory
enum : int {
    MW_ACTIVE = 0, MW_KS_LO, MW_KS_HI, MW_KE_LO, MW_KE_HI, MW_THR, MW_QUOTA, MW_PREFIX,
    MW_SA_LO, MW_SA_HI, MW_SB_LO, MW_SB_HI
};

IDX_DEVI long long meta_ll(const int* m, int lo) {
    return (long long)(((unsigned long long)(uint32_t)m[lo + 1] << 32) | (uint32_t)m[lo]);
}
IDX_DEVI void set_meta_ll(int* m, int lo, long long v) {
    m[lo] = (int)(uint32_t)((unsigned long long)v & 0xffffffffull);
    m[lo + 1] = (int)(uint32_t)((unsigned long long)v >> 32);
}

#ifndef IDX_EPI
#define IDX_EPI 5
#endif
#ifndef IDX_ONE_WAIT
#define IDX_ONE_WAIT 0
#endif
#ifndef IDX_SETMAXNREG
#define IDX_SETMAXNREG 0
#endif

// Per-head weights are stored pre-multiplied by this factor per head parity.
__host__ __device__ constexpr float epi_w_factor(int h) {
    return (IDX_EPI == 3 && (h & 1)) ? 0.5f : 1.0f;
}
// ... and the head sum is multiplied by this factor (with the key scale).
__host__ __device__ constexpr float epi_post() {
    return (IDX_EPI == 0 || IDX_EPI == 2 || IDX_EPI == 5) ? 0.5f : 1.0f;
}

// sum_h w[h] * ReLU(acc[h]) for one (row, key): the TMEM row of this thread,
// H consecutive columns from taddr, up to a constant factor (epi_post).
// Eight partial sums in a fixed combine order break the dependency chain.
template <int H>
IDX_DEVI float head_reduce(uint32_t taddr, const float* wr) {
    constexpr int CH = H >= 32 ? 32 : H;
#if IDX_EPI >= 3
    float2 acc2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc2[u] = make_float2(0.f, 0.f);
#else
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
#endif
#if IDX_ONE_WAIT
    float vv[H];
    if constexpr (CH == 32) {
#pragma unroll
        for (int c = 0; c < H / 32; ++c) tmem_ld32(taddr + c * 32, vv + c * 32);
    } else if constexpr (CH == 16) {
        tmem_ld16(taddr, vv);
    } else {
        tmem_ld8(taddr, vv);
    }
    tmem_ld_wait();  // one TMEM round trip per (row, tile)
#endif
#pragma unroll
    for (int c = 0; c < H / CH; ++c) {
#if IDX_ONE_WAIT
        const float* v = vv + c * CH;
#else
        float v[CH];
        if constexpr (CH == 32) tmem_ld32(taddr + c * 32, v);
        else if constexpr (CH == 16) tmem_ld16(taddr, v);
        else tmem_ld8(taddr, v);
        tmem_ld_wait();
#endif
#if IDX_EPI == 0
#pragma unroll
        for (int h = 0; h < CH; ++h)
            acc[h & 7] = fmaf(wr[c * CH + h], v[h] + fabsf(v[h]), acc[h & 7]);
#else
        const float4* w4 = reinterpret_cast<const float4*>(wr + c * CH);
#pragma unroll
        for (int h4 = 0; h4 < CH / 4; ++h4) {
            const float4 wq = w4[h4];
            float t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float x = v[4 * h4 + u];
#if IDX_EPI == 1 || IDX_EPI == 4
                t[u] = fmaxf(x, 0.f);
#elif IDX_EPI == 2 || IDX_EPI == 5
                t[u] = x + fabsf(x);
#else
                t[u] = (u & 1) ? x + fabsf(x) : fmaxf(x, 0.f);
#endif
            }
#if IDX_EPI >= 3
            acc2[(2 * h4) & 3] = __ffma2_rn(make_float2(wq.x, wq.y), make_float2(t[0], t[1]),
                                            acc2[(2 * h4) & 3]);
            acc2[(2 * h4 + 1) & 3] = __ffma2_rn(make_float2(wq.z, wq.w), make_float2(t[2], t[3]),
                                                acc2[(2 * h4 + 1) & 3]);
#else
            acc[(4 * h4 + 0) & 7] = fmaf(wq.x, t[0], acc[(4 * h4 + 0) & 7]);
            acc[(4 * h4 + 1) & 7] = fmaf(wq.y, t[1], acc[(4 * h4 + 1) & 7]);
            acc[(4 * h4 + 2) & 7] = fmaf(wq.z, t[2], acc[(4 * h4 + 2) & 7]);
            acc[(4 * h4 + 3) & 7] = fmaf(wq.w, t[3], acc[(4 * h4 + 3) & 7]);
#endif
        }
#endif
    }
#if IDX_EPI >= 3
    return ((acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y)) +
           ((acc2[2].x + acc2[2].y) + (acc2[3].x + acc2[3].y));
#else
    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
#endif
}

template <int DT, int H, int RB>
__global__ void __launch_bounds__(ScoreCfg<DT, H, RB>::THREADS, 1)
score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ ScoreArgs a) {
    using C = ScoreCfg<DT, H, RB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::NS;
    uint64_t* accf = bars + 2 * C::NS;
    uint64_t* acce = accf + 2;
    uint64_t* qfull = acce + 2;
    uint64_t* exch = qfull + 1;  // [NGROUPS]: the 4 warps of one row group, once per tile
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_TSLOT);
    float* w_s = reinterpret_cast<float*>(smem + C::OFF_W);
    int* meta = reinterpret_cast<int*>(smem + C::OFF_META);
    uint32_t* bal = reinterpret_cast<uint32_t*>(smem + C::OFF_BAL);
    long long* misc_ll = reinterpret_cast<long long*>(smem + C::OFF_MISC);  // [0] t0, [1] ntiles
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
    int* misc_i = reinterpret_cast<int*>(smem + C::OFF_MISC + 20);          // [0] phase

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * C::R;
    const int mode = a.mode;
    const long long phase =
        mode == SM_SAMPLE ? (long long)(hash32((uint32_t)blockIdx.x ^ a.phase_seed) % (uint32_t)a.S) : 0;

    // ---- per-row metadata
    if (tid < C::R) {
        int* m = meta + tid * C::META_WORDS;
        const int r = r0 + tid;
        long long ks = 0, ke = 0;
        int active = 0;
        uint32_t thr = 0, prefix = 0;
        int quota = 0;
        if (r < a.rows) {
            ks = a.ks[r];
            ke = a.ke[r];
            if (ks < 0 || ke > a.keys || ks > ke) {
                if (ke > ks || ks < 0) raise_status(a.d_status, IDX_DEV_RANGE);
                ks = ke = 0;
            }
            const long long n = ke - ks;
            switch (mode) {
                case SM_MATERIALISE:
                    active = n > 0;
                    if (n > a.out_stride) {
                        raise_status(a.d_status, IDX_DEV_RANGE);
                        active = 0;
                    }
                    break;
                case SM_SAMPLE: active = n > a.cap; break;
                case SM_EMIT:
                    // rows that see at most cap keys emit every key (page 1,
                    // section 1: blocks of short rows store every score)
                    active = n > a.topk;
                    if (active && n > a.cap) thr = a.plan[r].thr;
                    break;
                case SM_FB_HIST: {
                    const RowPlan p = a.plan[r];
                    active = n > 0 && p.state == ST_HIST && p.level == a.level;
                    prefix = p.prefix;
                } break;
                case SM_FB_EMIT: {
                    const RowPlan p = a.plan[r];
                    active = n > 0 && p.state == ST_EMIT;
                    thr = p.thr;
                    quota = p.quota;
                } break;
            }
        }
        m[MW_ACTIVE] = active;
        set_meta_ll(m, MW_KS_LO, ks);
        set_meta_ll(m, MW_KE_LO, ke);
        m[MW_THR] = (int)thr;
        m[MW_QUOTA] = quota;
        m[MW_PREFIX] = (int)prefix;
        if (mode == SM_SAMPLE) {
            const SampleSpan sp = sample_span(ks, ke, phase, a.S, a.nsamp);
            if (active && sp.b - sp.a > a.samp_stride) {
                raise_status(a.d_status, IDX_DEV_RANGE);  // longer than max_len
                active = 0;
                m[MW_ACTIVE] = 0;
            }
            set_meta_ll(m, MW_SA_LO, sp.a);
            set_meta_ll(m, MW_SB_LO, sp.b);
        } else {
            set_meta_ll(m, MW_SA_LO, ks);
            set_meta_ll(m, MW_SB_LO, ke);
        }
    }
    for (int i = tid; i < C::R * H; i += C::THREADS) {
        const long long r = r0 + i / H;
        w_s[i] = r < a.rows ? a.w[(long long)r0 * H + i] * epi_w_factor(i % H) : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        long long lo = 0x7fffffffffffffffll, hi = -1;
        for (int j = 0; j < C::R; ++j) {
            const int* m = meta + j * C::META_WORDS;
            if (!m[MW_ACTIVE]) continue;
            const long long sa = meta_ll(m, MW_SA_LO), sb = meta_ll(m, MW_SB_LO);
            if (sb <= sa) continue;
            lo = sa < lo ? sa : lo;
            hi = sb > hi ? sb : hi;
        }
        long long t0 = 0, nt = 0;
        if (hi > lo) {
            t0 = lo / C::M;
            nt = (hi + C::M - 1) / C::M - t0;
        }
        misc_ll[0] = t0;
        misc_ll[1] = nt;
        *abort_flag = 0;
        misc_i[0] = (int)phase;
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], C::EPI_WARPS);
        }
        mbar_init(qfull, 1);
        for (int i = 0; i < C::NGROUPS; ++i) mbar_init(&exch[i], 4);
        fence_barrier_init();
    }
    __syncthreads();
    const long long t0 = misc_ll[0];
    const long long ntiles = misc_ll[1];
    if (ntiles == 0) return;  // no active row in this block

    if (warp == 1) {
        __syncwarp();
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

#if IDX_SETMAXNREG
    // launch: 640 threads x 96 registers = 61440.  Warpgroup 0 (producer, MMA)
    // keeps 40, the four epilogue warpgroups take 104: 128*40 + 512*104 = 58368.
    if (warp < 4) setmaxnreg_dec<40>();
    else setmaxnreg_inc<104>();
#endif
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(mode == SM_SAMPLE ? (const void*)&tm_ks : (const void*)&tm_k);
            mbar_arrive_expect_tx(qfull, C::B_BYTES);
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c)
                tma_load_2d(smem + C::OFF_B + c * C::B_CHUNK, &tm_q, qfull, c * C::CHUNK_ELEMS,
                            r0 * H);
            long long issued = 0;
            for (long long i = 0; i < ntiles; ++i) {
                const int s = (int)(i % C::NS);
                const uint32_t use = (uint32_t)(i / C::NS);
                if (i >= C::NS && !mbar_wait(&empty[s], (use & 1u) ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    raise_status(a.d_status, IDX_DEV_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], C::A_BYTES);
                const int row0 = (int)((t0 + i) * C::M);
#pragma unroll
                for (int c = 0; c < C::NCHUNK; ++c) {
                    uint8_t* dst = smem + C::OFF_A + s * C::A_BYTES + c * C::A_CHUNK;
                    if (mode == SM_SAMPLE)
                        tma_load_3d(dst, &tm_ks, &full[s], c * C::CHUNK_ELEMS, (int)phase, row0);
                    else
                        tma_load_2d(dst, &tm_k, &full[s], c * C::CHUNK_ELEMS, row0);
                }
                issued = i + 1;
            }
            // do not leave with copies in flight: wait (bounded) for the last stages
            for (long long i = issued > C::NS ? issued - C::NS : 0; i < issued; ++i)
                mbar_wait(&full[i % C::NS], (uint32_t)((i / C::NS) & 1), nullptr, 1ll << 28);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a_base = smem_u32(smem + C::OFF_A);
            const uint32_t b_base = smem_u32(smem + C::OFF_B);
            bool ok = mbar_wait(qfull, 0, abort_flag);
            long long issued = 0;
            for (long long i = 0; ok && i < ntiles; ++i) {
                const int s = (int)(i % C::NS);
                const int b = (int)(i & 1);
                if (i >= 2 && !mbar_wait(&acce[b], (uint32_t)(((i >> 1) & 1) ^ 1), abort_flag)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&full[s], (uint32_t)((i / C::NS) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * C::N);
#pragma unroll
                for (int c = 0; c < C::NCHUNK; ++c) {
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS; ++kk) {
                        const uint64_t ad =
                            smem_desc(a_base + s * C::A_BYTES + c * C::A_CHUNK + kk * C::KSTEP_B,
                                      C::CHUNK_B);
                        const uint64_t bd =
                            smem_desc(b_base + c * C::B_CHUNK + kk * C::KSTEP_B, C::CHUNK_B);
                        const uint32_t acc = (c | kk) != 0;
                        if (DT == IDX_BF16)
                            mma_bf16(d, ad, bd, C::IDESC, acc);
                        else
                            mma_fp8(d, ad, bd, C::IDESC, acc);
                    }
                }
                mma_commit(&empty[s]);
                mma_commit(&accf[b]);
                issued = i + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                raise_status(a.d_status, IDX_DEV_TIMEOUT);
            }
            // wait (bounded) until the tensor core is done with TMEM
            if (issued > 0)
                mbar_wait(&accf[(issued - 1) & 1], (uint32_t)(((issued - 1) >> 1) & 1), nullptr,
                          1ll << 28);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;              // TMEM lane quarter
        const int grp = (warp - 4) >> 2;     // row group: rows [grp * RG, (grp + 1) * RG)
        const uint32_t lt = (1u << lane) - 1u;
        int cnt[C::RG];
        int ties[C::RG];
        // per-row visible range [lo, hi) in tile index space (sample indices in
        // SM_SAMPLE), empty for inactive rows, and the emit threshold key
        int rlo[C::RG], rhi[C::RG];
        uint32_t rthr[C::RG];
#pragma unroll
        for (int j = 0; j < C::RG; ++j) {
            cnt[j] = ties[j] = 0;
            const int* m = meta + (grp * C::RG + j) * C::META_WORDS;
            const bool span = mode == SM_MATERIALISE || mode == SM_SAMPLE;
            rlo[j] = m[MW_ACTIVE] ? (int)meta_ll(m, span ? MW_SA_LO : MW_KS_LO) : 0;
            rhi[j] = m[MW_ACTIVE] ? (int)meta_ll(m, span ? MW_SB_LO : MW_KE_LO) : 0;
            rthr[j] = (uint32_t)m[MW_THR];
        }

        // per-key scale of the next tile, loaded one tile ahead
        auto scale_of = [&](long long t) -> float {
            const long long ki = (t0 + t) * C::M + q * 32 + lane;
            const long long kk = mode == SM_SAMPLE ? phase + (long long)a.S * ki : ki;
            const bool ok = t < ntiles && (mode == SM_SAMPLE ? ki < a.nsamp : kk < a.keys);
            return ok ? __ldg(a.k_scale + kk) : 0.f;
        };
        float next_scale = scale_of(0);
        for (long long i = 0; i < ntiles; ++i) {
            const int b = (int)(i & 1);
            const float cur_scale = next_scale;
            next_scale = scale_of(i + 1);
            // warp-uniform outcome: the TMEM loads below are .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(&accf[b], (uint32_t)((i >> 1) & 1), abort_flag))) {
                *abort_flag = 1;
                if (lane == 0) raise_status(a.d_status, IDX_DEV_TIMEOUT);
                break;
            }
            tc_fence_after();
            const long long kidx = (t0 + i) * C::M + q * 32 + lane;  // key, or sample index
            const float post_scale = epi_post() * cur_scale;

            float sc[C::RG];
#pragma unroll
            for (int j = 0; j < C::RG; ++j) {
                const int rr = grp * C::RG + j;
                const uint32_t taddr =
                    tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::N + rr * H);
                sc[j] = head_reduce<H>(taddr, w_s + rr * H) * post_scale;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);

            const int k32 = (int)kidx;
            if (mode == SM_MATERIALISE || mode == SM_SAMPLE) {
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int off = k32 - rlo[j];
                    if ((uint32_t)off < (uint32_t)(rhi[j] - rlo[j])) {
                        const long long r = r0 + grp * C::RG + j;
                        if (mode == SM_MATERIALISE)
                            a.out[r * a.out_stride + off] = sc[j];
                        else
                            a.samp[r * a.samp_stride + off] = sc[j];
                    }
                }
            } else if (mode == SM_EMIT) {
                // main pass: each warp appends its keys >= T_r, in key order, to
                // its own run q of the row's slab; no cross-warp traffic
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int off = k32 - rlo[j];
                    const bool hit = (uint32_t)off < (uint32_t)(rhi[j] - rlo[j]) &&
                                     fkey(sc[j]) >= rthr[j];
                    const uint32_t A = __ballot_sync(0xffffffffu, hit);
                    if (A) {
                        const int pos = cnt[j] + __popc(A & lt);
                        if (hit && pos < a.cap_q) {
                            const long long slot =
                                ((long long)(r0 + grp * C::RG + j) * 4 + q) * a.cap_q + pos;
                            a.slab_s[slot] = sc[j];
                            a.slab_i[slot] = off;
                        }
                        cnt[j] += __popc(A);
                    }
                }
            } else if (mode == SM_FB_HIST) {
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int rr = grp * C::RG + j;
                    const int* m = meta + rr * C::META_WORDS;
                    const long long lo = meta_ll(m, MW_KS_LO), hi = meta_ll(m, MW_KE_LO);
                    const uint32_t kb = fkey(sc[j]);
                    const bool valid = m[MW_ACTIVE] && kidx >= lo && kidx < hi &&
                                       has_prefix(kb, a.level, (uint32_t)m[MW_PREFIX]);
                    const uint32_t dg = digit_of(kb, a.level);
                    const uint32_t same = __match_any_sync(0xffffffffu, valid ? dg : (0x80000000u | lane));
                    if (valid && lane == __ffs(same) - 1)
                        atomicAdd(&a.fb_hist[(long long)(r0 + rr) * kHistBins + dg], (uint32_t)__popc(same));
                }
            } else {
                // rescan re-emission (SM_FB_EMIT): one run per row in key order,
                // ties at the exact threshold limited to the first `quota`
                const int par = (int)(i & 1);
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int rr = grp * C::RG + j;
                    const int* m = meta + rr * C::META_WORDS;
                    const long long lo = meta_ll(m, MW_KS_LO), hi = meta_ll(m, MW_KE_LO);
                    const bool vis = m[MW_ACTIVE] && kidx >= lo && kidx < hi;
                    const uint32_t thr = (uint32_t)m[MW_THR];
                    const int quota = m[MW_QUOTA];
                    const uint32_t kb = fkey(sc[j]);
                    const bool above = vis && (quota > 0 ? kb > thr : kb >= thr);
                    const bool tie = vis && quota > 0 && kb == thr;
                    const uint32_t A = __ballot_sync(0xffffffffu, above);
                    const uint32_t T = __ballot_sync(0xffffffffu, tie);
                    if (lane == 0) {
                        uint32_t* e = bal + (((par * C::NGROUPS + grp) * C::RG + j) * 4 + q) * 2;
                        e[0] = A;
                        e[1] = T;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&exch[grp]);
                if (!__all_sync(0xffffffffu, mbar_wait(&exch[grp], (uint32_t)(i & 1), abort_flag))) {
                    *abort_flag = 1;
                    if (lane == 0) raise_status(a.d_status, IDX_DEV_TIMEOUT);
                    break;
                }
                const int run_cap = 4 * a.cap_q;
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int rr = grp * C::RG + j;
                    const int* m = meta + rr * C::META_WORDS;
                    const int quota = m[MW_QUOTA];
                    const uint32_t* e = bal + (((par * C::NGROUPS + grp) * C::RG + j) * 4) * 2;
                    int ab = 0, tb = 0, ta = 0, tt = 0;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const int pa = __popc(e[2 * qq]), pt = __popc(e[2 * qq + 1]);
                        if (qq < q) { ab += pa; tb += pt; }
                        ta += pa;
                        tt += pt;
                    }
                    if (ta == 0 && tt == 0) continue;
                    const uint32_t A = e[2 * q], T = e[2 * q + 1];
                    const int room = quota > ties[j] ? quota - ties[j] : 0;
                    const int above_before = ab + __popc(A & lt);
                    const int ties_before = tb + __popc(T & lt);
                    long long pos = -1;
                    if ((A >> lane) & 1u)
                        pos = cnt[j] + above_before + (ties_before < room ? ties_before : room);
                    else if (((T >> lane) & 1u) && ties_before < room)
                        pos = cnt[j] + above_before + ties_before;
                    if (pos >= 0 && pos < run_cap) {
                        const long long slot = (long long)(r0 + rr) * run_cap + pos;
                        a.slab_s[slot] = sc[j];
                        a.slab_i[slot] = (int)(kidx - meta_ll(m, MW_KS_LO));
                    }
                    const int took = tt < room ? tt : room;
                    cnt[j] += ta + took;
                    ties[j] += took;
                }
            }
        }
        if (lane == 0 && (mode == SM_EMIT || (mode == SM_FB_EMIT && q == 0))) {
#pragma unroll
            for (int j = 0; j < C::RG; ++j) {
                const int rr = grp * C::RG + j;
                const int* m = meta + rr * C::META_WORDS;
                if (!m[MW_ACTIVE]) continue;
                int* rc = a.run_cnt + (long long)(r0 + rr) * 4;
                if (mode == SM_EMIT) {
                    rc[q] = cnt[j];
                } else {
                    rc[0] = cnt[j];
                    rc[1] = rc[2] = rc[3] = 0;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace idx

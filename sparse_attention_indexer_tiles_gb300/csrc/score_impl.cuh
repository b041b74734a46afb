// The tcgen05 scoring kernel of libidx (sm_103a).
//
// Page "[sglang] logits를 쓰지 않는 top-k", section 1: a KV tile is the A
// operand (M = keys) of the tensor-core MMA, the accumulator lives in TMEM,
// and the heads are reduced per key in registers.  Here:
//   A = 128 keys x D        (TMA, 128/64-byte swizzle, a ring of stages)
//   B = 256 (row, head) x D (TMA, loaded once: rows_per_block = 256 / H rows)
//   D = 128 x 256 fp32 in TMEM, double buffered (2 x 256 columns).
// Warp roles (20 warps): 0 = TMA producer, 1 = TMEM owner + MMA issuer,
// 4..19 = epilogue in two teams of 8 warps.  Team t owns TMEM buffer t and the
// tiles i = t (mod 2), so one team reduces a tile while the other waits on
// the tensor core or on its TMEM loads.  Inside a team a warp owns the TMEM
// lane quarter warp % 4 (32 keys) and one of the two halves of the rows.  It
// reads its accumulators in the 16x256b shape (four threads share a key, each
// holding a quarter of the row's heads, whose weights stay in registers) and
// two butterfly steps finish every key's sum.
//
// Score of (row, key), heads summed in fp32 in a fixed order:
//   s = k_scale[key] * sum_h w[row,h] * ReLU(acc[h]).
// Every mode runs the same arithmetic, so the fused path compares exactly the
// scores that the materialising baseline writes.
//
// A launch may split row blocks' key tiles into contiguous parts, one CTA
// each (SPLIT instantiation): the blocks of the last, partly filled wave of an
// otherwise whole grid, or every block of a grid too small to fill the GPU.
// Each part of the emit pass fills runs of its own.
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
    static constexpr int TEAM_WARPS = 8;                    // per TMEM buffer
    static constexpr int EPI_WARPS = 2 * TEAM_WARPS;
    static constexpr int RG = R / 2;                        // rows per epilogue warp
    static constexpr int THREADS = 32 * (4 + EPI_WARPS);
    static constexpr uint32_t IDESC = instr_desc(DT == IDX_BF16 ? 1u : 0u, M, N);
    // q buffers: two let the next pass's q copy start during this pass
    static constexpr int QB = RB >= 256 ? 1 : 2;
    // shared memory carve (offsets from a 1024-byte aligned base)
    static constexpr int OFF_B = 0;
    static constexpr int OFF_A = QB * B_BYTES;
    static constexpr int OFF_BAR = OFF_A + NS * A_BYTES;
    // full[NS], empty[NS], accf[2], acce[2] (set up again by every pass), then,
    // kept for the whole kernel, qfull[QB] and pdone (the producer has issued
    // the pass's last key tile)
    static constexpr int NBAR = 2 * NS + 4 + QB + 1;
    static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
    static constexpr int OFF_CTL = OFF_TSLOT + 16;          // [0] abort flag, [1] next unit
    // two slots of pass metadata (the pass that runs, the one being prepared):
    // head weights [R * H], row words [R][META_WORDS], pass words [PASS_WORDS]
    static constexpr int OFF_W = (OFF_CTL + 16 + 15) / 16 * 16;
    static constexpr int OFF_META = OFF_W + 2 * R * H * 4;
    static constexpr int META_WORDS = 8;                    // per row
    static constexpr int OFF_MISC = OFF_META + 2 * R * META_WORDS * 4;
    static constexpr int PASS_WORDS = 16;
    static constexpr int SMEM_USED = OFF_MISC + 2 * PASS_WORDS * 4;
    // at least ~120 KB so that one CTA owns an SM (and its 512 TMEM columns)
    static constexpr int SMEM_ALLOC = (SMEM_USED + 1024 > 122880 ? SMEM_USED + 1024 : 122880);
};

// per-pass words of a metadata slot
enum : int {
    PW_T0 = 0,      // first key tile of the pass
    PW_NT,          // key tiles of the pass
    PW_ALL_LO,      // [all_lo, all_hi): keys every active row sees
    PW_ALL_HI,
    PW_PHASE,       // SM_SAMPLE: the block's sample phase
    PW_BLK,         // row block, part, parts
    PW_PART,
    PW_NPARTS,
};

// per-row metadata words in shared memory
enum : int {
    MW_ACTIVE = 0,  // row takes part in this pass
    MW_LO,          // visible range [lo, hi) in the tile index space (keys, or
    MW_HI,          //   sample indices in SM_SAMPLE); empty when inactive
    MW_KS,          // first visible key: index of key j is j - ks
    MW_THR,         // emit / histogram threshold key
    MW_CUT,         // emit: largest index taken among keys equal to thr
    MW_PREFIX,      // histogram: bits above the digit
    MW_THRF,        // emit: the float whose key is thr (keys compare as floats)
};

// Head reduce of one row for the 32 keys of a warp's TMEM lane quarter.
// The accumulator columns are read in the 16x256b shape: for each half of the
// quarter (16 lanes) thread t holds keys t/4 and t/4 + 8 at heads
// 8j + 2c, 8j + 2c + 1 (c = t % 4), so a thread needs only H/4 of the row's
// weights (held in registers for the whole kernel).  Each thread forms
//   P_k = sum over its heads of w[h] * (acc[h] + |acc[h]|)
// for its four keys k (x + |x| = 2 ReLU(x) stays on the FMA pipe; packed FFMA2
// takes two heads per instruction), and two butterfly steps over the four
// threads of a key group leave thread t with the full sum of one key,
// quarter offset key_off(t) = t/4 + 16 (t & 1) + 8 ((t >> 1) & 1).  The
// summation order is fixed, so every scoring mode gets the same bits.
IDX_DEVI int quad_key_off(int lane) { return (lane >> 2) + 16 * (lane & 1) + 8 * ((lane >> 1) & 1); }

template <int H>
IDX_DEVI float head_reduce_quad(uint32_t taddr, const float2* wq) {
    constexpr int REPS = H / 8;                   // 8-column groups of the row
    constexpr int RL = H >= 64 ? 2 : (REPS < 4 ? REPS : 4);       // repetitions per load
    const int lane = threadIdx.x & 31;
    float P[4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
#pragma unroll
        for (int j0 = 0; j0 < REPS; j0 += RL) {
            float v[4 * RL];
            tmem_ld16x256b<RL>(taddr + ((uint32_t)(half * 16) << 16) + (uint32_t)(j0 * 8), v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < RL; ++j) {
                const float* y = v + 4 * j;
                lo = __ffma2_rn(wq[j0 + j], make_float2(y[0] + fabsf(y[0]), y[1] + fabsf(y[1])), lo);
                hi = __ffma2_rn(wq[j0 + j], make_float2(y[2] + fabsf(y[2]), y[3] + fabsf(y[3])), hi);
            }
        }
        P[2 * half] = lo.x + lo.y;      // key t/4 + 16 half
        P[2 * half + 1] = hi.x + hi.y;  // key t/4 + 8 + 16 half
    }
    // P = keys g, g + 8, g + 16, g + 24 (g = t / 4); reduce over t % 4
    const bool b0 = lane & 1, b1 = (lane >> 1) & 1;
    const float s0 = b0 ? P[0] : P[2], s1 = b0 ? P[1] : P[3];
    const float r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
    const float r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
    const float k0 = (b0 ? P[2] : P[0]) + r0;  // key g (+16 when b0)
    const float k1 = (b0 ? P[3] : P[1]) + r1;  // key g + 8 (+16 when b0)
    const float sx = b1 ? k0 : k1;
    const float rx = __shfl_xor_sync(0xffffffffu, sx, 2);
    return (b1 ? k1 : k0) + rx;
}

// Head reduce of one row for H <= 32, one key per thread: the 32x32b shape
// gives thread t the accumulators of key t of the lane quarter at all H heads
// of the row, so no cross-thread sum is needed.  The row's weights are the
// same for every lane and come from shared memory (broadcast loads issued
// while the TMEM load is in flight).  Two packed accumulators take heads
// (4i, 4i + 1) and (4i + 2, 4i + 3); the order is fixed, so every scoring mode
// gets the same bits.  Loads of 16 columns keep the values and weights in
// flight within the register cap (32 columns spilled: 2.5 % slower at H = 32).
template <int H>
IDX_DEVI float head_reduce_lane(uint32_t taddr, const float* w_row) {
    constexpr int CH = H < 16 ? H : 16;  // columns per TMEM load
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c0 = 0; c0 < H; c0 += CH) {
        float v[CH];
        tmem_ld32x32b<CH>(taddr + (uint32_t)c0, v);
        float4 w4[CH / 4];
#pragma unroll
        for (int i = 0; i < CH / 4; ++i) w4[i] = reinterpret_cast<const float4*>(w_row + c0)[i];
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < CH / 4; ++i) {
            const float* y = v + 4 * i;
            a0 = __ffma2_rn(make_float2(w4[i].x, w4[i].y),
                            make_float2(y[0] + fabsf(y[0]), y[1] + fabsf(y[1])), a0);
            a1 = __ffma2_rn(make_float2(w4[i].z, w4[i].w),
                            make_float2(y[2] + fabsf(y[2]), y[3] + fabsf(y[3])), a1);
        }
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}

// The metadata of one pass over part `part` of `nparts` of row block blk in
// scoring mode `mode` (rescan histogram passes: digit `level`) into metadata
// slot `sl`: per row its visible range in the pass's index space, threshold
// words and head weights; per pass its key tiles.  Run by the nthr threads
// t = 0 .. nthr - 1 of a group that synchronises with bar() (the whole CTA
// before the first pass or a rescan pass; two warps while another pass runs).
template <int DT, int H, int RB, bool SPLIT, typename Bar>
IDX_DEVI void prep_pass(const ScoreArgs& a, uint8_t* smem, const int sl, const int blk,
                        const int part, const int nparts, const int mode, const int level,
                        const int t, const int nthr, Bar bar) {
    using C = ScoreCfg<DT, H, RB>;
    float* w_s = reinterpret_cast<float*>(smem + C::OFF_W) + sl * C::R * H;
    int* meta = reinterpret_cast<int*>(smem + C::OFF_META) + sl * C::R * C::META_WORDS;
    int* pw = reinterpret_cast<int*>(smem + C::OFF_MISC) + sl * C::PASS_WORDS;
    const int r0 = blk * C::R;
    const int phase =
        mode == SM_SAMPLE ? (int)(hash32((uint32_t)blk ^ a.phase_seed) % (uint32_t)a.S) : 0;
    if (t < C::R) {
        int* m = meta + t * C::META_WORDS;
        const int r = r0 + t;
        int ks = 0, ke = 0, active = 0, lo = 0, hi = 0, cut = kAllIdx;
        uint32_t thr = 0, prefix = 0;
        if (r < a.rows) {
            const long long ks_ = a.ks[r], ke_ = a.ke[r];
            if (ks_ < 0 || ke_ > a.keys || ks_ > ke_) {
                if (ke_ > ks_ || ks_ < 0) raise_status(a.d_status, IDX_DEV_RANGE);
            } else {
                ks = (int)ks_;
                ke = (int)ke_;
            }
            const int n = ke - ks;
            lo = ks;
            hi = ke;
            switch (mode) {
                case SM_MATERIALISE:
                    active = n > 0;
                    if (n > a.out_stride) {
                        raise_status(a.d_status, IDX_DEV_RANGE);
                        active = 0;
                    }
                    break;
                case SM_SAMPLE: {
                    active = n > a.cap;
                    const SampleSpan sp = sample_span(ks, ke, phase, a.S, a.nsamp);
                    lo = (int)sp.a;
                    hi = (int)sp.b;
                    if (active && hi - lo > a.samp_stride) {
                        raise_status(a.d_status, IDX_DEV_RANGE);  // longer than max_len
                        active = 0;
                    }
                } break;
                case SM_EMIT:
                    // rows that see at most cap keys emit every key (page 1,
                    // section 1: blocks of short rows store every score)
                    active = n > a.topk;
                    if (active && n > a.cap) {
                        if (a.sampled) {
                            thr = a.plan[r].thr;
                        } else {
                            // longer than the max_len the call was sized for: no
                            // threshold exists; emit nothing, so that the slab
                            // top-k reports the row (IDX_DEV_RANGE, -1 output)
                            thr = 0xffffffffu;
                            raise_status(a.d_status, IDX_DEV_RANGE);
                        }
                    }
                    break;
                case SM_FB_HIST: {
                    const RowPlan p = a.plan[r];
                    active = n > 0 && p.state == ST_HIST && p.level == level;
                    thr = p.thr;
                    prefix = p.prefix;
                } break;
                case SM_FB_EMIT: {
                    const RowPlan p = a.plan[r];
                    active = n > 0 && p.state == ST_EMIT;
                    thr = p.thr;
                    cut = p.idx_cut;
                } break;
            }
        }
        if (!active) lo = hi = 0;
        // a pass over a whole row block (the re-emission, or an emit CTA of a
        // block that the launch does not split) leaves the runs of the other
        // key splits empty
        if (SPLIT && active && (mode == SM_FB_EMIT || (mode == SM_EMIT && nparts == 1)))
            for (int c = kRuns; c < a.nruns; ++c) a.run_cnt[(long long)r * a.nruns + c] = 0;
        m[MW_ACTIVE] = active;
        m[MW_LO] = lo;
        m[MW_HI] = hi;
        m[MW_KS] = ks;
        m[MW_THR] = (int)thr;
        m[MW_CUT] = cut;
        m[MW_PREFIX] = (int)prefix;
        // the emit rule key > thr || (key == thr && idx <= cut) in floats: keys
        // below the one of -inf admit every score, whatever the index
        if (thr <= 0x007fffffu) cut = kAllIdx;
        m[MW_CUT] = cut;
        // rows that take no part: a threshold no score reaches
        m[MW_THRF] =
            __float_as_int(active && thr != 0xffffffffu ? key_floor_float(thr) : INFINITY);
    }
    for (int i = t; i < C::R * H; i += nthr) {
        const long long r = r0 + i / H;
        w_s[i] = r < a.rows ? a.w[(long long)r0 * H + i] : 0.f;
    }
    bar();
    if (t == 0) {
        int lo = 0x7fffffff, hi = -1, all_lo = -1, all_hi = 0x7fffffff;
        for (int j = 0; j < C::R; ++j) {
            const int* m = meta + j * C::META_WORDS;
            if (m[MW_HI] <= m[MW_LO]) continue;
            lo = m[MW_LO] < lo ? m[MW_LO] : lo;
            hi = m[MW_HI] > hi ? m[MW_HI] : hi;
            all_lo = m[MW_LO] > all_lo ? m[MW_LO] : all_lo;
            all_hi = m[MW_HI] < all_hi ? m[MW_HI] : all_hi;
        }
        pw[PW_ALL_LO] = all_lo;
        pw[PW_ALL_HI] = all_hi;
        int t0 = 0, nt = 0;
        if (hi > lo) {
            t0 = lo / C::M;
            nt = (hi + C::M - 1) / C::M - t0;
        }
        if (SPLIT) {
            // part `part` of nparts: a contiguous range of the block's tiles
            const int per = (nt + nparts - 1) / nparts;
            const int ts = part * per;
            const int te = ts + per < nt ? ts + per : nt;
            pw[PW_T0] = t0 + ts;
            pw[PW_NT] = te > ts ? te - ts : 0;
        } else {
            pw[PW_T0] = t0;
            pw[PW_NT] = nt;
        }
        pw[PW_PHASE] = phase;
        pw[PW_BLK] = blk;
        pw[PW_PART] = part;
        pw[PW_NPARTS] = nparts;
        // a new call: this block's rescan flag starts at 0
        if (mode == SM_SAMPLE && part == 0 && a.fb_bflag) a.fb_bflag[blk] = 0;
    }
    bar();
    if (SPLIT && mode == SM_EMIT && pw[PW_NT] == 0) {
        // nothing to score in this part: its runs of the active rows are empty
        for (int i = t; i < C::R * kRuns; i += nthr) {
            const int rr = i / kRuns;
            if (meta[rr * C::META_WORDS + MW_ACTIVE])
                a.run_cnt[(long long)(r0 + rr) * a.nruns + part * kRuns + i % kRuns] = 0;
        }
    }
}

// Issue the copy of row block blk's q rows into q buffer qs (thread of the
// caller's choice; the buffer and its barrier must be idle).
template <int DT, int H, int RB>
IDX_DEVI void issue_q(const CUtensorMap& tm_q, uint8_t* smem, const int qs, const int blk) {
    using C = ScoreCfg<DT, H, RB>;
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 2 * C::NS + 4;
    mbar_arrive_expect_tx(&qfull[qs], C::B_BYTES);
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_2d(smem + C::OFF_B + qs * C::B_BYTES + c * C::B_CHUNK, &tm_q, &qfull[qs],
                    c * C::CHUNK_ELEMS, blk * C::R * H);
}

// SPLIT: the launch splits row blocks over key ranges or addresses a slab
// with more than kRuns runs per row; without it the kernel is compiled with
// kRuns runs per row and no split arithmetic.
// One pass of the CTA over the part of a row block that metadata slot sl
// describes (prep_pass), in scoring mode `mode` (rescan histogram passes:
// digit `level`), with the block's q rows in q buffer qs (phase parity qpar of
// its barrier); q_at_start: thread 0 issues that copy here, else it was issued
// before.  Warps 2 and 3 run `side` meanwhile (the next pass's metadata, or
// nothing), in a pass with tiles once the producer is 2 NS tiles short of the
// pass's end (phase parity ppar of pdone): the next unit is taken late enough
// that a CTA does not commit to it long before it can start it, and early
// enough that its q copy and metadata are ready when the pass ends.  Every thread of the CTA calls it; it ends with the CTA
// synchronised, no MMA in flight and the pass's copies landed.  TMEM is taken
// by the first pass that has tiles to score and kept until the kernel ends
// (tslot[0] = address, tslot[1] = taken).
template <int DT, int H, int RB, bool SPLIT, typename Side>
IDX_DEVI void score_pass(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                         const CUtensorMap& tm_ks, const ScoreArgs& a, uint8_t* smem,
                         const int sl, const int qs, const uint32_t qpar, const bool q_at_start,
                         const uint32_t ppar, const int mode, const int level, Side side) {
    using C = ScoreCfg<DT, H, RB>;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::NS;
    uint64_t* accf = bars + 2 * C::NS;
    uint64_t* acce = accf + 2;
    uint64_t* qfull = acce + 2 + qs;
    uint64_t* pdone = acce + 2 + C::QB;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_TSLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_CTL);
    const float* w_s = reinterpret_cast<const float*>(smem + C::OFF_W) + sl * C::R * H;
    const int* meta = reinterpret_cast<const int*>(smem + C::OFF_META) + sl * C::R * C::META_WORDS;
    const int* pw = reinterpret_cast<const int*>(smem + C::OFF_MISC) + sl * C::PASS_WORDS;
    uint8_t* const qbuf = smem + C::OFF_B + qs * C::B_BYTES;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = pw[PW_BLK], part = pw[PW_PART];
    const int r0 = blk * C::R;
    const int phase = pw[PW_PHASE];
    const int t0 = pw[PW_T0];
    const int ntiles = pw[PW_NT];
    (void)part;

    // the pipeline's barriers, set up again for every pass (the previous pass
    // ended with none in use)
    if (tid == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], C::TEAM_WARPS);
        }
        fence_barrier_init();
        if (q_at_start) {
            prefetch_tmap(&tm_q);
            issue_q<DT, H, RB>(tm_q, smem, qs, blk);
        }
    }
    __syncthreads();
    if (ntiles == 0) {
        // nothing to score: the q copy is waited for (bounded)
        if (tid == 0) mbar_wait(qfull, qpar, nullptr, 1ll << 28);
        if (warp == 2 || warp == 3) side();
        __syncthreads();  // every thread is done with this pass's shared state
        return;
    }

    if (tslot[1] == 0) {
        // the CTA's first pass with tiles: take the 512 TMEM columns
        if (warp == 1) {
            __syncwarp();
            tmem_alloc(tslot, 512);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) tslot[1] = 1;
    }
    const uint32_t tmem = tslot[0];

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(mode == SM_SAMPLE ? (const void*)&tm_ks : (const void*)&tm_k);
            int issued = 0;
            // the side job may take the next unit once this many tiles are issued
            const int lead = ntiles > 2 * C::NS ? ntiles - 2 * C::NS : 0;
            bool told = false;
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % C::NS;
                const uint32_t use = (uint32_t)(i / C::NS);
                if (i == lead) {
                    mbar_arrive(pdone);
                    told = true;
                }
                if (i >= C::NS &&
                    !mbar_wait(&empty[s], (use & 1u) ^ 1u, abort_flag, a.wait_limit)) {
                    *abort_flag = 1;
                    raise_status(a.d_status, IDX_DEV_TIMEOUT);
                    break;
                }
                issued = i + 1;
                if (i == a.withhold_tile) continue;  // (test) no copy: its waits run out
                mbar_arrive_expect_tx(&full[s], C::A_BYTES);
                const int row0 = (t0 + i) * C::M;
#pragma unroll
                for (int c = 0; c < C::NCHUNK; ++c) {
                    uint8_t* dst = smem + C::OFF_A + s * C::A_BYTES + c * C::A_CHUNK;
                    if (mode == SM_SAMPLE)
                        tma_load_3d(dst, &tm_ks, &full[s], c * C::CHUNK_ELEMS, phase, row0);
                    else
                        tma_load_2d(dst, &tm_k, &full[s], c * C::CHUNK_ELEMS, row0);
                }
            }
            if (!told) mbar_arrive(pdone);  // (the loop stopped early)
            // do not leave with copies in flight: wait (bounded) for q and the last stages
            mbar_wait(qfull, qpar, nullptr, 1ll << 28);
            for (int i = issued > C::NS ? issued - C::NS : 0; i < issued; ++i)
                if (i != a.withhold_tile)
                    mbar_wait(&full[i % C::NS], (uint32_t)((i / C::NS) & 1), nullptr, 1ll << 28);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a_base = smem_u32(smem + C::OFF_A);
            const uint32_t b_base = smem_u32(qbuf);
            bool ok = mbar_wait(qfull, qpar, abort_flag, a.wait_limit);
            int issued = 0;
            for (int i = 0; ok && i < ntiles; ++i) {
                const int s = i % C::NS;
                const int b = i & 1;
                // buffer b is free once its team has read tile i - 2
                if (i >= 2 && !mbar_wait(&acce[b], (uint32_t)(((i >> 1) & 1) ^ 1), abort_flag,
                                         a.wait_limit)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&full[s], (uint32_t)((i / C::NS) & 1), abort_flag, a.wait_limit)) {
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
            // wait (bounded) until the tensor core is done with TMEM, and for the
            // arrivals of the last stages' release commits: the next pass
            // initialises these barriers again
            if (issued > 0)
                mbar_wait(&accf[(issued - 1) & 1], (uint32_t)(((issued - 1) >> 1) & 1), nullptr,
                          1ll << 28);
            for (int i = issued > C::NS ? issued - C::NS : 0; i < issued; ++i)
                mbar_wait(&empty[i % C::NS], (uint32_t)((i / C::NS) & 1), nullptr, 1ll << 28);
        }
    } else if (warp < 4) {
        // ------------------------------------------------ warps 2, 3: side job
        // once the producer is done (bounded: after a time-out it goes ahead)
        mbar_wait(pdone, ppar, abort_flag, a.wait_limit);
        side();
    } else {
        // ------------------------------------------------ epilogue
        const int e = warp - 4;
        const int team = e >> 3;             // TMEM buffer and tile parity
        const int q = warp & 3;              // TMEM lane quarter
        const int grp = (e >> 2) & 1;        // half of the rows
        const int run = q * 2 + team;        // candidate run of this warp (in its key split)
        // lanes whose key comes earlier (candidates are appended in key order)
        // H <= 32: one key per lane (32x32b loads); H = 64: four lanes per key
        // (16x256b loads and a butterfly)
        constexpr bool LANE_KEYS = H <= 32;
        uint32_t lt = 0u;
        if constexpr (LANE_KEYS) {
            lt = (1u << lane) - 1u;
        } else {
#pragma unroll
            for (int l = 0; l < 32; ++l)
                lt |= (quad_key_off(l) < quad_key_off(lane) ? 1u : 0u) << l;
        }
        int cnt[C::RG];
        // row metadata from shared memory; the emit words of up to 2 rows per
        // warp are held in registers across the tile loop
        const int* mrow = meta + grp * C::RG * C::META_WORDS;
        auto row_word = [&](int j, int word) -> int { return mrow[j * C::META_WORDS + word]; };
        constexpr bool HOIST = C::RG <= 2;
        constexpr int NH = HOIST ? C::RG : 1;
        int e_lo[NH], e_len[NH], e_cut[NH];
        float e_thr[NH];
#pragma unroll
        for (int j = 0; j < C::RG; ++j) {
            cnt[j] = 0;
            if constexpr (HOIST) {
                e_lo[j] = row_word(j, MW_LO);
                e_len[j] = row_word(j, MW_HI) - e_lo[j];
                e_cut[j] = row_word(j, MW_CUT);
                e_thr[j] = __int_as_float(row_word(j, MW_THRF));
            }
        }
        // this warp's runs of its rows, (score bits, index) pairs: row j's run
        // at pr + j * rstride
        const int nruns = SPLIT ? a.nruns : kRuns;
        const int split_run0 = SPLIT ? part * kRuns : 0;
        const long long rb = (long long)(r0 + grp * C::RG) * nruns + split_run0 + run;
        int2* const pr = a.slab ? a.slab + rb * a.cap_q : nullptr;
        const int rstride = nruns * a.cap_q;
#define RLO(j) row_word(j, MW_LO)
#define RHI(j) row_word(j, MW_HI)
#define RKS(j) row_word(j, MW_KS)
#define RTHR(j) ((uint32_t)row_word(j, MW_THR))
#define RCUT(j) row_word(j, MW_CUT)
#define RPRE(j) ((uint32_t)row_word(j, MW_PREFIX))
        // this thread's weights: row j, head pair (8 rep + 2c, 8 rep + 2c + 1)
        const int kq = LANE_KEYS ? lane : quad_key_off(lane);  // this thread's key in the quarter
        // Per-key scale of the team's next tile, loaded one tile ahead.  The
        // thread's tile index i (a key, or a sample index in SM_SAMPLE) grows
        // by 2 M per team tile; key = i, or phase + S i for the sample.
        // (keys < 2^31 - 256, so i stays an int; the key offset is only used
        // while i < ilim, so its 32-bit wrap past the end is harmless)
        const uint32_t kmul = mode == SM_SAMPLE ? (uint32_t)a.S : 1u;
        const int ilim = (int)(mode == SM_SAMPLE ? a.nsamp : a.keys);  // i must stay below
        int s_i = (t0 + team) * C::M + q * 32 + kq;
        uint32_t s_off = (mode == SM_SAMPLE ? (uint32_t)phase : 0u) + kmul * (uint32_t)s_i;
        const uint32_t s_step = kmul * 2u * C::M;
        // H = 64: this thread's weights of row j, head pair (8 rep + 2c, 8 rep + 2c + 1),
        // held in registers for the whole pass
        constexpr int WR = LANE_KEYS ? 1 : C::RG, WC = LANE_KEYS ? 1 : H / 8;
        float2 wq[WR][WC];
        if constexpr (!LANE_KEYS) {
#pragma unroll
            for (int j = 0; j < C::RG; ++j) {
                const float* wr = w_s + (grp * C::RG + j) * H + 2 * (lane & 3);
#pragma unroll
                for (int rp = 0; rp < H / 8; ++rp)
                    wq[j][rp] = make_float2(wr[8 * rp], wr[8 * rp + 1]);
            }
        }
        const int all_lo = pw[PW_ALL_LO], all_hi = pw[PW_ALL_HI];
        float next_scale = team < ntiles && s_i < ilim ? __ldg(a.k_scale + s_off) : 0.f;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(team * C::N);
        for (int i = team, un = 0; i < ntiles; i += 2, ++un) {
            // the team's tile count (accf parity): a counter of its own, or
            // i / 2 (team is 0 or 1) -- measured faster at H = 64 and at H <= 32
            // respectively (the register allocation differs)
            const uint32_t u = H <= 32 ? (uint32_t)i >> 1 : (uint32_t)un;
            const float cur_scale = next_scale;
            s_i += 2 * C::M;
            s_off += s_step;
            next_scale = i + 2 < ntiles && s_i < ilim ? __ldg(a.k_scale + s_off) : 0.f;
            // warp-uniform outcome: the TMEM loads below are .sync.aligned
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&accf[team], (uint32_t)(u & 1), abort_flag, a.wait_limit))) {
                *abort_flag = 1;
                if (lane == 0) raise_status(a.d_status, IDX_DEV_TIMEOUT);
                break;
            }
            tc_fence_after();
            const int kidx = (t0 + i) * C::M + q * 32 + kq;  // key, or sample index
            const float post_scale = 0.5f * cur_scale;
            float sc[C::RG];
#pragma unroll
            for (int j = 0; j < C::RG; ++j) {
                const int rr = grp * C::RG + j;
                if constexpr (LANE_KEYS)
                    sc[j] = head_reduce_lane<H>(tbase + (uint32_t)(rr * H), w_s + rr * H) *
                            post_scale;
                else
                    sc[j] = head_reduce_quad<H>(tbase + (uint32_t)(rr * H), wq[LANE_KEYS ? 0 : j]) *
                            post_scale;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[team]);

            if (mode == SM_MATERIALISE || mode == SM_SAMPLE) {
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int off = kidx - (HOIST ? e_lo[HOIST ? j : 0] : RLO(j));
                    const int len = HOIST ? e_len[HOIST ? j : 0] : RHI(j) - RLO(j);
                    if ((uint32_t)off < (uint32_t)len) {
                        const long long r = r0 + grp * C::RG + j;
                        if (mode == SM_MATERIALISE)
                            a.out[r * a.out_stride + off] = sc[j];
                        else
                            a.samp[r * a.samp_stride + off] = (uint16_t)(fkey(sc[j]) >> 16);
                    }
                }
            } else if (mode == SM_FB_HIST) {
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int off = kidx - RLO(j);
                    const bool vis = (uint32_t)off < (uint32_t)(RHI(j) - RLO(j));
                    const uint32_t kb = fkey(sc[j]);
                    const uint32_t ix = (uint32_t)(kidx - RKS(j));
                    const int lev = level;
                    bool valid;
                    uint32_t dg;
                    if (lev <= 2) {
                        valid = vis && has_prefix(kb, lev, RPRE(j));
                        dg = digit_of(kb, lev);
                    } else {
                        valid = vis && kb == RTHR(j) && idx_has_prefix(ix, lev, RPRE(j));
                        dg = idx_digit_of(ix, lev);
                    }
                    const uint32_t same =
                        __match_any_sync(0xffffffffu, valid ? dg : (0x80000000u | lane));
                    if (valid && lane == __ffs(same) - 1)
                        atomicAdd(&a.fb_hist[(long long)(r0 + grp * C::RG + j) * kHistBins + dg],
                                  (uint32_t)__popc(same));
                }
            } else if (mode == SM_EMIT && (t0 + i) * C::M >= all_lo &&
                       (t0 + i + 1) * C::M <= all_hi) {
                // SM_EMIT on a tile every active row sees whole: the rule is
                // s >= T_r (rows that take no part have T = +inf).  A lane's
                // place in the run is the number of hits of lower lanes
                // (earlier keys); a row whose 32 keys hold no hit (most of
                // them: about 1.5 topk candidates per row) costs one vote.
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const float thr = HOIST ? e_thr[HOIST ? j : 0]
                                            : __int_as_float(row_word(j, MW_THRF));
                    const bool hit = sc[j] >= thr;
                    const uint32_t A = __ballot_sync(0xffffffffu, hit);
                    if (A != 0u) {  // warp-uniform
                        const int pos = cnt[j] + __popc(A & lt);
                        if (hit && pos < a.cap_q)
                            pr[j * rstride + pos] =
                                make_int2(__float_as_int(sc[j]),
                                          kidx - (HOIST ? e_lo[HOIST ? j : 0] : RLO(j)));
                        cnt[j] += __popc(A);
                    }
                }
            } else {
                // SM_EMIT / SM_FB_EMIT: append every key that passes the row's
                // rule to this warp's run, in key order; no cross-warp traffic
#pragma unroll
                for (int j = 0; j < C::RG; ++j) {
                    const int lo = HOIST ? e_lo[HOIST ? j : 0] : RLO(j);
                    const int len = HOIST ? e_len[HOIST ? j : 0] : RHI(j) - RLO(j);
                    const float thr = HOIST ? e_thr[HOIST ? j : 0]
                                            : __int_as_float(row_word(j, MW_THRF));
                    const int cut = HOIST ? e_cut[HOIST ? j : 0] : RCUT(j);
                    const int off = kidx - lo;
                    const bool hit = (uint32_t)off < (uint32_t)len &&
                                     (sc[j] > thr || (sc[j] == thr && off <= cut));
                    const uint32_t A = __ballot_sync(0xffffffffu, hit);
                    if (A != 0u) {  // warp-uniform
                        const int pos = cnt[j] + __popc(A & lt);
                        if (hit && pos < a.cap_q)
                            pr[j * rstride + pos] = make_int2(__float_as_int(sc[j]), off);
                        cnt[j] += __popc(A);
                    }
                }
            }
        }
#undef RLO
#undef RHI
#undef RKS
#undef RTHR
#undef RCUT
#undef RPRE
        if (mode == SM_FB_HIST) {
            // this CTA saw every key of its rows: finish the digit step here
            __threadfence();  // the histogram atomics of every warp reached L2
            named_bar_sync(1, 32 * C::EPI_WARPS);
            for (int rr = e; rr < C::R; rr += C::EPI_WARPS) {
                if (!meta[rr * C::META_WORDS + MW_ACTIVE]) continue;
                rescan_pick_warp(a.plan + r0 + rr, a.fb_hist + (long long)(r0 + rr) * kHistBins,
                                 level, a.topk, a.cap, a.fb_cnt);
            }
        }
        if (lane == 0 && (mode == SM_EMIT || mode == SM_FB_EMIT)) {
#pragma unroll
            for (int j = 0; j < C::RG; ++j) {
                const int rr = grp * C::RG + j;
                if (meta[rr * C::META_WORDS + MW_ACTIVE])
                    a.run_cnt[(long long)(r0 + rr) * nruns + split_run0 + run] = cnt[j];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Key tiles of the pass in metadata slot sl.
template <int DT, int H, int RB>
IDX_DEVI int pw_nt(const uint8_t* smem, int sl) {
    using C = ScoreCfg<DT, H, RB>;
    return reinterpret_cast<const int*>(smem + C::OFF_MISC)[sl * C::PASS_WORDS + PW_NT];
}

// Unit u of a scoring launch: a row block, or a part of one (ScoreArgs::nwhole,
// ::ksplit), the blocks taken in ScoreArgs::order when there is one.
struct ScoreUnit {
    int blk, part, nparts;
};
IDX_DEVI ScoreUnit score_unit(const ScoreArgs& a, int u) {
    int i = u, part = 0, nparts = 1;
    if (u >= a.nwhole) {
        const int v = u - a.nwhole;
        i = a.nwhole + v / a.ksplit;
        part = v % a.ksplit;
        nparts = a.ksplit;
    }
    return {a.order ? __ldg(a.order + i) : i, part, nparts};
}

// The kernel.  A scoring launch (SM_MATERIALISE, SM_SAMPLE, SM_EMIT) is
// persistent: each CTA takes unit blockIdx.x, then the next unit of a launch
// counter (a.sched; without one, every gridDim.x-th unit), one pass each.
// While a pass runs, warps 2 and 3 take the next unit, start its q copy into
// the other q buffer and write its metadata into the other slot, so that the
// next pass starts with both at hand.  The exact rescan (SM_RESCAN) is a grid
// that strides over the device list of flagged row blocks and runs, per
// block, the histogram passes of the digits its rows still need and then the
// re-emission; each of those passes depends on the one before, so its
// metadata is read just before it.  A rescan launch with no block listed ends
// at once.
template <int DT, int H, int RB, bool SPLIT>
__global__ void __launch_bounds__(ScoreCfg<DT, H, RB>::THREADS, 1)
score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ ScoreArgs a) {
    using C = ScoreCfg<DT, H, RB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base (TMA swizzle atoms), derived from smem_raw by an
    // offset so that the compiler keeps every access in the shared space
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_TSLOT);
    volatile int* ctl = reinterpret_cast<volatile int*>(smem + C::OFF_CTL);
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 2 * C::NS + 4;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        tslot[1] = 0;
        ctl[0] = 0;  // abort flag: a wait that timed out releases every later wait
        for (int i = 0; i < C::QB; ++i) mbar_init(&qfull[i], 1);
        mbar_init(&qfull[C::QB], 1);  // pdone
        fence_barrier_init();
    }
    // (a launch that overlaps the kernel before it waits here for its results)
    pdl_wait();
    if (a.mode == SM_RESCAN && *(volatile int*)(a.fb_cnt + 7) == 0) return;  // none flagged
    // a new call: the rescan counters start at 0
    if (a.mode == SM_SAMPLE && blockIdx.x == 0 && tid < 8) a.fb_cnt[tid] = 0;
    __syncthreads();
    auto cta_bar = [] { __syncthreads(); };
    auto nothing = [] {};
    if (a.mode == SM_RESCAN) {
        const int nb = *(volatile int*)(a.fb_cnt + 7);
        int n = 0, ptiles = 0;
        for (int wi = (int)blockIdx.x; wi < nb; wi += (int)gridDim.x) {
            const int blk = a.fb_blocks[wi];
            for (int pass = 0; pass < 7; ++pass, ++n) {
                const int mode = pass < 6 ? SM_FB_HIST : SM_FB_EMIT;
                prep_pass<DT, H, RB, SPLIT>(a, smem, 0, blk, 0, 1, mode, pass, tid, C::THREADS,
                                            cta_bar);
                const bool tiles = pw_nt<DT, H, RB>(smem, 0) > 0;
                score_pass<DT, H, RB, SPLIT>(tm_q, tm_k, tm_ks, a, smem, 0, 0,
                                             (uint32_t)(n & 1), true, (uint32_t)(ptiles & 1),
                                             mode, pass, nothing);
                ptiles += tiles;
            }
        }
    } else {
        const int nblk = (a.rows + C::R - 1) / C::R;
        const int nunits = a.nwhole + (nblk - a.nwhole) * a.ksplit;
        int u = (int)blockIdx.x, n = 0, ptiles = 0;
        if (u < nunits) {
            const ScoreUnit x = score_unit(a, u);
            if (C::QB == 2 && tid == 0) {
                prefetch_tmap(&tm_q);
                issue_q<DT, H, RB>(tm_q, smem, 0, x.blk);
            }
            prep_pass<DT, H, RB, SPLIT>(a, smem, 0, x.blk, x.part, x.nparts, a.mode, a.level, tid,
                                        C::THREADS, cta_bar);
        }
        while (u < nunits) {
            const int sl = n & 1;
            // warps 2 and 3 during the pass: the next unit, its q copy and metadata
            auto next_job = [&] {
                const int t = tid - 64;
                if (t == 0) {
                    const int nx =
                        a.sched ? (int)gridDim.x + atomicAdd(a.sched, 1) : u + (int)gridDim.x;
                    ctl[1] = nx;
                    if (C::QB == 2 && nx < nunits)
                        issue_q<DT, H, RB>(tm_q, smem, (n + 1) & 1, score_unit(a, nx).blk);
                }
                named_bar_sync(2, 64);
                const int nx = ctl[1];
                if (nx < nunits) {
                    const ScoreUnit x = score_unit(a, nx);
                    prep_pass<DT, H, RB, SPLIT>(a, smem, sl ^ 1, x.blk, x.part, x.nparts, a.mode,
                                                a.level, t, 64, [] { named_bar_sync(2, 64); });
                }
            };
            const int qs = C::QB == 2 ? (n & 1) : 0;
            const uint32_t qpar = C::QB == 2 ? (uint32_t)((n >> 1) & 1) : (uint32_t)(n & 1);
            const bool tiles = pw_nt<DT, H, RB>(smem, sl) > 0;
            score_pass<DT, H, RB, SPLIT>(tm_q, tm_k, tm_ks, a, smem, sl, qs, qpar, C::QB == 1,
                                         (uint32_t)(ptiles & 1), a.mode, a.level, next_job);
            ptiles += tiles;
            const int nx = ctl[1];
            if (ctl[0]) {
                // a wait timed out: stop, once the next unit's q copy has landed
                if (tid == 0 && C::QB == 2 && nx < nunits)
                    mbar_wait(&qfull[(n + 1) & 1], (uint32_t)(((n + 1) >> 1) & 1), nullptr,
                              1ll << 28);
                break;
            }
            u = nx;
            ++n;
        }
    }
    __syncthreads();
    if (tslot[1] && warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tslot[0], 512);
    }
}

}  // namespace idx

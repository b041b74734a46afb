/*
 * idx.h - C ABI of libidx, the GB300 (sm_103a) sparse-attention prefill indexer.
 *
 * Problem (page "[sglang] logits를 쓰지 않는 top-k: SGLang의 LiteTopK prefill
 * indexer", introduction and section 1): for every query row r and every key j
 * that the row can see, ks[r] <= j < ke[r], the indexer score is
 *
 *     s[r,j] = k_scale[j] * sum_h w[r,h] * max(0, q[r,h,:] . k[j,:])
 *
 * and the row keeps the topk best keys.  This library returns the EXACT top-k:
 * keys ordered by (score descending, key index ascending), the first topk kept,
 * reported as row-relative indices j - ks[r] (page 1, section 1: candidate
 * indices are stored as key - ks[row]) in ascending order, followed by -1 when
 * the row sees fewer than topk keys (page 1, section 3: a consumer skips
 * negative positions).
 *
 * Conventions shared by every entry point
 *  - Tensor arguments are DEVICE pointers owned by the caller; the library
 *    keeps no pointer after the call returns and allocates no device memory.
 *    Scratch memory is the caller's workspace `ws` of at least the size its
 *    *_workspace query returns, 256-byte aligned.
 *  - All layouts are row-major and contiguous:
 *      q [rows, H, D], k [keys, D]  (both bf16 or both fp8 e4m3, see idx_dtype)
 *      k_scale [keys] float32 (> 0), w [rows, H] float32 (>= 0)
 *      ks, ke [rows] int32;  out_idx [rows, topk] int32
 *  - `stream` is a cudaStream_t (NULL is the legacy default stream).  Calls are
 *    asynchronous on that stream; the host never waits on the device.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns an error and launches nothing.  Errors met on the
 *    device (a visible range outside [0, keys], a wait that timed out) are
 *    OR-ed into the optional device status word options->d_status as
 *    IDX_DEV_* bits; nothing traps.
 *  - Preconditions not checked: scores, q, k, k_scale, w hold no NaN/Inf;
 *    k_scale > 0 and w >= 0 (the score formula relies on it).
 *  - Supported: sm_103a; H in {8, 16, 32, 64}; D in {64, 128};
 *    1 <= topk <= 4096; rows >= 0 (a row count of 0 is a no-op).
 *    Anything else returns IDX_EUNSUPPORTED.
 */
#ifndef IDX_H_
#define IDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    IDX_OK = 0,
    IDX_EINVAL = 1,        /* a null pointer, a negative size, topk < 1 ... */
    IDX_EALIGN = 2,        /* a tensor or the workspace is not 16 B (256 B for ws) aligned */
    IDX_EWORKSPACE = 3,    /* ws_bytes smaller than the query returned */
    IDX_EUNSUPPORTED = 4,  /* dtype, H, D, topk or the GPU architecture */
    IDX_ECUDA = 5,         /* a CUDA runtime/driver call failed */
    IDX_ETIMEOUT = 6       /* reserved for host-side reporting of IDX_DEV_TIMEOUT */
} idx_status;

/* bits OR-ed into *options->d_status by device code */
#define IDX_DEV_TIMEOUT 0x1   /* a bounded wait inside a kernel gave up */
#define IDX_DEV_RANGE   0x2   /* a row's [ks, ke) is not inside [0, keys] or exceeds max_len */
#define IDX_DEV_STATE   0x4   /* the exact fallback ran out of its refinement levels */

/* IDX_MXFP4 (the OCP MX format): e2m1 elements packed two per byte (element 2i in
 * the low nibble) with one e8m0 scale per 32 consecutive elements along D; only
 * the *_mxfp4 entry points below take it (they also take the scale arrays). */
typedef enum { IDX_BF16 = 1, IDX_FP8_E4M3 = 2, IDX_MXFP4 = 3 } idx_dtype;

/* Optional device-side counters (zero them before the call if you read them). */
typedef struct idx_stats {
    int emit_all_rows;   /* rows that see <= cap keys: every key became a candidate */
    int overflow_rows;   /* rows whose candidate count exceeded the slab cap */
    int short_rows;      /* rows with fewer than topk candidates although they see > cap keys */
    int fallback_rows;   /* rows re-selected by the exact full-row rescan */
    int max_count;       /* largest candidate count of any row */
    int split_rows;      /* rows the standalone top-k selected with a multi-block row split */
    int tie_rescan_rows; /* standalone top-k rows that needed the multi-pass path (the
                            one-pass candidate runs missed or overflowed) */
    int reserved;
} idx_stats;

/* Every field 0 selects the default.  Pass NULL for all defaults. */
typedef struct idx_options {
    float cap_factor;     /* candidate slab cap = ceil(cap_factor * topk) when given;
                             default min(max(ceil(3.5 * topk), 4096), 12288) (page 1
                             sizes its slab at about 2.25 x topk; the larger default
                             lets the threshold sample take a wider stride, so the
                             sample pass costs less than the extra candidates add).
                             Caps above 12288 are refused. */
    float target_factor;  /* expected candidates / topk that the sampled threshold aims
                             at; default sqrt(cap/topk).  Test knob to force short or
                             overflowing rows. */
    int sample_stride;    /* odd stride S of the threshold sample; 0 = automatic */
    int row_split;        /* standalone top-k row split, see below */
    int* d_status;        /* optional device int receiving IDX_DEV_* bits */
    idx_stats* d_stats;   /* optional device counters */
    int relative_rows;    /* idx_topk_from_scores: row r's visible scores start at
                             column 0 of its row (the layout idx_score_materialise
                             writes) instead of column ks[r] */
    int test_stall_us;    /* test only, 0 = off.  n > 0: the TMA producer of every
                             scoring pass issues no copy for key tile 1, and the
                             scoring kernel's waits give up after about n
                             microseconds (instead of about 2 s).  A pass with more
                             than one tile then stops early with IDX_DEV_TIMEOUT in
                             *d_status, leaving no copy or MMA in flight; the call
                             returns and its results are meaningless.  It exists to
                             run the timeout unwind on purpose. */
    void* const* stage_events; /* optional array of cudaEvent_t, recorded on `stream`
                             at stage boundaries (NULL entries are skipped).
                             idx_score_topk: [0] start, [1] after the sample and its
                             thresholds, [2] after the scoring/emit pass, [3] after
                             the slab top-k, [4] after the exact rescan (end).
                             The other entry points: [0] start, [1] end. */
} idx_options;

/* row_split: 0 = automatic (page "[sglang] ROCm DSA Indexer Top-K 최적화",
 * row_split function: split a row over g blocks when it is at least 65536 long
 * and g = min(SMs / rows, 32) >= 4), -1 or 1 = never split, g >= 2 = force
 * g blocks (at most 64).  Grids with more than 65535 rows never split.  A
 * split row is streamed once by g blocks, each over a contiguous slice; one
 * more block per row selects from what they kept, or re-selects the whole row
 * exactly when a slice kept more than it can hand over. */

/* ------------------------------------------------------------------------
 * idx_score_topk - fused score + exact top-k, without writing [rows, keys]
 * logits (page 1, "Sampled Threshold" and section 1).
 *
 * Per row: a threshold T_r is taken from an odd-stride single-key sample of
 * the row's own scores (page 1, section 2); one scoring pass emits only
 * (score, key) pairs with score >= T_r into a per-row candidate slab of `cap`
 * entries together with the exact count (page 1, section 1 parameter list);
 * an exact radix top-k then selects from the slab.  Rows whose count ended
 * below topk or above cap are re-selected exactly by a full-row rescan, so the
 * result never depends on the sample (the page's own kernel stays lossy here;
 * this library does not).
 *
 *   q, k, k_scale, w, ks, ke : inputs as in the conventions above
 *   rows, keys, H, D, topk   : sizes; keys < 2^31 - 256 and rows * H < 2^31 - 256
 *   max_len                  : an upper bound on ke[r] - ks[r] (0 = keys); it
 *                              sizes the workspace
 *   dt                       : element type of q and k
 *   out_idx                  : [rows, topk] int32 result
 *   ws, ws_bytes             : workspace, >= idx_score_topk_workspace(...)
 * Returns IDX_OK or an error from the list above.
 * ------------------------------------------------------------------------ */
size_t idx_score_topk_workspace(int rows, long long keys, long long max_len, int H, int D,
                                int topk, idx_dtype dt, const idx_options* opt);
idx_status idx_score_topk(const void* q, const void* k, const float* k_scale, const float* w,
                          const int* ks, const int* ke, int rows, long long keys,
                          long long max_len, int H, int D, int topk, idx_dtype dt,
                          int* out_idx, void* ws, size_t ws_bytes, const idx_options* opt,
                          void* stream);

/* ------------------------------------------------------------------------
 * idx_score_topk_host - idx_score_topk on inputs and output in HOST memory:
 * the call a host that holds q, k, ... (and wants the indices back) makes.
 * Page-locked host memory lets the copies run asynchronously and overlap the
 * compute; pageable memory gives the same result without the overlap.
 *
 * The rows are taken in two chunks (whole row blocks each).  k and
 * k_scale go up first, then each chunk's q, w, ks and ke on a copy stream;
 * chunk c is scored and selected on `stream` once its inputs are up, while
 * chunk c + 1 goes up and chunk c - 1's indices come back on a second copy
 * stream.  The call returns with everything enqueued and `stream` waiting
 * for the last copy back: once `stream` is synchronised, out_idx is
 * complete.  The copy streams and their events are the library's, one pair
 * per device; calls on one device are serialised on the host.
 *
 *   q, k, k_scale, w, ks, ke, out_idx : HOST pointers, shapes as for
 *                              idx_score_topk (no alignment needed)
 *   ws, ws_bytes             : DEVICE workspace (256-byte aligned), at least
 *                              idx_score_topk_host_workspace(...): the device
 *                              copies of the inputs and of out_idx, and the
 *                              fused workspace of one chunk
 *   opt                      : as for idx_score_topk; stage_events [0] start
 *                              and [1] end on `stream`
 * Returns IDX_OK or an error from the list above (arguments are checked
 * before anything is copied).
 * ------------------------------------------------------------------------ */
size_t idx_score_topk_host_workspace(int rows, long long keys, long long max_len, int H, int D,
                                     int topk, idx_dtype dt, const idx_options* opt);
idx_status idx_score_topk_host(const void* q, const void* k, const float* k_scale,
                               const float* w, const int* ks, const int* ke, int rows,
                               long long keys, long long max_len, int H, int D, int topk,
                               idx_dtype dt, int* out_idx, void* ws, size_t ws_bytes,
                               const idx_options* opt, void* stream);

/* ------------------------------------------------------------------------
 * idx_topk_from_scores - exact top-k of given fp32 scores (page "[sglang] ROCm
 * DSA Indexer Top-K 최적화": fp32 12-bit coarse histogram, radix tie
 * refinement, full-row rescan when the threshold bin overflows the tie
 * buffer, multi-block row split for long rows at low batch).
 *
 *   scores [rows, row_stride] fp32; row r's visible scores are
 *          scores[r*row_stride + j] for ks[r] <= j < ke[r]
 *          (or scores[r*row_stride + j - ks[r]] with options->relative_rows)
 *   ks may be NULL (all rows start at 0).
 *   out_idx [rows, topk]: ascending j - ks[r], then -1.
 * The result is bit-exact: ties at equal fp32 values (+0 == -0) go to the
 * lower index.  NaN scores are a precondition violation.
 * ws: idx_topk_workspace(...) bytes, 256-byte aligned (IDX_EWORKSPACE if
 * smaller, IDX_EALIGN if misaligned); 0 bytes, and ws may be NULL, unless
 * rows are split (row_split above): then 2 * 8192 * 4 + 8 bytes per block of
 * a split row, 8 bytes per row and 256.  The call allocates nothing, and the
 * workspace needs no clearing between calls.
 * ------------------------------------------------------------------------ */
size_t idx_topk_workspace(int rows, long long row_stride, int topk, const idx_options* opt);
idx_status idx_topk_from_scores(const float* scores, long long row_stride, const int* ks,
                                const int* ke, int rows, int topk, int* out_idx, void* ws,
                                size_t ws_bytes, const idx_options* opt, void* stream);

/* ------------------------------------------------------------------------
 * idx_score_materialise - the two-pass baseline's first pass (page 1,
 * introduction: the full [rows, keys] logits written to global memory).
 * Writes s[r,j] for ks[r] <= j < ke[r] to scores[r*row_stride + (j - ks[r])]
 * (row_stride >= the longest visible range); other entries are not touched.
 * Bit-identical to the scores the fused path compares against its threshold.
 * Feed the result to idx_topk_from_scores with options->relative_rows = 1.
 * ------------------------------------------------------------------------ */
idx_status idx_score_materialise(const void* q, const void* k, const float* k_scale,
                                 const float* w, const int* ks, const int* ke, int rows,
                                 long long keys, int H, int D, idx_dtype dt, float* scores,
                                 long long row_stride, const idx_options* opt, void* stream);

/* ------------------------------------------------------------------------
 * idx_score_topk_noalloc - idx_score_topk for callers that cannot allocate.
 * The paper has no counterpart to this entry point.
 *
 * Some callers only hold pointers to memory that someone else owns (a plugin
 * in a host framework that gives its extensions no allocator, or a serving
 * loop that must not call cudaMalloc, which can synchronize the device) and so
 * cannot pass a workspace.  This call takes the same arguments as
 * idx_score_topk without ws/ws_bytes and runs the same kernels on a scratch
 * array compiled into the library; it allocates no memory.
 *
 *  - Limit: the problem's idx_score_topk_workspace(...) must not exceed
 *    IDX_NOALLOC_SCRATCH_BYTES (32 MiB); larger problems return
 *    IDX_EWORKSPACE and launch nothing.  At topk 2048 with 64K-key rows that
 *    is about 480 query rows per call.
 *  - Every GPU that loads the library holds the 32 MiB array until the
 *    process exits.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - All calls share the one array, and each call leaves its contents behind
 *    (the kernels write every word they later read, so nothing needs
 *    clearing).  Calls whose executions overlap on the GPU, on any stream or
 *    from any thread, race on it: serialize them.
 * ------------------------------------------------------------------------ */
#define IDX_NOALLOC_SCRATCH_BYTES (32ull << 20)
idx_status idx_score_topk_noalloc(const void* q, const void* k, const float* k_scale,
                                  const float* w, const int* ks, const int* ke, int rows,
                                  long long keys, long long max_len, int H, int D, int topk,
                                  idx_dtype dt, int* out_idx, const idx_options* opt,
                                  void* stream);

/* ------------------------------------------------------------------------
 * idx_score_topk_routed - the same result as idx_score_topk, by the faster
 * path for the call's longest row (page "[sglang] logits를 쓰지 않는 top-k",
 * section 4: the fused path is used only when the longest row sees enough
 * keys; below that the filter passes most keys and the dense path is
 * faster).
 *
 * idx_route_fused(rows, max_len, topk) is the gate.  1 (the fused path)
 * when max_len <= max(ceil(2.25 topk), 4096) (every row fits the default
 * candidate slab: all keys are emitted, no sampling); else 0 (the two-pass
 * path: idx_score_materialise into the workspace, then idx_topk_from_scores)
 * for few rows, rows <= SMs / 4 with rows x max_len <= 2^25 (the logits are
 * small and the top-k splits each long row over >= 4 blocks, while the fused
 * path pays its sample, threshold and slab launches: at 8-32 rows x 1M keys,
 * H 32, the two-pass path is 1.36-1.02x faster); else 1 when max_len >= 24576
 * keys and 0 below.  24576 is the crossover measured on GB300 for e4m3
 * q/k with H = 32 and 64 and topk 512 and 2048 (4096 causal rows): the
 * two-pass path is faster from 6144 to 16384 keys, the two are within 1 % at
 * 24576 and 32768 (where the fused path needs no logits workspace), and the
 * fused one is faster at 65536; the page's own rule (8 x topk keys, 16384 at
 * topk 2048) sits below it.  Both
 * paths select exactly the same keys (they compare the same fp32 scores).
 * Arguments as idx_score_topk; max_len 0 = keys.  The workspace of the
 * two-pass route holds the [rows, max_len] fp32 logits.
 * ------------------------------------------------------------------------ */
int idx_route_fused(int rows, long long max_len, int topk);
size_t idx_score_topk_routed_workspace(int rows, long long keys, long long max_len, int H,
                                       int D, int topk, idx_dtype dt, const idx_options* opt);
idx_status idx_score_topk_routed(const void* q, const void* k, const float* k_scale,
                                 const float* w, const int* ks, const int* ke, int rows,
                                 long long keys, long long max_len, int H, int D, int topk,
                                 idx_dtype dt, int* out_idx, void* ws, size_t ws_bytes,
                                 const idx_options* opt, void* stream);

/* ------------------------------------------------------------------------
 * idx_page_table_transform - row-relative top-k positions to physical KV
 * slots of a paged cache (page "[sglang] logits를 쓰지 않는 top-k", section 3:
 * the page-table transform for paged output, page size 64).
 *
 *   idx   [rows, topk] int32, device, rewritten in place: every p >= 0
 *         becomes table[t, p / page_size] * page_size + p % page_size, with
 *         t = row_map[r] (or r when row_map is NULL); negative entries (the
 *         -1 padding) are left as they are.
 *   table [table_rows, table_stride] int32, device: physical page of each
 *         logical page of a table row.
 *   row_map [rows] int32, device, optional: the table row of each query row
 *         (all query rows of one request share its row).
 * A page past table_stride, or a table row outside [0, table_rows), gives -1
 * and raises IDX_DEV_RANGE in options->d_status.  The physical slot must fit
 * in int32 (a precondition, not checked).  Four entries per thread with one
 * 16-byte load and store when topk % 4 == 0 and idx is 16-byte aligned, one
 * otherwise.  No workspace; asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
idx_status idx_page_table_transform(int* idx, int rows, int topk, const int* table,
                                    int table_rows, long long table_stride, const int* row_map,
                                    int page_size, const idx_options* opt, void* stream);

/* ------------------------------------------------------------------------
 * MXFP4 inputs (page "[sglang] logits를 쓰지 않는 top-k", section 1: an fp4
 * indexer whose 128-element keys are 64 bytes).
 *
 * idx_mxfp4_to_e4m3 - n rows of D MXFP4 elements to e4m3, exactly.
 *   x   [n, D/2] bytes, device, 16-byte aligned: two e2m1 elements per byte,
 *       element 2i in the low nibble
 *   sf  [n, D/32] bytes, device: the e8m0 scale (2^(sf - 127)) of each block of
 *       32 consecutive elements
 *   out [n, D] e4m3 bytes, device, 16-byte aligned
 * An e2m1 value (0, ±0.5 ... ±6) times 2^e is an e4m3 value when e lies in
 * [-8, 6] (the OCP recipe e = floor(log2 max|x|) - 2 gives that range for
 * |x| in [2^-6, 2^8)); such elements are converted exactly.  Others (and the
 * NaN scale 255) are saturated to ±448 or flushed to zero and raise
 * IDX_DEV_RANGE.  D % 32 == 0 (IDX_EINVAL); misaligned x or out: IDX_EALIGN.
 *
 * idx_score_topk_mxfp4 / idx_score_materialise_mxfp4 - idx_score_topk and
 * idx_score_materialise on MXFP4 q [rows, H, D/2] + q_sf [rows, H, D/32] and
 * k [keys, D/2] + k_sf [keys, D/32]: q and k are expanded to e4m3 into the
 * workspace and scored by the e4m3 tensor-core path, so the scores are those of
 * the MXFP4 values (bit-identical to the e4m3 path on the same values).  Other
 * arguments as there; the workspaces are the e4m3 path's plus rows*H*D +
 * keys*D bytes (256-byte aligned regions).
 * ------------------------------------------------------------------------ */
idx_status idx_mxfp4_to_e4m3(const uint8_t* x, const uint8_t* sf, long long n, int D,
                             uint8_t* out, const idx_options* opt, void* stream);
size_t idx_score_topk_mxfp4_workspace(int rows, long long keys, long long max_len, int H,
                                      int D, int topk, const idx_options* opt);
idx_status idx_score_topk_mxfp4(const uint8_t* q, const uint8_t* q_sf, const uint8_t* k,
                                const uint8_t* k_sf, const float* k_scale, const float* w,
                                const int* ks, const int* ke, int rows, long long keys,
                                long long max_len, int H, int D, int topk, int* out_idx,
                                void* ws, size_t ws_bytes, const idx_options* opt,
                                void* stream);
size_t idx_score_materialise_mxfp4_workspace(int rows, long long keys, int H, int D);
idx_status idx_score_materialise_mxfp4(const uint8_t* q, const uint8_t* q_sf, const uint8_t* k,
                                       const uint8_t* k_sf, const float* k_scale,
                                       const float* w, const int* ks, const int* ke, int rows,
                                       long long keys, int H, int D, float* scores,
                                       long long row_stride, void* ws, size_t ws_bytes,
                                       const idx_options* opt, void* stream);

/* Static text for a status code. */
const char* idx_status_string(idx_status s);

/* Library version, (major << 16) | minor. */
int idx_version(void);

/* Text of the CUDA error behind the calling thread's last IDX_ECUDA or
 * IDX_EUNSUPPORTED that came from a CUDA call ("" when there was none). */
const char* idx_last_cuda_error(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads); a diagnostic for benchmarks. */
unsigned long long idx_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* IDX_H_ */

/*
 * fathom.h -- C ABI of libfathom, a GB300 (sm_103a) implementation of the
 * Fathom variable-depth bit-plane key scan for top-k sparse decode attention.
 *
 * Source of the method: the review page "Fathom: 쿼리마다 깊이를 바꾸는
 * 스캔으로 1M 토큰 디코딩을 1.67배 빠르게 하다" (jaehun.me, a summary of the
 * Fathom paper).  Section numbers below are the paper's, as that page cites
 * them (§2 evaluation protocol, §3.2 bit-plane K cache, §3.3 per-query read
 * depth, §3.5 rotated basis, §3.6 host-resident store, Appx. A toy example).
 *
 * Conventions shared by every call
 * --------------------------------
 * - A "unit" is one independent (sequence, layer, KV head) triple; units are
 *   packed row-major in that order and every array below has the unit as its
 *   outermost index.
 * - n tokens per unit, nb = ceil(n / 64) blocks of 64 tokens, D channels
 *   (1..128), G query heads sharing the KV head (1, 2, 4 or 8).
 * - Pointers are raw addresses.  "device" means device memory or any memory
 *   the GPU can load from directly (pinned host memory registered with CUDA:
 *   with unified addressing its host pointer is also its device pointer).
 *   The caller owns and allocates every buffer; the library never allocates.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call only enqueues work on that stream: no host
 *   synchronisation, no host read of device results.  Results are valid once
 *   the stream reaches them.  The kernels of fathom_plan, fathom_plan_fixed,
 *   fathom_scan_topk, fathom_scan, fathom_select, fathom_exact_topk, fathom_sparse_attn,
 *   fathom_sparse_attn_planes and fathom_sparse_attn_noalloc are launched with
 *   programmatic stream serialisation: each may be scheduled while the work before it on
 *   the stream is finishing, but it waits for that work to complete before
 *   it reads or writes memory, so the stream order is unchanged.
 * - Every call returns a fathom_status.  Argument errors return FATHOM_EINVAL
 *   before anything is enqueued; CUDA launch errors return FATHOM_ECUDA.
 *   fathom_last_error() returns the calling thread's last message.  Nothing
 *   throws across this ABI and nothing aborts the process.
 * - Inputs are never modified.  Outputs may not alias inputs.
 * - Fault injection (for testing a caller's error handling without a GPU
 *   fault): the environment variable FATHOM_FAULT, read once per process,
 *   holds a comma-separated list of sites.  "launch" makes every call that
 *   would enqueue GPU work return FATHOM_ECUDA after its argument checks,
 *   with nothing enqueued; "launch:<call name>" (e.g.
 *   launch:fathom_scan_topk) does so for that call only.  The message names
 *   the injected fault.  Unset, nothing is injected.
 *
 * Capacity
 * --------
 * The per-unit arrays (key and value rows, the bit-plane store) are laid out
 * for C = (n_cap ? n_cap : n) tokens, cb = ceil(C / 64) blocks: rows
 * [units][C][D], planes [units][D][4][cb], scales [units][D][cb].  Every call
 * reads and writes only the first n tokens (nb blocks) of each unit, so a store
 * allocated once for C tokens grows block by block during decoding
 * (fathom_append_block) and is scanned at its current length n.  With n_cap = 0
 * the layouts are exactly [units][n][D], [units][D][4][nb], [units][D][nb].
 */
#ifndef FATHOM_H
#define FATHOM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FATHOM_MAX_D 128
#define FATHOM_MAX_G 8
#define FATHOM_MAX_K 2048
#define FATHOM_PLANES 4
#define FATHOM_BLOCK 64

typedef enum {
    FATHOM_OK = 0,
    FATHOM_EINVAL = 1,   /* bad argument; nothing was enqueued */
    FATHOM_ECUDA = 2,    /* a CUDA call or launch failed */
    FATHOM_ENOMEM = 3,   /* a caller-provided buffer is too small */
    FATHOM_ETIMEOUT = 4  /* reserved for bounded device waits */
} fathom_status;

typedef enum { FATHOM_F32 = 0, FATHOM_BF16 = 1 } fathom_dtype;

typedef enum {
    FATHOM_WS_SCAN_TOPK = 0,
    FATHOM_WS_SPARSE_ATTN = 1,
    FATHOM_WS_DENSE_ATTN = 2,
    FATHOM_WS_KLT_ONLINE = 3
} fathom_workspace_kind;

/* Which copy of the bit-plane store a scan reads. */
typedef enum {
    FATHOM_SRC_STORE = 0,   /* the store in place, layout [U][D][4][cb] (HBM or pinned host memory) */
    FATHOM_SRC_STAGING = 1, /* the staging area written by fathom_gather (host-resident regime) */
    FATHOM_SRC_ROWS = 2     /* internal: the bf16 key rows (fathom_exact_topk) */
} fathom_source;

/* One slot of the fixed-size run list (§3.6): one per channel, zero length
 * when the channel is inactive.  Offsets count 64-bit plane words or fp16
 * scales, relative to the unit's store (src) and the unit's staging area
 * (dst).  Destinations are contiguous in ascending channel order. */
typedef struct {
    uint32_t src_word;   /* = j * 4 * cb: first plane word of channel j in the store */
    uint32_t n_words;    /* = t_j * nb: channel j's first t_j planes (one contiguous run when
                            cb = nb; planes cb words apart otherwise) */
    uint32_t dst_word;   /* = sum_{j' < j} t_j' * nb */
    uint32_t src_scale;  /* = j * cb */
    uint32_t n_scales;   /* = nb if t_j > 0 else 0 */
    uint32_t dst_scale;  /* = nb * #{j' < j : t_j' > 0} */
} fathom_run;

typedef struct {
    int32_t units;    /* >= 1 */
    int32_t n;        /* tokens per unit, 1 .. 2^28 */
    int32_t D;        /* channels, 1 .. 128 */
    int32_t G;        /* query heads per KV head: 1, 2, 4 or 8 */
    int32_t k;        /* tokens kept per query head, |forced| <= k <= min(n, 2048) */
    int32_t n_sink;   /* first tokens always kept (the pages use 4) */
    int32_t n_recent; /* last tokens always kept (the pages use 32) */
    int32_t n_cap;    /* tokens the per-unit arrays are laid out for: 0 means n, else n <= n_cap
                         (a store that grows during decoding; see "Capacity" above) */
    int32_t scan_ctas_per_sm; /* 0: the scan's grid fills every SM with as many CTAs as fit (3 for
                         G <= 4); 1..3: at most this many per SM, which leaves room on every SM for
                         kernels that other streams run beside the scan (a host-resident scan is
                         bound by the host link, not by its CTAs).  The workspace size follows it. */
} fathom_shape;

/* ---------------------------------------------------------------------- */

/* Calibration statistics (§3.3: Var(k_j) is measured once on calibration
 * keys).  For each unit and channel: mean and unbiased (ddof = 1) variance
 * over m calibration rows, accumulated in fp64 in row order and rounded to
 * fp32 once.
 *   calib [units][m][D] fp32 (device); mean_out (may be NULL), var_out
 *   [units][D] fp32 (device).  m >= 2. */
int fathom_calibrate(int32_t units, int32_t m, int32_t D, const float *calib,
                     float *mean_out, float *var_out, void *stream);

/* Rotated basis (§3.5), calibration.  For each calibration group g (one
 * layer and KV head) from m calibration rows: the mean mu_g (fp64, rows in
 * order), the covariance (fp64, ddof = 1) and its eigen-decomposition by
 * cyclic Jacobi rotations in fp64 (sweeps until the off-diagonal square sum
 * is <= 1e-30 of the total, at most 100): eigenvalues lambda_g in descending
 * order, eigenvectors as the columns of V_g, each with its largest-magnitude
 * component positive.  lambda_g takes the place of the variances in
 * fathom_plan for a rotated store.
 *   calib  [groups][m][D] fp32 (device), m >= 2
 *   mean   [groups][D] fp64 (out, device)
 *   V      [groups][D][D] fp64 (out, device): V[g][j][c] = component j of
 *          eigenvector c
 *   lambda [groups][D] fp32 (out, device)
 * An offline step (store build); fp64 throughout. */
int fathom_calibrate_klt(int32_t groups, int32_t m, int32_t D, const float *calib, double *mean,
                         double *V, float *lambda, void *stream);

/* Rotated keys (§3.5): out[u][i][c] = sum_j (k[u][i][j] - mu_g[j]) V_g[j][c]
 * for unit u in group g = u % groups (units packed sequence, layer, KV head:
 * groups = layers x KV heads shares a layer's and head's basis across the
 * sequences).  k - mu is formed in fp64 and rounded to fp32, V_g is rounded
 * to fp32, the sum is accumulated in fp32.  The result is the input of
 * fathom_quantize_pack (keys_dtype FATHOM_F32) for a rotated store.
 *   keys [units][C][D] fp32 or bf16 (keys_dtype), mean [groups][D] fp64,
 *   V [groups][D][D] fp64, out [units][C][D] fp32 (first n tokens written); all device.
 * Uses shape->units, n, D. */
int fathom_rotate_keys(const fathom_shape *shape, const void *keys, int keys_dtype, int32_t groups,
                       const double *mean, const double *V, float *out, void *stream);

/* Rotated queries (§3.5): q_rot[u][h][c] = sum_j q[u][h][j] V_g[j][c], g =
 * u % groups, fp32 accumulation.  The plan and the scan of a rotated store
 * take q_rot; the exact attention takes the original q.
 *   q [units][G][D] fp32, V [groups][D][D] fp64, q_rot [units][G][D] fp32
 *   (out); all device.  Uses shape->units, D, G. */
int fathom_rotate_query(const fathom_shape *shape, const float *q, int32_t groups, const double *V,
                        float *q_rot, void *stream);

/* Quantise and pack the K store (§3.2).  Per unit, channel j and 64-token
 * block beta: a = max_{i in beta} |k_ij| stored as fp16 (round to nearest
 * even, saturating at 65504); s = a / 8; code c = clip(floor(k / s), -8, 7) + 8
 * in [0, 16) (floor of the exact quotient; a == 0 gives code 8); bit p
 * (p = 0 the MSB) of the 64 codes of the block forms plane word P[beta][j][p],
 * token 64*beta + i at bit i.  Tail tokens past n have all-zero bits and do
 * not enter a.  Reading the first t planes of a channel then gives the t-bit
 * mid-rise code c >> (4 - t).
 *   keys   [units][C][D], fp32 or bf16 (keys_dtype), device (first n tokens read)
 *   planes [units][D][4][cb] uint64 (out, device; first nb blocks written): channel j's planes 0..3
 *          each contiguous over the sequence (§3.6)
 *   scales [units][D][cb] fp16 bit patterns (out, device)
 * Uses shape->units, n, D. */
int fathom_quantize_pack(const fathom_shape *shape, const void *keys, int keys_dtype,
                         uint64_t *planes, uint16_t *scales, void *stream);

/* Decode-time append (the step before the scan in a decode loop, §2, §3.2):
 * quantise block `block` (tokens 64*block .. 64*block + count - 1, 1 <= count
 * <= 64) of every unit into the store, exactly as fathom_quantize_pack would
 * code a sequence of 64*block + count tokens: a block that is still filling
 * is coded again as its tokens arrive (its maximum, and so its codes, can
 * change); tokens past `count` have all-zero bits and do not enter the
 * maximum.  Reads keys [units][C][D] (the rows buffer, fp32 or bf16) at that
 * block, writes its 4 plane words and its scale per channel; other blocks are
 * untouched.  Requires 64*block + count <= C (the shape's capacity); shape->n
 * is not used. */
int fathom_append_block(const fathom_shape *shape, const void *keys, int keys_dtype, int32_t block,
                        int32_t count, uint64_t *planes, uint16_t *scales, void *stream);

/* Per-query-group read plan (§3.3, §3.6).  Per unit:
 *   g_j = (sum_h q_hj^2) * var_j  (fp64, h ascending);
 *   depth t_j(theta) = #{m in 0..3 : g_j >= theta * 2^(2m+1)}
 *                    = clip(round(log4(g_j / theta)), 0, 4)  (ties round up);
 *   theta from 30 steps of geometric bisection mid = sqrt(lo * hi) on
 *   [lo, hi], keeping hi feasible (sum_j t_j(hi) <= budget), and the result is
 *   t(hi), theta = hi: the smallest probed theta that fits the budget.
 *   bracket NULL: hi = max_j g_j, lo = min_{g_j > 0} g_j / 512; if t(lo) fits
 *   the budget the bisection is skipped and theta = lo (budget not binding);
 *   if every g_j is 0, all depths are 0 and theta = 0.
 *   bracket non-NULL: [units][2] {lo, hi} fp64 used as given (hi must fit).
 * Every decision uses only IEEE-exact fp64 operations in a fixed order, so the
 * plan is reproducible bit for bit.
 *   q [units][G][D] fp32, var [units][D] fp32, budget [units] int32 >= 0
 *   depth [units][D] uint8 (out), theta [units] fp64 (out, or NULL),
 *   runs [units][D] fathom_run (out; see fathom_run).
 * theta NULL: theta is not written, and the depths and runs are the same as
 * with it.  Without an explicit bracket the call then skips the 30 dependent
 * bisection steps wherever they cannot change the depths: theta fits the
 * budget exactly when it lies above b*, the (budget + 1)-th largest of the
 * breakpoints g_j / 2^(2m+1), and the final theta lies within a factor
 * 1 + 4x of b* (x = (e + 1) ln2 / 2^30 + 2^-51, e the exponent span of the
 * bracket); when no breakpoint lies in that range the depths are those at the
 * next breakpoint above b*.  Otherwise the bisection runs as above.
 * All pointers device. */
int fathom_plan(const fathom_shape *shape, const float *q, const float *var,
                const int32_t *budget, const double *bracket, uint8_t *depth,
                double *theta, fathom_run *runs, void *stream);

/* Fixed-depth comparison plan: the n_channels channels of largest g_j (ties:
 * lower j) at depth depth_each, all others 0 (32 channels x 4 planes is the
 * byte-equivalent of a 136-bit scan).  Outputs as fathom_plan; theta is not
 * written.  1 <= n_channels <= D, 1 <= depth_each <= 4. */
int fathom_plan_fixed(const fathom_shape *shape, const float *q, const float *var,
                      int32_t n_channels, int32_t depth_each, uint8_t *depth,
                      fathom_run *runs, void *stream);

/* Gather (§3.6): for every unit and every channel, copy run[j].n_words plane
 * words from store_planes + src_word to stage_planes + dst_word (the first nb
 * words of each of the channel's t_j planes, which lie cb words apart) and
 * run[j].n_scales scales likewise; zero-length runs copy nothing, so the run
 * list needs no host synchronisation.  The store is typically pinned host
 * memory read over the host link; staging is device memory.
 *   store_planes/store_scales: the store as written by fathom_quantize_pack
 *   runs [units][D] from fathom_plan / fathom_plan_fixed
 *   stage_planes [units][stage_words], stage_scales [units][stage_nscales]
 *   (device): per-unit strides in words / scales
 * Runs whose destination would pass the unit's stage_words / stage_nscales
 * are clipped at that end (a plan that fits its budget B never is when
 * stage_words >= B * nb and stage_nscales >= min(B, D) * nb). */
int fathom_gather(const fathom_shape *shape, const uint64_t *store_planes,
                  const uint16_t *store_scales, const fathom_run *runs,
                  uint64_t *stage_planes, uint16_t *stage_scales, size_t stage_words,
                  size_t stage_nscales, void *stream);

/* Scan and select (§3.2, §3.3, §2).  For every unit, query head h and token i:
 *   s_h(i) = sum_{j : t_j > 0} q_hj * (c_t + 0.5 - 2^(t-1)) * a / 2^(t-1)
 * with t = t_j, c_t the code prefix read from channel j's first t planes and
 * a its block scale, accumulated in fp32 (one pass over the planned planes
 * serves all G heads).  Then per head the kept set is the first n_sink and
 * the last n_recent tokens plus the k - |forced| other tokens of largest
 * s_h (ties: lower index), written in ascending token order with their
 * scores.
 *   planes/scales: source (FATHOM_SRC_STORE: the store [U][D][4][cb] /
 *   [U][D][cb]; FATHOM_SRC_STAGING: staging [U][stage_words] /
 *   [U][stage_nscales] laid out by the run list; the strides are ignored
 *   for FATHOM_SRC_STORE)
 *   runs [units][D], q [units][G][D] fp32
 *   topk_idx [units][G][k] int32 (out), topk_score [units][G][k] fp32 (out)
 *   scores_opt NULL, or [units][G][n] fp32 (out): every token's score
 *   workspace: device scratch of at least
 *   fathom_workspace_size(shape, FATHOM_WS_SCAN_TOPK) bytes, 256-byte
 *   aligned, zero-filled before its first use; each call leaves it ready for
 *   the next call.  Calls that share a workspace must not overlap in time. */
int fathom_scan_topk(const fathom_shape *shape, const uint64_t *planes,
                     const uint16_t *scales, int source, size_t stage_words,
                     size_t stage_nscales, const fathom_run *runs, const float *q,
                     int32_t *topk_idx, float *topk_score, float *scores_opt,
                     void *workspace, size_t workspace_bytes, void *stream);

/* The two halves of fathom_scan_topk, for callers that overlap one group of
 * units' selection with the next group's scan on another stream.
 * fathom_scan (§3.2, §3.3) scores every token for all G heads and leaves each
 * CTA's candidate keys, threshold and the forced tokens' scores in the
 * workspace (scores_opt as in fathom_scan_topk).  fathom_select (§2) merges
 * those lists into the kept sets, rescans exactly any chunk whose threshold may
 * have dropped a winner (reading planes, scales, runs and q again), and writes
 * topk_idx and topk_score.  Together, with the same arguments and workspace and
 * fathom_select ordered after fathom_scan, they compute exactly what
 * fathom_scan_topk computes; until fathom_select has run, the workspace must
 * not be given to another scan.  Arguments, layouts and errors as in
 * fathom_scan_topk. */
int fathom_scan(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales, int source,
                size_t stage_words, size_t stage_nscales, const fathom_run *runs, const float *q,
                float *scores_opt, void *workspace, size_t workspace_bytes, void *stream);
int fathom_select(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales, int source,
                  size_t stage_words, size_t stage_nscales, const fathom_run *runs, const float *q,
                  int32_t *topk_idx, float *topk_score, void *workspace, size_t workspace_bytes,
                  void *stream);

/* Rotated basis without calibration data (Appx. D: the mean, eigenbasis and
 * eigenvalues of a session's own keys; the pages report this under 1 ms at
 * 100k tokens).  Per unit, over its n live key rows: mean mu (fp32 runs of 64
 * tokens folded in fp64), covariance (ddof = 1) of the rows centred on mu
 * rounded to fp32 (fp32 products, per-slice fp32 sums combined in fp64 in a
 * fixed order), eigen-decomposition by parallel cyclic Jacobi in fp32
 * (eigenvalues descending, each eigenvector's largest-magnitude component
 * positive).  Each unit is its own group: pass groups = units to
 * fathom_rotate_keys and fathom_rotate_query, and lambda to fathom_plan.
 *   k_rows [units][C][D] bf16 (device or pinned host), n >= 2 live tokens
 *   mean   [units][D] fp64 (out, device)
 *   V      [units][D][D] fp64 (out, device): V[u][j][c] = component j of
 *          eigenvector c (fp32 values)
 *   lambda [units][D] fp32 (out, device)
 *   workspace: at least fathom_workspace_size(shape, FATHOM_WS_KLT_ONLINE)
 *   bytes, 256-byte aligned (no zero-fill needed). */
int fathom_klt_online(const fathom_shape *shape, const uint16_t *k_rows, double *mean, double *V,
                      float *lambda, void *workspace, size_t workspace_bytes, void *stream);

/* Fidelity reference, exact top-k (§2 evaluation, the "exact top-k" the
 * pages compare against): the same kept set as fathom_scan_topk (first n_sink
 * and last n_recent tokens plus the k - |forced| others of largest score per
 * head, ties to the lower index, ascending output) with every token scored
 * exactly from its bf16 key row, s_h(i) = q_h . k_i in fp32, all D channels.
 *   k_rows [units][C][D] bf16 (device or pinned host), q [units][G][D] fp32
 *   topk_idx, topk_score, scores_opt, workspace: as fathom_scan_topk (the same
 *   workspace size). */
int fathom_exact_topk(const fathom_shape *shape, const uint16_t *k_rows, const float *q,
                      int32_t *topk_idx, float *topk_score, float *scores_opt,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Fidelity reference, dense attention (§2: the pages measure the relative
 * L2 error of the sparse output against full attention): per unit and head,
 * o_h = sum over all n tokens of softmax_i(q_h . k_i / sqrt(D)) v_i, bf16 rows,
 * fp32 accumulation; the same arithmetic as fathom_sparse_attn over every token.
 *   k_rows, v_rows [units][C][D] bf16 (device or pinned host), q [units][G][D]
 *   fp32, out [units][G][D] fp32 (out)
 *   workspace: at least fathom_workspace_size(shape, FATHOM_WS_DENSE_ATTN)
 *   bytes, 256-byte aligned, zero-filled before its first use; left ready
 *   for the next call. */
int fathom_dense_attn(const fathom_shape *shape, const uint16_t *k_rows, const uint16_t *v_rows,
                      const float *q, float *out, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Fidelity diagnostic, relative L2 error per row (§4, §5: the attention
 * output error the pages report): err[r] = ||a_r - ref_r||_2 / ||ref_r||_2
 * with both sums in fp64; ||a_r||_2 when ref_r is all zeros.
 *   a, ref [rows][D] fp32, err [rows] fp64 (out), all device memory.
 *   rows == 0 enqueues nothing. */
int fathom_rel_err(int32_t rows, int32_t D, const float *a, const float *ref, double *err,
                   void *stream);

/* Fidelity diagnostic, agreement of two kept sets (§5: agreement with the
 * exact top-k): count[r] = number of indices row r of a shares with row r of
 * b.  a, b [rows][k] int32, each row strictly ascending (as fathom_scan_topk
 * and fathom_exact_topk write them); count [rows] int32 (out); device memory.
 * Rows that are not ascending give an unspecified count. */
int fathom_set_overlap(int32_t rows, int32_t k, const int32_t *a, const int32_t *b,
                       int32_t *count, void *stream);

/* Greedy per-layer budgets (§3.4: bits go to the layer whose error falls the
 * most per bit, B_l in {24, ..., 128} around a target mean).  Host code, no
 * GPU.  The budget levels are b_min + step * i, i = 0 .. levels - 1, and
 * err [layers][levels] (host, fp64, finite) is each layer's measured error at
 * each level.  Every layer starts at b_min; layers * (b_mean - b_min) / step
 * times, `step` bits go to the layer with the largest err[l][i] - err[l][i+1]
 * at its current level i (ties to the lower layer; layers at the top level
 * take no more), so the budgets average exactly b_mean.
 *   budgets [layers] int32 (host, out).
 *   FATHOM_EINVAL when b_mean is not one of the levels. */
int fathom_greedy_budgets(int32_t layers, int32_t levels, const double *err, int32_t b_min,
                          int32_t step, int32_t b_mean, int32_t *budgets);

/* Exact sparse attention over the winners (§1, §2, §3.1).  The winners' rows
 * are fetched at full precision (bf16 K and V rows; at most G * k per unit),
 * and per head
 *   o_h = sum_{i in S_h} softmax_i(q_h . k_i / sqrt(D)) v_i
 * with fp32 accumulation and no mass for unselected tokens.  Each head reads
 * the rows of its own kept set, so a row kept by several heads is read once
 * per head (calls with more than 65535 (unit, head) pairs read the union of a
 * unit's kept sets once instead).
 *   k_rows, v_rows [units][C][D] bf16 bit patterns (device or pinned host)
 *   q [units][G][D] fp32, topk_idx [units][G][k] int32, each row strictly
 *   ascending as fathom_scan_topk writes it (other rows give an unspecified
 *   result; entries outside [0, n) are skipped, never read)
 *   out [units][G][D] fp32 (out)
 *   workspace: at least fathom_workspace_size(shape, FATHOM_WS_SPARSE_ATTN)
 *   bytes, same rules as fathom_scan_topk's. */
int fathom_sparse_attn(const fathom_shape *shape, const uint16_t *k_rows,
                       const uint16_t *v_rows, const float *q, const int32_t *topk_idx,
                       float *out, void *workspace, size_t workspace_bytes, void *stream);

/* Sparse attention with the winners' keys rebuilt from the bit-plane store
 * (§7 names this as the unbuilt next step: the 4-bit channel-major store as
 * the K cache itself, no bf16 K rows).  As fathom_sparse_attn, except that
 * the key of a winner i is read from all four planes of its block and
 * channel, k_ij = (c_ij - 7.5) a_{i/64, j} / 8 (the 4-bit mid-rise value, exact
 * in fp32).  Each winner reads 4 D plane words and D scales from separate
 * 32-byte sectors, against one 2 D-byte row: this is the single-token
 * reconstruction cost the pages name.
 *   planes [units][D][4][cb], scales [units][D][cb] (the store, device or
 *   pinned host), v_rows [units][C][D] bf16, q [units][G][D] fp32 (the scan's
 *   queries: for a rotated store q' = q V, whose logits differ from q . k by
 *   q . mu, the same for every token), topk_idx [units][G][k] ascending,
 *   out [units][G][D] fp32 (out), workspace: as fathom_sparse_attn. */
int fathom_sparse_attn_planes(const fathom_shape *shape, const uint64_t *planes,
                              const uint16_t *scales, const uint16_t *v_rows, const float *q,
                              const int32_t *topk_idx, float *out, void *workspace,
                              size_t workspace_bytes, void *stream);

/* fathom_sparse_attn without a workspace argument, for callers that cannot
 * allocate device memory for the library: a host framework that owns all
 * device memory and does not let plug-ins call cudaMalloc (which would also
 * synchronise the device), or a decode loop that must never allocate.  The
 * paper has no counterpart to this call; it is a packaging choice of this
 * library.  Same arguments, same results as fathom_sparse_attn.
 *   Scratch: a fixed 8 MiB array inside the library, held by every GPU that
 *   loads the library until the process exits; shapes whose
 *   fathom_workspace_size(shape, FATHOM_WS_SPARSE_ATTN) exceeds 8 MiB are
 *   rejected with FATHOM_EINVAL and nothing is enqueued.
 *   Every call looks up the array's device address with the calling thread's
 *   current device (a host-side query; nothing is cached, so the address stays
 *   right after cudaDeviceReset).  The first call on a device may load the
 *   library's device code there: make that first call before any stream
 *   capture.
 *   Every call clears the array's ticket words on `stream` and then uses the
 *   one shared array, so calls whose work overlaps on the GPU (other streams,
 *   other threads) race and must be serialised by the caller.
 *   Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. */
int fathom_sparse_attn_noalloc(const fathom_shape *shape, const uint16_t *k_rows,
                               const uint16_t *v_rows, const float *q, const int32_t *topk_idx,
                               float *out, void *stream);

/* Workspace bytes a call needs for this shape (0 if the shape is invalid). */
size_t fathom_workspace_size(const fathom_shape *shape, int which);

/* The calling thread's last error message ("" if none). */
const char *fathom_last_error(void);

/* Library version string. */
const char *fathom_version(void);

/* Bounds checks of a debug build (compiled with -DFATHOM_DEBUG; the paper has no
 * counterpart: they stand in for a memory checker).  In such a build every
 * load or store of the scan, gather and attention kernels whose index comes
 * from data (run lists, staged offsets, kept lists) first checks that the
 * index lies inside the buffer the call was given; a failed check skips the
 * access and records, per kernel file, the first failure as
 * (site << 48) | index, the sites being: 1-4 scan staging and loads of plane
 * words and scales, 5 a forced token's slot, 6-7 gather source and
 * destination, 8 an attention row.  This call synchronises the calling
 * thread's device and writes the records of the scan, gather and attention
 * files to first_failure[0..2] (0: no failure).  mode 0 reads them, mode 1
 * reads and clears them, mode 2 first plants a self-test record (site 15,
 * index 0x5e1f, no memory access) in each file and then reads, to test the
 * reporting path.  A build without the checks writes zeros and returns
 * FATHOM_EINVAL. */
int fathom_debug_status(int mode, uint64_t *first_failure);

#ifdef __cplusplus
}
#endif

#endif /* FATHOM_H */

// fathom_internal.cuh -- definitions shared by the libfathom CUDA sources.
// Method source: the Fathom review page ("Fathom: 쿼리마다 깊이를 바꾸는
// 스캔으로 1M 토큰 디코딩을 1.67배 빠르게 하다"); sections are the paper's.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "fathom.h"

namespace fathom {

// ---------------------------------------------------------------- errors
void set_error(const char *fmt, ...);
int launch_status(const char *what);   // FATHOM_OK or FATHOM_ECUDA (+ message)

// ---------------------------------------------------------------- debug checks
// A build with -DFATHOM_DEBUG checks, before each load or store whose index
// comes from data (run lists, kept lists, staged offsets), that the index lies
// inside the buffer the call was given.  A failed check records its site and
// the offending index in this translation unit's debug word (the first failure
// wins), and the access is skipped, so a bad index never reaches memory and
// the kernel still ends normally.  fathom_debug_status() reads the words.  In
// the default build every check is the constant true and costs nothing.
enum DebugSite : unsigned {
    kDbgScanStagePlanes = 1,   // scan: a staged plane word outside the store or staging area
    kDbgScanStageScales = 2,   // scan: a staged scale outside it
    kDbgScanLoadPlanes = 3,    // scan (synchronous staging): a plane word outside it
    kDbgScanLoadScales = 4,    // scan (synchronous staging): a scale outside it
    kDbgScanForced = 5,        // scan: a forced token's slot outside [0, |forced|)
    kDbgGatherSrc = 6,         // gather: a source word or scale outside the store
    kDbgGatherDst = 7,         // gather: a destination outside the staging area
    kDbgAttnRow = 8,           // attention: a kept row outside [0, n)
    kDbgSelfTest = 15          // a record planted on request, to test the reporting path
};
#ifdef FATHOM_DEBUG
static __device__ unsigned long long g_fathom_dbg;   // one per translation unit
__device__ __forceinline__ bool debug_check(bool ok, unsigned site, unsigned long long value) {
    if (!ok) atomicCAS(&g_fathom_dbg, 0ull, ((unsigned long long)site << 48) | (value & 0xffffffffffffull));
    return ok;
}
#define FATHOM_CHECK(cond, site, value) ::fathom::debug_check((cond), (site), (unsigned long long)(value))
// Each translation unit that checks defines its reader with this macro, and a
// one-thread kernel that plants a self-test record (no memory access).
#define FATHOM_DEBUG_READER(name)                                                        \
    __global__ void name##_plant_kernel() { FATHOM_CHECK(false, kDbgSelfTest, 0x5e1f); } \
    void name##_plant() { name##_plant_kernel<<<1, 1>>>(); }                            \
    unsigned long long name(bool reset) {                                               \
        unsigned long long v = 0;                                                       \
        cudaMemcpyFromSymbol(&v, g_fathom_dbg, sizeof v);                               \
        if (reset) { const unsigned long long z = 0; cudaMemcpyToSymbol(g_fathom_dbg, &z, sizeof z); } \
        return v;                                                                       \
    }
#else
#define FATHOM_CHECK(cond, site, value) (true)
#define FATHOM_DEBUG_READER(name)
#endif
#ifdef FATHOM_DEBUG
unsigned long long debug_read_scan(bool reset);
unsigned long long debug_read_gather(bool reset);
unsigned long long debug_read_attn(bool reset);
void debug_read_scan_plant();
void debug_read_gather_plant();
void debug_read_attn_plant();
#endif

// ---------------------------------------------------------------- geometry
__host__ __device__ inline int num_blocks(int n) { return (n + FATHOM_BLOCK - 1) / FATHOM_BLOCK; }

// Forced tokens (§2): the first n_sink and the last n_recent tokens.  With
// ns = min(n_sink, n) and r0 = max(ns, n - n_recent), token i is forced iff
// i < ns or i >= r0, and |forced| = ns + n - r0.
// Tokens and 64-token blocks the per-unit arrays are laid out for (the
// shape's capacity; n when no capacity is given).
inline int cap_tokens(const fathom_shape &s) { return s.n_cap > 0 ? s.n_cap : s.n; }
inline int cap_blocks(const fathom_shape &s) { return num_blocks(cap_tokens(s)); }

struct Forced {
    int ns, r0, nf;
};
__host__ __device__ inline Forced forced_range(int n, int n_sink, int n_recent) {
    Forced f;
    f.ns = n_sink < n ? n_sink : n;
    int r = n - n_recent;
    f.r0 = r > f.ns ? r : f.ns;
    f.nf = f.ns + (n - f.r0);
    return f;
}

// Scan decomposition: `chunks` CTAs per unit share its 32-block sub-chunks.  The
// grid is one-dimensional, units x chunks CTAs; CTA i works on unit i / chunks
// (chunk i % chunks), or with unit_fast on unit i % units (chunk i / units),
// so that every unit has a CTA among the first to start.
struct ScanGrid {
    int chunks;
    int unit_fast;
};
constexpr int kScanMaxChunks = 4096;
ScanGrid scan_grid(const fathom_shape &s);
int device_sm_count();
int scan_resident_ctas(int G);   // resident scan CTAs per SM (0: no device)

constexpr int kScanThreads = 256;
constexpr int kSubBlocks = 32;               // blocks per sub-chunk (8 threads per block)
constexpr int kSubTokens = kSubBlocks * 64;  // 2048
constexpr int kPruneSlack = 256;             // a pruned list keeps <= k' + slack keys

// Candidate list capacity per (CTA, head): after a prune a list holds at most
// k' + slack keys and a sub-chunk appends at most kSubTokens, so at least two
// sub-chunks fit between prunes.
int scan_cand_cap(const fathom_shape &s);

#define FATHOM_MERGE_MAX_LISTS 1024

// Per-CTA candidate target m: about four times a chunk's share of k', at
// least 64, at most k'.  Each chunk keeps its top-m per head in the first pass.
int scan_m_sel(int chunks, int k_sel);
int scan_m_first(int n_sub, int k_sel, int m_sel);
// Merge parts per (unit, head): about 8192 expected candidate keys per part.
int merge_parts(int chunks, int m_sel);

struct ScanWorkspace {
    int parts;
    size_t cand_off, cnt_off, tau_off, flags_off, forced_off, part_keys_off, part_cnt_off,
        ticket_off, dirty_off, sub_ctr_off, sub_owner_off, total;
};
ScanWorkspace scan_workspace_layout(const fathom_shape &s);

constexpr int kAttnThreads = 256;
constexpr int kAttnRowsMax = 512;   // kept-list entries per CTA, at most
// Two launch forms share one workspace: the union form (a unit's G heads in one
// grid row: every kept row fetched once, all G dot products computed for it) and
// the per-head form (each (unit, head) its own grid row: one dot product per
// fetched row, rows kept by several heads fetched once per head).  The partial
// states and the tickets are sized for whichever needs more.
struct AttnWorkspace {
    int rows;     // kept-list entries per CTA (union form)
    int splits;
    int ph_rows;  // the same for the per-head form (units x G rows of one head each)
    int ph_splits;
    size_t part_off, ticket_off, total;
};
AttnWorkspace attn_workspace_layout(const fathom_shape &s);
AttnWorkspace dense_workspace_layout(const fathom_shape &s);   // dense attention (fidelity reference)

// ---------------------------------------------------------------- selection keys
// A 64-bit key orders (score descending, token index ascending): the high
// word is the fp32 score mapped to an order-preserving unsigned integer
// (-0 folded onto +0), the low word is ~index.  Larger key = better token.
__device__ __forceinline__ uint32_t order_f32(float s) {
    s = s + 0.0f;                                   // -0 -> +0
    uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unorder_f32(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
    return __uint_as_float(u);
}
__device__ __forceinline__ uint64_t make_key(float s, uint32_t idx) {
    return ((uint64_t)order_f32(s) << 32) | (uint64_t)(0xffffffffu - idx);
}
__device__ __forceinline__ uint32_t key_index(uint64_t key) {
    return 0xffffffffu - (uint32_t)(key & 0xffffffffu);
}
__device__ __forceinline__ float key_score(uint64_t key) { return unorder_f32((uint32_t)(key >> 32)); }

// 16-byte asynchronous global -> shared copies (zero-filled when bytes == 0).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src, int bytes) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(gmem_src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Programmatic dependent launch.  The kernels of a decode step (plan, scan,
// merge, attention) are launched so that the next one may start while the
// previous one is finishing: every such kernel first waits until the kernel
// before it in the stream has completed and its writes are visible
// (griddepcontrol.wait, a no-op when the launch had no such dependency), then
// allows its own successor to launch.  Stream order is unchanged; only the
// launch latency between dependent kernels overlaps the previous kernel's
// tail.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, (KArgs)args...);
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device, size);
// later launches skip the driver call.
bool smem_attr_needed(const void *func, size_t bytes);   // thread-safe cache lookup/insert
template <typename F>
inline void ensure_smem(F *func, size_t bytes) {
    if (smem_attr_needed((const void *)func, bytes))
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// ---------------------------------------------------------------- launchers
int launch_calibrate(int units, int m, int D, const float *calib, float *mean, float *var,
                     cudaStream_t st);
int launch_calibrate_klt(int groups, int m, int D, const float *calib, double *mean, double *vec,
                         float *lambda, cudaStream_t st);
int launch_rotate_keys(const fathom_shape &s, const void *keys, int dtype, int groups, const double *mean,
                       const double *vec, float *out, cudaStream_t st);
int launch_rotate_query(const fathom_shape &s, const float *q, int groups, const double *vec, float *out,
                        cudaStream_t st);
int launch_append(const fathom_shape &s, const void *keys, int dtype, int block, int count, uint64_t *planes,
                  uint16_t *scales, cudaStream_t st);
int launch_quantize(const fathom_shape &s, const void *keys, int dtype, uint64_t *planes,
                    uint16_t *scales, cudaStream_t st);
int launch_plan(const fathom_shape &s, const float *q, const float *var, const int32_t *budget,
                const double *bracket, uint8_t *depth, double *theta, fathom_run *runs,
                cudaStream_t st);
int launch_plan_fixed(const fathom_shape &s, const float *q, const float *var, int n_sel,
                      int t_fixed, uint8_t *depth, fathom_run *runs, cudaStream_t st);
int launch_gather(const fathom_shape &s, const uint64_t *sp, const uint16_t *ss,
                  const fathom_run *runs, uint64_t *dp, uint16_t *ds, size_t stage_words,
                  size_t stage_scales, cudaStream_t st);
// Which launches of scan + top-k to enqueue: all of them, the first-pass scan
// only, or the selection only (merge, exact second pass, second merge).
enum ScanPart { SCAN_PART_ALL = 0, SCAN_PART_SCAN = 1, SCAN_PART_SELECT = 2 };
int launch_scan_topk(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                     int source, size_t stage_words, size_t stage_scales, const fathom_run *runs,
                     const float *q, int32_t *idx, float *score, float *scores_opt, void *ws,
                     cudaStream_t st, int part = SCAN_PART_ALL);
int launch_sparse_attn(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows,
                       const float *q, const int32_t *idx, float *out, void *ws, cudaStream_t st);
int launch_dense_attn(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows, const float *q,
                      float *out, void *ws, cudaStream_t st);
int launch_sparse_attn_planes(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                              const uint16_t *vrows, const float *q, const int32_t *idx, float *out, void *ws,
                              cudaStream_t st);
int launch_sparse_attn_noalloc(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows,
                               const float *q, const int32_t *idx, float *out, cudaStream_t st);

// Online rotated basis: partial sums per (unit, slice of tps tokens).
struct KltOnlineWs {
    int slices = 1, tps = 0;
    size_t mean_off = 0, cov_off = 0, total = 0;
};
KltOnlineWs klt_online_layout(const fathom_shape &s);
int launch_klt_online(const fathom_shape &s, const uint16_t *rows, double *mean, double *vec, float *lambda,
                      void *ws, cudaStream_t st);
int launch_rel_err(int rows, int D, const float *a, const float *ref, double *err, cudaStream_t st);
int launch_set_overlap(int rows, int k, const int32_t *a, const int32_t *b, int32_t *count, cudaStream_t st);
int greedy_budgets(int layers, int levels, const double *err, int b_min, int step, int b_mean, int32_t *budgets);

}  // namespace fathom

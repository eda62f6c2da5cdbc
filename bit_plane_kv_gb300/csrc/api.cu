// api.cu -- the extern "C" boundary of libfathom: argument checks, error
// reporting and workspace layouts.  All arithmetic lives in the kernels.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include <cmath>

#include "fathom_internal.cuh"

namespace fathom {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

int launch_status(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s: %s", what, cudaGetErrorString(e));
        return FATHOM_ECUDA;
    }
    return FATHOM_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool smem_attr_needed(const void *func, size_t bytes) {
    struct Entry { const void *f; int dev; size_t bytes; };
    static std::mutex mu;
    static Entry table[64];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        if (table[i].f == func && table[i].dev == dev) {
            if (table[i].bytes >= bytes) return false;
            table[i].bytes = bytes;
            return true;
        }
    }
    if (used < 64) table[used++] = Entry{func, dev, bytes};
    return true;
}

// Streaming multiprocessors of the current device (0 if no device answers).
int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev] = v;
    }
    return cache[dev];
}

// Makespan, in sub-chunk times, of a scan whose CTAs start in launch order as
// resident slots free up, CTA i working on unit i % units (unit_fast) or
// i / chunks.  A running CTA takes its unit's sub-chunks one at a time from a
// counter it shares with the unit's other CTAs (one time unit each) and ends
// with its fixed work (one unit: plan prologue, first threshold, final
// shrink); a CTA that finds the counter exhausted ends at once (0.1).
static double scan_makespan(long long units, int n_sub, int chunks, long long slots, bool unit_fast) {
    const long long total = units * chunks;
    std::vector<int> ctr((size_t)units, 0);
    std::vector<char> took((size_t)total, 0);
    using Ev = std::pair<double, long long>;
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> q;
    long long next = 0;
    for (; next < total && next < slots; ++next) q.push({0.0, next});
    double end = 0.0;
    while (!q.empty()) {
        const Ev e = q.top();
        q.pop();
        const long long i = e.second;
        const long long u = unit_fast ? i % units : i / chunks;
        if (ctr[(size_t)u] < n_sub) {
            ++ctr[(size_t)u];
            took[(size_t)i] = 1;
            q.push({e.first + 1.0, i});
            continue;
        }
        const double t = e.first + (took[(size_t)i] ? 1.0 : 0.1);
        end = t > end ? t : end;
        if (next < total) q.push({t, next++});
    }
    return end;
}

ScanGrid scan_grid(const fathom_shape &s) {
    // A unit's `chunks` CTAs share its sub-chunks (32 blocks) through a counter,
    // so a CTA that runs faster scores more of them.  With `slots` CTAs resident
    // at once (SMs x resident scan CTAs per SM; 152 x 3 on GB300 when no device
    // answers), the CTAs start in launch order as slots free up.  Launched
    // chunk-fastest, a unit's CTAs run together and the scan takes about
    // waves x (sub-chunks per CTA + 1) sub-chunk times.  With fewer units than
    // slots and no chunk count that fills the slots exactly, a unit-fastest
    // launch starts every unit at once and lets the later CTAs join the units
    // still running (the others find their counter spent and end at once):
    // its makespan comes from simulating that schedule.  Take the order and
    // chunk count with the smallest time (ties: chunk-fastest, fewer CTAs).
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;
    int res = scan_resident_ctas(s.G);
    if (res <= 0) res = (s.G <= 4) ? 3 : 1;
    if (s.scan_ctas_per_sm > 0 && s.scan_ctas_per_sm < res) res = s.scan_ctas_per_sm;
    const long long slots = (long long)sms * res;
    const int nb = num_blocks(s.n);
    const int n_sub = (nb + kSubBlocks - 1) / kSubBlocks;
    const int max_chunks = n_sub < kScanMaxChunks ? n_sub : kScanMaxChunks;
    int best = 1;
    double best_cost = -1.0;
    for (int c = 1; c <= max_chunks; ++c) {
        const long long waves = ((long long)s.units * c + slots - 1) / slots;
        const double cost = (double)(waves * ((n_sub + c - 1) / c + 1));
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = c; }
        if ((long long)s.units * c >= 8 * slots) break;   // more CTAs than this never pay
    }
    ScanGrid g;
    g.unit_fast = 0;
    if ((long long)s.units < slots && slots % s.units != 0 && (long long)s.units * n_sub <= 1000000) {
        static std::mutex mu;
        static long long key[16][3];
        static int val[16];
        static int used = 0, next_slot = 0;
        std::lock_guard<std::mutex> lock(mu);
        int hit = -1;
        for (int i = 0; i < used; ++i)
            if (key[i][0] == s.units && key[i][1] == n_sub && key[i][2] == slots) hit = i;
        int uf_best = 0;
        if (hit >= 0) {
            uf_best = val[hit];
        } else {
            double uf_cost = best_cost;
            const int q0 = (int)(slots / s.units) + 1;
            for (int c = q0; c <= 4 * q0 && c <= max_chunks; ++c) {
                const double t = scan_makespan(s.units, n_sub, c, slots, true);
                if (t < uf_cost) { uf_cost = t; uf_best = c; }
            }
            const int slot_i = used < 16 ? used++ : next_slot++ % 16;
            key[slot_i][0] = s.units; key[slot_i][1] = n_sub; key[slot_i][2] = slots;
            val[slot_i] = uf_best;
        }
        if (uf_best > 0) { best = uf_best; g.unit_fast = 1; }
    }
    g.chunks = best;
    return g;
}

int scan_cand_cap(const fathom_shape &s) {
    Forced f = forced_range(s.n, s.n_sink, s.n_recent);
    int k_sel = s.k - f.nf;
    if (k_sel < 0) k_sel = 0;
    int cap = k_sel + kPruneSlack + 2 * kSubTokens;
    return (cap + 255) / 256 * 256;   // <= 6400 for k <= 2048
}

int scan_m_sel(int chunks, int k_sel) {
    // keys each CTA hands to the merge (between m and 2m): four times its
    // expected share of the unit's k' winners, at least 32
    if (k_sel <= 0) return 0;
    int m = (4 * k_sel + chunks - 1) / chunks;
    m = m < 32 ? 32 : m;
    return m > k_sel ? k_sel : m;
}

int scan_m_first(int n_sub, int k_sel, int m_sel) {
    // Rank of the threshold taken from a CTA's first sub-chunk.  A sub-chunk that
    // holds at least this many of the unit's k' winners sets a threshold above the
    // k'-th key, and its CTA is rescanned exactly, so the rank is a tail bound of
    // the winners one sub-chunk holds: with the winners spread over the sequence
    // (lambda = k' / n_sub per sub-chunk on average, Poisson), the smallest m with
    // P(X >= m) <= 1e-6, at least 8, at most m_sel.  (Twice the mean, the earlier
    // rule, flagged about one (CTA, head) in twenty at lambda ~ 4.)
    if (k_sel <= 0) return 0;
    const double lam = (double)k_sel / (double)(n_sub > 0 ? n_sub : 1);
    int m;
    if (lam > 200.0) {
        m = (int)std::ceil(lam + 5.0 * std::sqrt(lam) + 5.0);   // normal tail, about 3e-7
    } else {
        double p = std::exp(-lam), cdf = p;   // P(X = 0), P(X <= m - 1) with m = 1
        m = 1;
        while (1.0 - cdf > 1e-6 && m < m_sel) {
            p *= lam / m;
            cdf += p;
            ++m;
        }
    }
    m = m < 8 ? 8 : m;
    return m > m_sel ? m_sel : m;
}

int merge_parts(int chunks, int m_sel) {
    // a list holds at most about 8m keys after the scan's final shrink, and
    // typically about 3m (the first threshold lets m1 .. 2 m1 keys per sub-chunk in)
    long long keys = (long long)chunks * 3 * (m_sel > 0 ? m_sel : 1);
    int p = (int)((keys + 8191) / 8192);
    if (p > chunks) p = chunks;
    if (p > FATHOM_MERGE_MAX_LISTS) p = FATHOM_MERGE_MAX_LISTS;
    return p < 1 ? 1 : p;
}

ScanWorkspace scan_workspace_layout(const fathom_shape &s) {
    ScanGrid g = scan_grid(s);
    Forced f = forced_range(s.n, s.n_sink, s.n_recent);
    int k_sel = s.k - f.nf;
    if (k_sel < 1) k_sel = 1;
    ScanWorkspace w;
    w.parts = merge_parts(g.chunks, scan_m_sel(g.chunks, k_sel));
    const size_t ctas = (size_t)s.units * g.chunks;
    const size_t uh = (size_t)s.units * s.G;
    w.cand_off = 0;
    w.cnt_off = align256(w.cand_off + ctas * s.G * (size_t)scan_cand_cap(s) * sizeof(uint64_t));
    w.tau_off = align256(w.cnt_off + ctas * s.G * sizeof(int32_t));
    w.flags_off = align256(w.tau_off + ctas * s.G * sizeof(uint64_t));
    w.forced_off = align256(w.flags_off + ctas * s.G * sizeof(int32_t));
    w.part_keys_off = align256(w.forced_off + uh * (f.nf > 0 ? f.nf : 1) * sizeof(float));
    w.part_cnt_off = align256(w.part_keys_off + uh * w.parts * (size_t)k_sel * sizeof(uint64_t));
    w.ticket_off = align256(w.part_cnt_off + uh * w.parts * sizeof(int32_t));
    w.dirty_off = align256(w.ticket_off + uh * sizeof(uint32_t));
    w.sub_ctr_off = align256(w.dirty_off + uh * sizeof(int32_t));
    const size_t n_sub = ((size_t)num_blocks(s.n) + kSubBlocks - 1) / kSubBlocks;
    w.sub_owner_off = align256(w.sub_ctr_off + (size_t)s.units * sizeof(int32_t));
    w.total = align256(w.sub_owner_off + (size_t)s.units * n_sub * sizeof(int32_t));
    return w;
}

// Kept-list entries per attention CTA for `pairs` grid rows of one head's list
// (G heads each): 128; 256 (fewer CTAs, each list loaded and searched fewer
// times) once 128 would need more than two waves of two CTAs per SM; 512 (one
// CTA per grid row and head) once that alone fills two waves (a 256-unit layer:
// 113 against 123 us; with few units it leaves the host link under-used: 115
// against 56 us for 8 units).
static int attn_rows_per_cta(long long units, int G, int k) {
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;
    const long long ctas128 = units * G * ((k + 127) / 128);
    const long long ctas512 = units * G * ((k + 511) / 512);
    return ctas512 >= 2LL * 2 * sms ? 512 : (ctas128 > 2LL * 2 * sms ? 256 : 128);
}

AttnWorkspace attn_workspace_layout(const fathom_shape &s) {
    AttnWorkspace w;
    w.rows = attn_rows_per_cta(s.units, s.G, s.k);
    w.splits = s.G * ((s.k + w.rows - 1) / w.rows);
    if (w.splits < 1) w.splits = 1;
    w.ph_rows = attn_rows_per_cta((long long)s.units * s.G, 1, s.k);
    w.ph_splits = (s.k + w.ph_rows - 1) / w.ph_rows;
    if (w.ph_splits < 1) w.ph_splits = 1;
    const size_t part_union = (size_t)s.units * w.splits * s.G * (s.D + 2);
    const size_t part_head = (size_t)s.units * s.G * w.ph_splits * (s.D + 2);
    w.part_off = 0;
    w.ticket_off = align256((part_union > part_head ? part_union : part_head) * sizeof(float));
    w.total = align256(w.ticket_off + (size_t)s.units * s.G * sizeof(uint32_t));
    return w;
}

AttnWorkspace dense_workspace_layout(const fathom_shape &s) {
    // about four waves of 2 CTAs per SM over the units, at most 64 splits, at
    // least 1024 tokens per split (a multiple of the 64-token block)
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;
    AttnWorkspace w;
    int splits = (4 * 2 * sms + s.units - 1) / s.units;
    const int max_splits = (s.n + 1023) / 1024;
    splits = splits < 1 ? 1 : (splits > 64 ? 64 : splits);
    splits = splits > max_splits ? max_splits : splits;
    w.rows = ((s.n + splits - 1) / splits + 63) / 64 * 64;
    w.splits = (s.n + w.rows - 1) / w.rows;
    w.ph_rows = w.rows;
    w.ph_splits = w.splits;
    w.part_off = 0;
    w.ticket_off = align256((size_t)s.units * w.splits * s.G * (s.D + 2) * sizeof(float));
    w.total = align256(w.ticket_off + (size_t)s.units * sizeof(uint32_t));
    return w;
}

}  // namespace fathom

using namespace fathom;

static int check_shape(const fathom_shape *s, bool need_select) {
    if (!s) { set_error("shape is NULL"); return FATHOM_EINVAL; }
    if (s->units < 1) { set_error("units must be >= 1 (got %d)", s->units); return FATHOM_EINVAL; }
    if (s->n < 1 || s->n > (1 << 28)) { set_error("n must be in [1, 2^28] (got %d)", s->n); return FATHOM_EINVAL; }
    if (s->D < 1 || s->D > FATHOM_MAX_D) { set_error("D must be in [1, %d] (got %d)", FATHOM_MAX_D, s->D); return FATHOM_EINVAL; }
    if (!(s->G == 1 || s->G == 2 || s->G == 4 || s->G == 8)) { set_error("G must be 1, 2, 4 or 8 (got %d)", s->G); return FATHOM_EINVAL; }
    if (s->n_cap != 0 && (s->n_cap < s->n || s->n_cap > (1 << 28))) {
        set_error("n_cap must be 0 or in [n, 2^28] (got n_cap=%d, n=%d)", s->n_cap, s->n); return FATHOM_EINVAL;
    }
    if (s->scan_ctas_per_sm < 0 || s->scan_ctas_per_sm > 8) {
        set_error("scan_ctas_per_sm must be in [0, 8] (got %d)", s->scan_ctas_per_sm); return FATHOM_EINVAL;
    }
    if ((size_t)s->units * s->D * FATHOM_PLANES * (size_t)cap_blocks(*s) >= ((size_t)1 << 40) ||
        (size_t)s->D * FATHOM_PLANES * (size_t)cap_blocks(*s) >= ((size_t)1 << 32)) {
        set_error("store too large"); return FATHOM_EINVAL;
    }
    if (need_select) {
        if (s->n_sink < 0 || s->n_recent < 0) { set_error("n_sink and n_recent must be >= 0"); return FATHOM_EINVAL; }
        if (s->k < 1 || s->k > s->n || s->k > FATHOM_MAX_K) {
            set_error("k must be in [1, min(n, %d)] (got k=%d, n=%d)", FATHOM_MAX_K, s->k, s->n);
            return FATHOM_EINVAL;
        }
        Forced f = forced_range(s->n, s->n_sink, s->n_recent);
        if (f.nf > s->k) {
            set_error("k=%d is smaller than the %d forced tokens", s->k, f.nf);
            return FATHOM_EINVAL;
        }
    }
    return FATHOM_OK;
}

#define NONNULL(p)                                               \
    do {                                                         \
        if (!(p)) { set_error("%s is NULL", #p); return FATHOM_EINVAL; } \
    } while (0)

// Host-side fault injection, for testing how callers handle a failed launch
// without faulting a GPU.  FATHOM_FAULT (read once per process) holds a
// comma-separated list of sites: "launch" makes every call that would enqueue
// GPU work fail, "launch:<name>" only the named call (e.g.
// launch:fathom_scan_topk).  A failing call has already validated its
// arguments; it enqueues nothing and returns FATHOM_ECUDA with a message that
// names the injected fault.  Unset (the default), nothing is injected.
static bool fault_injected(const char *entry) {
    static const char *spec = [] {
        const char *e = getenv("FATHOM_FAULT");
        return (e && *e) ? e : (const char *)nullptr;
    }();
    if (!spec) return false;
    const size_t n = strlen(entry);
    for (const char *p = spec; *p;) {
        const char *end = strchr(p, ',');
        const size_t len = end ? (size_t)(end - p) : strlen(p);
        if (len == 6 && strncmp(p, "launch", 6) == 0) return true;
        if (len == 7 + n && strncmp(p, "launch:", 7) == 0 && strncmp(p + 7, entry, n) == 0) return true;
        if (!end) break;
        p = end + 1;
    }
    return false;
}

#define FAULT_POINT(name)                                                              \
    do {                                                                               \
        if (fault_injected(name)) {                                                    \
            set_error("%s: injected launch failure (FATHOM_FAULT)", name);             \
            return FATHOM_ECUDA;                                                       \
        }                                                                              \
    } while (0)

extern "C" {

const char *fathom_last_error(void) { return g_err; }

const char *fathom_version(void) { return "fathom-gb300 0.2 (sm_103a)"; }

int fathom_debug_status(int mode, uint64_t *first_failure) {
    g_err[0] = 0;
    NONNULL(first_failure);
    if (mode < 0 || mode > 2) { set_error("debug_status: mode must be 0, 1 or 2"); return FATHOM_EINVAL; }
#ifdef FATHOM_DEBUG
    if (mode == 2) {   // plant a self-test record in every file's word first
        debug_read_scan_plant();
        debug_read_gather_plant();
        debug_read_attn_plant();
    }
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { set_error("debug_status: %s", cudaGetErrorString(e)); return FATHOM_ECUDA; }
    first_failure[0] = debug_read_scan(mode == 1);
    first_failure[1] = debug_read_gather(mode == 1);
    first_failure[2] = debug_read_attn(mode == 1);
    return launch_status("debug_status");
#else
    first_failure[0] = first_failure[1] = first_failure[2] = 0;
    set_error("debug_status: this library was built without the debug checks (-DFATHOM_DEBUG)");
    return FATHOM_EINVAL;
#endif
}

int fathom_calibrate(int32_t units, int32_t m, int32_t D, const float *calib, float *mean_out,
                     float *var_out, void *stream) {
    g_err[0] = 0;
    if (units < 1 || m < 2 || D < 1 || D > FATHOM_MAX_D) {
        set_error("calibrate: need units >= 1, m >= 2, 1 <= D <= %d", FATHOM_MAX_D);
        return FATHOM_EINVAL;
    }
    NONNULL(calib);
    NONNULL(var_out);
    FAULT_POINT("fathom_calibrate");
    return launch_calibrate(units, m, D, calib, mean_out, var_out, (cudaStream_t)stream);
}

int fathom_calibrate_klt(int32_t groups, int32_t m, int32_t D, const float *calib, double *mean,
                         double *V, float *lambda, void *stream) {
    g_err[0] = 0;
    if (groups < 1 || m < 2 || D < 1 || D > FATHOM_MAX_D) {
        set_error("calibrate_klt: need groups >= 1, m >= 2, 1 <= D <= %d", FATHOM_MAX_D);
        return FATHOM_EINVAL;
    }
    NONNULL(calib);
    NONNULL(mean);
    NONNULL(V);
    NONNULL(lambda);
    FAULT_POINT("fathom_calibrate_klt");
    return launch_calibrate_klt(groups, m, D, calib, mean, V, lambda, (cudaStream_t)stream);
}

int fathom_rotate_keys(const fathom_shape *shape, const void *keys, int keys_dtype, int32_t groups,
                       const double *mean, const double *V, float *out, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    if (keys_dtype != FATHOM_F32 && keys_dtype != FATHOM_BF16) {
        set_error("keys_dtype must be FATHOM_F32 or FATHOM_BF16"); return FATHOM_EINVAL;
    }
    if (groups < 1) { set_error("groups must be >= 1 (got %d)", groups); return FATHOM_EINVAL; }
    NONNULL(keys);
    NONNULL(mean);
    NONNULL(V);
    NONNULL(out);
    FAULT_POINT("fathom_rotate_keys");
    return launch_rotate_keys(*shape, keys, keys_dtype, groups, mean, V, out, (cudaStream_t)stream);
}

int fathom_rotate_query(const fathom_shape *shape, const float *q, int32_t groups, const double *V,
                        float *q_rot, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    if (groups < 1) { set_error("groups must be >= 1 (got %d)", groups); return FATHOM_EINVAL; }
    if (shape->units > 65535 * 32) { set_error("rotate_query: too many units"); return FATHOM_EINVAL; }
    NONNULL(q);
    NONNULL(V);
    NONNULL(q_rot);
    FAULT_POINT("fathom_rotate_query");
    return launch_rotate_query(*shape, q, groups, V, q_rot, (cudaStream_t)stream);
}

int fathom_append_block(const fathom_shape *shape, const void *keys, int keys_dtype, int32_t block,
                        int32_t count, uint64_t *planes, uint16_t *scales, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    if (keys_dtype != FATHOM_F32 && keys_dtype != FATHOM_BF16) {
        set_error("keys_dtype must be FATHOM_F32 or FATHOM_BF16"); return FATHOM_EINVAL;
    }
    if (block < 0 || count < 1 || count > FATHOM_BLOCK || (long long)FATHOM_BLOCK * block + count > cap_tokens(*shape)) {
        set_error("append_block: need block >= 0, 1 <= count <= 64 and 64 * block + count <= capacity %d "
                  "(got block=%d, count=%d)", cap_tokens(*shape), block, count);
        return FATHOM_EINVAL;
    }
    NONNULL(keys);
    NONNULL(planes);
    NONNULL(scales);
    FAULT_POINT("fathom_append_block");
    return launch_append(*shape, keys, keys_dtype, block, count, planes, scales, (cudaStream_t)stream);
}

int fathom_quantize_pack(const fathom_shape *shape, const void *keys, int keys_dtype,
                         uint64_t *planes, uint16_t *scales, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    if (keys_dtype != FATHOM_F32 && keys_dtype != FATHOM_BF16) {
        set_error("keys_dtype must be FATHOM_F32 or FATHOM_BF16"); return FATHOM_EINVAL;
    }
    NONNULL(keys);
    NONNULL(planes);
    NONNULL(scales);
    FAULT_POINT("fathom_quantize_pack");
    return launch_quantize(*shape, keys, keys_dtype, planes, scales, (cudaStream_t)stream);
}

int fathom_plan(const fathom_shape *shape, const float *q, const float *var, const int32_t *budget,
                const double *bracket, uint8_t *depth, double *theta, fathom_run *runs,
                void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    NONNULL(q);
    NONNULL(var);
    NONNULL(budget);
    NONNULL(depth);
    NONNULL(runs);
    FAULT_POINT("fathom_plan");
    return launch_plan(*shape, q, var, budget, bracket, depth, theta, runs, (cudaStream_t)stream);
}

int fathom_plan_fixed(const fathom_shape *shape, const float *q, const float *var,
                      int32_t n_channels, int32_t depth_each, uint8_t *depth, fathom_run *runs,
                      void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    if (n_channels < 1 || n_channels > shape->D || depth_each < 1 || depth_each > 4) {
        set_error("plan_fixed: need 1 <= n_channels <= D and 1 <= depth_each <= 4");
        return FATHOM_EINVAL;
    }
    NONNULL(q);
    NONNULL(var);
    NONNULL(depth);
    NONNULL(runs);
    FAULT_POINT("fathom_plan_fixed");
    return launch_plan_fixed(*shape, q, var, n_channels, depth_each, depth, runs,
                             (cudaStream_t)stream);
}

int fathom_gather(const fathom_shape *shape, const uint64_t *store_planes,
                  const uint16_t *store_scales, const fathom_run *runs, uint64_t *stage_planes,
                  uint16_t *stage_scales, size_t stage_words, size_t stage_scales_n, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    NONNULL(store_planes);
    NONNULL(store_scales);
    NONNULL(runs);
    NONNULL(stage_planes);
    NONNULL(stage_scales);
    if (stage_words < 1 || stage_scales_n < 1) { set_error("empty staging area"); return FATHOM_EINVAL; }
    FAULT_POINT("fathom_gather");
    return launch_gather(*shape, store_planes, store_scales, runs, stage_planes, stage_scales,
                         stage_words, stage_scales_n, (cudaStream_t)stream);
}

size_t fathom_workspace_size(const fathom_shape *shape, int which) {
    if (check_shape(shape, true)) return 0;
    if (which == FATHOM_WS_SCAN_TOPK) return scan_workspace_layout(*shape).total;
    if (which == FATHOM_WS_SPARSE_ATTN) return attn_workspace_layout(*shape).total;
    if (which == FATHOM_WS_DENSE_ATTN) return dense_workspace_layout(*shape).total;
    if (which == FATHOM_WS_KLT_ONLINE) {
        if (shape->n < 2) { set_error("klt_online needs n >= 2 tokens"); return 0; }
        return klt_online_layout(*shape).total;
    }
    return 0;
}

static int check_scan_args(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales, int source,
                           size_t stage_words, size_t stage_scales_n, const fathom_run *runs, const float *q,
                           void *workspace, size_t workspace_bytes) {
    int rc = check_shape(shape, true);
    if (rc) return rc;
    if (source != FATHOM_SRC_STORE && source != FATHOM_SRC_STAGING) {
        set_error("source must be FATHOM_SRC_STORE or FATHOM_SRC_STAGING"); return FATHOM_EINVAL;
    }
    if (source == FATHOM_SRC_STAGING && (stage_words < 1 || stage_scales_n < 1)) {
        set_error("staging strides must be >= 1"); return FATHOM_EINVAL;
    }
    NONNULL(planes);
    NONNULL(scales);
    NONNULL(runs);
    NONNULL(q);
    NONNULL(workspace);
    size_t need = scan_workspace_layout(*shape).total;
    if (workspace_bytes < need) {
        set_error("scan_topk workspace too small: %zu < %zu bytes", workspace_bytes, need);
        return FATHOM_ENOMEM;
    }
    if (((uintptr_t)workspace & 255) != 0) { set_error("workspace must be 256-byte aligned"); return FATHOM_EINVAL; }
    return FATHOM_OK;
}

int fathom_scan_topk(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales,
                     int source, size_t stage_words, size_t stage_scales_n, const fathom_run *runs,
                     const float *q, int32_t *topk_idx, float *topk_score, float *scores_opt,
                     void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_scan_args(shape, planes, scales, source, stage_words, stage_scales_n, runs, q, workspace,
                             workspace_bytes);
    if (rc) return rc;
    NONNULL(topk_idx);
    NONNULL(topk_score);
    FAULT_POINT("fathom_scan_topk");
    return launch_scan_topk(*shape, planes, scales, source, stage_words, stage_scales_n, runs, q,
                            topk_idx, topk_score, scores_opt, workspace, (cudaStream_t)stream, SCAN_PART_ALL);
}

int fathom_scan(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales, int source,
                size_t stage_words, size_t stage_scales_n, const fathom_run *runs, const float *q,
                float *scores_opt, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_scan_args(shape, planes, scales, source, stage_words, stage_scales_n, runs, q, workspace,
                             workspace_bytes);
    if (rc) return rc;
    FAULT_POINT("fathom_scan");
    return launch_scan_topk(*shape, planes, scales, source, stage_words, stage_scales_n, runs, q, nullptr,
                            nullptr, scores_opt, workspace, (cudaStream_t)stream, SCAN_PART_SCAN);
}

int fathom_select(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales, int source,
                  size_t stage_words, size_t stage_scales_n, const fathom_run *runs, const float *q,
                  int32_t *topk_idx, float *topk_score, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_scan_args(shape, planes, scales, source, stage_words, stage_scales_n, runs, q, workspace,
                             workspace_bytes);
    if (rc) return rc;
    NONNULL(topk_idx);
    NONNULL(topk_score);
    FAULT_POINT("fathom_select");
    return launch_scan_topk(*shape, planes, scales, source, stage_words, stage_scales_n, runs, q, topk_idx,
                            topk_score, nullptr, workspace, (cudaStream_t)stream, SCAN_PART_SELECT);
}

int fathom_exact_topk(const fathom_shape *shape, const uint16_t *k_rows, const float *q,
                      int32_t *topk_idx, float *topk_score, float *scores_opt,
                      void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, true);
    if (rc) return rc;
    NONNULL(k_rows);
    NONNULL(q);
    NONNULL(topk_idx);
    NONNULL(topk_score);
    NONNULL(workspace);
    size_t need = scan_workspace_layout(*shape).total;
    if (workspace_bytes < need) {
        set_error("exact_topk workspace too small: %zu < %zu bytes", workspace_bytes, need);
        return FATHOM_ENOMEM;
    }
    if (((uintptr_t)workspace & 255) != 0) { set_error("workspace must be 256-byte aligned"); return FATHOM_EINVAL; }
    FAULT_POINT("fathom_exact_topk");
    return launch_scan_topk(*shape, (const uint64_t *)k_rows, nullptr, FATHOM_SRC_ROWS, 0, 0, nullptr, q,
                            topk_idx, topk_score, scores_opt, workspace, (cudaStream_t)stream);
}

int fathom_sparse_attn_planes(const fathom_shape *shape, const uint64_t *planes, const uint16_t *scales,
                              const uint16_t *v_rows, const float *q, const int32_t *topk_idx, float *out,
                              void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, true);
    if (rc) return rc;
    NONNULL(planes);
    NONNULL(scales);
    NONNULL(v_rows);
    NONNULL(q);
    NONNULL(topk_idx);
    NONNULL(out);
    NONNULL(workspace);
    const size_t need = attn_workspace_layout(*shape).total;
    if (workspace_bytes < need) {
        set_error("sparse_attn_planes workspace too small: %zu < %zu bytes", workspace_bytes, need);
        return FATHOM_ENOMEM;
    }
    if (((uintptr_t)workspace & 255) != 0) { set_error("workspace must be 256-byte aligned"); return FATHOM_EINVAL; }
    FAULT_POINT("fathom_sparse_attn_planes");
    return launch_sparse_attn_planes(*shape, planes, scales, v_rows, q, topk_idx, out, workspace,
                                     (cudaStream_t)stream);
}

int fathom_dense_attn(const fathom_shape *shape, const uint16_t *k_rows, const uint16_t *v_rows,
                      const float *q, float *out, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    NONNULL(k_rows);
    NONNULL(v_rows);
    NONNULL(q);
    NONNULL(out);
    NONNULL(workspace);
    const size_t need = dense_workspace_layout(*shape).total;
    if (workspace_bytes < need) {
        set_error("dense_attn workspace too small: %zu < %zu bytes", workspace_bytes, need);
        return FATHOM_ENOMEM;
    }
    if (((uintptr_t)workspace & 255) != 0) { set_error("workspace must be 256-byte aligned"); return FATHOM_EINVAL; }
    FAULT_POINT("fathom_dense_attn");
    return launch_dense_attn(*shape, k_rows, v_rows, q, out, workspace, (cudaStream_t)stream);
}

int fathom_klt_online(const fathom_shape *shape, const uint16_t *k_rows, double *mean, double *V, float *lambda,
                      void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, false);
    if (rc) return rc;
    if (shape->n < 2) { set_error("klt_online needs n >= 2 tokens (n=%d)", shape->n); return FATHOM_EINVAL; }
    NONNULL(k_rows);
    NONNULL(mean);
    NONNULL(V);
    NONNULL(lambda);
    NONNULL(workspace);
    const size_t need = klt_online_layout(*shape).total;
    if (workspace_bytes < need) {
        set_error("klt_online workspace too small: %zu < %zu bytes", workspace_bytes, need);
        return FATHOM_ENOMEM;
    }
    if (((uintptr_t)workspace & 255) != 0) { set_error("workspace must be 256-byte aligned"); return FATHOM_EINVAL; }
    FAULT_POINT("fathom_klt_online");
    return launch_klt_online(*shape, k_rows, mean, V, lambda, workspace, (cudaStream_t)stream);
}

int fathom_rel_err(int32_t rows, int32_t D, const float *a, const float *ref, double *err, void *stream) {
    g_err[0] = 0;
    if (rows < 0 || D < 1) { set_error("rel_err: need rows >= 0 and D >= 1 (rows=%d, D=%d)", rows, D); return FATHOM_EINVAL; }
    if (rows == 0) return FATHOM_OK;
    NONNULL(a);
    NONNULL(ref);
    NONNULL(err);
    FAULT_POINT("fathom_rel_err");
    return launch_rel_err(rows, D, a, ref, err, (cudaStream_t)stream);
}

int fathom_set_overlap(int32_t rows, int32_t k, const int32_t *a, const int32_t *b, int32_t *count,
                       void *stream) {
    g_err[0] = 0;
    if (rows < 0 || k < 1) { set_error("set_overlap: need rows >= 0 and k >= 1 (rows=%d, k=%d)", rows, k); return FATHOM_EINVAL; }
    if (rows == 0) return FATHOM_OK;
    NONNULL(a);
    NONNULL(b);
    NONNULL(count);
    FAULT_POINT("fathom_set_overlap");
    return launch_set_overlap(rows, k, a, b, count, (cudaStream_t)stream);
}

int fathom_greedy_budgets(int32_t layers, int32_t levels, const double *err, int32_t b_min, int32_t step,
                          int32_t b_mean, int32_t *budgets) {
    g_err[0] = 0;
    if (layers < 1 || levels < 1 || step < 1 || b_min < 0) {
        set_error("greedy_budgets: need layers, levels, step >= 1 and b_min >= 0");
        return FATHOM_EINVAL;
    }
    const long long b_max = (long long)b_min + (long long)step * (levels - 1);
    if (b_mean < b_min || b_mean > b_max || (b_mean - b_min) % step != 0) {
        set_error("greedy_budgets: b_mean=%d must be one of the levels %d, %d, ..., %lld", b_mean, b_min,
                  b_min + step, b_max);
        return FATHOM_EINVAL;
    }
    NONNULL(err);
    NONNULL(budgets);
    for (long long i = 0; i < (long long)layers * levels; ++i)
        if (!std::isfinite(err[i])) { set_error("greedy_budgets: err[%lld] is not finite", i); return FATHOM_EINVAL; }
    return greedy_budgets(layers, levels, err, b_min, step, b_mean, budgets);
}

int fathom_sparse_attn(const fathom_shape *shape, const uint16_t *k_rows, const uint16_t *v_rows,
                       const float *q, const int32_t *topk_idx, float *out, void *workspace,
                       size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, true);
    if (rc) return rc;
    NONNULL(k_rows);
    NONNULL(v_rows);
    NONNULL(q);
    NONNULL(topk_idx);
    NONNULL(out);
    NONNULL(workspace);
    size_t need = attn_workspace_layout(*shape).total;
    if (workspace_bytes < need) {
        set_error("sparse_attn workspace too small: %zu < %zu bytes", workspace_bytes, need);
        return FATHOM_ENOMEM;
    }
    if (((uintptr_t)workspace & 255) != 0) { set_error("workspace must be 256-byte aligned"); return FATHOM_EINVAL; }
    FAULT_POINT("fathom_sparse_attn");
    return launch_sparse_attn(*shape, k_rows, v_rows, q, topk_idx, out, workspace,
                              (cudaStream_t)stream);
}

int fathom_sparse_attn_noalloc(const fathom_shape *shape, const uint16_t *k_rows,
                               const uint16_t *v_rows, const float *q, const int32_t *topk_idx,
                               float *out, void *stream) {
    g_err[0] = 0;
    int rc = check_shape(shape, true);
    if (rc) return rc;
    NONNULL(k_rows);
    NONNULL(v_rows);
    NONNULL(q);
    NONNULL(topk_idx);
    NONNULL(out);
    FAULT_POINT("fathom_sparse_attn_noalloc");
    return launch_sparse_attn_noalloc(*shape, k_rows, v_rows, q, topk_idx, out, (cudaStream_t)stream);
}

}  // extern "C"

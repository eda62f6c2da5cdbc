// plan.cu -- per-query-group read plan (Fathom §3.3 per-query read depth,
// §3.6 fixed-size run list).
//
// One warp per unit; lane l owns channels l, l+32, l+64, l+96.
//   g_j  = (sum_h q_hj^2) * var_j              (fp64, h ascending)
//   t_j(theta) = #{m in 0..3 : g_j >= theta * 2^(2m+1)}
// which is clip(round(log4(g_j / theta)), 0, 4) with ties rounding up, written
// with compares against exact power-of-two multiples of theta so that no
// logarithm (and no rounding of one) enters a decision.  theta comes from 30
// steps of geometric bisection mid = sqrt(lo * hi) that keep hi feasible
// (sum_j t_j(hi) <= B); the plan is t(hi).  Every fp64 operation is an
// explicitly rounded IEEE operation (no contraction), so the result is
// reproducible bit for bit on any IEEE machine.  The bisection's square roots
// come from exact_sqrt.cuh (the same bits as the fp64 square root, without its
// long latency on this part) whenever every lo * hi of the chain is a normal
// double.  The whole plan stays on the
// device: the run list has one slot per channel (zero length when t_j = 0),
// so nothing needs to come back to the host.
#include "exact_sqrt.cuh"
#include "fathom_internal.cuh"

namespace fathom {

constexpr int kPlanWarps = 1;   // one unit per CTA: the fp64 chains of many units spread over the SMs
constexpr int kCh = FATHOM_MAX_D / 32;   // channels per lane

// t(g, theta) = #{m in 0..3 : g >= theta * 2^(2m+1)}.  For a normal positive
// theta, theta * 2^e is the double whose bit pattern is bits(theta) + e * 2^52
// (no rounding: only the exponent changes), and positive doubles order like
// their bit patterns, so each compare is one exact 64-bit integer compare
// (negative or zero g compares below every positive threshold, as in fp64).
// Zero or subnormal theta takes the fp64 route.
__device__ __forceinline__ int depth_of(double g, double theta) {
    const long long tb = __double_as_longlong(theta);
    int t = 0;
    if ((tb >> 52) > 0 && (tb >> 52) < 0x7ff) {
        const long long gb = __double_as_longlong(g);
#pragma unroll
        for (int m = 0; m < 4; ++m) t += (gb >= tb + ((long long)(2 * m + 1) << 52)) ? 1 : 0;
    } else {
#pragma unroll
        for (int m = 0; m < 4; ++m) t += (g >= __dmul_rn(theta, (double)(2 << (2 * m)))) ? 1 : 0;
    }
    return t;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void importance(int u, int lane, int D, int G, const float *q,
                                           const float *var, double (&g)[kCh]) {
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
        const int j = lane + 32 * c;
        double gj = 0.0;
        if (j < D) {
            double s = 0.0;
            for (int h = 0; h < G; ++h) {
                const double x = (double)q[((size_t)u * G + h) * D + j];
                s = __dadd_rn(s, __dmul_rn(x, x));
            }
            gj = __dmul_rn(s, (double)var[(size_t)u * D + j]);
        }
        g[c] = gj;
    }
}

// Writes depth and the run list of one unit from per-lane depths t[c].
__device__ __forceinline__ void write_plan(int u, int lane, int D, int nb, int cb, const int (&t)[kCh],
                                           uint8_t *depth, fathom_run *runs) {
    uint32_t carry_w = 0, carry_s = 0;
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
        const int j = lane + 32 * c;
        const int tj = (j < D) ? t[c] : 0;
        const int act = tj > 0 ? 1 : 0;
        // inclusive warp scans of t and of "active"
        int st = tj, sa = act;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yt = __shfl_up_sync(0xffffffffu, st, o);
            const int ya = __shfl_up_sync(0xffffffffu, sa, o);
            if (lane >= o) { st += yt; sa += ya; }
        }
        if (j < D) {
            depth[(size_t)u * D + j] = (uint8_t)tj;
            fathom_run r;
            r.src_word = (uint32_t)j * FATHOM_PLANES * cb;
            r.n_words = (uint32_t)tj * nb;
            r.dst_word = (carry_w + (uint32_t)(st - tj)) * nb;
            r.src_scale = (uint32_t)j * cb;
            r.n_scales = act ? (uint32_t)nb : 0u;
            r.dst_scale = (carry_s + (uint32_t)(sa - act)) * nb;
            runs[(size_t)u * D + j] = r;
        }
        carry_w += (uint32_t)__shfl_sync(0xffffffffu, st, 31);
        carry_s += (uint32_t)__shfl_sync(0xffffffffu, sa, 31);
    }
}

// The (B+1)-th largest breakpoint b_{j,m} = g_j * 2^-(2m+1) over the warp's
// channels (with multiplicity), by an MSD radix select on the bit patterns
// (positive doubles order like their bit patterns), ranking the last bucket's
// keys directly once it holds at most 32.  `bp` holds the lane's 16 patterns
// (0 for channels past D or g_j <= 0); hist is the warp's 256 bins (also the
// 32 candidate slots of the final ranking).  Requires more than B positive
// breakpoints.
__device__ unsigned long long critical_breakpoint(const unsigned long long (&bp)[4 * kCh], int B,
                                                  unsigned *hist) {
    const int lane = threadIdx.x & 31;
    unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll
    for (int e = 0; e < 4 * kCh; ++e)
        if (bp[e]) { mn = min(mn, bp[e]); mx = max(mx, bp[e]); }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (mn == mx) return mn;
    int hi_bit = 63 - __clzll((long long)(mn ^ mx));
    unsigned long long pmask = (hi_bit == 63) ? 0ull : ~((2ull << hi_bit) - 1ull);
    unsigned long long prefix = mn & pmask;
    int need = B + 1;   // rank (from the top) still to find within the current bucket
    while (true) {
        const int lo = hi_bit >= 7 ? hi_bit - 7 : 0;
        const unsigned long long dmask = (2ull << (hi_bit - lo)) - 1ull;
#pragma unroll
        for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0;
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 4 * kCh; ++e)
            if (bp[e] && (bp[e] & pmask) == prefix) atomicAdd(&hist[(bp[e] >> lo) & dmask], 1u);
        __syncwarp();
        // lane l owns bins 255-8l .. 248-8l (descending)
        unsigned loc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) loc += hist[255 - 8 * lane - i];
        unsigned incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned excl = incl - loc;
        int digit = -1, above = 0, bucket = 0;
        if (excl < (unsigned)need && (unsigned)need <= incl) {
            unsigned c = excl;
            for (int i = 0; i < 8; ++i) {
                const int bin = 255 - 8 * lane - i;
                const unsigned hb = hist[bin];
                if (c + hb >= (unsigned)need) { digit = bin; above = (int)c; bucket = (int)hb; break; }
                c += hb;
            }
        }
        const unsigned owner = __ballot_sync(0xffffffffu, digit >= 0);
        const int src = __ffs(owner) - 1;
        digit = __shfl_sync(0xffffffffu, digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        bucket = __shfl_sync(0xffffffffu, bucket, src);
        __syncwarp();
        prefix |= (unsigned long long)digit << lo;
        pmask |= dmask << lo;
        need -= above;
        if (lo == 0) return prefix;              // every bit decided: this value
        if (bucket <= 32) {
            // few candidates left: gather them (lane order) and rank each against
            // the others; the need-th largest is the one with fewer than `need`
            // candidates above it and at least `need` at or above it
            unsigned long long *cand = reinterpret_cast<unsigned long long *>(hist);   // 32 slots
            int mine = 0;
#pragma unroll
            for (int e = 0; e < 4 * kCh; ++e) mine += (bp[e] && (bp[e] & pmask) == prefix) ? 1 : 0;
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            __syncwarp();
            int pos = incl - mine;
#pragma unroll
            for (int e = 0; e < 4 * kCh; ++e)
                if (bp[e] && (bp[e] & pmask) == prefix) cand[pos++] = bp[e];
            __syncwarp();
            const unsigned long long x = lane < bucket ? cand[lane] : 0ull;
            int gt = 0, ge = 0;
            for (int j = 0; j < bucket; ++j) {
                const unsigned long long y = cand[j];
                gt += y > x ? 1 : 0;
                ge += y >= x ? 1 : 0;
            }
            const bool hit = lane < bucket && gt < need && ge >= need;
            const unsigned who = __ballot_sync(0xffffffffu, hit);
            const unsigned long long v = __shfl_sync(0xffffffffu, x, __ffs(who) - 1);
            __syncwarp();
            return v;
        }
        hi_bit = lo - 1;
    }
}

__global__ void __launch_bounds__(32 * kPlanWarps)
plan_kernel(int units, int n, int cb, int D, int G, const float *__restrict__ q,
            const float *__restrict__ var, const int32_t *__restrict__ budget,
            const double *__restrict__ bracket, uint8_t *__restrict__ depth,
            double *__restrict__ theta_out, fathom_run *__restrict__ runs) {
    pdl_enter();
    const int u = blockIdx.x * kPlanWarps + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (u >= units) return;
    const int nb = num_blocks(n);
    double g[kCh];
    importance(u, lane, D, G, q, var, g);
    const int B = budget[u];

    auto total = [&](double th) {
        int s = 0;
#pragma unroll
        for (int c = 0; c < kCh; ++c) s += depth_of(g[c], th);
        return warp_sum(s);
    };

    double lo, hi;
    bool bisect = true;
    if (bracket) {
        lo = bracket[2 * (size_t)u];
        hi = bracket[2 * (size_t)u + 1];
    } else {
        double gmax = 0.0, gmin = CUDART_INF;
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
            gmax = fmax(gmax, g[c]);
            if (g[c] > 0.0) gmin = fmin(gmin, g[c]);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            gmax = fmax(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
            gmin = fmin(gmin, __shfl_xor_sync(0xffffffffu, gmin, o));
        }
        if (gmax == 0.0) {                       // nothing worth reading
            int t0[kCh] = {0};
            write_plan(u, lane, D, nb, cb, t0, depth, runs);
            if (lane == 0) theta_out[u] = 0.0;
            return;
        }
        hi = gmax;
        lo = __dmul_rn(gmin, 1.0 / 512.0);        // exact power-of-two scaling
        if (total(lo) <= B) { hi = lo; bisect = false; }   // budget not binding
    }
    if (bisect) {
        // total(theta) = #{breakpoints b_{j,m} = g_j 2^-(2m+1) >= theta}, so theta
        // fits the budget iff theta > b*, the (B+1)-th largest breakpoint: each
        // step is then one exact compare instead of a count over the channels.
        // The breakpoints are exact (power-of-two scaling) unless g is within
        // 2^7 of the subnormal range; then, and with an explicit bracket, count.
        bool exact_bp = !bracket && B >= 0;
        unsigned long long bp[4 * kCh];
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
            const long long gb = __double_as_longlong(g[c]);
            const bool pos = g[c] > 0.0;
            exact_bp = exact_bp && (!pos || (gb >> 52) > 16);
#pragma unroll
            for (int m = 0; m < 4; ++m)
                bp[4 * c + m] = pos ? (unsigned long long)(gb - ((long long)(2 * m + 1) << 52)) : 0ull;
        }
        exact_bp = __all_sync(0xffffffffu, exact_bp);
        if (exact_bp) {
            __shared__ __align__(16) unsigned hist_s[kPlanWarps][256];   // 8-byte slots reuse it
            const double bstar = __longlong_as_double(
                (long long)critical_breakpoint(bp, B, hist_s[threadIdx.x / 32]));
            const long long elo = __double_as_longlong(lo) >> 52, ehi = __double_as_longlong(hi) >> 52;
            if (elo >= 1023 - 511 && ehi <= 1023 + 510) {
                // lo * hi stays a normal double on every step: integer square root
                for (int it = 0; it < 30; ++it) {
                    const double mid = __longlong_as_double(
                        (long long)xsqrt::sqrt_rn((uint64_t)__double_as_longlong(__dmul_rn(lo, hi))));
                    if (mid > bstar) hi = mid; else lo = mid;
                }
            } else {
                for (int it = 0; it < 30; ++it) {
                    const double mid = __dsqrt_rn(__dmul_rn(lo, hi));
                    if (mid > bstar) hi = mid; else lo = mid;
                }
            }
        } else {
            for (int it = 0; it < 30; ++it) {
                const double mid = __dsqrt_rn(__dmul_rn(lo, hi));
                if (total(mid) <= B) hi = mid; else lo = mid;
            }
        }
    }
    int t[kCh];
#pragma unroll
    for (int c = 0; c < kCh; ++c) t[c] = depth_of(g[c], hi);
    write_plan(u, lane, D, nb, cb, t, depth, runs);
    if (lane == 0) theta_out[u] = hi;
}

// Fixed-depth comparison plan: the n_sel channels of largest g (ties: lower
// index) at depth t_fixed.
__global__ void __launch_bounds__(32 * kPlanWarps)
plan_fixed_kernel(int units, int n, int cb, int D, int G, const float *__restrict__ q,
                  const float *__restrict__ var, int n_sel, int t_fixed,
                  uint8_t *__restrict__ depth, fathom_run *__restrict__ runs) {
    pdl_enter();
    __shared__ double gs[kPlanWarps][FATHOM_MAX_D];
    const int w = threadIdx.x / 32;
    const int u = blockIdx.x * kPlanWarps + w;
    const int lane = threadIdx.x & 31;
    if (u >= units) return;   // whole warps exit together; no block barrier below
    const int nb = num_blocks(n);
    double g[kCh];
    importance(u, lane, D, G, q, var, g);
#pragma unroll
    for (int c = 0; c < kCh; ++c) gs[w][lane + 32 * c] = g[c];
    __syncwarp();
    int t[kCh];
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
        const int j = lane + 32 * c;
        int better = 0;
        for (int i = 0; i < D; ++i) {
            const double gi = gs[w][i];
            better += (gi > g[c] || (gi == g[c] && i < j)) ? 1 : 0;
        }
        t[c] = (j < D && better < n_sel) ? t_fixed : 0;
    }
    write_plan(u, lane, D, nb, cb, t, depth, runs);
}

int launch_plan(const fathom_shape &s, const float *q, const float *var, const int32_t *budget,
                const double *bracket, uint8_t *depth, double *theta, fathom_run *runs,
                cudaStream_t st) {
    const int grid = (s.units + kPlanWarps - 1) / kPlanWarps;
    const cudaError_t e = launch_pdl(plan_kernel, dim3(grid), dim3(32 * kPlanWarps), 0, st, s.units, s.n,
                                     cap_blocks(s), s.D, s.G, q, var, budget, bracket, depth, theta, runs);
    if (e != cudaSuccess) { set_error("plan_kernel: %s", cudaGetErrorString(e)); return FATHOM_ECUDA; }
    return launch_status("plan_kernel");
}

int launch_plan_fixed(const fathom_shape &s, const float *q, const float *var, int n_sel,
                      int t_fixed, uint8_t *depth, fathom_run *runs, cudaStream_t st) {
    const int grid = (s.units + kPlanWarps - 1) / kPlanWarps;
    const cudaError_t e = launch_pdl(plan_fixed_kernel, dim3(grid), dim3(32 * kPlanWarps), 0, st, s.units, s.n,
                                     cap_blocks(s), s.D, s.G, q, var, n_sel, t_fixed, depth, runs);
    if (e != cudaSuccess) { set_error("plan_fixed_kernel: %s", cudaGetErrorString(e)); return FATHOM_ECUDA; }
    return launch_status("plan_fixed_kernel");
}

}  // namespace fathom

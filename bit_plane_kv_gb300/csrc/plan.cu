// plan.cu -- per-query-group read plan (Fathom §3.3 per-query read depth,
// §3.6 fixed-size run list).
//
// One CTA of 128 threads per unit; thread j owns channel j.
//   g_j  = (sum_h q_hj^2) * var_j              (fp64, h ascending)
//   t_j(theta) = #{m in 0..3 : g_j >= theta * 2^(2m+1)}
// which is clip(round(log4(g_j / theta)), 0, 4) with ties rounding up, written
// with compares against exact power-of-two multiples of theta so that no
// logarithm (and no rounding of one) enters a decision.  theta comes from 30
// steps of geometric bisection mid = sqrt(lo * hi) that keep hi feasible
// (sum_j t_j(hi) <= B); the plan is t(hi).  Every fp64 operation is an
// explicitly rounded IEEE operation (no contraction), so the result is
// reproducible bit for bit on any IEEE machine.  theta itself is an optional
// output: without it the depths come straight from the critical breakpoint
// whenever that provably gives t(hi) of the 30-step bisection (see below), and
// from the bisection otherwise.  The bisection's square roots
// come from exact_sqrt.cuh (the same bits as the fp64 square root, without its
// long latency on this part) whenever every lo * hi of the chain is a normal
// double.  The whole plan stays on the
// device: the run list has one slot per channel (zero length when t_j = 0),
// so nothing needs to come back to the host.
#include "exact_sqrt.cuh"
#include "fathom_internal.cuh"

namespace fathom {

constexpr int kPlanWarps = 1;   // the fixed plan: one warp per unit
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

// ---------------------------------------------------------------------------
// The plan kernel: one CTA of kPT = 128 threads per unit, thread j owning
// channel j (its importance and its four breakpoints), so that the importance,
// the critical-breakpoint selection and the run-list scans are spread over the
// CTA instead of being looped over by one warp.
constexpr int kPT = FATHOM_MAX_D;
constexpr int kPW = kPT / 32;

struct PlanSmem {
    unsigned hist[256];
    unsigned long long cand[32];
    unsigned long long red64[2][kPW];
    double redd[2][kPW];
    int redi[2][kPW];
    int digit, above, bucket, ncand;
    unsigned long long result;
    double hi_out;
};

__device__ __forceinline__ int cta_sum(PlanSmem &sm, int v) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) sm.redi[0][w] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int i = 0; i < kPW; ++i) t += sm.redi[0][i];
    return t;
}

// The (B+1)-th largest breakpoint over the CTA (4 per thread, 0 = none), as in
// critical_breakpoint: an MSD radix select on the bit patterns, the last bucket
// of at most 32 keys ranked directly.  Requires more than B positive breakpoints.
__device__ unsigned long long cta_critical_breakpoint(PlanSmem &sm, const unsigned long long (&bp)[4], int B) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (bp[e]) { mn = min(mn, bp[e]); mx = max(mx, bp[e]); }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    __syncthreads();
    if (lane == 0) { sm.red64[0][w] = mn; sm.red64[1][w] = mx; }
    __syncthreads();
    mn = ~0ull; mx = 0ull;
#pragma unroll
    for (int i = 0; i < kPW; ++i) { mn = min(mn, sm.red64[0][i]); mx = max(mx, sm.red64[1][i]); }
    if (mn == mx) return mn;
    int hi_bit = 63 - __clzll((long long)(mn ^ mx));
    unsigned long long pmask = (hi_bit == 63) ? 0ull : ~((2ull << hi_bit) - 1ull);
    unsigned long long prefix = mn & pmask;
    int need = B + 1;
    while (true) {
        const int lo = hi_bit >= 7 ? hi_bit - 7 : 0;
        const unsigned long long dmask = (2ull << (hi_bit - lo)) - 1ull;
        for (int i = tid; i < 256; i += kPT) sm.hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (bp[e] && (bp[e] & pmask) == prefix) atomicAdd(&sm.hist[(bp[e] >> lo) & dmask], 1u);
        __syncthreads();
        if (w == 0) {   // lane l owns bins 255-8l .. 248-8l (descending)
            unsigned loc = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) loc += sm.hist[255 - 8 * lane - i];
            unsigned incl = loc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned excl = incl - loc;
            if (excl < (unsigned)need && (unsigned)need <= incl) {
                unsigned c = excl;
                for (int i = 0; i < 8; ++i) {
                    const int bin = 255 - 8 * lane - i;
                    const unsigned hb = sm.hist[bin];
                    if (c + hb >= (unsigned)need) {
                        sm.digit = bin; sm.above = (int)c; sm.bucket = (int)hb;
                        break;
                    }
                    c += hb;
                }
            }
            if (lane == 0) sm.ncand = 0;
        }
        __syncthreads();
        const int digit = sm.digit, above = sm.above, bucket = sm.bucket;
        prefix |= (unsigned long long)digit << lo;
        pmask |= dmask << lo;
        need -= above;
        if (lo == 0) return prefix;               // every bit decided: this value
        if (bucket <= 32) {
            // few candidates left: gather them and rank each against the others; the
            // need-th largest has fewer than `need` above it and at least `need` at or above
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (bp[e] && (bp[e] & pmask) == prefix) sm.cand[atomicAdd(&sm.ncand, 1)] = bp[e];
            __syncthreads();
            if (w == 0) {
                const unsigned long long x = lane < bucket ? sm.cand[lane] : 0ull;
                int gt = 0, ge = 0;
                for (int j = 0; j < bucket; ++j) {
                    const unsigned long long y = sm.cand[j];
                    gt += y > x ? 1 : 0;
                    ge += y >= x ? 1 : 0;
                }
                const bool hit = lane < bucket && gt < need && ge >= need;
                const unsigned who = __ballot_sync(0xffffffffu, hit);
                const unsigned long long v = __shfl_sync(0xffffffffu, x, __ffs(who) - 1);
                if (lane == 0) sm.result = v;
            }
            __syncthreads();
            return sm.result;
        }
        hi_bit = lo - 1;
    }
}

// Writes depth and the run list of one unit, thread j for channel j: block
// exclusive scans of t_j and of "t_j > 0" give the staging destinations.
__device__ void cta_write_plan(PlanSmem &sm, int u, int D, int nb, int cb, int t, uint8_t *depth,
                               fathom_run *runs) {
    const int j = threadIdx.x, lane = j & 31, w = j >> 5;
    const int tj = (j < D) ? t : 0;
    const int act = tj > 0 ? 1 : 0;
    int st = tj, sa = act;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yt = __shfl_up_sync(0xffffffffu, st, o);
        const int ya = __shfl_up_sync(0xffffffffu, sa, o);
        if (lane >= o) { st += yt; sa += ya; }
    }
    __syncthreads();
    if (lane == 31) { sm.redi[0][w] = st; sm.redi[1][w] = sa; }
    __syncthreads();
    int bt = 0, ba = 0;
    for (int i = 0; i < w; ++i) { bt += sm.redi[0][i]; ba += sm.redi[1][i]; }
    if (j < D) {
        depth[(size_t)u * D + j] = (uint8_t)tj;
        fathom_run r;
        r.src_word = (uint32_t)j * FATHOM_PLANES * cb;
        r.n_words = (uint32_t)tj * nb;
        r.dst_word = (uint32_t)(bt + st - tj) * nb;
        r.src_scale = (uint32_t)j * cb;
        r.n_scales = act ? (uint32_t)nb : 0u;
        r.dst_scale = (uint32_t)(ba + sa - act) * nb;
        runs[(size_t)u * D + j] = r;
    }
}

__global__ void __launch_bounds__(kPT)
plan_kernel(int units, int n, int cb, int D, int G, const float *__restrict__ q,
            const float *__restrict__ var, const int32_t *__restrict__ budget,
            const double *__restrict__ bracket, uint8_t *__restrict__ depth,
            double *__restrict__ theta_out, fathom_run *__restrict__ runs) {
    pdl_enter();
    __shared__ PlanSmem sm;
    const int u = blockIdx.x;
    const int j = threadIdx.x, lane = j & 31, w = j >> 5;
    if (u >= units) return;                       // the whole CTA
    const int nb = num_blocks(n);
    // g_j = (sum_h q_hj^2) var_j in fp64, h ascending
    double g = 0.0;
    if (j < D) {
        double sq = 0.0;
        for (int h = 0; h < G; ++h) {
            const double x = (double)q[((size_t)u * G + h) * D + j];
            sq = __dadd_rn(sq, __dmul_rn(x, x));
        }
        g = __dmul_rn(sq, (double)var[(size_t)u * D + j]);
    }
    const int B = budget[u];
    auto total = [&](double th) { return cta_sum(sm, depth_of(g, th)); };

    double lo, hi;
    bool bisect = true;
    if (bracket) {
        lo = bracket[2 * (size_t)u];
        hi = bracket[2 * (size_t)u + 1];
    } else {
        double gmax = g, gmin = g > 0.0 ? g : CUDART_INF;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            gmax = fmax(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
            gmin = fmin(gmin, __shfl_xor_sync(0xffffffffu, gmin, o));
        }
        if (lane == 0) { sm.redd[0][w] = gmax; sm.redd[1][w] = gmin; }
        __syncthreads();
        gmax = 0.0; gmin = CUDART_INF;
#pragma unroll
        for (int i = 0; i < kPW; ++i) { gmax = fmax(gmax, sm.redd[0][i]); gmin = fmin(gmin, sm.redd[1][i]); }
        if (gmax == 0.0) {                        // nothing worth reading
            cta_write_plan(sm, u, D, nb, cb, 0, depth, runs);
            if (j == 0 && theta_out) theta_out[u] = 0.0;
            return;
        }
        hi = gmax;
        lo = __dmul_rn(gmin, 1.0 / 512.0);        // exact power-of-two scaling
        if (total(lo) <= B) { hi = lo; bisect = false; }   // budget not binding
    }
    if (bisect) {
        // total(theta) = #{breakpoints g_j 2^-(2m+1) >= theta}, so theta fits iff
        // theta > b*, the (B+1)-th largest breakpoint.  The breakpoints are exact
        // unless g is within 2^7 of the subnormal range; then, and with an
        // explicit bracket, count at every step.
        const long long gb = __double_as_longlong(g);
        const bool pos = g > 0.0;
        unsigned long long bp[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) bp[m] = pos ? (unsigned long long)(gb - ((long long)(2 * m + 1) << 52)) : 0ull;
        const bool exact_bp = !bracket && B >= 0 && __syncthreads_and(!pos || (gb >> 52) > 16);
        if (exact_bp) {
            const unsigned long long bs_bits = cta_critical_breakpoint(sm, bp, B);
            const double bstar = __longlong_as_double((long long)bs_bits);
            const long long elo = __double_as_longlong(lo) >> 52, ehi = __double_as_longlong(hi) >> 52;
            const bool normal_chain = elo >= 1023 - 511 && ehi <= 1023 + 510;
            if (!theta_out && normal_chain) {
                // No theta wanted: the depths are t(hi) for the bisection's final hi, and
                // hi_30 <= b* exp(w), w = ln(hi0 / lo0) 2^-30 + 3.2 u (each step halves the
                // log-width of [lo, hi] up to 1.6 u of rounding, and lo stays <= b*).  If
                // the next breakpoint above b* lies beyond b* (1 + 4x) >= b* exp(w), with
                // x >= w bounding w from the exponents, no breakpoint lies in (b*, hi_30],
                // so t(hi_30) = t(b_next) and the 30 dependent steps are not needed.
                unsigned long long nx = ~0ull;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (bp[e] > bs_bits && bp[e] < nx) nx = bp[e];
#pragma unroll
                for (int o = 16; o; o >>= 1) nx = min(nx, __shfl_xor_sync(0xffffffffu, nx, o));
                __syncthreads();
                if (lane == 0) sm.red64[0][w] = nx;
                __syncthreads();
                nx = ~0ull;
#pragma unroll
                for (int i = 0; i < kPW; ++i) nx = min(nx, sm.red64[0][i]);
                const double x = __dadd_rn(__dmul_rn((double)(ehi - elo + 1), 0.6931471805599453 * 0x1p-30),
                                           0x1p-51);
                const double ub = __dmul_rn(bstar, __dadd_rn(1.0, __dmul_rn(4.0, x)));
                const double bnext = (nx == ~0ull) ? CUDART_INF : __longlong_as_double((long long)nx);
                if (bnext > ub) {
                    cta_write_plan(sm, u, D, nb, cb, depth_of(g, bnext), depth, runs);
                    return;
                }
            }
            // the 30 dependent steps, on one thread
            if (j == 0) {
                if (normal_chain) {
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
                sm.hi_out = hi;
            }
            __syncthreads();
            hi = sm.hi_out;
        } else {
            for (int it = 0; it < 30; ++it) {
                const double mid = __dsqrt_rn(__dmul_rn(lo, hi));
                if (total(mid) <= B) hi = mid; else lo = mid;
            }
        }
    }
    cta_write_plan(sm, u, D, nb, cb, depth_of(g, hi), depth, runs);
    if (j == 0 && theta_out) theta_out[u] = hi;
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
    const cudaError_t e = launch_pdl(plan_kernel, dim3(s.units), dim3(kPT), 0, st, s.units, s.n,
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

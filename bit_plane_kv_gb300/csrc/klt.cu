// klt.cu -- rotated basis (Fathom §3.5): per calibration group (one layer
// and KV head) the mean mu and the eigenvectors V / eigenvalues lambda of the
// key covariance; the store holds the bit planes of (k - mu) V, queries are
// rotated q' = q V, and the plan weighs channel j of the rotated basis by
// g_j = sum_h q'_hj^2 lambda_j.  q' . (k - mu) V = q . (k - mu): the ranking
// of the tokens is that of q . k (q . mu is the same for every token).
//
// Unit u belongs to group u % groups (units are packed sequence, layer, KV
// head, so with groups = layers x KV heads every sequence shares its layer's
// and head's basis).
//
//   klt_mean_kernel    fp64 mean per channel, rows in order
//   klt_cov_kernel     fp64 covariance (ddof = 1) of the centred rows, 4 x 4
//                      entries per thread, centred rows staged in shared memory
//   klt_eigh_kernel    cyclic Jacobi (row-cyclic pairs p < r, the rotation
//                      that zeroes A[p][r]) in fp64, one CTA per group with A in
//                      shared memory; then eigenvalues in descending order and
//                      each eigenvector's largest-magnitude component positive
//   klt_rotate_keys    (k - mu) V per token, fp32 tiles of 64 tokens
//   klt_rotate_query   q V per head, V_g staged once for several units
#include "fathom_internal.cuh"

namespace fathom {

constexpr int kCovThreads = 256;
constexpr int kCovRows = 32;          // centred rows staged per round
constexpr int kEigThreads = 128;
constexpr int kRotTokens = 64;        // tokens per rotation tile
constexpr int kRotThreads = 256;

__global__ void klt_mean_kernel(int m, int D, const float *__restrict__ calib, double *__restrict__ mean) {
    const int g = blockIdx.x, j = threadIdx.x;
    if (j >= D) return;
    const float *x = calib + (size_t)g * m * D + j;
    double s = 0.0;
    for (int i = 0; i < m; ++i) s = __dadd_rn(s, (double)x[(size_t)i * D]);
    mean[(size_t)g * D + j] = __ddiv_rn(s, (double)m);
}

// Grid (groups, 4): CTA y covers covariance rows [32 y, 32 y + 32); thread t
// the 4 x 4 entries rows 32 y + 4 (t / 32) + 0..3, columns 4 (t % 32) + 0..3.
__global__ void __launch_bounds__(kCovThreads)
klt_cov_kernel(int m, int D, const float *__restrict__ calib, const double *__restrict__ mean,
               double *__restrict__ cov) {
    __shared__ double xc[kCovRows][FATHOM_MAX_D];
    __shared__ double mu[FATHOM_MAX_D];
    const int g = blockIdx.x, tid = threadIdx.x;
    const int a0 = 32 * blockIdx.y + 4 * (tid / 32), b0 = 4 * (tid % 32);
    for (int j = tid; j < FATHOM_MAX_D; j += kCovThreads) mu[j] = j < D ? mean[(size_t)g * D + j] : 0.0;
    double acc[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.0;
    const float *base = calib + (size_t)g * m * D;
    for (int i0 = 0; i0 < m; i0 += kCovRows) {
        __syncthreads();
        for (int e = tid; e < kCovRows * FATHOM_MAX_D; e += kCovThreads) {
            const int i = e / FATHOM_MAX_D, j = e % FATHOM_MAX_D;
            xc[i][j] = (i0 + i < m && j < D) ? (double)base[(size_t)(i0 + i) * D + j] - mu[j] : 0.0;
        }
        __syncthreads();
        const int rows = min(kCovRows, m - i0);
        for (int i = 0; i < rows; ++i) {
            double va[4], vb[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) { va[x] = xc[i][a0 + x]; vb[x] = xc[i][b0 + x]; }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fma(va[x], vb[y], acc[x][y]);
        }
    }
    const double inv = 1.0 / (double)(m - 1);
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y)
            if (a0 + x < D && b0 + y < D) cov[((size_t)g * D + a0 + x) * D + b0 + y] = acc[x][y] * inv;
}

__device__ __forceinline__ double block_sum(double v, double *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double s = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    return s;
}

// One CTA per group, thread x owns row and column x.  On entry vec holds the
// covariance; on exit the eigenvectors (columns).
__global__ void __launch_bounds__(kEigThreads)
klt_eigh_kernel(int D, double *__restrict__ vec, float *__restrict__ lambda) {
    extern __shared__ __align__(16) double A[];   // [D][D]
    __shared__ double red[kEigThreads / 32];
    __shared__ double lam_s[FATHOM_MAX_D];
    __shared__ int rank_s[FATHOM_MAX_D];
    const int g = blockIdx.x, x = threadIdx.x;
    double *V = vec + (size_t)g * D * D;
    for (int e = x; e < D * D; e += kEigThreads) A[e] = V[e];
    __syncthreads();
    for (int e = x; e < D * D; e += kEigThreads) V[e] = (e / D == e % D) ? 1.0 : 0.0;
    __syncthreads();
    for (int sweep = 0; sweep < 100; ++sweep) {
        double off = 0.0, tot = 0.0;
        if (x < D)
            for (int b = 0; b < D; ++b) {
                const double v = A[x * D + b] * A[x * D + b];
                tot += v;
                if (b != x) off += v;
            }
        off = block_sum(off, red);
        tot = block_sum(tot, red);
        if (off <= 1e-30 * tot || off == 0.0) break;
        for (int p = 0; p < D - 1; ++p)
            for (int r = p + 1; r < D; ++r) {
                const double apr = A[p * D + r];
                if (apr == 0.0) continue;                 // uniform: every thread reads the same value
                const double app = A[p * D + p], arr = A[r * D + r];
                const double tau = (arr - app) / (2.0 * apr);
                const double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                const double c = 1.0 / sqrt(1.0 + t * t), s = t * c;
                __syncthreads();                          // everyone has read A[p][r], A[p][p], A[r][r]
                if (x < D) {                              // columns p and r
                    const double axp = A[x * D + p], axr = A[x * D + r];
                    A[x * D + p] = c * axp - s * axr;
                    A[x * D + r] = s * axp + c * axr;
                    const double vxp = V[x * D + p], vxr = V[x * D + r];
                    V[x * D + p] = c * vxp - s * vxr;
                    V[x * D + r] = s * vxp + c * vxr;
                }
                __syncthreads();
                if (x < D) {                              // rows p and r
                    const double apx = A[p * D + x], arx = A[r * D + x];
                    A[p * D + x] = c * apx - s * arx;
                    A[r * D + x] = s * apx + c * arx;
                }
                __syncthreads();
            }
    }
    // eigenvalues in descending order (ties: lower index first), vectors permuted alike
    if (x < D) lam_s[x] = A[x * D + x];
    __syncthreads();
    if (x < D) {
        int rk = 0;
        for (int y = 0; y < D; ++y) rk += (lam_s[y] > lam_s[x] || (lam_s[y] == lam_s[x] && y < x)) ? 1 : 0;
        rank_s[x] = rk;
        lambda[(size_t)g * D + rk] = __double2float_rn(lam_s[x]);
    }
    __syncthreads();
    for (int e = x; e < D * D; e += kEigThreads) {   // A <- V with columns moved to their ranks
        const int row = e / D, col = e % D;
        A[row * D + rank_s[col]] = V[e];
    }
    __syncthreads();
    if (x < D) {   // column x: its largest-magnitude component (first of equals) positive
        int arg = 0;
        for (int y = 1; y < D; ++y)
            if (fabs(A[y * D + x]) > fabs(A[arg * D + x])) arg = y;
        const double sg = A[arg * D + x] < 0.0 ? -1.0 : 1.0;
        for (int y = 0; y < D; ++y) A[y * D + x] *= sg;
    }
    __syncthreads();
    for (int e = x; e < D * D; e += kEigThreads) V[e] = A[e];
}

// Grid (chunks, units): CTA x of unit u rotates token tiles x, x + chunks, ...
// of 64 tokens with V_g staged once in fp32.  Thread t computes tokens
// 8 (t / 32) + 0..7 of a tile and output channels (t % 32) + 32 c, c = 0..3;
// the centred tile is fp32 ((k - mu) rounded once from fp64).
template <typename T>
__global__ void __launch_bounds__(kRotThreads)
klt_rotate_keys_kernel(int n, int ctok, int D, int groups, const T *__restrict__ keys, const double *__restrict__ mean,
                       const double *__restrict__ vec, float *__restrict__ out) {
    extern __shared__ __align__(16) float rsm[];
    float *Vs = rsm;                                   // [128][128]
    float *xs = rsm + FATHOM_MAX_D * FATHOM_MAX_D;     // [64][129]
    constexpr int XS = FATHOM_MAX_D + 1;
    const int u = blockIdx.y, g = u % groups, tid = threadIdx.x;
    const double *Vg = vec + (size_t)g * D * D;
    for (int e = tid; e < FATHOM_MAX_D * FATHOM_MAX_D; e += kRotThreads) {
        const int j = e / FATHOM_MAX_D, c = e % FATHOM_MAX_D;
        Vs[e] = (j < D && c < D) ? __double2float_rn(Vg[(size_t)j * D + c]) : 0.0f;
    }
    const int tr = tid / 32, tc = tid % 32;
    for (int i0 = blockIdx.x * kRotTokens; i0 < n; i0 += gridDim.x * kRotTokens) {
        __syncthreads();   // the previous tile's reads of xs are done
        const T *kb = keys + ((size_t)u * ctok + i0) * D;
        for (int e = tid; e < kRotTokens * FATHOM_MAX_D; e += kRotThreads) {
            const int i = e / FATHOM_MAX_D, j = e % FATHOM_MAX_D;
            float v = 0.0f;
            if (i0 + i < n && j < D) {
                double k;
                if constexpr (sizeof(T) == 2) k = (double)__uint_as_float(((uint32_t)kb[(size_t)i * D + j]) << 16);
                else k = (double)kb[(size_t)i * D + j];
                v = __double2float_rn(k - mean[(size_t)g * D + j]);
            }
            xs[i * XS + j] = v;
        }
        __syncthreads();
        float acc[8][4];
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = 0.0f;
        for (int j = 0; j < D; ++j) {
            float va[8], vb[4];
#pragma unroll
            for (int a = 0; a < 8; ++a) va[a] = xs[(8 * tr + a) * XS + j];
#pragma unroll
            for (int c = 0; c < 4; ++c) vb[c] = Vs[j * FATHOM_MAX_D + tc + 32 * c];
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(va[a], vb[c], acc[a][c]);
        }
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const int i = i0 + 8 * tr + a;
            if (i >= n) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = tc + 32 * c;
                if (col < D) out[((size_t)u * ctok + i) * D + col] = acc[a][c];
            }
        }
    }
}

// Grid (groups, ceil(units_per_group / kQUnits)): a CTA stages V_g once in fp32
// (every thread keeps 32 independent 16-byte loads in flight) and rotates the
// queries of up to kQUnits units of group g (units g, g + groups, ...);
// thread t computes output channel t % 128 of half of the (unit, head) rows.
constexpr int kQUnits = 1;
constexpr int kQThreads = 256;
__global__ void __launch_bounds__(kQThreads)
klt_rotate_query_kernel(int units, int G, int D, int groups, const float *__restrict__ q,
                        const double *__restrict__ vec, float *__restrict__ out) {
    extern __shared__ __align__(16) float qsm[];
    float *Vs = qsm;                                        // [D][D] (row stride FATHOM_MAX_D)
    float *qs = qsm + FATHOM_MAX_D * FATHOM_MAX_D;          // [kQUnits * G][FATHOM_MAX_D]
    const int g = blockIdx.x, tid = threadIdx.x;
    const int t0 = blockIdx.y * kQUnits;
    const double *Vg = vec + (size_t)g * D * D;
    if (D == FATHOM_MAX_D && ((uintptr_t)Vg & 15) == 0) {
        constexpr int kPer = FATHOM_MAX_D * FATHOM_MAX_D / 2 / kQThreads;   // double2 per thread
        double2 r[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) r[i] = __ldg(reinterpret_cast<const double2 *>(Vg) + tid + i * kQThreads);
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            reinterpret_cast<float2 *>(Vs)[tid + i * kQThreads] = make_float2(__double2float_rn(r[i].x),
                                                                              __double2float_rn(r[i].y));
    } else {
        for (int e = tid; e < D * D; e += kQThreads) Vs[(e / D) * FATHOM_MAX_D + e % D] = __double2float_rn(Vg[e]);
    }
    int nu = 0;
    for (int t = 0; t < kQUnits; ++t) {
        const long long u = (long long)g + (long long)groups * (t0 + t);
        if (u >= units) break;
        for (int e = tid; e < G * D; e += kQThreads) qs[(t * G + e / D) * FATHOM_MAX_D + e % D] = q[u * G * D + e];
        ++nu;
    }
    __syncthreads();
    const int c = tid % FATHOM_MAX_D, part = tid / FATHOM_MAX_D;
    if (c >= D) return;
    constexpr int kRows = kQUnits * FATHOM_MAX_G / 2;      // (unit, head) rows per thread
    const int rows = nu * G, r0 = part * kRows;
    float acc[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) acc[i] = 0.0f;
    for (int j = 0; j < D; ++j) {
        const float v = Vs[j * FATHOM_MAX_D + c];
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            if (r0 + i < rows) acc[i] = fmaf(qs[(r0 + i) * FATHOM_MAX_D + j], v, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        if (r0 + i < rows) {
            const long long u = (long long)g + (long long)groups * (t0 + (r0 + i) / G);
            out[(u * G + (r0 + i) % G) * D + c] = acc[i];
        }
    }
}

int launch_calibrate_klt(int groups, int m, int D, const float *calib, double *mean, double *vec,
                         float *lambda, cudaStream_t st) {
    if (groups > 65535) { set_error("calibrate_klt: too many groups for one launch"); return FATHOM_EINVAL; }
    klt_mean_kernel<<<groups, FATHOM_MAX_D, 0, st>>>(m, D, calib, mean);
    int rc = launch_status("klt_mean_kernel");
    if (rc) return rc;
    klt_cov_kernel<<<dim3(groups, 4), kCovThreads, 0, st>>>(m, D, calib, mean, vec);
    rc = launch_status("klt_cov_kernel");
    if (rc) return rc;
    const size_t smem = (size_t)D * D * sizeof(double);
    ensure_smem(klt_eigh_kernel, smem);
    klt_eigh_kernel<<<groups, kEigThreads, smem, st>>>(D, vec, lambda);
    return launch_status("klt_eigh_kernel");
}

int launch_rotate_keys(const fathom_shape &s, const void *keys, int dtype, int groups, const double *mean,
                       const double *vec, float *out, cudaStream_t st) {
    if (s.units > 65535) { set_error("rotate_keys: too many units for one launch"); return FATHOM_EINVAL; }
    const size_t smem = ((size_t)FATHOM_MAX_D * FATHOM_MAX_D + (size_t)kRotTokens * (FATHOM_MAX_D + 1)) * sizeof(float);
    const int tiles = (s.n + kRotTokens - 1) / kRotTokens;
    const dim3 grid(tiles < 16 ? tiles : 16, s.units);   // each CTA stages V_g once for several tiles
    if (dtype == FATHOM_F32) {
        ensure_smem(klt_rotate_keys_kernel<float>, smem);
        klt_rotate_keys_kernel<float><<<grid, kRotThreads, smem, st>>>(s.n, cap_tokens(s), s.D, groups, (const float *)keys, mean,
                                                                       vec, out);
    } else {
        ensure_smem(klt_rotate_keys_kernel<uint16_t>, smem);
        klt_rotate_keys_kernel<uint16_t><<<grid, kRotThreads, smem, st>>>(s.n, cap_tokens(s), s.D, groups, (const uint16_t *)keys,
                                                                          mean, vec, out);
    }
    return launch_status("klt_rotate_keys_kernel");
}

int launch_rotate_query(const fathom_shape &s, const float *q, int groups, const double *vec, float *out,
                        cudaStream_t st) {
    const int per_group = (s.units + groups - 1) / groups;   // units of the most populous group
    const dim3 grid(groups < s.units ? groups : s.units, (per_group + kQUnits - 1) / kQUnits);
    if (grid.x > 65535 * 32 || grid.y > 65535) { set_error("rotate_query: too many units"); return FATHOM_EINVAL; }
    const size_t smem = ((size_t)FATHOM_MAX_D * FATHOM_MAX_D + (size_t)kQUnits * FATHOM_MAX_G * FATHOM_MAX_D) * sizeof(float);
    ensure_smem(klt_rotate_query_kernel, smem);
    klt_rotate_query_kernel<<<grid, kQThreads, smem, st>>>(s.units, s.G, s.D, groups, q, vec, out);
    return launch_status("klt_rotate_query_kernel");
}


// ---------------------------------------------------------------- online basis
// A session's own keys give its basis (Fathom Appx. D: mean, eigenbasis and
// eigenvalues without calibration data).  fp64 runs at a small fraction of
// the fp32 rate on this part, so the per-token work is fp32 with fp64 only
// where partial results are combined:
//   klt_online_mean_kernel  fp32 sums over runs of 64 tokens, folded in fp64,
//                           one partial per (unit, slice)
//   klt_online_cov_kernel   the slices' partials summed in a fixed order give
//                           mu; rows centred in fp32 and staged 32 tokens at a
//                           time; each thread accumulates an 8 x 8 tile of the
//                           upper triangle (a per-stage fp32 sum added into a
//                           running fp32 total), one partial per slice
//   klt_online_reduce_kernel  covariance = fixed-order fp64 sum of the
//                           slices' partials / (n - 1), mirrored
//   klt_eigh32_kernel       parallel cyclic Jacobi in fp32 (round-robin
//                           ordering: D / 2 disjoint pairs rotated at once)
constexpr int kOnThreads = 160;       // 136 upper-triangle tiles of 8 x 8 (+ staging helpers)
constexpr int kOnTiles = 136;
constexpr int kOnStage = 32;          // tokens staged per round
constexpr int kOnMeanThreads = 256;
constexpr int kEig32Threads = 512;
constexpr int kEigPad = FATHOM_MAX_D + 1;

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Grid (slices, units).  Thread t sums channel t % 128 over the slice's tokens
// of parity t / 128, in fp32 runs of 64 tokens folded into fp64.
__global__ void __launch_bounds__(kOnMeanThreads)
klt_online_mean_kernel(int n, int ctok, int D, int tps, const uint16_t *__restrict__ rows,
                       double *__restrict__ part) {
    __shared__ double red[kOnMeanThreads];
    const int s = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
    const int j = tid % FATHOM_MAX_D, par = tid / FATHOM_MAX_D;
    const int i0 = s * tps, i1 = min(n, i0 + tps);
    double acc = 0.0;
    if (j < D) {
        const uint16_t *base = rows + (size_t)u * ctok * D + j;
        for (int r0 = i0 + par; r0 < i1; r0 += 128) {
            float run = 0.0f;
            const int r1 = min(i1, r0 + 128);
            for (int i = r0; i < r1; i += 2) run += bf16_to_f32(__ldg(base + (size_t)i * D));
            acc += (double)run;
        }
    }
    red[tid] = acc;
    __syncthreads();
    if (tid < FATHOM_MAX_D && tid < D)
        part[((size_t)u * gridDim.x + s) * FATHOM_MAX_D + tid] = red[tid] + red[tid + FATHOM_MAX_D];
}

// Grid (slices, units), kOnThreads threads.
__global__ void __launch_bounds__(kOnThreads)
klt_online_cov_kernel(int n, int ctok, int D, int tps, const uint16_t *__restrict__ rows,
                      const double *__restrict__ mean_part, double *__restrict__ mean_out,
                      float *__restrict__ cov_part) {
    __shared__ __align__(16) float xs[kOnStage][FATHOM_MAX_D];
    __shared__ float mu[FATHOM_MAX_D];
    const int s = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
    const int S = gridDim.x;
    if (tid < FATHOM_MAX_D) {
        double m = 0.0;
        if (tid < D) {
            for (int q = 0; q < S; ++q) m += mean_part[((size_t)u * S + q) * FATHOM_MAX_D + tid];
            m /= (double)n;
            if (s == 0) mean_out[(size_t)u * D + tid] = m;
        }
        mu[tid] = __double2float_rn(m);
    }
    // this thread's tile (ti <= tj) of the upper triangle
    int ti = 0, tj = 0;
    {
        int t = tid < kOnTiles ? tid : 0;
        while (t >= 16 - ti) { t -= 16 - ti; ++ti; }
        tj = ti + t;
    }
    float tot[8][8], stg[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) tot[a][b] = 0.0f;
    const int i0 = s * tps, i1 = min(n, i0 + tps);
    const uint16_t *base = rows + (size_t)u * ctok * D;
    for (int r0 = i0; r0 < i1; r0 += kOnStage) {
        __syncthreads();   // mu ready / the previous stage's reads are done
        for (int e = tid; e < kOnStage * FATHOM_MAX_D; e += kOnThreads) {
            const int i = e / FATHOM_MAX_D, j = e % FATHOM_MAX_D;
            float v = 0.0f;
            if (r0 + i < i1 && j < D) v = bf16_to_f32(__ldg(base + (size_t)(r0 + i) * D + j)) - mu[j];
            xs[i][j] = v;
        }
        __syncthreads();
        if (tid < kOnTiles) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) stg[a][b] = 0.0f;
            const int rn = min(kOnStage, i1 - r0);
            for (int i = 0; i < rn; ++i) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&xs[i][8 * ti]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&xs[i][8 * ti + 4]);
                const float4 b0 = *reinterpret_cast<const float4 *>(&xs[i][8 * tj]);
                const float4 b1 = *reinterpret_cast<const float4 *>(&xs[i][8 * tj + 4]);
                const float va[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float vb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int a = 0; a < 8; ++a)
#pragma unroll
                    for (int b = 0; b < 8; ++b) stg[a][b] = fmaf(va[a], vb[b], stg[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) tot[a][b] += stg[a][b];
        }
    }
    if (tid < kOnTiles) {
        float *P = cov_part + ((size_t)u * S + s) * FATHOM_MAX_D * FATHOM_MAX_D;
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            float4 *dst = reinterpret_cast<float4 *>(P + (size_t)(8 * ti + a) * FATHOM_MAX_D + 8 * tj);
            dst[0] = make_float4(tot[a][0], tot[a][1], tot[a][2], tot[a][3]);
            dst[1] = make_float4(tot[a][4], tot[a][5], tot[a][6], tot[a][7]);
        }
    }
}

// Grid (D * D / 256 rounded up, units): one entry per thread, fp64 sum over the
// slices in order, / (n - 1); entries below the diagonal read the mirror.
__global__ void __launch_bounds__(256)
klt_online_reduce_kernel(int n, int D, int S, const float *__restrict__ cov_part, double *__restrict__ cov) {
    const int u = blockIdx.y;
    const int e = blockIdx.x * 256 + threadIdx.x;
    if (e >= D * D) return;
    const int a = e / D, b = e % D;
    const int lo = min(a, b), hi = max(a, b);
    const float *P = cov_part + (size_t)u * S * FATHOM_MAX_D * FATHOM_MAX_D + (size_t)lo * FATHOM_MAX_D + hi;
    double acc = 0.0;
    for (int q = 0; q < S; ++q) acc += (double)P[(size_t)q * FATHOM_MAX_D * FATHOM_MAX_D];
    cov[(size_t)u * D * D + e] = acc / (double)(n - 1);
}

// One CTA per unit.  On entry vec holds the covariance (fp64); on exit the
// eigenvectors (unit-length columns, fp32 values widened), eigenvalues descending, each
// vector's largest-magnitude component positive.  Round-robin ordering over
// Dp = D rounded up to even indices: in step t, pair 0 is (0, 1 + t mod (Dp - 1))
// and pair i > 0 is (1 + (t + i) mod (Dp - 1), 1 + (t - i) mod (Dp - 1)); every
// pair meets once per sweep of Dp - 1 steps.  A pair rotates when |a_pr| exceeds
// both 2^-23 sqrt(|a_pp a_rr|) and 2^-22 ||A||_F (fp32 rounding leaves
// off-diagonal entries of about 2^-24 ||A|| that no rotation removes); sweeps
// stop when one rotates nothing or after 24 sweeps.  Warp w applies the
// rotations of pairs w, w + 16, ... with its lanes over the rows.
__global__ void __launch_bounds__(kEig32Threads)
klt_eigh32_kernel(int D, double *__restrict__ vec, float *__restrict__ lambda) {
    extern __shared__ __align__(16) float esm[];
    float *A = esm;                                  // [128][129]
    float *V = esm + FATHOM_MAX_D * kEigPad;         // [128][129]
    __shared__ int pp[FATHOM_MAX_D / 2], pr[FATHOM_MAX_D / 2];
    __shared__ float pc[FATHOM_MAX_D / 2], ps[FATHOM_MAX_D / 2];
    __shared__ float red[kEig32Threads / 32];
    __shared__ float lam_s[FATHOM_MAX_D];
    __shared__ int rank_s[FATHOM_MAX_D];
    constexpr int NW = kEig32Threads / 32;
    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Dp = D + (D & 1), half = Dp / 2;
    double *Vg = vec + (size_t)u * D * D;
    for (int x = warp; x < Dp; x += NW)
        for (int y = lane; y < Dp; y += 32) {
            A[x * kEigPad + y] = (x < D && y < D) ? __double2float_rn(Vg[(size_t)x * D + y]) : 0.0f;
            V[x * kEigPad + y] = (x == y) ? 1.0f : 0.0f;
        }
    __syncthreads();
    for (int sweep = 0; sweep < 24; ++sweep) {
        float tot = 0.0f;
        for (int x = warp; x < Dp; x += NW)
            for (int y = lane; y < Dp; y += 32) tot = fmaf(A[x * kEigPad + y], A[x * kEigPad + y], tot);
#pragma unroll
        for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane == 0) red[warp] = tot;
        __syncthreads();
        tot = 0.0f;
        for (int w = 0; w < NW; ++w) tot += red[w];
        const float floor_abs = 2.384185791e-7f * sqrtf(tot);      // 2^-22 ||A||_F
        int rotated = 0;
        for (int t = 0; t < Dp - 1; ++t) {
            if (tid < half) {
                int p, r;
                if (tid == 0) { p = 0; r = 1 + t % (Dp - 1); }
                else {
                    p = 1 + (t + tid) % (Dp - 1);
                    r = 1 + (t - tid + (Dp - 1)) % (Dp - 1);
                }
                if (p > r) { const int q = p; p = r; r = q; }
                const float apr = A[p * kEigPad + r], app = A[p * kEigPad + p], arr = A[r * kEigPad + r];
                float c = 1.0f, sn = 0.0f;
                const float aa = fabsf(apr);
                if (aa > floor_abs && aa > 1.1920929e-7f * sqrtf(fabsf(app * arr))) {
                    const float th = (arr - app) / (2.0f * apr);
                    const float tt = fabsf(th) > 1e18f ? 0.5f / th
                                                       : (th >= 0.0f ? 1.0f : -1.0f) / (fabsf(th) + sqrtf(1.0f + th * th));
                    c = 1.0f / sqrtf(1.0f + tt * tt);
                    sn = tt * c;
                    rotated = 1;
                }
                pp[tid] = p; pr[tid] = r; pc[tid] = c; ps[tid] = sn;
            }
            __syncthreads();
            for (int i = warp; i < half; i += NW) {          // columns p and r of A and V
                const int p = pp[i], r = pr[i];
                const float c = pc[i], sn = ps[i];
                if (sn == 0.0f) continue;                     // uniform across the warp
                for (int x = lane; x < Dp; x += 32) {
                    const float axp = A[x * kEigPad + p], axr = A[x * kEigPad + r];
                    A[x * kEigPad + p] = c * axp - sn * axr;
                    A[x * kEigPad + r] = sn * axp + c * axr;
                    const float vxp = V[x * kEigPad + p], vxr = V[x * kEigPad + r];
                    V[x * kEigPad + p] = c * vxp - sn * vxr;
                    V[x * kEigPad + r] = sn * vxp + c * vxr;
                }
            }
            __syncthreads();
            for (int i = warp; i < half; i += NW) {          // rows p and r of A
                const int p = pp[i], r = pr[i];
                const float c = pc[i], sn = ps[i];
                if (sn == 0.0f) continue;
                for (int x = lane; x < Dp; x += 32) {
                    const float apx = A[p * kEigPad + x], arx = A[r * kEigPad + x];
                    A[p * kEigPad + x] = c * apx - sn * arx;
                    A[r * kEigPad + x] = sn * apx + c * arx;
                }
            }
            __syncthreads();
        }
        if (!__syncthreads_or(rotated)) break;
    }
    // eigenvalues in descending order (ties: lower index first), vectors permuted alike
    if (tid < D) lam_s[tid] = A[tid * kEigPad + tid];
    __syncthreads();
    if (tid < D) {
        int rk = 0;
        for (int y = 0; y < D; ++y) rk += (lam_s[y] > lam_s[tid] || (lam_s[y] == lam_s[tid] && y < tid)) ? 1 : 0;
        rank_s[tid] = rk;
        lambda[(size_t)u * D + rk] = lam_s[tid];
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kEig32Threads) {   // A <- V with columns moved to their ranks
        const int row = e / D, col = e % D;
        A[row * kEigPad + rank_s[col]] = V[row * kEigPad + col];
    }
    __syncthreads();
    if (tid < D) {
        // column tid: unit length again (the fp32 rotations let c^2 + s^2 drift from
        // 1 by an ulp each, which accumulates over the sweeps; norm in fp64) and its
        // largest-magnitude component (first of equals) positive
        int arg = 0;
        double nn = 0.0;
        for (int y = 0; y < D; ++y) {
            const float a = A[y * kEigPad + tid];
            nn += (double)a * (double)a;
            if (fabsf(a) > fabsf(A[arg * kEigPad + tid])) arg = y;
        }
        const float sc = (float)((A[arg * kEigPad + tid] < 0.0f ? -1.0 : 1.0) / sqrt(nn));
        for (int y = 0; y < D; ++y) A[y * kEigPad + tid] *= sc;
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kEig32Threads) Vg[e] = (double)A[(e / D) * kEigPad + e % D];
}

static size_t klt_align(size_t x) { return (x + 255) & ~(size_t)255; }

KltOnlineWs klt_online_layout(const fathom_shape &s) {
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;
    KltOnlineWs w;
    // about four CTAs per SM over the units, at least 512 tokens per slice
    int S = (4 * sms + s.units - 1) / s.units;
    const int max_s = (s.n + 511) / 512;
    S = S < 1 ? 1 : (S > max_s ? max_s : S);
    w.tps = ((s.n + S - 1) / S + kOnStage - 1) / kOnStage * kOnStage;
    w.slices = (s.n + w.tps - 1) / w.tps;
    w.mean_off = 0;
    w.cov_off = klt_align((size_t)s.units * w.slices * FATHOM_MAX_D * sizeof(double));
    w.total = klt_align(w.cov_off + (size_t)s.units * w.slices * FATHOM_MAX_D * FATHOM_MAX_D * sizeof(float));
    return w;
}

int launch_klt_online(const fathom_shape &s, const uint16_t *rows, double *mean, double *vec, float *lambda,
                      void *ws, cudaStream_t st) {
    if (s.units > 65535) { set_error("klt_online: too many units for one launch"); return FATHOM_EINVAL; }
    const KltOnlineWs w = klt_online_layout(s);
    char *base = (char *)ws;
    double *mpart = (double *)(base + w.mean_off);
    float *cpart = (float *)(base + w.cov_off);
    const int ctok = cap_tokens(s);
    klt_online_mean_kernel<<<dim3(w.slices, s.units), kOnMeanThreads, 0, st>>>(s.n, ctok, s.D, w.tps, rows, mpart);
    int rc = launch_status("klt_online_mean_kernel");
    if (rc) return rc;
    klt_online_cov_kernel<<<dim3(w.slices, s.units), kOnThreads, 0, st>>>(s.n, ctok, s.D, w.tps, rows, mpart, mean,
                                                                          cpart);
    rc = launch_status("klt_online_cov_kernel");
    if (rc) return rc;
    klt_online_reduce_kernel<<<dim3((s.D * s.D + 255) / 256, s.units), 256, 0, st>>>(s.n, s.D, w.slices, cpart, vec);
    rc = launch_status("klt_online_reduce_kernel");
    if (rc) return rc;
    const size_t smem = 2 * (size_t)FATHOM_MAX_D * kEigPad * sizeof(float);
    ensure_smem(klt_eigh32_kernel, smem);
    klt_eigh32_kernel<<<s.units, kEig32Threads, smem, st>>>(s.D, vec, lambda);
    return launch_status("klt_eigh32_kernel");
}

}  // namespace fathom

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

}  // namespace fathom

// Fidelity diagnostics and per-layer budgets.
//
// The Fathom review page ("Fathom: 쿼리마다 깊이를 바꾸는 스캔으로 1M 토큰 디코딩을
// 1.67배 빠르게 하다"), §4 and §5, measures the sparse path by the relative L2
// error of its attention output against dense attention and against exact
// top-k attention, and by how far the kept sets agree with the exact top-k;
// §3.4 gives the greedy per-layer plan that hands bits to the layer with the
// largest error reduction per bit.  These are off the decode path: one warp
// per output row for the two reductions, plain host code for the allocation.
#include "fathom_internal.cuh"

namespace fathom {

namespace {

constexpr int kFidThreads = 256;
constexpr int kFidWarps = kFidThreads / 32;

// err[r] = ||a_r - ref_r|| / ||ref_r||, both sums in fp64 over lanes then a
// fixed shuffle tree; ||a_r|| when ref_r is all zeros.
__global__ void __launch_bounds__(kFidThreads)
rel_err_kernel(int rows, int D, const float *__restrict__ a, const float *__restrict__ ref,
               double *__restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kFidWarps + (threadIdx.x >> 5);
    if (r >= rows) return;
    const float *ar = a + (size_t)r * D, *rr = ref + (size_t)r * D;
    double num = 0.0, den = 0.0;
    for (int j = lane; j < D; j += 32) {
        const double x = (double)ar[j], y = (double)rr[j];
        num += (x - y) * (x - y);
        den += y * y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        num += __shfl_xor_sync(0xffffffffu, num, o);
        den += __shfl_xor_sync(0xffffffffu, den, o);
    }
    if (lane == 0) err[r] = den > 0.0 ? sqrt(num) / sqrt(den) : sqrt(num);
}

// count[r] = |{a_r} ∩ {b_r}| for strictly ascending lists of length k: each
// element of a_r is looked up in b_r by binary search.
__global__ void __launch_bounds__(kFidThreads)
set_overlap_kernel(int rows, int k, const int32_t *__restrict__ a, const int32_t *__restrict__ b,
                   int32_t *__restrict__ count) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kFidWarps + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int32_t *ar = a + (size_t)r * k, *br = b + (size_t)r * k;
    int c = 0;
    for (int i = lane; i < k; i += 32) {
        const int32_t x = ar[i];
        int lo = 0, hi = k;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (br[mid] < x) lo = mid + 1; else hi = mid;
        }
        c += (lo < k && br[lo] == x) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) count[r] = c;
}

}  // namespace

int launch_rel_err(int rows, int D, const float *a, const float *ref, double *err, cudaStream_t st) {
    if (rows == 0) return FATHOM_OK;
    const int blocks = (rows + kFidWarps - 1) / kFidWarps;
    rel_err_kernel<<<blocks, kFidThreads, 0, st>>>(rows, D, a, ref, err);
    return launch_status("rel_err_kernel");
}

int launch_set_overlap(int rows, int k, const int32_t *a, const int32_t *b, int32_t *count, cudaStream_t st) {
    if (rows == 0) return FATHOM_OK;
    const int blocks = (rows + kFidWarps - 1) / kFidWarps;
    set_overlap_kernel<<<blocks, kFidThreads, 0, st>>>(rows, k, a, b, count);
    return launch_status("set_overlap_kernel");
}

// Every layer starts at b_min; each of layers (b_mean - b_min) / step
// increments of `step` bits goes to the layer whose error falls the most on
// its next level (ties to the lower layer), layers at the top level take no more.
int greedy_budgets(int layers, int levels, const double *err, int b_min, int step, int b_mean,
                   int32_t *budgets) {
    const long long incs = (long long)layers * (b_mean - b_min) / step;
    int *lev = new int[layers];
    for (int l = 0; l < layers; ++l) lev[l] = 0;
    for (long long it = 0; it < incs; ++it) {
        int best = -1;
        double best_gain = 0.0;
        for (int l = 0; l < layers; ++l) {
            if (lev[l] + 1 >= levels) continue;
            const double gain = err[(size_t)l * levels + lev[l]] - err[(size_t)l * levels + lev[l] + 1];
            if (best < 0 || gain > best_gain) { best = l; best_gain = gain; }
        }
        if (best < 0) break;
        ++lev[best];
    }
    for (int l = 0; l < layers; ++l) budgets[l] = b_min + step * lev[l];
    delete[] lev;
    return FATHOM_OK;
}

}  // namespace fathom

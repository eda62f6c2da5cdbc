// calibrate.cu -- per-channel calibration statistics (Fathom §3.3: Var(k_j)
// is measured once on calibration keys).  fp64 accumulation in row order with
// explicitly rounded operations (no contraction), so the result is the same
// on any IEEE machine; rounded to fp32 once at the end.
#include "fathom_internal.cuh"

namespace fathom {

__global__ void calibrate_kernel(int m, int D, const float *__restrict__ calib,
                                 float *__restrict__ mean_out, float *__restrict__ var_out) {
    const int u = blockIdx.x;
    const int j = threadIdx.x;
    if (j >= D) return;
    const float *x = calib + (size_t)u * m * D + j;
    double s = 0.0;
    for (int i = 0; i < m; ++i) s = __dadd_rn(s, (double)x[(size_t)i * D]);
    const double mean = __ddiv_rn(s, (double)m);
    double v = 0.0;
    for (int i = 0; i < m; ++i) {
        double d = __dsub_rn((double)x[(size_t)i * D], mean);
        v = __dadd_rn(v, __dmul_rn(d, d));
    }
    const double var = __ddiv_rn(v, (double)(m - 1));
    if (mean_out) mean_out[(size_t)u * D + j] = __double2float_rn(mean);
    var_out[(size_t)u * D + j] = __double2float_rn(var);
}

int launch_calibrate(int units, int m, int D, const float *calib, float *mean, float *var,
                     cudaStream_t st) {
    calibrate_kernel<<<units, 128, 0, st>>>(m, D, calib, mean, var);
    return launch_status("calibrate_kernel");
}

}  // namespace fathom

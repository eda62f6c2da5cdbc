// Host build of the plan's integer square root (bit_plane_kv_gb300/csrc/exact_sqrt.cuh),
// exported over plain arrays so that a CPU test can compare it with IEEE sqrt bit for bit.
#include <stddef.h>
#include <stdint.h>

#include "exact_sqrt.cuh"

extern "C" void xsqrt_many(size_t n, const uint64_t *x, float seed_scale, uint64_t *out) {
    for (size_t i = 0; i < n; ++i) out[i] = fathom::xsqrt::sqrt_rn(x[i], seed_scale);
}

// gather.cu -- contiguous-run gather from the (host-resident) store into an
// HBM staging area (Fathom §3.6: with the whole sequence one channel-major
// block, channel j's first t_j planes are one t_j * n / 8-byte run; a gather
// kernel copies one run plus the scales per active channel, and the run list
// has a fixed slot per channel so no host synchronisation is needed).
//
// The destination of a unit is dense (runs are packed in channel order), so
// the work is laid over destination space in windows of W words: a CTA of
// unit u copies windows x, x + gridDim.x, ..., finding the runs that overlap
// each window from the run list in shared memory.  Every thread keeps several
// 16-byte loads in flight before storing, which is what a long-latency host
// link needs; about two CTAs per SM saturate the link.
#include "fathom_internal.cuh"

namespace fathom {

constexpr int kGThreads = 256;
constexpr int kGChunkWords = 8192;     // 64 KiB of plane words per CTA
constexpr int kGChunkScales = 16384;   // 32 KiB of scales per CTA
constexpr int kGUnroll = 4;

template <typename T, typename V>
__device__ __forceinline__ void copy_span(const T *__restrict__ src, T *__restrict__ dst, uint32_t len,
                                          bool vec_ok) {
    constexpr int E = sizeof(V) / sizeof(T);
    if (vec_ok) {
        const uint32_t nv = len / E;
        const V *s = reinterpret_cast<const V *>(src);
        V *d = reinterpret_cast<V *>(dst);
        uint32_t i = threadIdx.x;
        for (; i + (kGUnroll - 1) * kGThreads < nv; i += kGUnroll * kGThreads) {
            V r[kGUnroll];
#pragma unroll
            for (int k = 0; k < kGUnroll; ++k) r[k] = __ldcs(s + i + k * kGThreads);
#pragma unroll
            for (int k = 0; k < kGUnroll; ++k) d[i + k * kGThreads] = r[k];
        }
        for (; i < nv; i += kGThreads) d[i] = __ldcs(s + i);
        for (uint32_t e = nv * E + threadIdx.x; e < len; e += kGThreads) dst[e] = src[e];
    } else {
        for (uint32_t e = threadIdx.x; e < len; e += kGThreads) dst[e] = src[e];
    }
}

__global__ void __launch_bounds__(kGThreads)
gather_kernel(int D, int nb, int cb, int x_planes, int x_total, const uint64_t *__restrict__ store_planes,
              const uint16_t *__restrict__ store_scales, const fathom_run *__restrict__ runs,
              uint64_t *__restrict__ stage_planes, uint16_t *__restrict__ stage_scales,
              size_t stage_words, size_t stage_scales_n, int vec_planes, int vec_scales) {
    __shared__ fathom_run r[FATHOM_MAX_D];
    const int u = blockIdx.y;
    for (int j = threadIdx.x; j < D; j += kGThreads) {
        fathom_run v = runs[(size_t)u * D + j];
        // The source fields must be the ones the plan writes for channel j: the run
        // starts at the channel's own planes and scales, covers whole planes (at most
        // four) and at most one scale per block.  Any other run would read outside
        // channel j's part of the store, so it copies nothing.
        const bool ok = v.src_word == (uint32_t)j * FATHOM_PLANES * (uint32_t)cb &&
                        v.src_scale == (uint32_t)j * (uint32_t)cb &&
                        v.n_words <= (uint32_t)FATHOM_PLANES * (uint32_t)nb && v.n_words % (uint32_t)nb == 0 &&
                        v.n_scales <= (uint32_t)nb;
        if (!ok) { v.n_words = 0; v.n_scales = 0; }
        r[j] = v;
    }
    __syncthreads();
    // grid-stride over the unit's destination windows: plane windows, then scale windows
    for (int x = blockIdx.x; x < x_total; x += gridDim.x) {
        const bool do_planes = x < x_planes;
        const size_t win = do_planes ? kGChunkWords : kGChunkScales;
        const size_t cap = do_planes ? stage_words : stage_scales_n;
        const size_t d0 = (size_t)(do_planes ? x : x - x_planes) * win;
        if (d0 >= cap) continue;
        const size_t d1 = min(d0 + win, cap);
        for (int j = 0; j < D; ++j) {
            const size_t rs = do_planes ? r[j].dst_word : r[j].dst_scale;
            const size_t rl = do_planes ? r[j].n_words : r[j].n_scales;
            const size_t lo = max(rs, d0), hi = min(rs + rl, d1);
            if (lo >= hi) continue;
            if (do_planes) {
                // the run is the first nb words of t planes that lie cb words apart in the
                // store (one contiguous span when cb = nb); copy it plane by plane
                const uint64_t *sbase = store_planes + (size_t)u * D * FATHOM_PLANES * cb + r[j].src_word;
                size_t d = lo;
                while (d < hi) {
                    const size_t p = (d - rs) / nb, o = (d - rs) - p * nb;
                    const size_t seg = (cb == nb) ? hi - d : min(hi - d, nb - o);
                    const size_t src0 = p * cb + o;
                    const size_t sidx = (size_t)u * D * FATHOM_PLANES * cb + r[j].src_word + src0;
                    (void)sidx;   // read by the debug build's checks only
                    if (FATHOM_CHECK(sidx + seg <= (size_t)gridDim.y * D * FATHOM_PLANES * cb, kDbgGatherSrc, sidx) &&
                        FATHOM_CHECK(d + seg <= stage_words, kDbgGatherDst, d + seg))
                        copy_span<uint64_t, uint4>(sbase + src0, stage_planes + (size_t)u * stage_words + d,
                                                   (uint32_t)seg,
                                                   vec_planes && (((r[j].src_word + src0) | d) % 2 == 0));
                    d += seg;
                }
            } else {
                const size_t src0 = r[j].src_scale + (lo - rs);
                const size_t sidx = (size_t)u * D * cb + src0;
                (void)sidx;   // read by the debug build's checks only
                if (FATHOM_CHECK(sidx + (hi - lo) <= (size_t)gridDim.y * D * cb, kDbgGatherSrc, sidx) &&
                    FATHOM_CHECK(hi <= stage_scales_n, kDbgGatherDst, hi))
                    copy_span<uint16_t, uint4>(store_scales + (size_t)u * D * cb + src0,
                                               stage_scales + (size_t)u * stage_scales_n + lo,
                                               (uint32_t)(hi - lo), vec_scales && ((src0 | lo) % 8 == 0));
            }
        }
    }
}

FATHOM_DEBUG_READER(debug_read_gather)

int launch_gather(const fathom_shape &s, const uint64_t *sp, const uint16_t *ss,
                  const fathom_run *runs, uint64_t *dp, uint16_t *ds, size_t stage_words,
                  size_t stage_scales, cudaStream_t st) {
    const int nb = num_blocks(s.n), cb = cap_blocks(s);
    // windows past the largest possible destination (every plane, every scale) never copy
    const size_t max_w = (size_t)s.D * FATHOM_PLANES * nb, max_s = (size_t)s.D * nb;
    const size_t wcap = stage_words < max_w ? stage_words : max_w;
    const size_t scap = stage_scales < max_s ? stage_scales : max_s;
    const int xp = (int)((wcap + kGChunkWords - 1) / kGChunkWords);
    const int xs = (int)((scap + kGChunkScales - 1) / kGChunkScales);
    if (s.units > 65535) { set_error("gather: too many units for one launch"); return FATHOM_EINVAL; }
    const uintptr_t a = (uintptr_t)sp | (uintptr_t)dp;
    const int vec_planes = (a % 16 == 0) && (stage_words % 2 == 0) && (nb % 2 == 0) && (cb % 2 == 0);
    const uintptr_t b = (uintptr_t)ss | (uintptr_t)ds;
    const int vec_scales = (b % 16 == 0) && (stage_scales % 8 == 0) && (nb % 8 == 0) && (cb % 8 == 0);
    // a copy over the host link needs enough bytes in flight (each thread keeps
    // 4 x 16 B outstanding) but not every SM: about two CTAs per SM in all, which
    // leaves room for kernels that run beside the gather
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;   // no device answered: the GB300's count
    int per_unit = (2 * sms + s.units - 1) / s.units;
    if (per_unit > xp + xs) per_unit = xp + xs;
    dim3 grid(per_unit, s.units);
    gather_kernel<<<grid, kGThreads, 0, st>>>(s.D, nb, cb, xp, xp + xs, sp, ss, runs, dp, ds, stage_words,
                                              stage_scales, vec_planes, vec_scales);
    return launch_status("gather_kernel");
}

}  // namespace fathom

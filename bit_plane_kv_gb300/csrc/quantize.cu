// quantize.cu -- 4-bit symmetric per-channel quantiser and channel-major
// bit-plane packing (Fathom §3.2, bit-plane K cache).
//
// One CTA takes four consecutive 64-token blocks of one unit (decode-time
// appends launch the same kernel over one block).  Each block is
// staged row-major in shared memory (coalesced loads of whole key rows), then
// thread (channel j, half h) reduces its 32 tokens' |k|, combines the two
// halves into the block maximum a, rounds a to fp16 and codes its 32 tokens:
//     c = clip(floor(k / s), -8, 7) + 8,   s = a16 / 8,
// with floor taken of the exact quotient (fp32 division, then an exact
// product check moves the result by one where the division rounded across
// an integer).  The four bits of the codes go straight into the 32-bit halves
// of the four plane words (bit p = 0 is the MSB, token i of the block at bit
// i), which are collected in shared memory and written as 32-byte runs
// [j][p][beta .. beta+3] of the channel-major store.
#include "fathom_internal.cuh"

namespace fathom {

constexpr int kQBlocks = 4;          // 64-token blocks per CTA
constexpr int kQThreads = 256;

__device__ __forceinline__ int code_of(float k, float a16) {
    if (a16 == 0.0f) return 8;
    const float s = a16 * 0.125f;                    // exact
    const float qv = __fdiv_rn(k, s);
    if (qv >= 16.0f) return 15;
    if (qv <= -16.0f) return 0;
    float f = floorf(qv);
    // |f| <= 16 and s has 11 significant bits: both products are exact
    if (__fmul_rn(f, s) > k) f -= 1.0f;
    else if (__fmul_rn(f + 1.0f, s) <= k) f += 1.0f;
    f = fminf(fmaxf(f, -8.0f), 7.0f);
    return (int)f + 8;
}

template <typename T>
__device__ __forceinline__ float load_key(const T *p);
template <>
__device__ __forceinline__ float load_key<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_key<uint16_t>(const uint16_t *p) {
    return __uint_as_float(((uint32_t)__ldg(p)) << 16);   // bf16 -> fp32, exact
}

struct QSmem {
    float tile[64][FATHOM_MAX_D + 1];
    float half_max[2][FATHOM_MAX_D];
    uint32_t words[FATHOM_MAX_D][FATHOM_PLANES][kQBlocks][2];
    uint16_t sc[FATHOM_MAX_D][kQBlocks];
};

// Blocks [block0, block1) of every unit of a sequence of n tokens; keys rows
// `ctok` tokens apart per unit, planes and scales `cb` blocks apart per
// (channel, plane).
template <typename T>
__global__ void __launch_bounds__(kQThreads)
quantize_kernel(int n, int D, int ctok, int cb, int block0, int block1, const T *__restrict__ keys,
                uint64_t *__restrict__ planes, uint16_t *__restrict__ scales) {
    extern __shared__ __align__(16) unsigned char qsmem[];
    QSmem &sm = *reinterpret_cast<QSmem *>(qsmem);
    auto &tile = sm.tile;
    auto &half_max = sm.half_max;
    auto &words = sm.words;
    auto &sc = sm.sc;

    const int u = blockIdx.y;
    const int beta0 = block0 + blockIdx.x * kQBlocks;
    const int nbl = min(kQBlocks, block1 - beta0);
    const int tid = threadIdx.x;
    const T *K = keys + (size_t)u * ctok * D;

    for (int bl = 0; bl < nbl; ++bl) {
        const int i0 = (beta0 + bl) * 64;
        const int nv = min(64, n - i0);
        __syncthreads();
        for (int e = tid; e < nv * D; e += kQThreads) {
            const int i = e / D, j = e - (e / D) * D;
            tile[i][j] = load_key<T>(K + (size_t)(i0 + i) * D + j);
        }
        __syncthreads();
        const bool active = tid < 2 * D;
        const int j = tid % D;
        const int h = tid / D;            // 0 or 1 for active threads
        float amax = 0.0f;
        if (active) {
            for (int i = h * 32; i < min(nv, h * 32 + 32); ++i) amax = fmaxf(amax, fabsf(tile[i][j]));
            half_max[h][j] = amax;
        }
        __syncthreads();
        if (active) {
            const float a = fmaxf(half_max[0][j], half_max[1][j]);
            __half ah = (a >= 65504.0f) ? __ushort_as_half((unsigned short)0x7bff) : __float2half_rn(a);
            const float a16 = __half2float(ah);
            uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
            for (int i = h * 32; i < min(nv, h * 32 + 32); ++i) {
                const uint32_t c = (uint32_t)code_of(tile[i][j], a16);
                const int b = i - h * 32;
                w0 |= ((c >> 3) & 1u) << b;
                w1 |= ((c >> 2) & 1u) << b;
                w2 |= ((c >> 1) & 1u) << b;
                w3 |= (c & 1u) << b;
            }
            words[j][0][bl][h] = w0;
            words[j][1][bl][h] = w1;
            words[j][2][bl][h] = w2;
            words[j][3][bl][h] = w3;
            if (h == 0) sc[j][bl] = __half_as_ushort(ah);
        }
    }
    __syncthreads();
    // plane words: planes[u][j][p][beta0 + bl]
    uint64_t *P = planes + (size_t)u * D * FATHOM_PLANES * cb;
    for (int e = tid; e < D * FATHOM_PLANES * nbl; e += kQThreads) {
        const int bl = e % nbl;
        const int jp = e / nbl;
        const int j = jp / FATHOM_PLANES, p = jp % FATHOM_PLANES;
        const uint64_t w = (uint64_t)words[j][p][bl][0] | ((uint64_t)words[j][p][bl][1] << 32);
        P[(size_t)jp * cb + beta0 + bl] = w;
    }
    uint16_t *S = scales + (size_t)u * D * cb;
    for (int e = tid; e < D * nbl; e += kQThreads) {
        const int bl = e % nbl, j = e / nbl;
        S[(size_t)j * cb + beta0 + bl] = sc[j][bl];
    }
}

static int launch_blocks(const fathom_shape &s, int n, int block0, int block1, const void *keys, int dtype,
                         uint64_t *planes, uint16_t *scales, cudaStream_t st, const char *what) {
    dim3 grid((block1 - block0 + kQBlocks - 1) / kQBlocks, s.units);
    if (grid.y > 65535) { set_error("%s: too many units for one launch", what); return FATHOM_EINVAL; }
    const size_t smem = sizeof(QSmem);
    const int ctok = cap_tokens(s), cb = cap_blocks(s);
    if (dtype == FATHOM_F32) {
        ensure_smem(quantize_kernel<float>, smem);
        quantize_kernel<float><<<grid, kQThreads, smem, st>>>(n, s.D, ctok, cb, block0, block1,
                                                              (const float *)keys, planes, scales);
    } else {
        ensure_smem(quantize_kernel<uint16_t>, smem);
        quantize_kernel<uint16_t><<<grid, kQThreads, smem, st>>>(n, s.D, ctok, cb, block0, block1,
                                                                 (const uint16_t *)keys, planes, scales);
    }
    return launch_status("quantize_kernel");
}

int launch_quantize(const fathom_shape &s, const void *keys, int dtype, uint64_t *planes,
                    uint16_t *scales, cudaStream_t st) {
    return launch_blocks(s, s.n, 0, num_blocks(s.n), keys, dtype, planes, scales, st, "quantize");
}

int launch_append(const fathom_shape &s, const void *keys, int dtype, int block, int count, uint64_t *planes,
                  uint16_t *scales, cudaStream_t st) {
    return launch_blocks(s, 64 * block + count, block, block + 1, keys, dtype, planes, scales, st, "append_block");
}

}  // namespace fathom

// scan_topk.cu -- variable-depth bit-plane scan and top-k selection
// (Fathom §3.2 prefix dequantisation, §3.3 active channels and a plan shared
// by the G query heads, §2 forced sink/recent tokens, §7 one multiply-add per
// active channel, token and head).
//
// Grid: (chunks, units).  A CTA streams its chunk of 64-token blocks in
// sub-chunks of 32 blocks (2048 tokens).  For each sub-chunk the planned
// plane words of the active channels (grouped so that at most 64 planes are
// staged at a time) and per-block weights are staged in shared memory, then
// each thread scores 8 tokens of one block for all G heads:
//
//   thread (block b, r in 0..7) takes tokens r, r+8, r+16, r+24 from the low
//   and the high 32-bit half of every plane word.  (w >> r) & 0x01010101
//   puts those four tokens' bits in four byte lanes; t shift-and-add steps
//   over a channel's t planes build the t-bit code prefixes c_t byte-wise,
//   one more step makes every byte 2 c_t + 1 (at most 31, so no carries);
//   a byte permute drops one byte under the exponent of 2^23 and one fp32
//   subtraction of 2^23 + 2^t gives exactly 2 (c_t + 0.5 - 2^(t-1)).  With
//   the block weight w_hj = q_hj * a_j * 2^-t, one fma per head adds
//   q_hj * (c_t + 0.5 - 2^(t-1)) * a_j / 2^(t-1), i.e. q_hj times the t-bit
//   mid-rise value, with no rounding before the multiply.
//
// Selection never materialises all scores.  Each CTA keeps, per head, a
// candidate list of 64-bit keys (score, ~index) in the workspace and a
// threshold key tau: a token is appended only if its key >= tau.  When a
// list could overflow, an in-CTA radix select finds a key T such that at
// least k' (and at most k' + slack) keys are >= T, keeps those and sets
// tau = T.  Any token of the CTA's top-k' is always kept, so the union of the
// CTAs' lists contains the unit's top-k'.  A second kernel, one CTA per
// (unit, head), selects the exact top-k' from that union, adds the forced
// tokens and writes the kept set in ascending index order.
#include "fathom_internal.cuh"

namespace fathom {

constexpr int kPG = 64;                 // plane words staged per group
constexpr int kPWStride = kPG + 2;      // padded row (uint2 units) -> distinct banks per block
constexpr int NT = kScanThreads;

template <int G>
struct ScanCfg {
    static constexpr int CHG = (G <= 4) ? 64 : 32;     // channels per staged group
    static constexpr int WStride = CHG * G + 4;        // padded weight row (floats)
};

struct GroupDesc {
    int a0, p0, n4, n3, n2, n1;   // first active channel, first plane slot, channels per depth
};

template <int G>
struct ScanSmem {
    uint2 pw[kSubBlocks][kPWStride];
    float w[kSubBlocks][ScanCfg<G>::WStride];
    uint64_t plane_src[FATHOM_PLANES * FATHOM_MAX_D];   // word offset of (active channel, plane)
    uint64_t ch_scale[FATHOM_MAX_D];                   // scale offset of active channel
    float qs[FATHOM_MAX_D][G];                          // q_hj * 2^-t_j, active channels
    int ch_t[FATHOM_MAX_D];                             // depth of active channel (sorted)
    int raw_t[FATHOM_MAX_D];
    GroupDesc grp[FATHOM_MAX_D];
    int n_groups, n_active;
    int cnt[G];
    int cur[G];
    uint64_t tau[G];
    float tau_s[G];
    // radix select scratch
    unsigned hist[256];
    unsigned lane_sum[32];
    int sel_digit, sel_above, sel_bucket;
    int new_cnt;
};

// ---------------------------------------------------------------------------
// Inner loop: channels [a_lo, a_hi) of depth T of the current group.
template <int G, int T>
__device__ __forceinline__ void accum_depth(const uint2 *__restrict__ pwrow,
                                            const float *__restrict__ wrow, int a_lo, int a_hi,
                                            int slot, uint32_t r, float (&acc)[8][G]) {
    constexpr float K = 8388608.0f + (float)(1 << T);
#pragma unroll 2
    for (int a = a_lo; a < a_hi; ++a, slot += T) {
        uint32_t ylo = 0, yhi = 0;
#pragma unroll
        for (int p = 0; p < T; ++p) {
            const uint2 w = pwrow[slot + p];
            ylo = (ylo << 1) + ((w.x >> r) & 0x01010101u);
            yhi = (yhi << 1) + ((w.y >> r) & 0x01010101u);
        }
        ylo = (ylo << 1) + 0x01010101u;
        yhi = (yhi << 1) + 0x01010101u;
        float f[8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            f[b] = __uint_as_float(__byte_perm(ylo, 0x4B000000u, 0x7650u | b)) - K;
            f[4 + b] = __uint_as_float(__byte_perm(yhi, 0x4B000000u, 0x7650u | b)) - K;
        }
        float wv[G];
        if constexpr (G == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(wrow + a * G);
            wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
        } else if constexpr (G == 8) {
            const float4 v0 = *reinterpret_cast<const float4 *>(wrow + a * G);
            const float4 v1 = *reinterpret_cast<const float4 *>(wrow + a * G + 4);
            wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
            wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
        } else if constexpr (G == 2) {
            const float2 v = *reinterpret_cast<const float2 *>(wrow + a * G);
            wv[0] = v.x; wv[1] = v.y;
        } else {
            wv[0] = wrow[a];
        }
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int h = 0; h < G; ++h) acc[m][h] = fmaf(wv[h], f[m], acc[m][h]);
    }
}

// ---------------------------------------------------------------------------
// CTA-wide radix select over `count` keys at `src`.  Finds T with
// #{keys >= T} in [target, target + slack] (slack = 0: exactly target) and
// returns #{keys >= T}.  target >= 1 and count >= target.
template <typename Sm>
__device__ uint64_t radix_threshold(Sm &sm, const uint64_t *src, int count, int target, int slack,
                                    int *kept) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    uint64_t prefix = 0, pmask = 0;
    int above = 0;   // keys strictly above the current bucket
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) sm.hist[i] = 0;
        __syncthreads();
        for (int e = tid; e < count; e += blockDim.x) {
            const uint64_t key = src[e];
            if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l (descending)
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
            const unsigned need = (unsigned)(target - above);
            if (excl < need && need <= incl) {
                unsigned c = excl;
                for (int i = 0; i < 8; ++i) {
                    const int bin = 255 - 8 * lane - i;
                    const unsigned hb = sm.hist[bin];
                    if (c + hb >= need) {
                        sm.sel_digit = bin;
                        sm.sel_above = (int)c;
                        sm.sel_bucket = (int)hb;
                        break;
                    }
                    c += hb;
                }
            }
        }
        __syncthreads();
        const int d = sm.sel_digit;
        above += sm.sel_above;
        const int hb = sm.sel_bucket;
        prefix |= (uint64_t)d << shift;
        pmask |= (uint64_t)255 << shift;
        __syncthreads();   // everyone has read sel_* before the next pass rewrites them
        if (above + hb == target || above + hb <= target + slack || shift == 0) {
            *kept = above + hb;
            return prefix;
        }
    }
    *kept = target;
    return prefix;
}

// Keep the keys >= T of list (count) by copying them to dst; returns new count.
template <typename Sm>
__device__ int compact_keys(Sm &sm, const uint64_t *src, int count, uint64_t T, uint64_t *dst,
                            int dst_cap) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) sm.new_cnt = 0;
    __syncthreads();
    for (int e0 = 0; e0 < count; e0 += blockDim.x) {
        const int e = e0 + tid;
        uint64_t key = 0;
        bool keep = false;
        if (e < count) { key = src[e]; keep = key >= T; }
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&sm.new_cnt, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (keep && pos < dst_cap) dst[pos] = key;
    }
    __syncthreads();
    return min(sm.new_cnt, dst_cap);
}

// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(NT)
scan_kernel(int n, int D, int chunk_blocks, int source, size_t stage_words, size_t stage_scales,
            const uint64_t *__restrict__ planes, const uint16_t *__restrict__ scales,
            const fathom_run *__restrict__ runs, const float *__restrict__ q, int k_sel, int ns,
            int r0, int nf, int cap, float *__restrict__ scores_opt, uint64_t *__restrict__ cand,
            int *__restrict__ cand_cnt, float *__restrict__ forced_scores) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem<G> &sm = *reinterpret_cast<ScanSmem<G> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31;
    const int u = blockIdx.y;
    const int chunk = blockIdx.x;
    const int nb = num_blocks(n);
    const int b_begin = chunk * chunk_blocks;
    const int b_end = min(nb, b_begin + chunk_blocks);
    const size_t cta = (size_t)u * gridDim.x + chunk;

    // ---- prologue: active channels sorted by depth (desc), ties by channel
    if (tid < D) {
        const fathom_run rr = runs[(size_t)u * D + tid];
        int t = (int)(rr.n_words / (uint32_t)nb);
        t = t > FATHOM_PLANES ? FATHOM_PLANES : t;
        // a channel whose staged run or scales would pass the unit's staging
        // stride (a plan larger than the staging area) is not read at all
        if (source == FATHOM_SRC_STAGING &&
            ((uint64_t)rr.dst_word + (uint64_t)t * nb > stage_words ||
             (uint64_t)rr.dst_scale + (t > 0 ? (uint64_t)nb : 0) > stage_scales))
            t = 0;
        if (source == FATHOM_SRC_STORE && rr.src_word != (uint32_t)tid * FATHOM_PLANES * nb) t = 0;
        sm.raw_t[tid] = t;
    }
    if (tid == 0) { sm.sel_digit = 0; sm.sel_above = 0; sm.sel_bucket = 0; }
    if (tid < G) {
        sm.cnt[tid] = 0;
        sm.cur[tid] = 0;
        sm.tau[tid] = 0;
        sm.tau_s[tid] = -CUDART_INF_F;
    }
    __syncthreads();
    if (tid < D) {
        const int t = sm.raw_t[tid];
        if (t > 0) {
            int pos = 0;
            for (int i = 0; i < D; ++i) {
                const int ti = sm.raw_t[i];
                pos += (ti > t || (ti == t && i < tid)) ? 1 : 0;
            }
            const fathom_run rr = runs[(size_t)u * D + tid];
            const uint64_t wbase = (source == FATHOM_SRC_STORE)
                                       ? ((uint64_t)u * D + tid) * FATHOM_PLANES * nb
                                       : (uint64_t)u * stage_words + rr.dst_word;
            const uint64_t sbase = (source == FATHOM_SRC_STORE)
                                       ? ((uint64_t)u * D + tid) * nb
                                       : (uint64_t)u * stage_scales + rr.dst_scale;
            sm.ch_t[pos] = t;
            sm.ch_scale[pos] = sbase;
            const float sc = ldexpf(1.0f, -t);
            for (int h = 0; h < G; ++h) sm.qs[pos][h] = q[((size_t)u * G + h) * D + tid] * sc;
            // plane slots are assigned after the sort; stash the base for now
            sm.plane_src[pos] = wbase;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int A = 0;
        for (int i = 0; i < D; ++i) A += sm.raw_t[i] > 0 ? 1 : 0;
        sm.n_active = A;
        // expand plane slots (in place from the back: slot index >= channel index)
        int P = 0;
        for (int a = 0; a < A; ++a) P += sm.ch_t[a];
        int slot = P;
        for (int a = A - 1; a >= 0; --a) {
            const int t = sm.ch_t[a];
            const uint64_t base = sm.plane_src[a];
            slot -= t;
            for (int p = t - 1; p >= 0; --p) sm.plane_src[slot + p] = base + (uint64_t)p * nb;
        }
        // groups of consecutive channels: <= kPG planes and <= CHG channels
        int ng = 0, a = 0, p0 = 0;
        while (a < A) {
            GroupDesc g;
            g.a0 = a;
            g.p0 = p0;
            g.n4 = g.n3 = g.n2 = g.n1 = 0;
            int planes_in = 0, chans = 0;
            while (a < A && planes_in + sm.ch_t[a] <= kPG && chans < ScanCfg<G>::CHG) {
                const int t = sm.ch_t[a];
                if (t == 4) ++g.n4; else if (t == 3) ++g.n3; else if (t == 2) ++g.n2; else ++g.n1;
                planes_in += t;
                ++chans;
                ++a;
            }
            p0 += planes_in;
            sm.grp[ng++] = g;
        }
        sm.n_groups = ng;
    }
    __syncthreads();

    const int ng = sm.n_groups;
    const int bl = tid >> 3;                 // block within the sub-chunk
    const uint32_t r = (uint32_t)(tid & 7);  // token offset within a byte lane

    for (int sb = b_begin; sb < b_end; sb += kSubBlocks) {
        const int nblk = min(kSubBlocks, b_end - sb);
        // make room in every head's candidate list before this sub-chunk
        if (k_sel > 0) {
            for (int h = 0; h < G; ++h) {
                if (sm.cnt[h] + kSubTokens > cap) {
                    uint64_t *base = cand + (cta * G + h) * 2 * (size_t)cap;
                    const uint64_t *srcl = base + (size_t)sm.cur[h] * cap;
                    uint64_t *dstl = base + (size_t)(1 - sm.cur[h]) * cap;
                    int kept;
                    const int cnt_h = min(sm.cnt[h], cap);
                    const uint64_t T = radix_threshold(sm, srcl, cnt_h, k_sel, kPruneSlack, &kept);
                    const int c = compact_keys(sm, srcl, cnt_h, T, dstl, cap);
                    if (tid == 0) {
                        sm.cnt[h] = c;
                        sm.cur[h] = 1 - sm.cur[h];
                        sm.tau[h] = T;
                        const uint32_t hi = (uint32_t)(T >> 32);
                        sm.tau_s[h] = (hi <= 0x00800000u) ? -CUDART_INF_F : unorder_f32(hi);
                    }
                    __syncthreads();
                }
            }
        }

        float acc[8][G];
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int h = 0; h < G; ++h) acc[m][h] = 0.0f;

        for (int gi = 0; gi < ng; ++gi) {
            const GroupDesc g = sm.grp[gi];
            const int nch = g.n4 + g.n3 + g.n2 + g.n1;
            const int npl = 4 * g.n4 + 3 * g.n3 + 2 * g.n2 + g.n1;
            __syncthreads();
            // stage plane words: slot-major, 32 consecutive blocks per slot
            for (int e = tid; e < npl * kSubBlocks; e += NT) {
                const int s = e / kSubBlocks, b = e % kSubBlocks;
                uint2 v = make_uint2(0u, 0u);
                if (b < nblk) {
                    const uint64_t wd = __ldg(planes + sm.plane_src[g.p0 + s] + sb + b);
                    v = make_uint2((uint32_t)wd, (uint32_t)(wd >> 32));
                }
                sm.pw[b][s] = v;
            }
            // stage block weights w_hj = q_hj * 2^-t_j * a_{beta,j}
            for (int e = tid; e < nch * kSubBlocks; e += NT) {
                const int al = e / kSubBlocks, b = e % kSubBlocks;
                const int a = g.a0 + al;
                float a16 = 0.0f;
                if (b < nblk) a16 = __half2float(__ushort_as_half(__ldg(scales + sm.ch_scale[a] + sb + b)));
#pragma unroll
                for (int h = 0; h < G; ++h) sm.w[b][al * G + h] = sm.qs[a][h] * a16;
            }
            __syncthreads();
            if (bl < nblk) {
                const uint2 *pwrow = sm.pw[bl];
                const float *wrow = sm.w[bl];
                int a = 0, slot = 0;
                accum_depth<G, 4>(pwrow, wrow, a, a + g.n4, slot, r, acc);
                a += g.n4; slot += 4 * g.n4;
                accum_depth<G, 3>(pwrow, wrow, a, a + g.n3, slot, r, acc);
                a += g.n3; slot += 3 * g.n3;
                accum_depth<G, 2>(pwrow, wrow, a, a + g.n2, slot, r, acc);
                a += g.n2; slot += 2 * g.n2;
                accum_depth<G, 1>(pwrow, wrow, a, a + g.n1, slot, r, acc);
            }
        }

        // ---- epilogue: debug scores, forced tokens, candidates
        const int beta = sb + bl;
        uint64_t pass = 0;   // bit m * G + h
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = beta * 64 + (int)r + 8 * (m & 3) + 32 * (m >> 2);
            const bool valid = (bl < nblk) && (i < n);
            if (!valid) continue;
            if (scores_opt) {
#pragma unroll
                for (int h = 0; h < G; ++h) scores_opt[((size_t)u * G + h) * n + i] = acc[m][h];
            }
            if (i < ns || i >= r0) {
                const int slot = (i < ns) ? i : ns + (i - r0);
#pragma unroll
                for (int h = 0; h < G; ++h) forced_scores[((size_t)u * G + h) * nf + slot] = acc[m][h];
            } else if (k_sel > 0) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    if (acc[m][h] >= sm.tau_s[h]) pass |= 1ull << (m * G + h);
            }
        }
        if (__any_sync(0xffffffffu, pass != 0)) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                uint64_t *lst = cand + (cta * G + h) * 2 * (size_t)cap + (size_t)sm.cur[h] * cap;
                const uint64_t tau = sm.tau[h];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int i = beta * 64 + (int)r + 8 * (m & 3) + 32 * (m >> 2);
                    uint64_t key = 0;
                    bool p = (pass >> (m * G + h)) & 1ull;
                    if (p) {
                        key = make_key(acc[m][h], (uint32_t)i);
                        p = key >= tau;
                    }
                    const unsigned bal = __ballot_sync(0xffffffffu, p);
                    if (bal) {
                        int base = 0;
                        const int leader = __ffs(bal) - 1;
                        if (lane == leader) base = atomicAdd(&sm.cnt[h], __popc(bal));
                        base = __shfl_sync(0xffffffffu, base, leader);
                        const int pos = base + __popc(bal & ((1u << lane) - 1u));
                        if (p && pos < cap) lst[pos] = key;
                    }
                }
            }
        }
        __syncthreads();
    }

    // ---- final prune to at most k' + slack keys per head, then publish
    if (k_sel > 0) {
        for (int h = 0; h < G; ++h) {
            if (sm.cnt[h] > k_sel + kPruneSlack) {
                uint64_t *base = cand + (cta * G + h) * 2 * (size_t)cap;
                const uint64_t *srcl = base + (size_t)sm.cur[h] * cap;
                uint64_t *dstl = base + (size_t)(1 - sm.cur[h]) * cap;
                int kept;
                const int cnt_h = min(sm.cnt[h], cap);
                const uint64_t T = radix_threshold(sm, srcl, cnt_h, k_sel, kPruneSlack, &kept);
                const int c = compact_keys(sm, srcl, cnt_h, T, dstl, cap);
                if (tid == 0) {
                    sm.cnt[h] = c;
                    sm.cur[h] = 1 - sm.cur[h];
                }
                __syncthreads();
            }
        }
    }
    if (tid < G) cand_cnt[cta * G + tid] = min(sm.cnt[tid], cap) | (sm.cur[tid] << 30);
}

// ---------------------------------------------------------------------------
// Merge: one CTA per (head, unit).  Exact top-k' of the chunks' candidate
// lists, plus the forced tokens, ascending by index.
constexpr int kMThreads = 512;

struct MergeSmem {
    unsigned hist[256];
    unsigned lane_sum[32];
    int sel_digit, sel_above, sel_bucket;
    int new_cnt;
    int total;
    uint64_t sel[FATHOM_MAX_K];
};

// radix select over the union of `chunks` lists (exact).
__device__ uint64_t merge_threshold(MergeSmem &sm, const uint64_t *cand, const int *cnts, int chunks,
                                    size_t list_stride, size_t cap, int target) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    uint64_t prefix = 0, pmask = 0;
    int above = 0;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) sm.hist[i] = 0;
        __syncthreads();
        for (int c = 0; c < chunks; ++c) {
            const int cc = cnts[(size_t)c * list_stride];
            const int cnt = min(cc & 0x3fffffff, (int)cap), half = (cc >> 30) & 1;
            const uint64_t *lst = cand + (size_t)c * list_stride * 2 * cap + (size_t)half * cap;
            for (int e = tid; e < cnt; e += blockDim.x) {
                const uint64_t key = lst[e];
                if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255], 1u);
            }
        }
        __syncthreads();
        if (warp == 0) {
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
            const unsigned need = (unsigned)(target - above);
            if (excl < need && need <= incl) {
                unsigned c = excl;
                for (int i = 0; i < 8; ++i) {
                    const int bin = 255 - 8 * lane - i;
                    const unsigned hb = sm.hist[bin];
                    if (c + hb >= need) {
                        sm.sel_digit = bin;
                        sm.sel_above = (int)c;
                        sm.sel_bucket = (int)hb;
                        break;
                    }
                    c += hb;
                }
            }
        }
        __syncthreads();
        const int d = sm.sel_digit;
        above += sm.sel_above;
        const int hb = sm.sel_bucket;
        prefix |= (uint64_t)d << shift;
        pmask |= (uint64_t)255 << shift;
        __syncthreads();
        if (above + hb == target || shift == 0) return prefix;
    }
    return prefix;
}

__global__ void __launch_bounds__(kMThreads)
merge_kernel(int n, int G, int k, int k_sel, int ns, int r0, int nf, int chunks, int cap,
             const uint64_t *__restrict__ cand, const int *__restrict__ cand_cnt,
             const float *__restrict__ forced_scores, int32_t *__restrict__ out_idx,
             float *__restrict__ out_score) {
    extern __shared__ __align__(16) unsigned char msmem_raw[];
    MergeSmem &sm = *reinterpret_cast<MergeSmem *>(msmem_raw);
    const int h = blockIdx.x, u = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31;
    int32_t *oi = out_idx + ((size_t)u * G + h) * k;
    float *os = out_score + ((size_t)u * G + h) * k;
    const float *fs = forced_scores + ((size_t)u * G + h) * nf;
    // forced tokens: sinks first, recent last
    for (int e = tid; e < ns; e += blockDim.x) { oi[e] = e; os[e] = fs[e]; }
    for (int e = tid; e < n - r0; e += blockDim.x) {
        oi[ns + k_sel + e] = r0 + e;
        os[ns + k_sel + e] = fs[ns + e];
    }
    if (k_sel == 0) return;

    if (tid == 0) { sm.sel_digit = 0; sm.sel_above = 0; sm.sel_bucket = 0; }
    for (int e = tid; e < FATHOM_MAX_K; e += blockDim.x) sm.sel[e] = 0;
    __syncthreads();
    const uint64_t *c0 = cand + ((size_t)u * chunks * G + h) * 2 * (size_t)cap;
    const int *n0 = cand_cnt + (size_t)u * chunks * G + h;
    const uint64_t T = merge_threshold(sm, c0, n0, chunks, (size_t)G, (size_t)cap, k_sel);

    // gather the k' keys >= T
    if (tid == 0) sm.new_cnt = 0;
    __syncthreads();
    for (int c = 0; c < chunks; ++c) {
        const int cc = n0[(size_t)c * G];
        const int cnt = min(cc & 0x3fffffff, cap), half = (cc >> 30) & 1;
        const uint64_t *lst = c0 + (size_t)c * G * 2 * cap + (size_t)half * cap;
        for (int e0 = 0; e0 < cnt; e0 += blockDim.x) {
            const int e = e0 + tid;
            uint64_t key = 0;
            bool keep = false;
            if (e < cnt) { key = lst[e]; keep = key >= T; }
            const unsigned bal = __ballot_sync(0xffffffffu, keep);
            int base = 0;
            if (lane == 0 && bal) base = atomicAdd(&sm.new_cnt, __popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            const int pos = base + __popc(bal & ((1u << lane) - 1u));
            if (keep && pos < k_sel) sm.sel[pos] = key;
        }
    }
    __syncthreads();
    // bitonic sort by token index ascending (key_index); pad with index 0xffffffff
    int P = 1;
    while (P < k_sel) P <<= 1;
    for (int e = k_sel + tid; e < P; e += blockDim.x) sm.sel[e] = 0;   // key 0 -> index 0xffffffff
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int e = tid; e < P / 2; e += blockDim.x) {
                const int lo = 2 * stride * (e / stride) + (e % stride);
                const int hi = lo + stride;
                const bool up = ((lo & size) == 0);
                const uint64_t a = sm.sel[lo], b = sm.sel[hi];
                const bool swap = up ? (key_index(a) > key_index(b)) : (key_index(a) < key_index(b));
                if (swap) { sm.sel[lo] = b; sm.sel[hi] = a; }
            }
            __syncthreads();
        }
    }
    for (int e = tid; e < k_sel; e += blockDim.x) {
        const uint64_t key = sm.sel[e];
        oi[ns + e] = (int32_t)key_index(key);
        os[ns + e] = key_score(key);
    }
}

// ---------------------------------------------------------------------------
template <int G>
static int launch_g(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                    int source, size_t stage_words, size_t stage_scales, const fathom_run *runs,
                    const float *q, int32_t *idx, float *score, float *scores_opt, void *ws,
                    cudaStream_t st) {
    const ScanGrid sg = scan_grid(s.units, s.n);
    const Forced f = forced_range(s.n, s.n_sink, s.n_recent);
    const ScanWorkspace wl = scan_workspace_layout(s);
    const int k_sel = s.k - f.nf;
    const int cap = scan_cand_cap(s);
    char *w = (char *)ws;
    uint64_t *cand = (uint64_t *)(w + wl.cand_off);
    int *cnt = (int *)(w + wl.cnt_off);
    float *forced = (float *)(w + wl.forced_off);
    const size_t smem = sizeof(ScanSmem<G>);
    if (s.units > 65535) { set_error("scan: too many units for one launch"); return FATHOM_EINVAL; }
    ensure_smem(scan_kernel<G>, smem);
    dim3 grid(sg.chunks, s.units);
    scan_kernel<G><<<grid, NT, smem, st>>>(s.n, s.D, sg.chunk_blocks, source, stage_words,
                                           stage_scales, planes, scales, runs, q, k_sel, f.ns, f.r0,
                                           f.nf > 0 ? f.nf : 1, cap, scores_opt, cand, cnt, forced);
    int rc = launch_status("scan_kernel");
    if (rc) return rc;
    const size_t msmem = sizeof(MergeSmem);
    ensure_smem(merge_kernel, msmem);
    merge_kernel<<<dim3(s.G, s.units), kMThreads, msmem, st>>>(s.n, s.G, s.k, k_sel, f.ns, f.r0,
                                                               f.nf > 0 ? f.nf : 1, sg.chunks, cap,
                                                               cand, cnt, forced, idx, score);
    return launch_status("merge_kernel");
}

int launch_scan_topk(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                     int source, size_t stage_words, size_t stage_scales, const fathom_run *runs,
                     const float *q, int32_t *idx, float *score, float *scores_opt, void *ws,
                     cudaStream_t st) {
    switch (s.G) {
        case 1: return launch_g<1>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st);
        case 2: return launch_g<2>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st);
        case 4: return launch_g<4>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st);
        case 8: return launch_g<8>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st);
        default: set_error("unsupported G=%d", s.G); return FATHOM_EINVAL;
    }
}

}  // namespace fathom

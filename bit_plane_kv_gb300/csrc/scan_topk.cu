// scan_topk.cu -- variable-depth bit-plane scan and top-k selection
// (Fathom §3.2 prefix dequantisation, §3.3 active channels and a plan shared
// by the G query heads, §2 forced sink/recent tokens, §7 one multiply-add per
// active channel, token and head).
//
// Grid: units x chunks CTAs, one-dimensional (chunk-fastest, or unit-fastest
// when the units do not fill the resident slots evenly; see scan_grid).  A CTA
// streams sub-chunks of 32 blocks (2048 tokens)
// of its unit, taking the next one from a per-unit counter as it goes (so a
// CTA that runs faster scores more of them).  For each sub-chunk the planned
// plane words of the active channels (grouped so that at most 64 planes are
// staged at a time) and per-block weights are staged in shared memory, then
// each thread scores 8 tokens of one block for all G heads:
//
//   thread (block b, r in 0..7) takes tokens r, r+8, r+16, r+24 from the low
//   and the high 32-bit half of every plane word.  Rotating plane p's half
//   word right by (r - (t - p)) mod 32 puts those four tokens' bits on bit
//   t - p of four byte lanes; merged under a mask into 0x01010101, the t planes
//   make every byte 2 c_t + 1 (c_t the t-bit code prefix; at most 31, so no
//   carries);
//   a byte permute drops one byte under the exponent of 2^23 and one fp32
//   subtraction of 2^23 + 2^t gives exactly 2 (c_t + 0.5 - 2^(t-1)).  With
//   the block weight w_hj = q_hj * a_j * 2^-t, one fma per head adds
//   q_hj * (c_t + 0.5 - 2^(t-1)) * a_j / 2^(t-1), i.e. q_hj times the t-bit
//   mid-rise value, with no rounding before the multiply.  Tokens m and m + 4
//   of a thread share byte lanes, so the subtraction and the fmas run as
//   packed f32x2 operations (each half an ordinary round-to-nearest fp32 op).
//
// Selection never materialises all scores.  Tokens are ordered by a 64-bit
// key (score, ~index).  Each CTA keeps, per head, a candidate list of keys in
// the workspace and a threshold key tau; a token is appended only if its key
// >= tau.  tau starts as a key of the CTA's first sub-chunk (selected straight
// from registers for all heads at once: m1 of the threads' best keys, and so
// at least m1 of the sub-chunk's keys, lie at or above it), m1 being a tail
// bound of the winners a sub-chunk holds (P <= 1e-6 that it holds more, for
// winners spread over the sequence; at least 8); at the end a list
// longer than 8m is cut back to m .. 2m keys, m being four times the CTA's
// expected share of the k' winners for the sub-chunks it scored.  The merge kernel streams
// the lists through shared memory (P CTAs per (unit, head), the last of
// which, by an atomic ticket, merges the P partial results), selects the
// exact top-k', adds the forced tokens and writes the kept set in ascending
// index order.  Any CTA whose tau lies above the k'-th key may have dropped
// a winner: the merge flags it, and a second pass rescans exactly the
// sub-chunks that CTA scored (keeping their exact top-k') before a second
// merge.
#include <cstddef>
#include <mutex>
#include <type_traits>

#include "fathom_internal.cuh"

namespace fathom {

constexpr int kCHG = 32;                // channels per staged group (fixed runs of the sorted order)
constexpr int kPG = kCHG * FATHOM_PLANES;   // plane words staged per group, at most
constexpr int NT = kScanThreads;

template <int G>
struct ScanCfg {
    static constexpr int WStride = kCHG * G + 4;       // padded weight row (floats)
};

struct GroupDesc {
    int a0, p0, n4, n3, n2, n1;   // first active channel, first plane slot, channels per depth
};

// Scratch of up to S simultaneous CTA-wide threshold selections.
constexpr int kMaxWarps = 16;
template <int S>
struct SelScratch {
    unsigned hist[S][256];
    unsigned long long red[2][S][kMaxWarps];
    int red_n[S][kMaxWarps];
    int digit[S], above[S], bucket[S];
    int new_cnt;
};

template <int G>
struct ScanSmem {
    // plane words, slot-major: pw[slot][block].  The synchronous path stages up
    // to kPG slots of one group; the pipelined path ping-pongs between the two
    // halves [0, kPG/2) and [kPG/2, kPG).
    uint2 pw[kPG][kSubBlocks];
    uint16_t scb[2][kCHG][kSubBlocks];                  // prefetched fp16 scales (pipelined path)
    float w[kSubBlocks][ScanCfg<G>::WStride];
    uint64_t plane_src[FATHOM_PLANES * FATHOM_MAX_D];   // word offset of (active channel, plane)
    uint64_t ch_scale[FATHOM_MAX_D];                   // scale offset of active channel
    float qs[FATHOM_MAX_D][G];                          // q_hj * 2^-t_j, active channels
    int ch_t[FATHOM_MAX_D];                             // depth of active channel (sorted)
    int raw_t[FATHOM_MAX_D];
    GroupDesc grp[FATHOM_MAX_D / kCHG];
    int wcnt[FATHOM_PLANES + 1][FATHOM_MAX_D / 32];   // channels of each depth per warp
    int n_groups;
    int sq0[2];                                         // first two sub-chunks of this CTA
    int sq[2];                                          // next sub-chunk of this CTA (double-buffered)
    int fix_pos;                                        // second pass: where the owner search resumes
    int cnt[G];
    uint64_t tau[G];
    SelScratch<G> selg;   // first-sub-chunk selection, all heads at once
    SelScratch<1> sel1;   // list prunes
};


// ---------------------------------------------------------------------------
// Per-thread scores of 8 tokens x G heads.  Token m (m = 0..7, token r + 8 m of
// the block) lives in v[m & 3][h].x for m < 4 and .y for m >= 4: tokens m and
// m + 4 come from the same byte lane of the low and the high half of a plane
// word, so one packed (f32x2) instruction updates both.  Each half of a packed
// operation is an ordinary IEEE single-precision operation (round to nearest),
// so the scores are the same as with scalar fmaf.
template <int G>
struct Acc8 {
    float2 v[4][G];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int h = 0; h < G; ++h) v[b][h] = make_float2(0.0f, 0.0f);
    }
    __device__ __forceinline__ float &operator()(int m, int h) { return m < 4 ? v[m][h].x : v[m - 4][h].y; }
    __device__ __forceinline__ float operator()(int m, int h) const { return m < 4 ? v[m][h].x : v[m - 4][h].y; }
};

// Rotation amounts of thread r: rot[k] = (r - k) mod 32, so that rotating a
// plane half-word right by rot[k] moves token r + 8m (bit r + 8m) to bit
// 8m + k, for the four tokens m = 0..3 at once.
struct DecodeRot {
    uint32_t rot[FATHOM_PLANES + 1];
};

// ---------------------------------------------------------------------------
// Inner loop: channels [a_lo, a_hi) of depth T of the current group.
// pwcol points at this thread's block in slot 0 of the staged group: slot s of
// the block is pwcol[s * kSubBlocks] (the lanes of a warp read 4 adjacent words).
// Byte m of y is built as 1 + sum_p b_p 2^(T - p): plane p's bit of token
// r + 8m is rotated to bit T - p of byte m and merged in (one funnel shift and
// one three-input logic op per plane and half word), so y's bytes are
// 2 c_T + 1 with c_T the T-bit code prefix (at most 31: no carries).
template <int G, int T>
__device__ __forceinline__ void accum_depth(const uint2 *__restrict__ pwcol,
                                            const float *__restrict__ wrow, int a_lo, int a_hi,
                                            int slot, const DecodeRot &dr, Acc8<G> &acc) {
    constexpr float K = 8388608.0f + (float)(1 << T);
    const float2 negK = make_float2(-K, -K);
#pragma unroll 1
    for (int a = a_lo; a < a_hi; ++a, slot += T) {
        uint32_t ylo = 0x01010101u, yhi = 0x01010101u;
#pragma unroll
        for (int p = 0; p < T; ++p) {
            const uint2 w = pwcol[(slot + p) * kSubBlocks];
            const uint32_t m = 0x01010101u << (T - p);
            ylo |= __funnelshift_r(w.x, w.x, dr.rot[T - p]) & m;
            yhi |= __funnelshift_r(w.y, w.y, dr.rot[T - p]) & m;
        }
        // byte b of each half under the exponent of 2^23, minus 2^23 + 2^T (exact)
        float2 f[4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
            f[b] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(ylo, 0x4B000000u, 0x7650u | b)),
                                          __uint_as_float(__byte_perm(yhi, 0x4B000000u, 0x7650u | b))),
                              negK);
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
        for (int h = 0; h < G; ++h) {
            const float2 w2 = make_float2(wv[h], wv[h]);
#pragma unroll
            for (int b = 0; b < 4; ++b) acc.v[b][h] = __ffma2_rn(w2, f[b], acc.v[b][h]);
        }
    }
}


// ---------------------------------------------------------------------------
// CTA-wide threshold selection, S selections at once.
//
// For every selection s, finds T[s] such that #{keys of s >= T[s]} lies in
// [target, target + slack] (slack = 0: T[s] is exactly the target-th largest
// key); a selection with fewer than `target` keys gets T[s] = 0 (keep all).
// Keys are unique within a selection.  visit(f) calls f(s, valid, key) for
// every key from every thread in lock step (invalid entries pass
// valid = false), so warp collectives inside f are safe.
//
// MSD radix select that starts at the highest bit in which the selection's
// keys differ (a min/max reduction finds it), so the first 8-bit digit
// already splits the live range of scores rather than the sign and exponent
// bits every candidate shares.  (Plain shared-memory atomics for the
// histogram measured faster here than aggregating equal digits per warp.)
// Compile-time loop: f(integral_constant<int, I>) for I in [B, E).
template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F &&f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

template <int S, typename Visit>
__device__ void select_thresholds(SelScratch<S> &sm, Visit visit, int target, int slack,
                                  uint64_t (&T)[S], int (&kept)[S]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    unsigned long long kmin[S], kmax[S];
    int cnt[S];
    static_for<0, S>([&](auto s) { kmin[s] = ~0ull; kmax[s] = 0ull; cnt[s] = 0; });
    visit([&](auto s, bool valid, uint64_t key) {
        if (valid) {
            kmin[s] = min(kmin[s], (unsigned long long)key);
            kmax[s] = max(kmax[s], (unsigned long long)key);
            ++cnt[s];
        }
    });
    static_for<0, S>([&](auto s) {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            kmin[s] = min(kmin[s], __shfl_xor_sync(0xffffffffu, kmin[s], o));
            kmax[s] = max(kmax[s], __shfl_xor_sync(0xffffffffu, kmax[s], o));
            cnt[s] += __shfl_xor_sync(0xffffffffu, cnt[s], o);
        }
        if (lane == 0) { sm.red[0][s][warp] = kmin[s]; sm.red[1][s][warp] = kmax[s]; sm.red_n[s][warp] = cnt[s]; }
    });
    __syncthreads();
    uint64_t prefix[S], pmask[S];
    int hi_bit[S], above[S];
    bool done[S];
    static_for<0, S>([&](auto s) {
        unsigned long long mn = ~0ull, mx = 0ull;
        int c = 0;
        for (int w = 0; w < nw; ++w) { mn = min(mn, sm.red[0][s][w]); mx = max(mx, sm.red[1][s][w]); c += sm.red_n[s][w]; }
        above[s] = 0;
        prefix[s] = 0; pmask[s] = 0; hi_bit[s] = 0;
        if (c < target || c == 0) { T[s] = 0; kept[s] = c; done[s] = true; }
        else if (mn == mx) { T[s] = mn; kept[s] = 1; done[s] = true; }
        else {
            done[s] = false;
            hi_bit[s] = 63 - __clzll((long long)(mn ^ mx));
            pmask[s] = (hi_bit[s] == 63) ? 0ull : ~((2ull << hi_bit[s]) - 1ull);
            prefix[s] = mn & pmask[s];
            T[s] = 0; kept[s] = c;
        }
    });
    __syncthreads();
    while (true) {
        bool all_done = true;
        static_for<0, S>([&](auto s) { all_done = all_done && done[s]; });
        if (all_done) break;
        int lo[S];
        uint64_t dmask[S];
        static_for<0, S>([&](auto s) {
            lo[s] = hi_bit[s] >= 7 ? hi_bit[s] - 7 : 0;
            dmask[s] = (2ull << (hi_bit[s] - lo[s])) - 1ull;    // digit bits [hi_bit .. lo]
        });
        for (int i = tid; i < S * 256; i += blockDim.x) (&sm.hist[0][0])[i] = 0;
        __syncthreads();
        visit([&](auto s, bool valid, uint64_t key) {
            if (valid && !done[s] && ((key & pmask[s]) == prefix[s]))
                atomicAdd(&sm.hist[s][(unsigned)((key >> lo[s]) & dmask[s])], 1u);
        });
        __syncthreads();
        bool warp_live = false;   // this warp searches selection `warp`
        int need_w = 0;
        static_for<0, S>([&](auto s) {
            if (warp == s && !done[s]) { warp_live = true; need_w = target - above[s]; }
        });
        if (warp_live) {
            const int s = warp;
            // lane l owns bins 255-8l .. 248-8l (descending)
            unsigned loc = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) loc += sm.hist[s][255 - 8 * lane - i];
            unsigned incl = loc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned excl = incl - loc;
            const unsigned need = (unsigned)need_w;
            if (lane == 31 && incl < need) { sm.digit[s] = -1; sm.above[s] = 0; sm.bucket[s] = 0; }
            if (excl < need && need <= incl) {
                unsigned c = excl;
                for (int i = 0; i < 8; ++i) {
                    const int bin = 255 - 8 * lane - i;
                    const unsigned hb = sm.hist[s][bin];
                    if (c + hb >= need) {
                        sm.digit[s] = bin;
                        sm.above[s] = (int)c;
                        sm.bucket[s] = (int)hb;
                        break;
                    }
                    c += hb;
                }
            }
        }
        __syncthreads();
        static_for<0, S>([&](auto s) {
            if (done[s]) return;
            const int d = sm.digit[s];
            if (d < 0) {                      // cannot happen for unique keys; keep everything
                T[s] = 0; done[s] = true;
                return;
            }
            above[s] += sm.above[s];
            const int hb = sm.bucket[s];
            prefix[s] |= (uint64_t)d << lo[s];
            pmask[s] |= dmask[s] << lo[s];
            if (above[s] + hb == target || above[s] + hb <= target + slack || lo[s] == 0) {
                T[s] = prefix[s];
                kept[s] = above[s] + hb;
                done[s] = true;
            } else {
                hi_bit[s] = lo[s] - 1;
            }
        });
        __syncthreads();   // everyone has read the results before the next pass rewrites them
    }
}

// Bin of a score among 256 equal-width bins from smin (explicitly rounded
// operations, so both passes below compute the same bin; monotone in s).
__device__ __forceinline__ int score_bin(float s, float smin, float inv) {
    const int b = (int)__fmul_rn(__fsub_rn(s, smin), inv);
    return b < 0 ? 0 : (b > 255 ? 255 : b);
}

// For every selection h (S at once), a threshold key T[h] with at least m of
// the visited keys at or above it and, unless the scores bunch into one bin,
// at most 2m (T[h] = 0: fewer than m keys, keep them all).  One histogram of
// the scores over 256 equal-width bins between their minimum and maximum
// (value space, so the sparse upper tail gets fine bins), the boundary bin
// found from the top, and T the smallest key in the bins at or above it.
// Bins are monotone in the score, so exactly the keys in those bins are >= T.
// visit(f) calls f(s, valid, score, key) for every item of every thread, in
// lock step.  Three passes over registers and four barriers, no refinement
// rounds: the callers only need a bound, not an exact rank.
template <int S, typename Visit>
__device__ void hist_thresholds(SelScratch<S> &sm, Visit visit, int m, uint64_t (&T)[S]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = tid; i < S * 256; i += blockDim.x) (&sm.hist[0][0])[i] = 0;
    float lo[S], hi[S];
    int cnt[S];
#pragma unroll
    for (int h = 0; h < S; ++h) { lo[h] = CUDART_INF_F; hi[h] = -CUDART_INF_F; cnt[h] = 0; }
    visit([&](auto h, bool valid, float sc, uint64_t) {
        if (valid) { lo[h] = fminf(lo[h], sc); hi[h] = fmaxf(hi[h], sc); ++cnt[h]; }
    });
#pragma unroll
    for (int h = 0; h < S; ++h) {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            lo[h] = fminf(lo[h], __shfl_xor_sync(0xffffffffu, lo[h], o));
            hi[h] = fmaxf(hi[h], __shfl_xor_sync(0xffffffffu, hi[h], o));
            cnt[h] += __shfl_xor_sync(0xffffffffu, cnt[h], o);
        }
        if (lane == 0) {
            sm.red[0][h][warp] = __float_as_uint(lo[h]);
            sm.red[1][h][warp] = __float_as_uint(hi[h]);
            sm.red_n[h][warp] = cnt[h];
        }
    }
    __syncthreads();
    float smin[S], inv[S];
    bool use[S];
#pragma unroll
    for (int h = 0; h < S; ++h) {
        float a = CUDART_INF_F, z = -CUDART_INF_F;
        int c = 0;
        for (int w = 0; w < nw; ++w) {
            a = fminf(a, __uint_as_float((uint32_t)sm.red[0][h][w]));
            z = fmaxf(z, __uint_as_float((uint32_t)sm.red[1][h][w]));
            c += sm.red_n[h][w];
        }
        use[h] = c >= m && c > 0;
        const float span = __fsub_rn(z, a);
        smin[h] = a;
        inv[h] = (span > 0.0f && span < CUDART_INF_F) ? __fdiv_rn(256.0f, span) : 0.0f;
    }
    visit([&](auto h, bool valid, float sc, uint64_t) {
        if (valid && use[h]) atomicAdd(&sm.hist[h][score_bin(sc, smin[h], inv[h])], 1u);
    });
    __syncthreads();
    if (warp < S) {   // warp h finds selection h's boundary: lane l owns bins 255-8l .. 248-8l
        const int h = warp;
        unsigned loc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) loc += sm.hist[h][255 - 8 * lane - i];
        unsigned incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned excl = incl - loc, need = (unsigned)m;
        bool uh = false;
        static_for<0, S>([&](auto hh) { if (h == hh) uh = use[hh]; });
        if (lane == 0 && !uh) sm.digit[h] = -1;
        if (uh && excl < need && need <= incl) {
            unsigned c = excl;
            for (int i = 0; i < 8; ++i) {
                const int bin = 255 - 8 * lane - i;
                c += sm.hist[h][bin];
                if (c >= need) { sm.digit[h] = bin; break; }
            }
        }
    }
    __syncthreads();
    int bnd[S];
    unsigned long long kmin[S];
#pragma unroll
    for (int h = 0; h < S; ++h) { bnd[h] = sm.digit[h]; kmin[h] = ~0ull; }
    visit([&](auto h, bool valid, float sc, uint64_t key) {
        if (valid && bnd[h] >= 0 && score_bin(sc, smin[h], inv[h]) >= bnd[h])
            kmin[h] = min(kmin[h], (unsigned long long)key);
    });
#pragma unroll
    for (int h = 0; h < S; ++h) {
#pragma unroll
        for (int o = 16; o; o >>= 1) kmin[h] = min(kmin[h], __shfl_xor_sync(0xffffffffu, kmin[h], o));
        if (lane == 0) sm.red[0][h][warp] = kmin[h];
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < S; ++h) {
        unsigned long long k = ~0ull;
        for (int w = 0; w < nw; ++w) k = min(k, sm.red[0][h][w]);
        T[h] = bnd[h] >= 0 ? k : 0ull;
    }
    __syncthreads();   // sm.red and sm.digit are reused by the next selection
}

// Appends the valid keys >= T (one per thread) to dst at a shared counter.
template <int S>
__device__ __forceinline__ void append_if(SelScratch<S> &sm, bool keep, uint64_t key, uint64_t *dst,
                                          int dst_cap) {
    const int lane = threadIdx.x & 31;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (bal) {
        int base = 0;
        if (lane == __ffs(bal) - 1) base = atomicAdd(&sm.new_cnt, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, __ffs(bal) - 1);
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (keep && pos < dst_cap) dst[pos] = key;
    }
}

// Prunes a list of `count` keys (global or shared memory) in place to the
// keys >= T found by select_thresholds(target, slack): the keys are read into
// registers once (KPT per thread, KPT * blockDim.x >= count), so the radix
// passes never go back to memory.  Returns the new count and T.
template <int KPT>
__device__ int prune_list(SelScratch<1> &sm, uint64_t *lst, int count, int target, int slack,
                          uint64_t *T_out) {
    const int tid = threadIdx.x;
    // only the first `used` register slots hold keys (a block-uniform bound)
    const int used = (count + (int)blockDim.x - 1) / (int)blockDim.x;
    uint64_t r[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        const int e = i * (int)blockDim.x + tid;
        r[i] = (i < used && e < count) ? lst[e] : 0ull;
    }
    uint64_t T[1];
    int kept[1];
    select_thresholds<1>(sm, [&](auto f) {
#pragma unroll
        for (int i = 0; i < KPT; ++i)
            if (i < used) f(std::integral_constant<int, 0>{}, i * (int)blockDim.x + tid < count, r[i]);
    }, target, slack, T, kept);
    if (tid == 0) sm.new_cnt = 0;
    __syncthreads();   // all keys are in registers: the list may be overwritten
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        if (i < used) {
            const bool keep = (i * (int)blockDim.x + tid < count) && r[i] >= T[0];
            append_if<1>(sm, keep, r[i], lst, count);
        }
    }
    __syncthreads();
    *T_out = T[0];
    return min(sm.new_cnt, count);
}

// ---------------------------------------------------------------------------
constexpr int kListKPT = 26;   // register keys per thread for list prunes (cap <= 26 * 256)
constexpr int kMultiKPT = 4;   // register keys per thread and head for the final shrink
// A first-pass list is cut back at the end only when it is longer than this many
// times m: the merge streams longer lists for less than the cut costs (a cut at
// 4m took 6 us of a 105 us scan of eight 1M-token units, and the merge was no
// faster for the shorter lists).
constexpr int kShrinkAbove = 8;

// kFix = false: the first pass (histogram thresholds, no exact selection; a
// list that would overflow publishes tau = max so that the merge flags it).
// kFix = true: the exact second pass over the chunks the merge flagged.
// kScores: also write every token's score (a diagnostic output; kept out of
// the other instantiations so that their loop stays small).
// kRows: score every token exactly from its bf16 key row (q . k in fp32, all
// channels; `planes` holds the rows [units][ctok][D]) instead of the planned
// planes; the selection is the same.  The exact top-k of a fidelity check.
template <int G, bool kFix, bool kScores, bool kRows>
__global__ void __launch_bounds__(NT, (G <= 4) ? 3 : 1)
scan_kernel(int n, int cb, int ctok, int D, int chunks, int unit_fast, int source, size_t stage_words, size_t stage_scales,
            const uint64_t *__restrict__ planes, const uint16_t *__restrict__ scales,
            const fathom_run *__restrict__ runs, const float *__restrict__ q, int k_sel, int m_sel,
            int m_first, int ns, int r0, int nf, int cap, int vec, float *__restrict__ scores_opt,
            uint64_t *__restrict__ cand, int *__restrict__ cand_cnt, uint64_t *__restrict__ cand_tau,
            int *__restrict__ flags, float *__restrict__ forced_scores, int *__restrict__ sub_ctr,
            int *__restrict__ sub_owner) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem<G> &sm = *reinterpret_cast<ScanSmem<G> *>(smem_raw);
    const int tid = threadIdx.x;
    const int units = (int)(gridDim.x / (unsigned)chunks);
    const int u = unit_fast ? (int)(blockIdx.x % (unsigned)units) : (int)(blockIdx.x / (unsigned)chunks);
    const int chunk = unit_fast ? (int)(blockIdx.x / (unsigned)units) : (int)(blockIdx.x % (unsigned)chunks);
    const int nb = num_blocks(n);
    const int n_sub = (nb + kSubBlocks - 1) / kSubBlocks;
    const size_t cta = (size_t)u * chunks + chunk;
    if (kFix) {
        // second pass: only chunks the merge flagged run again, keeping their exact top-k'
        bool any = false;
        for (int h = 0; h < G; ++h) any |= flags[cta * G + h] != 0;
        if (!any) return;
        m_sel = m_first = k_sel;
    } else {
        // the first sub-chunk is taken before the prologue: a CTA that starts after
        // its unit's sub-chunks are all taken publishes an empty list and ends
        if (tid == 0) {
            const int q0 = atomicAdd(sub_ctr + u, 1);
            sm.sq0[0] = q0 < n_sub ? q0 : n_sub;
        }
        __syncthreads();
        if (sm.sq0[0] >= n_sub) {
            if (tid < G) {
                cand_cnt[cta * G + tid] = 0;
                cand_tau[cta * G + tid] = 0ull;
            }
            return;
        }
    }

    // ---- prologue: active channels sorted by depth (desc), ties by channel:
    // a stable partition by depth from per-warp ballots over the D <= 128
    // channels; plane slots and the fixed 32-channel staging groups follow
    // arithmetically from the per-depth totals.
    const int lane = tid & 31, wid = tid >> 5;
    int t = 0;
    fathom_run rr = {0, 0, 0, 0, 0, 0};
    if (!kRows && tid < D) {
        rr = runs[(size_t)u * D + tid];
        t = (int)(rr.n_words / (uint32_t)nb);
        t = t > FATHOM_PLANES ? FATHOM_PLANES : t;
        // a channel whose staged run or scales would pass the unit's staging
        // stride (a plan larger than the staging area) is not read at all
        if (source == FATHOM_SRC_STAGING &&
            ((uint64_t)rr.dst_word + (uint64_t)t * nb > stage_words ||
             (uint64_t)rr.dst_scale + (t > 0 ? (uint64_t)nb : 0) > stage_scales))
            t = 0;
        if (source == FATHOM_SRC_STORE && rr.src_word != (uint32_t)tid * FATHOM_PLANES * cb) t = 0;
    }
    unsigned my_mask = 0;   // lanes of this warp with the same depth as this thread
    if (tid < FATHOM_MAX_D) {
#pragma unroll
        for (int v = 1; v <= FATHOM_PLANES; ++v) {
            const unsigned m = __ballot_sync(0xffffffffu, t == v);
            if (t == v) my_mask = m;
            if (lane == 0) sm.wcnt[v][wid] = __popc(m);
        }
    }
    if (tid < G) {
        sm.cnt[tid] = 0;
        sm.tau[tid] = 0;
    }
    __syncthreads();
    int tot[FATHOM_PLANES + 1], start[FATHOM_PLANES + 1];   // per depth: count, first sorted index
    {
        int acc_start = 0;
#pragma unroll
        for (int v = FATHOM_PLANES; v >= 1; --v) {
            int c = 0;
#pragma unroll
            for (int w2 = 0; w2 < FATHOM_MAX_D / 32; ++w2) c += sm.wcnt[v][w2];
            tot[v] = c;
            start[v] = acc_start;
            acc_start += c;
        }
        tot[0] = start[0] = 0;
    }
    const int A = tot[1] + tot[2] + tot[3] + tot[4];
    // first plane slot of sorted channel a: planes of all channels before it
    auto slot_of = [&](int a) {
        int sl = 0;
#pragma unroll
        for (int v = 1; v <= FATHOM_PLANES; ++v) {
            const int lo = start[v], hi = start[v] + tot[v];
            const int ov = max(0, min(a, hi) - lo);
            sl += v * ov;
        }
        return sl;
    };
    if (tid < D && t > 0) {
        int pos = start[t] + __popc(my_mask & ((1u << lane) - 1u));
        for (int w2 = 0; w2 < wid; ++w2) pos += sm.wcnt[t][w2];
        const uint64_t wbase = (source == FATHOM_SRC_STORE)
                                   ? ((uint64_t)u * D + tid) * FATHOM_PLANES * cb
                                   : (uint64_t)u * stage_words + rr.dst_word;
        const uint64_t sbase = (source == FATHOM_SRC_STORE)
                                   ? ((uint64_t)u * D + tid) * cb
                                   : (uint64_t)u * stage_scales + rr.dst_scale;
        sm.ch_t[pos] = t;
        sm.ch_scale[pos] = sbase;
        const float sc = ldexpf(1.0f, -t);
        for (int h = 0; h < G; ++h) sm.qs[pos][h] = q[((size_t)u * G + h) * D + tid] * sc;
        const int sl = slot_of(pos);
        // the store keeps a channel's planes cb words apart, staging packs them nb apart
        const uint64_t pstride = (source == FATHOM_SRC_STORE) ? (uint64_t)cb : (uint64_t)nb;
        for (int p = 0; p < t; ++p) sm.plane_src[sl + p] = wbase + (uint64_t)p * pstride;
    }
    const int n_groups = (A + kCHG - 1) / kCHG;
    if (tid < n_groups) {
        GroupDesc g;
        g.a0 = tid * kCHG;
        const int a1 = min(A, g.a0 + kCHG);
        g.p0 = slot_of(g.a0);
        int nv[FATHOM_PLANES + 1];
#pragma unroll
        for (int v = 1; v <= FATHOM_PLANES; ++v)
            nv[v] = max(0, min(a1, start[v] + tot[v]) - max(g.a0, start[v]));
        g.n4 = nv[4]; g.n3 = nv[3]; g.n2 = nv[2]; g.n1 = nv[1];
        sm.grp[tid] = g;
    }
    // Sub-chunks are handed out dynamically: the first pass takes the next one of
    // its unit from a counter, so CTAs that run faster take more of them, and
    // records which CTA scored each one; the second pass rescans exactly the
    // sub-chunks the flagged CTA scored.
    auto grab = [&]() -> int {   // thread 0 only
        if (kFix) {
            for (int q2 = sm.fix_pos; q2 < n_sub; ++q2)
                if (sub_owner[(size_t)u * n_sub + q2] == chunk) { sm.fix_pos = q2 + 1; return q2; }
            sm.fix_pos = n_sub;
            return n_sub;
        }
        const int q2 = atomicAdd(sub_ctr + u, 1);
        return q2 < n_sub ? q2 : n_sub;
    };
    if (tid == 0) {
        sm.n_groups = n_groups;
        sm.fix_pos = 0;
        if (kFix) sm.sq0[0] = grab();   // (the first pass took its first sub-chunk above)
        sm.sq0[1] = sm.sq0[0] < n_sub ? grab() : n_sub;
    }
    if constexpr (kRows) {   // every channel, unscaled queries
        for (int e = tid; e < D * G; e += NT) sm.qs[e / G][e % G] = q[((size_t)u * G + e % G) * D + e / G];
    }
    __syncthreads();

    const int ng = sm.n_groups;
    const int bl = tid >> 3;                 // block within the sub-chunk
    const uint32_t r = (uint32_t)(tid & 7);  // token offset within a byte lane
    DecodeRot dr;
#pragma unroll
    for (int k = 0; k <= FATHOM_PLANES; ++k) dr.rot[k] = (r - (uint32_t)k) & 31u;
    int s_cur = sm.sq0[0], s_next = sm.sq0[1], iter = 0;

    uint64_t tau[G];                         // per-head thresholds (same in every thread)
    float tf[G];                             // the score part of tau (-inf: keep everything)
#pragma unroll
    for (int h = 0; h < G; ++h) { tau[h] = 0; tf[h] = -CUDART_INF_F; }
    auto refresh_tf = [&]() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint32_t thi = (uint32_t)(tau[h] >> 32);
            tf[h] = (thi <= order_f32(-CUDART_INF_F)) ? -CUDART_INF_F : unorder_f32(thi);
        }
    };
    bool first = true;

    // The unit's CTAs take sub-chunks in order from the counter, so they sweep the
    // sequence together and the addresses in use at any moment stay within a
    // narrow band (few pages, few DRAM rows).  The usual plan (one staging group of at most kPG / 2 planes, aligned runs)
    // is double-buffered: while a sub-chunk is scored, cp.async already moves the
    // next one's plane words and scales into the other half of the staging
    // area, so loads stay in flight the whole time (this is what keeps a store
    // across the host link busy).  Other plans stage synchronously.
    const GroupDesc g0 = sm.grp[0];
    const int nch0 = g0.n4 + g0.n3 + g0.n2 + g0.n1;
    const int npl0 = 4 * g0.n4 + 3 * g0.n3 + 2 * g0.n2 + g0.n1;
    const bool piped = vec && ng == 1 && npl0 <= kPG / 2;
    // words and scales of the buffer the scan reads (store or staging), for the debug checks
    const uint64_t src_words = (source == FATHOM_SRC_STORE) ? (uint64_t)units * D * FATHOM_PLANES * cb
                                                             : (uint64_t)units * stage_words;
    const uint64_t src_scales = (source == FATHOM_SRC_STORE) ? (uint64_t)units * D * cb
                                                              : (uint64_t)units * stage_scales;
    (void)src_words;
    (void)src_scales;
    auto stage_async = [&](int half, int sbx) {
        for (int e = tid; e < npl0 * (kSubBlocks / 2); e += NT) {
            const int sl = e / (kSubBlocks / 2), c = e % (kSubBlocks / 2);
            const bool ok = sbx + 2 * c < nb &&              // nb even: both words in range or neither
                            FATHOM_CHECK(sm.plane_src[sl] + sbx + 2 * c + 2 <= src_words, kDbgScanStagePlanes,
                                         sm.plane_src[sl] + sbx + 2 * c);
            const uint64_t *src = ok ? planes + sm.plane_src[sl] + sbx + 2 * c : planes;
            cp_async16(&sm.pw[half * (kPG / 2) + sl][2 * c], src, ok ? 16 : 0);
        }
        for (int e = tid; e < nch0 * (kSubBlocks / 8); e += NT) {
            const int al = e / (kSubBlocks / 8), c = e % (kSubBlocks / 8);
            const bool ok = sbx + 8 * c < nb &&              // nb % 8 == 0 on this path
                            FATHOM_CHECK(sm.ch_scale[al] + sbx + 8 * c + 8 <= src_scales, kDbgScanStageScales,
                                         sm.ch_scale[al] + sbx + 8 * c);
            const uint16_t *src = ok ? scales + sm.ch_scale[al] + sbx + 8 * c : scales;
            cp_async16(&sm.scb[half][al][8 * c], src, ok ? 16 : 0);
        }
    };
    int half = 0;
    if (piped && s_cur < n_sub) stage_async(0, s_cur * kSubBlocks);
    if (piped) cp_async_commit();

    while (s_cur < n_sub) {
        const int sb = s_cur * kSubBlocks;
        const int nblk = min(kSubBlocks, nb - sb);
        // (second pass) make room in every head's candidate list before this sub-chunk
        if (kFix && k_sel > 0) {
#pragma unroll 1
            for (int h = 0; h < G; ++h) {
                const int c = sm.cnt[h];
                if (c + kSubTokens > cap) {
                    uint64_t *lst = cand + (cta * G + h) * (size_t)cap;
                    uint64_t T;
                    const int nc = prune_list<kListKPT>(sm.sel1, lst, min(c, cap), m_sel, kPruneSlack, &T);
                    if (tid == 0) { sm.cnt[h] = nc; sm.tau[h] = max((unsigned long long)sm.tau[h], (unsigned long long)T); }
                    __syncthreads();
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) tau[h] = sm.tau[h];
            refresh_tf();
        }

        Acc8<G> acc;
        acc.zero();

        if constexpr (kRows) {
            // exact scores: 4 channels of q (all heads) at a time from shared memory,
            // then the 8 tokens' key rows (8-byte loads of 4 bf16 channels)
            const uint16_t *rows = reinterpret_cast<const uint16_t *>(planes);
            const int beta = sb + bl;
            for (int j0 = 0; j0 < D; j0 += 4) {
                float qv[4][G];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int h = 0; h < G; ++h) qv[c][h] = (j0 + c < D) ? sm.qs[j0 + c][h] : 0.0f;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int i = beta * 64 + (int)r + 8 * m;
                    if (bl < nblk && i < n) {
                        const uint16_t *kr = rows + ((size_t)u * ctok + i) * D + j0;
                        float kf[4];
                        if (vec) {
                            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(kr));
                            kf[0] = __uint_as_float(v.x << 16); kf[1] = __uint_as_float(v.x & 0xffff0000u);
                            kf[2] = __uint_as_float(v.y << 16); kf[3] = __uint_as_float(v.y & 0xffff0000u);
                        } else {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                kf[c] = (j0 + c < D) ? __uint_as_float(((uint32_t)__ldg(kr + c)) << 16) : 0.0f;
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int h = 0; h < G; ++h) acc(m, h) = fmaf(qv[c][h], kf[c], acc(m, h));
                    }
                }
            }
        } else {
            // one staging group at a time: the pipelined plan has a single group whose
            // copies were issued one sub-chunk ahead; other plans stage each group here
            for (int gi = 0; gi < (piped ? 1 : ng); ++gi) {
                const GroupDesc g = piped ? g0 : sm.grp[gi];
                const int nch = g.n4 + g.n3 + g.n2 + g.n1;
                const uint2 *pwbase;
                if (piped) {
                    if (s_next < n_sub) stage_async(half ^ 1, s_next * kSubBlocks);
                    cp_async_commit();
                    cp_async_wait<1>();                 // this sub-chunk's copies have landed
                    __syncthreads();
                    // block weights w_hj = q_hj * 2^-t_j * a_{beta,j} from the prefetched scales
                    for (int e = tid; e < nch * kSubBlocks; e += NT) {
                        const int al = e / kSubBlocks, b = e % kSubBlocks;
                        const float a16 = __half2float(__ushort_as_half(sm.scb[half][al][b]));
#pragma unroll
                        for (int h = 0; h < G; ++h) sm.w[b][al * G + h] = sm.qs[al][h] * a16;
                    }
                    pwbase = &sm.pw[half * (kPG / 2)][0];
                } else {
                    const int npl = 4 * g.n4 + 3 * g.n3 + 2 * g.n2 + g.n1;
                    __syncthreads();
                    // stage plane words (slot-major) and block weights; with aligned runs
                    // and a full sub-chunk every load is 16 bytes
                    if (vec && nblk == kSubBlocks) {
                        for (int e = tid; e < npl * (kSubBlocks / 2); e += NT) {
                            const int sl = e / (kSubBlocks / 2), c = e % (kSubBlocks / 2);
                            const uint64_t w0 = sm.plane_src[g.p0 + sl] + sb + 2 * c;
                            *reinterpret_cast<uint4 *>(&sm.pw[sl][2 * c]) =
                                FATHOM_CHECK(w0 + 2 <= src_words, kDbgScanLoadPlanes, w0)
                                    ? __ldg(reinterpret_cast<const uint4 *>(planes + w0))
                                    : make_uint4(0u, 0u, 0u, 0u);
                        }
                    } else {
                        for (int e = tid; e < npl * kSubBlocks; e += NT) {
                            const int sl = e / kSubBlocks, b = e % kSubBlocks;
                            uint2 v = make_uint2(0u, 0u);
                            if (b < nblk && FATHOM_CHECK(sm.plane_src[g.p0 + sl] + sb + b < src_words,
                                                         kDbgScanLoadPlanes, sm.plane_src[g.p0 + sl] + sb + b)) {
                                const uint64_t wd = __ldg(planes + sm.plane_src[g.p0 + sl] + sb + b);
                                v = make_uint2((uint32_t)wd, (uint32_t)(wd >> 32));
                            }
                            sm.pw[sl][b] = v;
                        }
                    }
                    for (int e = tid; e < nch * kSubBlocks; e += NT) {
                        const int al = e / kSubBlocks, b = e % kSubBlocks;
                        const int a = g.a0 + al;
                        float a16 = 0.0f;
                        if (b < nblk && FATHOM_CHECK(sm.ch_scale[a] + sb + b < src_scales, kDbgScanLoadScales,
                                                     sm.ch_scale[a] + sb + b))
                            a16 = __half2float(__ushort_as_half(__ldg(scales + sm.ch_scale[a] + sb + b)));
#pragma unroll
                        for (int h = 0; h < G; ++h) sm.w[b][al * G + h] = sm.qs[a][h] * a16;
                    }
                    pwbase = &sm.pw[0][0];
                }
                __syncthreads();
                if (bl < nblk) {
                    const uint2 *pwcol = pwbase + bl;
                    const float *wrow = sm.w[bl];
                    int a = 0, slot = 0;
                    accum_depth<G, 4>(pwcol, wrow, a, a + g.n4, slot, dr, acc);
                    a += g.n4; slot += 4 * g.n4;
                    accum_depth<G, 3>(pwcol, wrow, a, a + g.n3, slot, dr, acc);
                    a += g.n3; slot += 3 * g.n3;
                    accum_depth<G, 2>(pwcol, wrow, a, a + g.n2, slot, dr, acc);
                    a += g.n2; slot += 2 * g.n2;
                    accum_depth<G, 1>(pwcol, wrow, a, a + g.n1, slot, dr, acc);
                }
            }
        }

        // ---- epilogue: debug scores, forced tokens, then the candidates' keys
        const int beta = sb + bl;
        unsigned cvm = 0;                        // bit m: a candidate (valid, not forced)
        // a block inside the sequence and clear of the forced tokens: all 8 are candidates
        const bool interior = !kScores && bl < nblk && beta * 64 >= ns && beta * 64 + 64 <= r0 && beta * 64 + 64 <= n;
        if (interior) cvm = 0xffu;
#pragma unroll
        for (int m = 0; m < 8 && !interior; ++m) {
            const int i = beta * 64 + (int)r + 8 * (m & 3) + 32 * (m >> 2);
            const bool valid = (bl < nblk) && (i < n);
            const bool forced = (i < ns || i >= r0);
            if (valid && !forced) cvm |= 1u << m;
            if (kScores && valid) {
#pragma unroll
                for (int h = 0; h < G; ++h) scores_opt[((size_t)u * G + h) * n + i] = acc(m, h);
            }
            if (valid && forced) {
                const int slot = (i < ns) ? i : ns + (i - r0);
                if (FATHOM_CHECK(slot >= 0 && slot < nf, kDbgScanForced, slot)) {
#pragma unroll
                    for (int h = 0; h < G; ++h) forced_scores[((size_t)u * G + h) * nf + slot] = acc(m, h);
                }
            }
        }
        auto key_of = [&](int m, int h) -> uint64_t {
            const uint32_t i = (uint32_t)(beta * 64 + (int)r + 8 * (m & 3) + 32 * (m >> 2));
            return ((uint64_t)order_f32(acc(m, h)) << 32) | (uint64_t)(0xffffffffu - i);
        };
        if (k_sel > 0 && first) {
            // a threshold from this first sub-chunk, all heads at once, from registers:
            // at least m1 of its keys are >= it (m1: a tail bound of the winners one
            // sub-chunk holds; the second pass: exactly k' .. 2k')
            uint64_t T[G];
            auto visit = [&](auto f) {
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    static_for<0, G>([&](auto h) { f(h, (cvm >> m) & 1u, acc(m, h), key_of(m, h)); });
            };
            if constexpr (kFix) {
                int kept[G];
                select_thresholds<G>(sm.selg, [&](auto f) {
                    visit([&](auto h, bool v, float, uint64_t key) { f(h, v, key); });
                }, m_first, m_first, T, kept);
            } else {
                // each thread's best key per head (its 8 tokens); the threshold puts
                // m1 of these maxima at or above it, so at least m1 keys pass
                float mx[G];
                uint64_t mk[G];
                bool any = false;
#pragma unroll
                for (int h = 0; h < G; ++h) { mx[h] = -CUDART_INF_F; mk[h] = 0ull; }
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    if ((cvm >> m) & 1u) {
                        any = true;
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            const uint64_t kk = key_of(m, h);
                            if (kk > mk[h]) { mk[h] = kk; mx[h] = acc(m, h); }
                        }
                    }
                }
                hist_thresholds<G>(sm.selg, [&](auto f) {
                    static_for<0, G>([&](auto h) { f(h, any, mx[h], mk[h]); });
                }, m_first, T);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) tau[h] = T[h];
            refresh_tf();
            if (tid < G) sm.tau[tid] = T[tid];
            first = false;
        }
        if (k_sel > 0) {
            // append every key >= tau (few, about m1 .. 2 m1 per sub-chunk and head):
            // a mask of the heads whose score reaches tau's score (one float compare
            // each; tau = 0 keeps everything), then per token a short loop over them
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                unsigned hm = 0;
#pragma unroll
                for (int h = 0; h < G; ++h)
                    if (((cvm >> m) & 1u) && acc(m, h) >= tf[h]) hm |= 1u << h;
                while (hm) {
                    const int h = __ffs(hm) - 1;
                    hm &= hm - 1;
                    float sc = acc(m, 0);
                    uint64_t th = tau[0];
                    static_for<1, G>([&](auto hh) {
                        if (h == hh) { sc = acc(m, hh); th = tau[hh]; }
                    });
                    const uint64_t kk = make_key(sc, (uint32_t)(beta * 64 + (int)r + 8 * (m & 3) + 32 * (m >> 2)));
                    if (kk >= th) {
                        const int pos = atomicAdd(&sm.cnt[h], 1);
                        if (pos < cap) cand[(cta * G + h) * (size_t)cap + pos] = kk;
                    }
                }
            }
        }
        if (tid == 0) {
            if (!kFix) sub_owner[(size_t)u * n_sub + s_cur] = chunk;
            sm.sq[iter & 1] = s_next < n_sub ? grab() : n_sub;
        }
        __syncthreads();   // staging buffers and counters are reused by the next sub-chunk
        s_cur = s_next;
        s_next = sm.sq[iter & 1];
        ++iter;
        half ^= 1;
    }
    if (piped) cp_async_wait<0>();

    // ---- shrink long lists (first pass: lists longer than 8m to about m .. 2m keys
    // by one histogram pass; second pass: exactly k'), then publish counts and thresholds: every
    // key this CTA dropped is < its threshold
    if constexpr (!kFix) {
        if (k_sel > 0) {
            // m: four times this CTA's expected share of the k' winners, for the
            // sub-chunks it actually scored (a CTA that took more of them may hold
            // more winners; cutting its list to the average share would raise its
            // threshold above the k'-th key and force a rescan)
            const int m_eff = min(k_sel, max(m_sel, (int)(((long long)4 * k_sel * iter + n_sub - 1) / n_sub)));
            int cs[G];
            bool fits = true, any_long = false;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                cs[h] = min(sm.cnt[h], cap);
                fits = fits && cs[h] <= kMultiKPT * NT;
                any_long = any_long || cs[h] > kShrinkAbove * m_eff;
            }
            if (fits && any_long) {
                uint64_t *lists = cand + cta * G * (size_t)cap;
                uint64_t rk[G][kMultiKPT];
#pragma unroll
                for (int i = 0; i < kMultiKPT; ++i)
                    static_for<0, G>([&](auto h) {
                        const int e = i * NT + tid;
                        rk[h][i] = e < cs[h] ? lists[h * (size_t)cap + e] : 0ull;
                    });
                uint64_t T[G];
                hist_thresholds<G>(sm.selg, [&](auto f) {
#pragma unroll
                    for (int i = 0; i < kMultiKPT; ++i)
                        static_for<0, G>([&](auto h) { f(h, i * NT + tid < cs[h], key_score(rk[h][i]), rk[h][i]); });
                }, m_eff, T);
                if (tid < G) sm.cnt[tid] = 0;
                __syncthreads();   // every key is in registers: the lists may be overwritten
                const int lane_ = tid & 31;
#pragma unroll
                for (int i = 0; i < kMultiKPT; ++i)
                    static_for<0, G>([&](auto h) {
                        const bool keep = i * NT + tid < cs[h] && rk[h][i] >= T[h];
                        const unsigned bal = __ballot_sync(0xffffffffu, keep);
                        if (bal) {
                            const int leader = __ffs(bal) - 1;
                            int base = 0;
                            if (lane_ == leader) base = atomicAdd(&sm.cnt[h], __popc(bal));
                            base = __shfl_sync(0xffffffffu, base, leader);
                            if (keep) lists[h * (size_t)cap + base + __popc(bal & ((1u << lane_) - 1u))] = rk[h][i];
                        }
                    });
                // a list that kept everything (T = 0) keeps its earlier threshold
                if (tid < G) sm.tau[tid] = max((unsigned long long)sm.tau[tid], (unsigned long long)T[tid]);
                __syncthreads();
            }
        }
        if (tid < G) {
            const int c = sm.cnt[tid];
            cand_cnt[cta * G + tid] = min(c, cap);
            // an overflowed list lost keys >= tau: the largest threshold makes the merge
            // flag this chunk for the exact second pass
            cand_tau[cta * G + tid] = c > cap ? ~0ull : sm.tau[tid];
        }
    } else {
        if (k_sel > 0) {
#pragma unroll 1
            for (int h = 0; h < G; ++h) {
                const int c = min(sm.cnt[h], cap);
                if (c > k_sel) {
                    uint64_t *lst = cand + (cta * G + h) * (size_t)cap;
                    uint64_t T;
                    const int nc = prune_list<kListKPT>(sm.sel1, lst, c, k_sel, 0, &T);
                    if (tid == 0) { sm.cnt[h] = nc; sm.tau[h] = T; }
                    __syncthreads();
                }
            }
        }
        if (tid < G) {
            cand_cnt[cta * G + tid] = min(sm.cnt[tid], cap);
            cand_tau[cta * G + tid] = sm.tau[tid];
            flags[cta * G + tid] = 0;   // handled
        }
    }
}

// ---------------------------------------------------------------------------
// Merge: grid (parts, G, units).  Part p of (unit, head) streams the
// candidate lists of chunks [p S / P, (p + 1) S / P) through a shared-memory
// buffer, pruning it to the exact top-k' whenever the next window would not
// fit; it writes its top-k' to the workspace and takes a ticket.  The last
// part to finish streams the P partial lists the same way, sorts the exact
// top-k' by token index and writes it between the forced sink and recent
// tokens.  With P = 1 the single part finishes directly.
// Two builds of the merge: 512 threads and an 8192-key buffer (one CTA per SM:
// for calls with few (unit, head) pairs), and 256 threads with a 2048-key
// buffer and at most 64 registers a thread (four CTAs per SM: for calls with
// many pairs, such as a 256-unit layer's 1024, whose merges would otherwise
// run in seven waves).  Both compute the same result; a buffer that fills is
// cut to its exact top-k' and streaming goes on.
constexpr int kMThreads = 512;
constexpr int kMBuf = 8192;                  // keys in the shared-memory buffer
constexpr int kMThreadsS = 256;
constexpr int kMBufS = 2048;

constexpr int kMSmall = 1024;              // keys of the boundary bin ranked directly, at most
template <int NTH, int MBUF>
struct MergeSmem {
    static constexpr int kThreads = NTH, kBuf = MBUF;
    static constexpr int kKPT = MBUF / NTH;  // register keys per thread for a buffer prune
    SelScratch<1> sel;
    uint64_t buf[MBUF];
    uint64_t small[kMSmall];                 // the boundary bin's keys (exact selection)
    float fred[2][NTH / 32];
    int bin_sel, bin_above, n_small;
    int off[FATHOM_MERGE_MAX_LISTS + 1];     // prefix sums of the streamed lists' counts
    int count;
    int is_last;
    uint64_t thresh;                         // the k'-th key of what was streamed (0: fewer keys)
};

// Cuts sm.buf[0 .. count) to its exact top-k keys (keys are unique) and
// returns the k-th key.  One histogram of the scores over 256 equal-width
// bins between their minimum and maximum finds the bin b holding the k-th
// key; every key in the bins above b is kept, and the keys of bin b (few: the
// bins are fine where the k-th key falls) are ranked against each other to
// find the k-th exactly.  A bin of more than kMSmall keys (scores bunched
// together) takes the radix select instead.  Requires count > k.
template <class SM>
__device__ uint64_t merge_exact_top(SM &sm, int count, int k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    float lo = CUDART_INF_F, hi = -CUDART_INF_F;
    for (int e = tid; e < count; e += blockDim.x) {
        const float sc = key_score(sm.buf[e]);
        lo = fminf(lo, sc);
        hi = fmaxf(hi, sc);
    }
    for (int i = tid; i < 256; i += blockDim.x) sm.sel.hist[0][i] = 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) { sm.fred[0][warp] = lo; sm.fred[1][warp] = hi; }
    if (tid == 0) sm.n_small = 0;
    __syncthreads();
    lo = CUDART_INF_F; hi = -CUDART_INF_F;
    for (int w = 0; w < nw; ++w) { lo = fminf(lo, sm.fred[0][w]); hi = fmaxf(hi, sm.fred[1][w]); }
    const float span = __fsub_rn(hi, lo);
    const float inv = (span > 0.0f && span < CUDART_INF_F) ? __fdiv_rn(256.0f, span) : 0.0f;
    for (int e = tid; e < count; e += blockDim.x) atomicAdd(&sm.sel.hist[0][score_bin(key_score(sm.buf[e]), lo, inv)], 1u);
    __syncthreads();
    if (warp == 0) {   // lane l owns bins 255-8l .. 248-8l; find the bin of the k-th key from the top
        unsigned loc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) loc += sm.sel.hist[0][255 - 8 * lane - i];
        unsigned incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned excl = incl - loc;
        if (excl < (unsigned)k && (unsigned)k <= incl) {
            unsigned c = excl;
            for (int i = 0; i < 8; ++i) {
                const int bin = 255 - 8 * lane - i;
                const unsigned hb = sm.sel.hist[0][bin];
                if (c + hb >= (unsigned)k) { sm.bin_sel = bin; sm.bin_above = (int)c; break; }
                c += hb;
            }
        }
    }
    __syncthreads();
    const int b = sm.bin_sel, above = sm.bin_above;
    if ((int)sm.sel.hist[0][b] > kMSmall) {   // bunched scores: radix select
        uint64_t T;
        const int nc = prune_list<SM::kKPT>(sm.sel, sm.buf, count, k, 0, &T);
        __syncthreads();
        if (tid == 0) { sm.count = nc; sm.thresh = T; }
        __syncthreads();
        return T;
    }
    for (int e = tid; e < count; e += blockDim.x) {
        const uint64_t key = sm.buf[e];
        if (score_bin(key_score(key), lo, inv) == b) sm.small[atomicAdd(&sm.n_small, 1)] = key;
    }
    __syncthreads();
    const int ns = sm.n_small, need = k - above;     // the need-th largest key of bin b is the k-th overall
    for (int e = tid; e < ns; e += blockDim.x) {
        const uint64_t x = sm.small[e];
        int rank = 0;
        for (int j = 0; j < ns; ++j) rank += sm.small[j] > x ? 1 : 0;
        if (rank == need - 1) sm.thresh = x;
    }
    __syncthreads();
    const uint64_t T = sm.thresh;
    // every key is >= T or not: keep the k keys >= T, compacted in place through registers
    uint64_t r[SM::kKPT];
    const int used = (count + (int)blockDim.x - 1) / (int)blockDim.x;
#pragma unroll
    for (int i = 0; i < SM::kKPT; ++i) {
        const int e = i * (int)blockDim.x + tid;
        r[i] = (i < used && e < count) ? sm.buf[e] : 0ull;
    }
    if (tid == 0) sm.sel.new_cnt = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < SM::kKPT; ++i)
        if (i < used) append_if<1>(sm.sel, (i * (int)blockDim.x + tid < count) && r[i] >= T, r[i], sm.buf, count);
    __syncthreads();
    if (tid == 0) sm.count = sm.sel.new_cnt;
    __syncthreads();
    return T;
}

// Streams `nl` lists (list l: base(l), count(l)) into sm.buf and leaves the
// exact top-k' (or everything, if fewer) in sm.buf[0 .. sm.count).
template <class SM, typename Base, typename Count>
__device__ void stream_select(SM &sm, int nl, Base base, Count count, int k_sel) {
    const int tid = threadIdx.x;
    // all list counts in one round of loads, then an exclusive scan by warp 0
    // (lane l sums a run of ceil(nl / 32) consecutive counts)
    for (int l = tid; l < nl; l += blockDim.x) sm.off[l + 1] = count(l);
    __syncthreads();
    if (tid < 32) {
        const int per = (nl + 31) / 32;
        const int l0 = min(nl, tid * per), l1 = min(nl, l0 + per);
        int run = 0;
        for (int l = l0; l < l1; ++l) run += sm.off[l + 1];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += y;
        }
        int acc = incl - run;
        for (int l = l0; l < l1; ++l) {
            const int c = sm.off[l + 1];
            sm.off[l] = acc;
            acc += c;
        }
        if (tid == 31) { sm.off[nl] = incl; sm.count = 0; }
    }
    __syncthreads();
    const int total = sm.off[nl];
    int done = 0;
    while (done < total) {
        int room = SM::kBuf - sm.count;
        if (room < SM::kThreads) {           // make room: cut the buffer to its exact top-k'
            merge_exact_top(sm, sm.count, k_sel);
            room = SM::kBuf - sm.count;
        }
        const int take = min(room, total - done);
        const int c0 = sm.count;
        // one warp per list: the lanes copy consecutive keys of the part of the list
        // that falls in this window (flattened positions [done, done + take))
        const int lane = tid & 31, warp = tid >> 5, nwarps = (int)blockDim.x >> 5;
        for (int l = warp; l < nl; l += nwarps) {
            const int a = max(sm.off[l], done), b = min(sm.off[l + 1], done + take);
            if (a >= b) continue;
            const uint64_t *src = base(l) + (a - sm.off[l]);
            uint64_t *dst = sm.buf + c0 + (a - done);
            for (int e = lane; e < b - a; e += 32) dst[e] = src[e];
        }
        __syncthreads();
        if (tid == 0) sm.count = c0 + take;
        __syncthreads();
        done += take;
    }
    if (sm.count > k_sel) {
        merge_exact_top(sm, sm.count, k_sel);    // leaves the k'-th key in sm.thresh
    } else {
        // k' keys or fewer: the threshold is the smallest of them (0: fewer than k')
        const int c = sm.count;
        unsigned long long mn = ~0ull;
        for (int e = tid; e < c; e += blockDim.x) mn = min(mn, (unsigned long long)sm.buf[e]);
#pragma unroll
        for (int o = 16; o; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        if ((tid & 31) == 0) sm.sel.red[0][0][tid >> 5] = mn;
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mn = min(mn, sm.sel.red[0][0][w]);
            sm.thresh = (c == k_sel) ? mn : 0ull;
        }
    }
    __syncthreads();
}

template <int NTH, int MBUF>
__global__ void __launch_bounds__(NTH, (NTH <= 256 ? 4 : 1))
merge_kernel(int n, int G, int k, int k_sel, int ns, int r0, int nf, int chunks, int parts, int cap,
             int second, const uint64_t *__restrict__ cand, const int *__restrict__ cand_cnt,
             const uint64_t *__restrict__ cand_tau, int *__restrict__ flags, int *__restrict__ dirty,
             const float *__restrict__ forced_scores, uint64_t *__restrict__ part_keys,
             int *__restrict__ part_cnt, unsigned *__restrict__ ticket, int32_t *__restrict__ out_idx,
             float *__restrict__ out_score, int *__restrict__ sub_ctr) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char msmem_raw[];
    MergeSmem<NTH, MBUF> &sm = *reinterpret_cast<MergeSmem<NTH, MBUF> *>(msmem_raw);
    const int p = blockIdx.x, h = blockIdx.y, u = blockIdx.z;
    const int tid = threadIdx.x;
    const size_t uh = (size_t)u * G + h;
    // the scan that ran before this merge took all of the unit's sub-chunks: its
    // counter starts again from zero for the next call
    if (!second && p == 0 && h == 0 && tid == 0) sub_ctr[u] = 0;
    if (second && !dirty[uh]) return;        // nothing was flagged for this (unit, head)
    int32_t *oi = out_idx + uh * k;
    float *os = out_score + uh * k;
    if (p == 0 && !second) {
        // forced tokens: sinks first, recent last
        const float *fs = forced_scores + uh * nf;
        for (int e = tid; e < ns; e += blockDim.x) { oi[e] = e; os[e] = fs[e]; }
        for (int e = tid; e < n - r0; e += blockDim.x) {
            oi[ns + k_sel + e] = r0 + e;
            os[ns + k_sel + e] = fs[ns + e];
        }
    }
    if (k_sel == 0) return;

    const int c_lo = (int)((long long)p * chunks / parts);
    const int c_hi = (int)((long long)(p + 1) * chunks / parts);
    stream_select(sm, c_hi - c_lo,
                  [&](int l) { return cand + (((size_t)u * chunks + c_lo + l) * G + h) * (size_t)cap; },
                  [&](int l) { return min(cand_cnt[((size_t)u * chunks + c_lo + l) * G + h], cap); },
                  k_sel);
    if (parts > 1) {
        uint64_t *pk = part_keys + (uh * parts + p) * (size_t)k_sel;
        for (int e = tid; e < sm.count; e += blockDim.x) pk[e] = sm.buf[e];
        if (tid == 0) part_cnt[uh * parts + p] = sm.count;
        __threadfence();
        __syncthreads();
        if (tid == 0) sm.is_last = (atomicAdd(ticket + uh, 1u) == (unsigned)parts - 1u) ? 1 : 0;
        __syncthreads();
        if (!sm.is_last) return;
        __threadfence();
        stream_select(sm, parts,
                      [&](int l) { return (const uint64_t *)(part_keys + (uh * parts + l) * (size_t)k_sel); },
                      [&](int l) { return __ldcg(part_cnt + uh * parts + l); }, k_sel);
        if (tid == 0) ticket[uh] = 0u;   // ready for the next call
    }
    // exactness: a chunk whose threshold lies above the k'-th key T may have
    // dropped keys >= T; flag it for the second pass (which rescans it exactly)
    if (!second) {
        const uint64_t T = sm.thresh;
        int any = 0;
        for (int c = tid; c < chunks; c += blockDim.x) {
            const size_t ch = ((size_t)u * chunks + c) * G + h;
            if (cand_tau[ch] > T) { flags[ch] = 1; any = 1; }
        }
        any = __syncthreads_or(any);
        if (tid == 0 && any) dirty[uh] = 1;
    } else if (tid == 0) {
        dirty[uh] = 0;
    }
    // bitonic sort of the k' winners by token index; padding keys 0 (index 0xffffffff) sort last
    int P2 = 1;
    while (P2 < k_sel) P2 <<= 1;
    if (P2 <= NTH) {
        // one key per thread: compare-exchange partners within a warp by shuffles,
        // farther ones through two alternating shared-memory buffers
        uint64_t x = (tid < sm.count) ? sm.buf[tid] : 0ull;
        __syncthreads();
        uint64_t *xb[2] = {sm.buf, sm.buf + NTH};
        int pb = 0;
        for (int size = 2; size <= P2; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                uint64_t y;
                if (stride >= 32) {
                    xb[pb][tid] = x;
                    __syncthreads();
                    y = xb[pb][tid ^ stride];
                    pb ^= 1;
                } else {
                    y = __shfl_xor_sync(0xffffffffu, x, stride);
                }
                const bool take_min = ((tid & stride) == 0) == ((tid & size) == 0);
                const bool x_first = key_index(x) < key_index(y);
                x = (take_min == x_first) ? x : y;
            }
        }
        __syncthreads();
        sm.buf[tid] = x;
        __syncthreads();
    } else {
        for (int e = sm.count + tid; e < P2; e += blockDim.x) sm.buf[e] = 0;
        __syncthreads();
        for (int size = 2; size <= P2; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int e = tid; e < P2 / 2; e += blockDim.x) {
                    const int lo = 2 * stride * (e / stride) + (e % stride);
                    const int hi = lo + stride;
                    const bool up = ((lo & size) == 0);
                    const uint64_t a = sm.buf[lo], b = sm.buf[hi];
                    const bool swap = up ? (key_index(a) > key_index(b)) : (key_index(a) < key_index(b));
                    if (swap) { sm.buf[lo] = b; sm.buf[hi] = a; }
                }
                __syncthreads();
            }
        }
    }
    for (int e = tid; e < k_sel; e += blockDim.x) {
        const uint64_t key = sm.buf[e];
        oi[ns + e] = (int32_t)key_index(key);
        os[ns + e] = key_score(key);
    }
}

// ---------------------------------------------------------------------------
template <int G>
static int launch_g(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                    int source, size_t stage_words, size_t stage_scales, const fathom_run *runs,
                    const float *q, int32_t *idx, float *score, float *scores_opt, void *ws,
                    cudaStream_t st, int part) {
    const ScanGrid sg = scan_grid(s);
    const Forced f = forced_range(s.n, s.n_sink, s.n_recent);
    const ScanWorkspace wl = scan_workspace_layout(s);
    const int k_sel = s.k - f.nf;
    const int cap = scan_cand_cap(s);
    if (cap > kListKPT * NT) { set_error("scan: candidate capacity %d too large", cap); return FATHOM_EINVAL; }
    char *w = (char *)ws;
    uint64_t *cand = (uint64_t *)(w + wl.cand_off);
    int *cnt = (int *)(w + wl.cnt_off);
    float *forced = (float *)(w + wl.forced_off);
    uint64_t *pkeys = (uint64_t *)(w + wl.part_keys_off);
    int *pcnt = (int *)(w + wl.part_cnt_off);
    unsigned *ticket = (unsigned *)(w + wl.ticket_off);
    const int m_sel = scan_m_sel(sg.chunks, k_sel);
    const int m_first = scan_m_first((num_blocks(s.n) + kSubBlocks - 1) / kSubBlocks, k_sel, m_sel);
    uint64_t *ctau = (uint64_t *)(w + wl.tau_off);
    int *flags = (int *)(w + wl.flags_off);
    int *dirty = (int *)(w + wl.dirty_off);
    int *sub_ctr = (int *)(w + wl.sub_ctr_off);
    int *sub_owner = (int *)(w + wl.sub_owner_off);
    // 16-byte staging loads need every plane-row and scale-row start 16-byte aligned:
    // nb a multiple of 8 (n a multiple of 512), aligned strides and bases
    const int nb = num_blocks(s.n);
    const bool aligned_src = (source == FATHOM_SRC_STORE) || (stage_words % 2 == 0 && stage_scales % 8 == 0);
    const int cb = cap_blocks(s);
    const bool rows_src = source == FATHOM_SRC_ROWS;
    // rows: 8-byte loads of 4 bf16 channels need D % 4 == 0 and an aligned base
    const int vec = rows_src ? (s.D % 4 == 0 && (uintptr_t)planes % 8 == 0)
                             : (nb % 8 == 0) && (source != FATHOM_SRC_STORE || cb % 8 == 0) && aligned_src &&
                                   ((uintptr_t)planes % 16 == 0) && ((uintptr_t)scales % 16 == 0);
    const size_t smem = sizeof(ScanSmem<G>);
    if ((long long)s.units * sg.chunks > 0x7fffffffLL) { set_error("scan: too many units for one launch"); return FATHOM_EINVAL; }
    ensure_smem(scan_kernel<G, false, false, false>, smem);
    ensure_smem(scan_kernel<G, false, true, false>, smem);
    ensure_smem(scan_kernel<G, true, false, false>, smem);
    ensure_smem(scan_kernel<G, false, false, true>, smem);
    ensure_smem(scan_kernel<G, false, true, true>, smem);
    ensure_smem(scan_kernel<G, true, false, true>, smem);
    // the merge build: four 256-thread CTAs per SM once the (unit, head) pairs (times
    // the parts of each) would fill two waves of one 512-thread CTA per SM
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;
    // (and k' at most half its buffer, so that a cut buffer keeps room to stream)
    const bool small_merge = (long long)s.units * s.G * wl.parts >= 2LL * sms && k_sel <= kMBufS / 2;
    const size_t msmem = small_merge ? sizeof(MergeSmem<kMThreadsS, kMBufS>) : sizeof(MergeSmem<kMThreads, kMBuf>);
    if (small_merge) ensure_smem(merge_kernel<kMThreadsS, kMBufS>, msmem);
    else ensure_smem(merge_kernel<kMThreads, kMBuf>, msmem);
    const int nf = f.nf > 0 ? f.nf : 1;
    dim3 grid((unsigned)(s.units * sg.chunks));
    cudaError_t le = cudaSuccess;
    for (int pass = 0; pass < 2; ++pass) {
        // part SCAN: the first-pass scan only; part SELECT: everything after it
        const bool do_scan = pass == 1 ? part != SCAN_PART_SCAN : part != SCAN_PART_SELECT;
        const bool do_merge = part != SCAN_PART_SCAN;
#define FATHOM_SCAN_LAUNCH(FIX, SC, RW)                                                                    \
    le = launch_pdl(scan_kernel<G, FIX, SC, RW>, grid, dim3(NT), smem, st, s.n, cb, cap_tokens(s), s.D,        \
                    sg.chunks, sg.unit_fast, source, stage_words, stage_scales, planes, scales, runs, q, k_sel, m_sel, \
                    m_first, f.ns, f.r0, nf, cap, vec, SC ? scores_opt : nullptr, cand, cnt, ctau, flags,      \
                    forced, sub_ctr, sub_owner)
        if (do_scan) {
            if (rows_src) {
                if (pass == 1) FATHOM_SCAN_LAUNCH(true, false, true);
                else if (scores_opt) FATHOM_SCAN_LAUNCH(false, true, true);
                else FATHOM_SCAN_LAUNCH(false, false, true);
            } else {
                if (pass == 1) FATHOM_SCAN_LAUNCH(true, false, false);
                else if (scores_opt) FATHOM_SCAN_LAUNCH(false, true, false);
                else FATHOM_SCAN_LAUNCH(false, false, false);
            }
            if (le != cudaSuccess) { set_error("scan_kernel: %s", cudaGetErrorString(le)); return FATHOM_ECUDA; }
            const int rc0 = launch_status("scan_kernel");
            if (rc0) return rc0;
        }
#undef FATHOM_SCAN_LAUNCH
        if (!do_merge) break;
#define FATHOM_MERGE_LAUNCH(NTH, MBUF)                                                                    \
    le = launch_pdl(merge_kernel<NTH, MBUF>, dim3(wl.parts, s.G, s.units), dim3(NTH), msmem, st, s.n, s.G, s.k, k_sel, \
                    f.ns, f.r0, nf, sg.chunks, wl.parts, cap, pass, (const uint64_t *)cand, (const int *)cnt,     \
                    (const uint64_t *)ctau, flags, dirty, (const float *)forced, pkeys, pcnt, ticket, idx, score,  \
                    sub_ctr)
        if (small_merge) FATHOM_MERGE_LAUNCH(kMThreadsS, kMBufS);
        else FATHOM_MERGE_LAUNCH(kMThreads, kMBuf);
#undef FATHOM_MERGE_LAUNCH
        if (le != cudaSuccess) { set_error("merge_kernel: %s", cudaGetErrorString(le)); return FATHOM_ECUDA; }
        const int rc = launch_status("merge_kernel");
        if (rc) return rc;
        if (k_sel == 0) break;   // nothing selected: no second pass needed
    }
    return FATHOM_OK;
}

// Resident CTAs of scan_kernel<G> per SM on the current device, with its
// shared memory (0 when no device answers); cached per device.
template <int G>
static int resident_g() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        const size_t smem = sizeof(ScanSmem<G>);
        ensure_smem(scan_kernel<G, false, false, false>, smem);
        int nbk = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nbk, scan_kernel<G, false, false, false>, NT, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev] = nbk;
    }
    return cache[dev];
}

FATHOM_DEBUG_READER(debug_read_scan)

int scan_resident_ctas(int G) {
    switch (G) {
        case 1: return resident_g<1>();
        case 2: return resident_g<2>();
        case 4: return resident_g<4>();
        case 8: return resident_g<8>();
        default: return 0;
    }
}

int launch_scan_topk(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                     int source, size_t stage_words, size_t stage_scales, const fathom_run *runs,
                     const float *q, int32_t *idx, float *score, float *scores_opt, void *ws,
                     cudaStream_t st, int part) {
    switch (s.G) {
        case 1: return launch_g<1>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st, part);
        case 2: return launch_g<2>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st, part);
        case 4: return launch_g<4>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st, part);
        case 8: return launch_g<8>(s, planes, scales, source, stage_words, stage_scales, runs, q, idx, score, scores_opt, ws, st, part);
        default: set_error("unsupported G=%d", s.G); return FATHOM_EINVAL;
    }
}

}  // namespace fathom

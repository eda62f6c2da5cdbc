// sparse_attn.cu -- exact attention over the winners (Fathom §1 / §3.1: the
// winners' rows at full precision; §2: each head attends exactly over its own
// selected set, with no mass redistribution for the rest).
//
// Two launch forms of one kernel.  One head per grid row (the usual one): the
// kernel runs with G = 1 over units x G grid rows, row (u, h) reading unit u's
// K and V rows with head h's query and kept list; CTA c of a row takes entries
// [c R, c R + R) of the list, and a row kept by several heads is read once per
// head.  The union form (keys rebuilt from the store, or more than 65535
// (unit, head) pairs): grid (G * ceil(k / R), units), CTA (h, c) takes entries
// [c R, c R + R) of head h's list and handles the rows that h owns -- the rows
// no lower head lists -- so every row of the union is fetched exactly once; the
// CTA first finds, for its R rows, which other heads list them (one binary
// search per (row, head) pair, all threads at once).  In both forms each warp
// loads a batch of rows (K and V, bf16) and computes the dot products of every
// (row, head) slot of the batch with one transpose reduction across the warp,
// updates an online softmax state (running max, sum, weighted V) per head, and
// the CTA merges its warps into one partial state per head.  The last CTA of
// the grid row (an atomic ticket, no waiting) merges the partial states of all
// CTAs of the row and writes o_h.

#include <mutex>

#include "fathom_internal.cuh"

namespace fathom {

constexpr int NA = kAttnThreads;
constexpr int kWarps = NA / 32;

// Where the batch step reads K: bf16 rows [units][ctok][D], or the 4-bit store
// ([units][D][4][cb] planes, [units][D][cb] fp16 scales) with every winner's key
// rebuilt from all four planes.
struct KSource {
    const uint16_t *rows;
    const uint64_t *planes;
    const uint16_t *scales;
    int cb;
};

// Rows per warp batch: RB rows x G heads = S dot products, reduced together
// (16 rows for one head per grid row: twice the loads in flight, and the
// batch's reduction and softmax update spread over twice the rows).
template <int G>
struct AttnBatch {
    static constexpr int RB = G == 1 ? 16 : ((32 / G) < 8 ? (32 / G) : 8);
    static constexpr int S = RB * G;   // <= 32, a power of two
};

struct AttnHeader {
    int is_last;
    int rows[kAttnRowsMax];
    unsigned rmask[kAttnRowsMax];
    float wm[kWarps][FATHOM_MAX_G];
    float wl[kWarps][FATHOM_MAX_G];
    float wf[kWarps][FATHOM_MAX_G];
    float cl[FATHOM_MAX_G];
    float pbuf[kWarps][32];
};

// Heads merged per round by the last CTA: all of them when their partial
// states fit in about 96 KiB of shared memory, else one at a time.
__host__ __device__ inline int attn_merge_heads(int G, int splits, int D) {
    const size_t per_head = (size_t)splits * (D + 2) * sizeof(float);
    return (size_t)G * per_head <= ((size_t)96 << 10) ? G : 1;
}

struct AttnLayout {
    size_t lists, wo, merge, total;
};

// header, then the G index lists and the warps' weighted-V states; the last
// CTA's merge buffer ([splits][heads of the round][D + 2] floats) reuses the
// same bytes once they are no longer read
__host__ __device__ inline AttnLayout attn_smem_layout(int G, int k, int D, int splits) {
    AttnLayout L;
    L.lists = (sizeof(AttnHeader) + 15) & ~(size_t)15;
    L.wo = (L.lists + (size_t)G * k * sizeof(int) + 15) & ~(size_t)15;
    const size_t end_main = L.wo + (size_t)kWarps * G * D * sizeof(float);
    L.merge = L.lists;
    const size_t end_merge =
        L.merge + (size_t)attn_merge_heads(G, splits, D) * splits * (D + 2) * sizeof(float);
    L.total = ((end_main > end_merge ? end_main : end_merge) + 15) & ~(size_t)15;
    return L;
}

__device__ __forceinline__ bool contains(const int *lst, int k, int x) {
    int lo = 0, hi = k;   // first position with lst[pos] >= x
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (lst[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo < k && lst[lo] == x;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Warp merge, this CTA's partial state per head, and (last CTA of the unit, by
// an atomic ticket) the merge of all partial states into o_h.  m_h, l_h, o_h:
// this thread's online-softmax state (lane l holds channels 4l..4l+3, kVec, or
// l + 32 e).  Shared by the sparse and the dense attention.
template <int G, bool kVec>
__device__ __forceinline__ void attn_finish(AttnHeader &sm, unsigned char *asmem_raw, const AttnLayout &lay,
                                            int D, int s, int u, int splits, const float (&m_h)[G],
                                            const float (&l_h)[G], float (&o_h)[G][4], float *__restrict__ out,
                                            float *__restrict__ part, unsigned *__restrict__ ticket) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *wo = reinterpret_cast<float *>(asmem_raw + lay.wo);          // [warp][h][D]
    // ---- merge the warps: rescale each warp's state to the CTA maximum
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) { sm.wm[warp][h] = m_h[h]; sm.wl[warp][h] = l_h[h]; }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][h]);
        const float f = (m_h[h] == -CUDART_INF_F) ? 0.0f : expf(m_h[h] - M);
        if (lane == 0) sm.wf[warp][h] = f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = kVec ? 4 * lane + c : lane + 32 * c;
            if (j < D) wo[((size_t)warp * G + h) * D + j] = o_h[h][c] * f;
        }
    }
    __syncthreads();
    float *pp = part + ((size_t)u * splits + s) * G * (D + 2);
    for (int e = tid; e < G * (D + 2); e += NA) {
        const int h = e / (D + 2), c = e % (D + 2);
        float acc = 0.0f;
        if (c == 0) {
            acc = -CUDART_INF_F;
            for (int w = 0; w < kWarps; ++w) acc = fmaxf(acc, sm.wm[w][h]);
        } else if (c == 1) {
            for (int w = 0; w < kWarps; ++w) acc = fmaf(sm.wf[w][h], sm.wl[w][h], acc);
        } else {
            for (int w = 0; w < kWarps; ++w) acc += wo[((size_t)w * G + h) * D + (c - 2)];
        }
        pp[e] = acc;
    }
    // ---- the last CTA of the unit merges the partial states
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(ticket + u, 1u);
        sm.is_last = (t == (unsigned)splits - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!sm.is_last) return;
    __threadfence();
    const float *p0 = part + (size_t)u * splits * G * (D + 2);
    float *mg = reinterpret_cast<float *>(asmem_raw + lay.merge);   // [splits][nh][D + 2]
    const int hc = attn_merge_heads(G, splits, D);
    for (int h0 = 0; h0 < G; h0 += hc) {
        const int nh = min(hc, G - h0), row = nh * (D + 2);
        for (int e = tid; e < splits * row; e += NA) {
            const int sp = e / row, c = e % row;
            mg[e] = __ldcg(p0 + ((size_t)sp * G + h0) * (D + 2) + c);
        }
        __syncthreads();
        if (warp < nh) {   // warp hh: the head's maximum, split weights (in place of m) and sum
            float M = -CUDART_INF_F;
            for (int sp = lane; sp < splits; sp += 32) M = fmaxf(M, mg[(size_t)sp * row + warp * (D + 2)]);
            M = warp_max(M);
            float L = 0.0f;
            for (int sp = lane; sp < splits; sp += 32) {
                float *b = mg + (size_t)sp * row + warp * (D + 2);
                const float f = (b[0] == -CUDART_INF_F) ? 0.0f : expf(b[0] - M);
                b[0] = f;
                L = fmaf(f, b[1], L);
            }
            L = warp_sum(L);
            if (lane == 0) sm.cl[warp] = L;
        }
        __syncthreads();
        for (int e = tid; e < nh * D; e += NA) {
            const int hh = e / D, j = e % D;
            float O = 0.0f;
            for (int sp = 0; sp < splits; ++sp) {
                const float *b = mg + (size_t)sp * row + hh * (D + 2);
                O = fmaf(b[0], b[2 + j], O);
            }
            out[((size_t)u * G + h0 + hh) * D + j] = O / sm.cl[hh];
        }
        __syncthreads();
    }
    if (tid == 0) ticket[u] = 0u;   // ready for the next call
}

// One batch of RB rows (token ti[r] of the unit, attended by the heads in
// mask[r]; mask 0: no row): loads K (bf16 rows, or kPlanes: rebuilt from the
// store's four planes) and V (bf16), the G dot products of every
// row with one transpose reduction across the warp, and the online-softmax
// update of every head's state.
template <int G, bool kVec, bool kPlanes>
__device__ __forceinline__ void attn_batch(const unsigned (&mask)[AttnBatch<G>::RB], const int (&ti)[AttnBatch<G>::RB],
                                           const KSource &ks, const uint16_t *__restrict__ vrows, int u,
                                           size_t ubase, int D, float scale, const float (&qv)[G][4],
                                           float (&m_h)[G], float (&l_h)[G], float (&o_h)[G][4], float *pb) {
    constexpr int RB = AttnBatch<G>::RB, S = AttnBatch<G>::S;
    const int lane = threadIdx.x & 31;
    const int v = lane & (S - 1), vr = v / G, vh = v % G;   // this lane's (row, head) slot
    uint2 kp[RB], vp[RB];                      // bf16 pairs (kVec)
    float kv[RB][4], vv[RB][4];                // general path (and keys rebuilt from the planes)
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const unsigned m = mask[r];
        const uint16_t *kr = ks.rows + (ubase + (m ? ti[r] : 0)) * D;
        const uint16_t *vr_ = vrows + (ubase + (m ? ti[r] : 0)) * D;
        if constexpr (kPlanes) {
            // code c of token i, channel j: bit i % 64 of the block's four plane
            // words (plane 0 = MSB); the key is (c - 7.5) a / 8, exact in fp32
            const int beta = m ? (ti[r] >> 6) : 0, sh = m ? (ti[r] & 63) : 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = kVec ? 4 * lane + c : lane + 32 * c;
                float kx = 0.0f;
                if (m && j < D) {
                    const size_t ch = (size_t)u * D + j;
                    const uint64_t *pw = ks.planes + ch * 4 * (size_t)ks.cb + beta;
                    const uint32_t code = (uint32_t)((__ldg(pw) >> sh) & 1u) << 3 |
                                          (uint32_t)((__ldg(pw + ks.cb) >> sh) & 1u) << 2 |
                                          (uint32_t)((__ldg(pw + 2 * (size_t)ks.cb) >> sh) & 1u) << 1 |
                                          (uint32_t)((__ldg(pw + 3 * (size_t)ks.cb) >> sh) & 1u);
                    const float a = __half2float(__ushort_as_half(__ldg(ks.scales + ch * ks.cb + beta)));
                    kx = ((float)code - 7.5f) * (a * 0.125f);
                }
                kv[r][c] = kx;
            }
            if (kVec) vp[r] = m ? __ldg(reinterpret_cast<const uint2 *>(vr_) + lane) : make_uint2(0u, 0u);
            else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = lane + 32 * c;
                    vv[r][c] = (m && j < D) ? __uint_as_float(((uint32_t)__ldg(vr_ + j)) << 16) : 0.0f;
                }
            }
        } else if (kVec) {
            kp[r] = m ? __ldg(reinterpret_cast<const uint2 *>(kr) + lane) : make_uint2(0u, 0u);
            vp[r] = m ? __ldg(reinterpret_cast<const uint2 *>(vr_) + lane) : make_uint2(0u, 0u);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = lane + 32 * c;
                const bool ok = m && j < D;
                kv[r][c] = ok ? __uint_as_float(((uint32_t)__ldg(kr + j)) << 16) : 0.0f;
                vv[r][c] = ok ? __uint_as_float(((uint32_t)__ldg(vr_ + j)) << 16) : 0.0f;
            }
        }
    }
        // partial dots of every (row, head) slot, then one transpose reduction:
        // afterwards lane l holds the full dot of slot l mod S
        float a[S];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float kk[4];
            if (kVec && !kPlanes) {
                kk[0] = bf16lo(kp[r].x); kk[1] = bf16hi(kp[r].x); kk[2] = bf16lo(kp[r].y); kk[3] = bf16hi(kp[r].y);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) kk[c] = kv[r][c];
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float d = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) d = fmaf(qv[h][c], kk[c], d);
                a[r * G + h] = d;
            }
        }
#pragma unroll
        for (int w = S / 2; w >= 1; w >>= 1) {
            const bool up = (lane & w) != 0;
#pragma unroll
            for (int i = 0; i < w; ++i) {
                const float send = up ? a[i] : a[i + w];
                const float keep = up ? a[i + w] : a[i];
                a[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
        }
#pragma unroll
        for (int o = S; o < 32; o <<= 1) a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
        // online softmax for slot (vr, vh), then per head across the batch's rows
        unsigned mv = 0;
        float mo = -CUDART_INF_F;
#pragma unroll
        for (int r = 0; r < RB; ++r) mv = (r == vr) ? mask[r] : mv;
#pragma unroll
        for (int h = 0; h < G; ++h) mo = (h == vh) ? m_h[h] : mo;
        const bool live = (mv >> vh) & 1u;
        const float logit = live ? a[0] * scale : -CUDART_INF_F;
        float mn = logit;
#pragma unroll
        for (int o = G; o < S; o <<= 1) mn = fmaxf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mn = fmaxf(mn, mo);
        float p = 0.0f, corr = 1.0f;
        if (mn != -CUDART_INF_F) {
            p = live ? expf(logit - mn) : 0.0f;
            corr = expf(mo - mn);
        }
        float ps = p;
#pragma unroll
        for (int o = G; o < S; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        if (lane < S) pb[lane] = p;
        __syncwarp();
#pragma unroll
        for (int h = 0; h < G; ++h) {   // lane h holds slot (row 0, head h)
            const float c = __shfl_sync(0xffffffffu, corr, h);
            l_h[h] = l_h[h] * c + __shfl_sync(0xffffffffu, ps, h);
            m_h[h] = __shfl_sync(0xffffffffu, mn, h);
#pragma unroll
            for (int e = 0; e < 4; ++e) o_h[h][e] *= c;
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float vx[4];
            if (kVec) {
                vx[0] = bf16lo(vp[r].x); vx[1] = bf16hi(vp[r].x); vx[2] = bf16lo(vp[r].y); vx[3] = bf16hi(vp[r].y);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) vx[c] = vv[r][c];
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pr = pb[r * G + h];
#pragma unroll
                for (int e = 0; e < 4; ++e) o_h[h][e] = fmaf(pr, vx[e], o_h[h][e]);
            }
        }
        __syncwarp();
}

// Lane l holds channels 4l .. 4l+3 (kVec: D = 128, one 8-byte load of K and one
// of V per row) or channels l + 32 e (any D <= 128).
template <int G, bool kVec, bool kPlanes>
__global__ void __launch_bounds__(NA, G >= 8 ? 1 : 2)
attn_kernel(int n, int ctok, int D, int k, int rows_cta, int cph, int splits, int hdiv, const KSource ks,
            const uint16_t *__restrict__ vrows, const float *__restrict__ q,
            const int32_t *__restrict__ topk, float *__restrict__ out, float *__restrict__ part,
            unsigned *__restrict__ ticket) {
    pdl_enter();
    constexpr int RB = AttnBatch<G>::RB;
    extern __shared__ __align__(16) unsigned char asmem_raw[];
    AttnHeader &sm = *reinterpret_cast<AttnHeader *>(asmem_raw);
    const AttnLayout lay = attn_smem_layout(G, k, D, splits);
    int *lists = reinterpret_cast<int *>(asmem_raw + lay.lists);
    const int s = blockIdx.x, u = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hown = s / cph;
    const int e_begin = (s % cph) * rows_cta;
    const int R = min(k, e_begin + rows_cta) - e_begin;

    // ---- the G sorted lists, then this CTA's rows and their head masks
    const int32_t *src = topk + (size_t)u * G * k;
    if ((k & 3) == 0 && ((uintptr_t)src & 15) == 0) {
        for (int e = tid; e < G * k / 4; e += NA)
            reinterpret_cast<int4 *>(lists)[e] = __ldg(reinterpret_cast<const int4 *>(src) + e);
    } else {
        for (int e = tid; e < G * k; e += NA) lists[e] = __ldg(src + e);
    }
    __syncthreads();
    for (int r = tid; r < R; r += NA) {
        const int i = r < R ? lists[hown * k + e_begin + r] : -1;
        sm.rows[r] = i;
        sm.rmask[r] = (r < R && i >= 0 && i < n) ? (1u << hown) : 0u;
    }
    __syncthreads();
    for (int p = tid; p < R * G; p += NA) {
        const int r = p % R, h2 = p / R;
        if (h2 != hown && r < R && contains(lists + h2 * k, k, sm.rows[r])) atomicOr(&sm.rmask[r], 1u << h2);
    }
    __syncthreads();

    const float scale = 1.0f / sqrtf((float)D);   // 1/sqrt(D), correctly rounded
    float m_h[G], l_h[G], o_h[G][4], qv[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_h[h] = -CUDART_INF_F;
        l_h[h] = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o_h[h][e] = 0.0f;
            const int j = kVec ? 4 * lane + e : lane + 32 * e;
            qv[h][e] = (j < D) ? q[((size_t)u * G + h) * D + j] : 0.0f;
        }
    }
    float *pb = sm.pbuf[warp];
    const unsigned below = (1u << hown) - 1u;
    for (int r0 = warp * RB; r0 < R; r0 += kWarps * RB) {
        unsigned mask[RB];
        int ti[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int rr = r0 + r;
            unsigned m = 0;
            int i = 0;
            if (rr < R) {
                m = sm.rmask[rr];
                i = sm.rows[rr];
                if (!((m >> hown) & 1u) || (m & below)) m = 0;   // invalid, or a lower head owns it
                if (m && !FATHOM_CHECK(i >= 0 && i < n, kDbgAttnRow, (unsigned)i)) m = 0;
            }
            mask[r] = m;
            ti[r] = i;
        }
        attn_batch<G, kVec, kPlanes>(mask, ti, ks, vrows, u / hdiv, (size_t)(u / hdiv) * ctok, D, scale, qv, m_h,
                                     l_h, o_h, pb);
    }
    attn_finish<G, kVec>(sm, asmem_raw, lay, D, s, u, splits, m_h, l_h, o_h, out, part, ticket);
}

// Dense attention over every token (the fidelity reference): grid (splits, units),
// CTA c attends all G heads over tokens [c R, c R + R) with the same batch step,
// then the same partial states and last-CTA merge.
template <int G, bool kVec>
__global__ void __launch_bounds__(NA, G >= 8 ? 1 : 2)
dense_attn_kernel(int n, int ctok, int D, int rows_cta, int splits, const KSource ks,
                  const uint16_t *__restrict__ vrows, const float *__restrict__ q, float *__restrict__ out,
                  float *__restrict__ part, unsigned *__restrict__ ticket) {
    constexpr int RB = AttnBatch<G>::RB;
    extern __shared__ __align__(16) unsigned char asmem_raw[];
    AttnHeader &sm = *reinterpret_cast<AttnHeader *>(asmem_raw);
    const AttnLayout lay = attn_smem_layout(G, 0, D, splits);
    const int s = blockIdx.x, u = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i_begin = s * rows_cta;
    const int R = max(0, min(n, i_begin + rows_cta) - i_begin);
    const float scale = 1.0f / sqrtf((float)D);
    float m_h[G], l_h[G], o_h[G][4], qv[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_h[h] = -CUDART_INF_F;
        l_h[h] = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o_h[h][e] = 0.0f;
            const int j = kVec ? 4 * lane + e : lane + 32 * e;
            qv[h][e] = (j < D) ? q[((size_t)u * G + h) * D + j] : 0.0f;
        }
    }
    float *pb = sm.pbuf[warp];
    for (int r0 = warp * RB; r0 < R; r0 += kWarps * RB) {
        unsigned mask[RB];
        int ti[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            mask[r] = (r0 + r < R) ? (1u << G) - 1u : 0u;
            ti[r] = i_begin + r0 + r;
        }
        attn_batch<G, kVec, false>(mask, ti, ks, vrows, u, (size_t)u * ctok, D, scale, qv, m_h, l_h, o_h, pb);
    }
    attn_finish<G, kVec>(sm, asmem_raw, lay, D, s, u, splits, m_h, l_h, o_h, out, part, ticket);
}

int launch_dense_attn(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows, const float *q,
                      float *out, void *ws, cudaStream_t st) {
    const AttnWorkspace wl = dense_workspace_layout(s);
    char *w = (char *)ws;
    float *part = (float *)(w + wl.part_off);
    unsigned *ticket = (unsigned *)(w + wl.ticket_off);
    if (s.units > 65535) { set_error("dense_attn: too many units for one launch"); return FATHOM_EINVAL; }
    const size_t smem = attn_smem_layout(s.G, 0, s.D, wl.splits).total;
    const bool vec = s.D == 128 && ((uintptr_t)krows % 8 == 0) && ((uintptr_t)vrows % 8 == 0);
    const dim3 grid(wl.splits, s.units);
    const KSource ks{krows, nullptr, nullptr, 0};
#define FATHOM_DENSE_LAUNCH(GG, VV)                                                                       \
    do {                                                                                                  \
        ensure_smem(dense_attn_kernel<GG, VV>, smem);                                                     \
        dense_attn_kernel<GG, VV><<<grid, NA, smem, st>>>(s.n, cap_tokens(s), s.D, wl.rows, wl.splits, ks, \
                                                          vrows, q, out, part, ticket);                   \
    } while (0)
    switch (s.G * 2 + (vec ? 1 : 0)) {
        case 2: FATHOM_DENSE_LAUNCH(1, false); break;
        case 3: FATHOM_DENSE_LAUNCH(1, true); break;
        case 4: FATHOM_DENSE_LAUNCH(2, false); break;
        case 5: FATHOM_DENSE_LAUNCH(2, true); break;
        case 8: FATHOM_DENSE_LAUNCH(4, false); break;
        case 9: FATHOM_DENSE_LAUNCH(4, true); break;
        case 16: FATHOM_DENSE_LAUNCH(8, false); break;
        case 17: FATHOM_DENSE_LAUNCH(8, true); break;
        default: set_error("dense_attn: unsupported G=%d", s.G); return FATHOM_EINVAL;
    }
#undef FATHOM_DENSE_LAUNCH
    return launch_status("dense_attn_kernel");
}

static int launch_sparse_attn_src(const fathom_shape &s, const KSource &ks, const uint16_t *vrows,
                                  const float *q, const int32_t *idx, float *out, void *ws, cudaStream_t st);

int launch_sparse_attn(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows,
                       const float *q, const int32_t *idx, float *out, void *ws, cudaStream_t st) {
    return launch_sparse_attn_src(s, KSource{krows, nullptr, nullptr, 0}, vrows, q, idx, out, ws, st);
}

int launch_sparse_attn_planes(const fathom_shape &s, const uint64_t *planes, const uint16_t *scales,
                              const uint16_t *vrows, const float *q, const int32_t *idx, float *out, void *ws,
                              cudaStream_t st) {
    return launch_sparse_attn_src(s, KSource{nullptr, planes, scales, cap_blocks(s)}, vrows, q, idx, out, ws, st);
}

static int launch_sparse_attn_src(const fathom_shape &s, const KSource &ks, const uint16_t *vrows,
                                  const float *q, const int32_t *idx, float *out, void *ws, cudaStream_t st) {
    const bool planes = ks.planes != nullptr;
    const AttnWorkspace wl = attn_workspace_layout(s);
    char *w = (char *)ws;
    float *part = (float *)(w + wl.part_off);
    unsigned *ticket = (unsigned *)(w + wl.ticket_off);
    const bool vec = s.D == 128 && (planes || (uintptr_t)ks.rows % 8 == 0) && ((uintptr_t)vrows % 8 == 0);
    // One head per grid row: each (unit, head) attends its own list with one dot
    // product per fetched row; a row kept by several heads (about a tenth of them) is
    // read once per head.  Faster for rows in HBM (a 256-unit layer: 72 against 113
    // us) and in pinned host memory (an 8-unit 1M-token layer: 54 against 60-73 us),
    // where the union form's G dot products per row delayed the next rows' loads.  The
    // union form (every kept row fetched once for all G heads) stays for keys rebuilt
    // from the store, whose rebuild costs more than the arithmetic, and for calls
    // with more than 65535 (unit, head) pairs.
    const bool per_head = !planes && s.G > 1 && (long long)s.units * s.G <= 65535;
    const int gg = per_head ? 1 : s.G;
    const int units = per_head ? s.units * s.G : s.units;
    const int rows = per_head ? wl.ph_rows : wl.rows;
    const int splits = per_head ? wl.ph_splits : wl.splits;
    const int hdiv = per_head ? s.G : 1;
    if (units > 65535) { set_error("sparse_attn: too many units for one launch"); return FATHOM_EINVAL; }
    const size_t smem = attn_smem_layout(gg, s.k, s.D, splits).total;
    const int cph = (s.k + rows - 1) / rows;   // CTAs per head
    const dim3 grid(splits, units);
#define FATHOM_ATTN_LAUNCH(GG, VV)                                                                        \
    do {                                                                                                  \
        if (planes) {                                                                                     \
            ensure_smem(attn_kernel<GG, VV, true>, smem);                                                 \
            le = launch_pdl(attn_kernel<GG, VV, true>, grid, dim3(NA), smem, st, s.n, cap_tokens(s), s.D, s.k, \
                            rows, cph, splits, hdiv, ks, vrows, q, idx, out, part, ticket);               \
        } else {                                                                                          \
            ensure_smem(attn_kernel<GG, VV, false>, smem);                                                \
            le = launch_pdl(attn_kernel<GG, VV, false>, grid, dim3(NA), smem, st, s.n, cap_tokens(s), s.D,  \
                            s.k, rows, cph, splits, hdiv, ks, vrows, q, idx, out, part, ticket);          \
        }                                                                                                 \
    } while (0)
    cudaError_t le = cudaSuccess;
    switch (gg * 2 + (vec ? 1 : 0)) {
        case 2: FATHOM_ATTN_LAUNCH(1, false); break;
        case 3: FATHOM_ATTN_LAUNCH(1, true); break;
        case 4: FATHOM_ATTN_LAUNCH(2, false); break;
        case 5: FATHOM_ATTN_LAUNCH(2, true); break;
        case 8: FATHOM_ATTN_LAUNCH(4, false); break;
        case 9: FATHOM_ATTN_LAUNCH(4, true); break;
        case 16: FATHOM_ATTN_LAUNCH(8, false); break;
        case 17: FATHOM_ATTN_LAUNCH(8, true); break;
        default: set_error("sparse_attn: unsupported G=%d", s.G); return FATHOM_EINVAL;
    }
#undef FATHOM_ATTN_LAUNCH
    if (le != cudaSuccess) { set_error("attn_kernel: %s", cudaGetErrorString(le)); return FATHOM_ECUDA; }
    return launch_status("attn_kernel");
}

FATHOM_DEBUG_READER(debug_read_attn)

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot hand the library a workspace
// of their own: a host framework that owns every byte of device memory and
// forbids plug-ins from calling cudaMalloc (it would also synchronise the
// device and fragment the framework's pool), or a latency-critical decode loop
// that must not allocate at all.  For them the scratch (partial softmax
// states and per-unit tickets) lives in this file-scope device array, which
// every GPU that loads the library keeps until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

// The array's device address on the current device.  In host code the symbol
// is only a host-side stand-in, so the address is looked up with the device
// current, on every call: the lookup is a host-side query, and a cached address
// would go stale after cudaDeviceReset or under another primary context.  The
// first lookup on a device may load the library's device code there.
static void *noalloc_scratch_ptr(int *status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("sparse_attn_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        *status = FATHOM_ECUDA;
        return nullptr;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || !p) {
        set_error("sparse_attn_noalloc: cudaGetSymbolAddress on device %d: %s", dev, cudaGetErrorString(e));
        *status = FATHOM_ECUDA;
        return nullptr;
    }
    *status = FATHOM_OK;
    return p;
}

int launch_sparse_attn_noalloc(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows,
                               const float *q, const int32_t *idx, float *out, cudaStream_t st) {
    const AttnWorkspace wl = attn_workspace_layout(s);
    if (wl.total > kNoAllocScratchBytes) {
        set_error("sparse_attn_noalloc: this shape needs %zu bytes of scratch, more than the "
                  "library's fixed %zu (use fathom_sparse_attn with a workspace)",
                  wl.total, kNoAllocScratchBytes);
        return FATHOM_EINVAL;
    }
    int rc = FATHOM_OK;
    char *scratch = (char *)noalloc_scratch_ptr(&rc);
    if (rc) return rc;
    // the tickets must start at zero; the partial states are written before they are read
    cudaError_t e = cudaMemsetAsync(scratch + wl.ticket_off, 0, wl.total - wl.ticket_off, st);
    if (e != cudaSuccess) {
        set_error("sparse_attn_noalloc: cudaMemsetAsync: %s", cudaGetErrorString(e));
        return FATHOM_ECUDA;
    }
    return launch_sparse_attn(s, krows, vrows, q, idx, out, scratch, st);
}

}  // namespace fathom

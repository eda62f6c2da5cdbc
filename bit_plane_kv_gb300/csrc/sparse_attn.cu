// sparse_attn.cu -- exact attention over the winners (Fathom §1 / §3.1: the
// union of the G heads' winners, k_union <= G k rows, is fetched once at full
// precision; §2: each head attends exactly over its own selected set, with no
// mass redistribution for the rest).
//
// Grid: (G * ceil(k / kAttnRows), units).  A CTA takes a slice of one head's
// sorted kept list and handles the rows that head owns (the first head, in
// order, that lists the token), so the union of the heads' winners is fetched
// exactly once; a row's head mask comes from binary searches in the other
// lists.  Each warp keeps several rows in flight (K and V, bf16), computes
// q_h . k / sqrt(D) for the heads in the row's mask and keeps an online
// softmax state (running max, sum, weighted V) per head.  Warp states are
// merged per CTA and written to the workspace; the last CTA of the unit (an
// atomic ticket, no waiting) merges the splits and writes o_h.
#include <mutex>

#include "fathom_internal.cuh"

namespace fathom {

constexpr int NA = kAttnThreads;
constexpr int kWarps = NA / 32;

// Shared memory: a fixed header, then wo[warps][G][D] floats and the G
// index lists (G * k ints), laid out by attn_smem_layout.
struct AttnHeader {
    int is_last;
    float wm[kWarps][FATHOM_MAX_G];
    float wl[kWarps][FATHOM_MAX_G];
};

struct AttnLayout {
    size_t wo, lists, merge, total;
};

// wo[warps][G][D] floats, lists[G * k] ints, merge[splits][D + 2] floats (one head
// of the final combine at a time)
__host__ __device__ inline AttnLayout attn_smem_layout(int G, int k, int D) {
    AttnLayout L;
    const int splits = G * ((k + kAttnRows - 1) / kAttnRows);
    L.wo = (sizeof(AttnHeader) + 15) & ~(size_t)15;
    L.lists = L.wo + (size_t)kWarps * G * D * sizeof(float);
    L.merge = (L.lists + (size_t)G * k * sizeof(int) + 15) & ~(size_t)15;
    L.total = (L.merge + (size_t)splits * (D + 2) * sizeof(float) + 15) & ~(size_t)15;
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

constexpr int kRowsInFlight = 8;   // rows a warp loads before using them

// Grid: (G * chunks_per_head, units).  CTA (h, c) takes entries [c R, c R + R)
// of head h's sorted list and handles the rows that h owns, i.e. that no lower
// head lists: every row of the union is fetched exactly once.  The row's head
// mask (which heads attend to it) comes from binary searches in the other
// heads' lists.  Lane l holds channels 4l .. 4l+3 (D = 128: one 8-byte load of
// K and one of V per row); other D take the general path with channel
// j = l + 32 e.
template <int G, bool kVec>
__global__ void __launch_bounds__(NA, 2)
attn_kernel(int n, int D, int k, int cph, int splits, const uint16_t *__restrict__ krows,
            const uint16_t *__restrict__ vrows, const float *__restrict__ q,
            const int32_t *__restrict__ topk, float *__restrict__ out, float *__restrict__ part,
            unsigned *__restrict__ ticket) {
    extern __shared__ __align__(16) unsigned char asmem_raw[];
    AttnHeader &sm = *reinterpret_cast<AttnHeader *>(asmem_raw);
    const AttnLayout lay = attn_smem_layout(G, k, D);
    float *wo = reinterpret_cast<float *>(asmem_raw + lay.wo);          // [warp][h][D]
    int *lists = reinterpret_cast<int *>(asmem_raw + lay.lists);
    const int s = blockIdx.x, u = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int GK = G * k;
    const int hown = s / cph;
    const int e_begin = (s % cph) * kAttnRows;
    const int e_end = min(k, e_begin + kAttnRows);

    for (int e = tid; e < GK; e += NA) lists[e] = topk[(size_t)u * GK + e];
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
    const int *own = lists + (size_t)hown * k;
    for (int e0 = e_begin + warp * kRowsInFlight; e0 < e_end; e0 += kWarps * kRowsInFlight) {
        unsigned mask[kRowsInFlight];
        uint2 kp[kRowsInFlight], vp[kRowsInFlight];        // bf16 pairs, unpacked at use
        float kv[kRowsInFlight][4], vv[kRowsInFlight][4];  // general path only
#pragma unroll
        for (int r = 0; r < kRowsInFlight; ++r) {
            const int e = e0 + r;
            int i = -1;
            unsigned m = 0;
            if (e < e_end) {
                i = own[e];
                m = 1u << hown;
                for (int h2 = 0; h2 < G; ++h2) {
                    if (h2 == hown) continue;
                    if (contains(lists + (size_t)h2 * k, k, i)) {
                        if (h2 < hown) { m = 0; break; }   // a lower head owns this row
                        m |= 1u << h2;
                    }
                }
                if (i < 0 || i >= n) m = 0;                 // not a token of this unit
            }
            mask[r] = m;
            const uint16_t *kr = krows + ((size_t)u * n + (m ? i : 0)) * D;
            const uint16_t *vr = vrows + ((size_t)u * n + (m ? i : 0)) * D;
            if (kVec) {
                kp[r] = m ? __ldg(reinterpret_cast<const uint2 *>(kr) + lane) : make_uint2(0u, 0u);
                vp[r] = m ? __ldg(reinterpret_cast<const uint2 *>(vr) + lane) : make_uint2(0u, 0u);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = lane + 32 * c;
                    const bool ok = m && j < D;
                    kv[r][c] = ok ? __uint_as_float(((uint32_t)__ldg(kr + j)) << 16) : 0.0f;
                    vv[r][c] = ok ? __uint_as_float(((uint32_t)__ldg(vr + j)) << 16) : 0.0f;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsInFlight; ++r) {
            if (!mask[r]) continue;                         // warp-uniform
            float kk[4], vx[4];
            if (kVec) {
                kk[0] = bf16lo(kp[r].x); kk[1] = bf16hi(kp[r].x); kk[2] = bf16lo(kp[r].y); kk[3] = bf16hi(kp[r].y);
                vx[0] = bf16lo(vp[r].x); vx[1] = bf16hi(vp[r].x); vx[2] = bf16lo(vp[r].y); vx[3] = bf16hi(vp[r].y);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) { kk[c] = kv[r][c]; vx[c] = vv[r][c]; }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (!((mask[r] >> h) & 1u)) continue;
                float d = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) d = fmaf(qv[h][c], kk[c], d);
#pragma unroll
                for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                const float logit = d * scale;
                const float mn = fmaxf(m_h[h], logit);
                const float corr = expf(m_h[h] - mn);
                const float p = expf(logit - mn);
                l_h[h] = l_h[h] * corr + p;
#pragma unroll
                for (int c = 0; c < 4; ++c) o_h[h][c] = o_h[h][c] * corr + p * vx[c];
                m_h[h] = mn;
            }
        }
    }
    // ---- merge warps
#pragma unroll
    for (int h = 0; h < G; ++h) {
        if (lane == 0) { sm.wm[warp][h] = m_h[h]; sm.wl[warp][h] = l_h[h]; }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = kVec ? 4 * lane + c : lane + 32 * c;
            if (j < D) wo[((size_t)warp * G + h) * D + j] = o_h[h][c];
        }
    }
    __syncthreads();
    float *pp = part + ((size_t)u * splits + s) * G * (D + 2);
    for (int e = tid; e < G * (D + 2); e += NA) {
        const int h = e / (D + 2), c = e % (D + 2);
        float M = -CUDART_INF_F;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][h]);
        float acc = 0.0f;
        if (c == 0) acc = M;
        else {
            for (int w = 0; w < kWarps; ++w) {
                const float f = (sm.wm[w][h] == -CUDART_INF_F) ? 0.0f : expf(sm.wm[w][h] - M);
                acc += f * (c == 1 ? sm.wl[w][h] : wo[((size_t)w * G + h) * D + (c - 2)]);
            }
        }
        pp[e] = acc;
    }
    // ---- last CTA of the unit merges the splits
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
    float *mg = reinterpret_cast<float *>(asmem_raw + lay.merge);   // [splits][D + 2], one head
    for (int h = 0; h < G; ++h) {
        // all of the head's partial states in one round of independent loads
        for (int e = tid; e < splits * (D + 2); e += NA) {
            const int sp = e / (D + 2), c = e % (D + 2);
            mg[e] = __ldcg(p0 + ((size_t)sp * G + h) * (D + 2) + c);
        }
        __syncthreads();
        for (int j = tid; j < D; j += NA) {
            float M = -CUDART_INF_F;
            for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, mg[sp * (D + 2)]);
            float L = 0.0f, O = 0.0f;
            for (int sp = 0; sp < splits; ++sp) {
                const float ms = mg[sp * (D + 2)];
                if (ms == -CUDART_INF_F) continue;
                const float f = expf(ms - M);
                L += f * mg[sp * (D + 2) + 1];
                O += f * mg[sp * (D + 2) + 2 + j];
            }
            out[((size_t)u * G + h) * D + j] = O / L;
        }
        __syncthreads();
    }
    if (tid == 0) ticket[u] = 0u;   // ready for the next call
}

int launch_sparse_attn(const fathom_shape &s, const uint16_t *krows, const uint16_t *vrows,
                       const float *q, const int32_t *idx, float *out, void *ws, cudaStream_t st) {
    const AttnWorkspace wl = attn_workspace_layout(s);
    char *w = (char *)ws;
    float *part = (float *)(w + wl.part_off);
    unsigned *ticket = (unsigned *)(w + wl.ticket_off);
    if (s.units > 65535) { set_error("sparse_attn: too many units for one launch"); return FATHOM_EINVAL; }
    const size_t smem = attn_smem_layout(s.G, s.k, s.D).total;
    const int cph = (s.k + kAttnRows - 1) / kAttnRows;   // CTAs per head
    const bool vec = s.D == 128 && ((uintptr_t)krows % 8 == 0) && ((uintptr_t)vrows % 8 == 0);
    const dim3 grid(wl.splits, s.units);
#define FATHOM_ATTN_LAUNCH(GG, VV)                                                               \
    do {                                                                                         \
        ensure_smem(attn_kernel<GG, VV>, smem);                                                  \
        attn_kernel<GG, VV><<<grid, NA, smem, st>>>(s.n, s.D, s.k, cph, wl.splits, krows, vrows, \
                                                    q, idx, out, part, ticket);                  \
    } while (0)
    switch (s.G * 2 + (vec ? 1 : 0)) {
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
    return launch_status("attn_kernel");
}

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

// The array's device address, looked up once per device with that device
// current (in host code the symbol is only a host-side stand-in).
static void *noalloc_scratch_ptr(int *status) {
    static std::mutex mu;
    static void *ptrs[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        set_error("sparse_attn_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        *status = FATHOM_ECUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p) {
            set_error("sparse_attn_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            *status = FATHOM_ECUDA;
            return nullptr;
        }
        ptrs[dev] = p;
    }
    *status = FATHOM_OK;
    return ptrs[dev];
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

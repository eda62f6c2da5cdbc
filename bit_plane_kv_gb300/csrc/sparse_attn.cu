// sparse_attn.cu -- exact attention over the winners (Fathom §1 / §3.1: the
// union of the G heads' winners, k_union <= G k rows, is fetched once at full
// precision; §2: each head attends exactly over its own selected set, with no
// mass redistribution for the rest).
//
// Grid: (splits, units).  Every CTA rebuilds the unit's union in shared
// memory from the G sorted index lists (an entry is owned by the first head
// that lists it; its head mask comes from binary searches in the other
// lists), then takes a slice of kAttnRows union rows.  Each warp streams rows
// (K and V, bf16, loaded once for all heads that selected the row), computes
// q_h . k / sqrt(D) for the heads in the row's mask and keeps an online
// softmax state (running max, sum, weighted V) per head.  Warp states are
// merged per CTA and written to the workspace; the last CTA of the unit (an
// atomic ticket, no waiting) merges the splits and writes o_h.
#include "fathom_internal.cuh"

namespace fathom {

constexpr int NA = kAttnThreads;
constexpr int kWarps = NA / 32;

// Shared memory: a fixed header, then wo[warps][G][D] floats, lists[G*k] and
// uidx[G*k] ints and umask[G*k] bytes, laid out by attn_smem_layout.
struct AttnHeader {
    int wsum[kWarps];
    int is_last;
    float wm[kWarps][FATHOM_MAX_G];
    float wl[kWarps][FATHOM_MAX_G];
};

struct AttnLayout {
    size_t wo, lists, uidx, umask, total;
};

__host__ __device__ inline AttnLayout attn_smem_layout(int G, int k, int D) {
    AttnLayout L;
    L.wo = (sizeof(AttnHeader) + 15) & ~(size_t)15;
    L.lists = L.wo + (size_t)kWarps * G * D * sizeof(float);
    L.uidx = L.lists + (size_t)G * k * sizeof(int);
    L.umask = L.uidx + (size_t)G * k * sizeof(int);
    L.total = (L.umask + (size_t)G * k + 15) & ~(size_t)15;
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

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__global__ void __launch_bounds__(NA)
attn_kernel(int n, int D, int G, int k, int splits, const uint16_t *__restrict__ krows,
            const uint16_t *__restrict__ vrows, const float *__restrict__ q,
            const int32_t *__restrict__ topk, float *__restrict__ out, float *__restrict__ part,
            unsigned *__restrict__ ticket) {
    extern __shared__ __align__(16) unsigned char asmem_raw[];
    AttnHeader &sm = *reinterpret_cast<AttnHeader *>(asmem_raw);
    const AttnLayout lay = attn_smem_layout(G, k, D);
    float *wo = reinterpret_cast<float *>(asmem_raw + lay.wo);          // [warp][h][D]
    int *lists = reinterpret_cast<int *>(asmem_raw + lay.lists);
    int *uidx = reinterpret_cast<int *>(asmem_raw + lay.uidx);
    unsigned char *umask = asmem_raw + lay.umask;
    const int s = blockIdx.x, u = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int GK = G * k;

    for (int e = tid; e < GK; e += NA) lists[e] = topk[(size_t)u * GK + e];
    __syncthreads();

    // ---- union: entry e = (h, r) is owned if no lower head lists the same token
    // pass 1: counts per warp (entries processed in chunks of NA, in order)
    int running = 0;
    for (int e0 = 0; e0 < GK; e0 += NA) {
        const int e = e0 + tid;
        bool own = false;
        unsigned char mask = 0;
        int x = 0;
        if (e < GK) {
            const int h = e / k;
            x = lists[e];
            own = true;
            mask = (unsigned char)(1u << h);
            for (int h2 = 0; h2 < G; ++h2) {
                if (h2 == h) continue;
                if (contains(lists + h2 * k, k, x)) {
                    mask |= (unsigned char)(1u << h2);
                    if (h2 < h) own = false;
                }
            }
        }
        const unsigned bal = __ballot_sync(0xffffffffu, own);
        if (lane == 0) sm.wsum[warp] = __popc(bal);
        __syncthreads();
        int before = running;
        for (int w = 0; w < warp; ++w) before += sm.wsum[w];
        int chunk_total = 0;
        for (int w = 0; w < kWarps; ++w) chunk_total += sm.wsum[w];
        if (own) {
            const int pos = before + __popc(bal & ((1u << lane) - 1u));
            uidx[pos] = x;
            umask[pos] = mask;
        }
        running += chunk_total;
        __syncthreads();
    }
    const int nu = running;

    // ---- this CTA's slice of union rows
    const int r_begin = s * kAttnRows;
    const int r_end = min(nu, r_begin + kAttnRows);
    const float scale = 1.0f / sqrtf((float)D);   // 1/sqrt(D), correctly rounded
    const int EPL = (D + 31) / 32;          // elements per lane (<= 4)
    float m_h[FATHOM_MAX_G], l_h[FATHOM_MAX_G], o_h[FATHOM_MAX_G][4];
    float qv[FATHOM_MAX_G][4];
#pragma unroll
    for (int h = 0; h < FATHOM_MAX_G; ++h) {
        m_h[h] = -CUDART_INF_F;
        l_h[h] = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o_h[h][e] = 0.0f;
            const int j = lane + 32 * e;
            qv[h][e] = (h < G && e < EPL && j < D) ? q[((size_t)u * G + h) * D + j] : 0.0f;
        }
    }
    for (int rr = r_begin + warp; rr < r_end; rr += kWarps) {
        const int i = uidx[rr];
        if (i < 0 || i >= n) continue;    // not a token of this unit: contributes nothing
        const unsigned mask = umask[rr];
        const uint16_t *kr = krows + ((size_t)u * n + i) * D;
        const uint16_t *vr = vrows + ((size_t)u * n + i) * D;
        float kv[4], vv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = lane + 32 * e;
            const bool ok = e < EPL && j < D;
            kv[e] = ok ? bf16f(__ldg(kr + j)) : 0.0f;
            vv[e] = ok ? bf16f(__ldg(vr + j)) : 0.0f;
        }
#pragma unroll
        for (int h = 0; h < FATHOM_MAX_G; ++h) {
            if (h >= G || !((mask >> h) & 1u)) continue;
            float d = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) d = fmaf(qv[h][e], kv[e], d);
#pragma unroll
            for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            const float logit = d * scale;
            const float mn = fmaxf(m_h[h], logit);
            const float corr = expf(m_h[h] - mn);
            const float p = expf(logit - mn);
            l_h[h] = l_h[h] * corr + p;
#pragma unroll
            for (int e = 0; e < 4; ++e) o_h[h][e] = o_h[h][e] * corr + p * vv[e];
            m_h[h] = mn;
        }
    }
    // ---- merge warps
#pragma unroll
    for (int h = 0; h < FATHOM_MAX_G; ++h) {
        if (h >= G) continue;
        if (lane == 0) { sm.wm[warp][h] = m_h[h]; sm.wl[warp][h] = l_h[h]; }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = lane + 32 * e;
            if (e < EPL && j < D) wo[((size_t)warp * G + h) * D + j] = o_h[h][e];
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
    for (int e = tid; e < G * D; e += NA) {
        const int h = e / D, j = e % D;
        float M = -CUDART_INF_F;
        for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, __ldcg(p0 + ((size_t)sp * G + h) * (D + 2)));
        float L = 0.0f, O = 0.0f;
        for (int sp = 0; sp < splits; ++sp) {
            const float *ph = p0 + ((size_t)sp * G + h) * (D + 2);
            const float ms = __ldcg(ph);
            if (ms == -CUDART_INF_F) continue;
            const float f = expf(ms - M);
            L += f * __ldcg(ph + 1);
            O += f * __ldcg(ph + 2 + j);
        }
        out[((size_t)u * G + h) * D + j] = O / L;
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
    ensure_smem(attn_kernel, smem);
    attn_kernel<<<dim3(wl.splits, s.units), NA, smem, st>>>(s.n, s.D, s.G, s.k, wl.splits, krows,
                                                           vrows, q, idx, out, part, ticket);
    return launch_status("attn_kernel");
}

}  // namespace fathom

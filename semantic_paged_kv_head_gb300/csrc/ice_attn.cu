// Paged sparse GQA attention over the selected pages ("IceCache", Figure 2
// step 3: all tokens of the selected pages attend with q).
//
// One 256-thread block per unit. Warp w takes pages w, w + 8, ... of the
// unit's list; within a warp two tokens are processed at a time, 16 lanes per
// token, each lane owning 8 of the 128 dimensions (one 16-byte load per K or V
// row for bf16). All rows of a page chunk are requested before any is used.
// Scores for the G query heads of the group run through an fp32 online
// softmax per half-warp; the half-warps, then the warps, are merged in a fixed
// order in shared memory, so the result does not depend on scheduling.
#include "ice_internal.cuh"

namespace ice {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTokUnr = 4;  // token pairs requested ahead per warp (8 rows of K and V)
static_assert(2 * kAttnThreads >= 512, "two list slots per thread cover the longest list");

// 8 consecutive elements as floats.
template <typename T> struct Row8;
template <> struct Row8<__nv_bfloat16> {
    uint4 r;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { r = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ void get(float (&x)[8]) const {
        const unsigned a[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(a[k] << 16);
            x[2 * k + 1] = __uint_as_float(a[k] & 0xFFFF0000u);
        }
    }
};
template <> struct Row8<float> {
    float4 r0, r1;
    __device__ __forceinline__ void load(const float* p) {
        r0 = __ldg(reinterpret_cast<const float4*>(p));
        r1 = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void get(float (&x)[8]) const {
        x[0] = r0.x; x[1] = r0.y; x[2] = r0.z; x[3] = r0.w;
        x[4] = r1.x; x[5] = r1.y; x[6] = r1.z; x[7] = r1.w;
    }
};

template <typename T, int G>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_kernel(IndexView v, const T* __restrict__ q,
                                                              const int32_t* __restrict__ page_ids,
                                                              const int32_t* __restrict__ n_pages,
                                                              int page_stride, T* __restrict__ out) {
    __shared__ float s_part[kAttnWarps][G][kD + 2];  // per-warp {acc[kD], m, l}
    __shared__ int s_pid[512];
    __shared__ int s_cnt[512];
    pdl_wait_then_release();
    const int u = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = v.P;

    // ---- page list and counts, all pages at once --------------------------------------
    // the list length, the allocated page count and every slot of the list's row are
    // read together (page_stride <= 2 * kAttnThreads), then the counts of the pages
    int np = n_pages[u];
    const int nalloc = v.next_id[v.ul(u, 0)];
    int pids[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = tid + k * kAttnThreads;
        pids[k] = i < page_stride ? page_ids[(long long)u * page_stride + i] : -1;
    }
    if (np < 0 || np > page_stride) {
        if (tid == 0) set_status(v.status, ICE_ERR_BOUNDS);
        np = np < 0 ? 0 : page_stride;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = tid + k * kAttnThreads;
        if (i >= np) continue;
        const int pid = pids[k];
        int c = 0;
        if (pid < 0 || pid >= nalloc || pid >= v.C) {
            set_status(v.status, ICE_ERR_BOUNDS);
        } else {
            c = v.list_cnt[v.leaf_base(u, 0) + pid];
            c = c < 0 ? 0 : (c > P ? P : c);
        }
        s_pid[i] = pid;
        s_cnt[i] = c;
    }

    // ---- query registers: half-warp lane hl owns dims [8 hl, 8 hl + 8) -----------------
    const int hl = lane & 15, half = lane >> 4;
    float qr[G][8];
    {
        const T* qu = q + (long long)u * G * kD;
        const float sc = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            Row8<T> r;
            r.load(qu + (long long)h * kD + 8 * hl);
            float x[8];
            r.get(x);
#pragma unroll
            for (int k = 0; k < 8; ++k) qr[h][k] = x[k] * sc;
        }
    }
    __syncthreads();

    float m[G], lsum[G], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[h][k] = 0.0f;
    }
    const T* pk = reinterpret_cast<const T*>(v.page_k);
    const T* pv = reinterpret_cast<const T*>(v.page_v);
    for (int pi = warp; pi < np; pi += kAttnWarps) {  // warp-uniform
        const int c = s_cnt[pi];
        if (c == 0) continue;
        const long long row0 = v.page_row(u, s_pid[pi], 0);
        for (int t0 = 0; t0 < c; t0 += 2 * kTokUnr) {
            Row8<T> kr[kTokUnr], vr[kTokUnr];
#pragma unroll
            for (int k = 0; k < kTokUnr; ++k) {
                const int t = t0 + 2 * k + half;
                if (t < c) {
                    kr[k].load(pk + (row0 + t) * kD + 8 * hl);
                    vr[k].load(pv + (row0 + t) * kD + 8 * hl);
                }
            }
#pragma unroll
            for (int k = 0; k < kTokUnr; ++k) {
                if (t0 + 2 * k >= c) break;  // warp-uniform
                const bool valid = t0 + 2 * k + half < c;
                float kx[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (valid) kr[k].get(kx);
                float s[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float a = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) a = fmaf(qr[h][i], kx[i], a);
                    a += __shfl_xor_sync(0xffffffffu, a, 1);
                    a += __shfl_xor_sync(0xffffffffu, a, 2);
                    a += __shfl_xor_sync(0xffffffffu, a, 4);
                    a += __shfl_xor_sync(0xffffffffu, a, 8);
                    s[h] = a;
                }
                if (valid) {
                    float vx[8];
                    vr[k].get(vx);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float mn = fmaxf(m[h], s[h]);
                        const float corr = exp2_approx(m[h] - mn);
                        const float p = exp2_approx(s[h] - mn);
                        lsum[h] = lsum[h] * corr + p;
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(p, vx[i], acc[h][i] * corr);
                        m[h] = mn;
                    }
                }
            }
        }
    }
    // merge the two half-warps (lane hl with lane hl + 16)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[h], 16);
        const float lo = __shfl_xor_sync(0xffffffffu, lsum[h], 16);
        const float mn = fmaxf(m[h], mo);
        const float ca = mn == -INFINITY ? 0.0f : exp2_approx(m[h] - mn);
        const float cb = mn == -INFINITY ? 0.0f : exp2_approx(mo - mn);
        lsum[h] = lsum[h] * ca + lo * cb;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float ao = __shfl_xor_sync(0xffffffffu, acc[h][i], 16);
            acc[h][i] = acc[h][i] * ca + ao * cb;
        }
        m[h] = mn;
    }
    if (half == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int i = 0; i < 8; ++i) s_part[warp][h][8 * hl + i] = acc[h][i];
            if (hl == 0) {
                s_part[warp][h][kD] = m[h];
                s_part[warp][h][kD + 1] = lsum[h];
            }
        }
    }
    __syncthreads();
    // ---- merge the warps in fixed order and write the output ----------------------------
    T* ou = out + (long long)u * G * kD;
    for (int e = tid; e < G * kD; e += kAttnThreads) {
        const int h = e / kD, dcol = e % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_part[w][h][kD]);
        float Lt = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float mw = s_part[w][h][kD];
                if (mw == -INFINITY) continue;
                const float cf = exp2_approx(mw - M);
                Lt = fmaf(s_part[w][h][kD + 1], cf, Lt);
                O = fmaf(s_part[w][h][dcol], cf, O);
            }
        }
        ou[e] = from_f<T>(Lt > 0.0f ? O / Lt : 0.0f);
    }
}

template <typename T>
static cudaError_t launch_attn_dt(const IndexView& v, const void* q, const int32_t* page_ids,
                                  const int32_t* n_pages, int page_stride, void* out,
                                  cudaStream_t s) {
    const T* qq = (const T*)q;
    T* oo = (T*)out;
    switch (v.G) {
        case 1: return launch_pdl(attn_kernel<T, 1>, dim3(v.U), dim3(kAttnThreads), 0, s, v, qq, page_ids, n_pages, page_stride, oo);
        case 2: return launch_pdl(attn_kernel<T, 2>, dim3(v.U), dim3(kAttnThreads), 0, s, v, qq, page_ids, n_pages, page_stride, oo);
        case 4: return launch_pdl(attn_kernel<T, 4>, dim3(v.U), dim3(kAttnThreads), 0, s, v, qq, page_ids, n_pages, page_stride, oo);
        case 8: return launch_pdl(attn_kernel<T, 8>, dim3(v.U), dim3(kAttnThreads), 0, s, v, qq, page_ids, n_pages, page_stride, oo);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn(const IndexView& v, const void* q, const int32_t* page_ids,
                        const int32_t* n_pages, int page_stride, void* out, cudaStream_t s) {
    if (v.dtype == ICE_BF16)
        return launch_attn_dt<__nv_bfloat16>(v, q, page_ids, n_pages, page_stride, out, s);
    return launch_attn_dt<float>(v, q, page_ids, n_pages, page_stride, out, s);
}

}  // namespace ice

// Paged sparse GQA attention over the selected pages ("IceCache", Figure 2
// step 3: all tokens of the selected pages attend with q).
//
// One thread-block cluster per unit; CTA r of the cluster owns pages
// [r*ppc, (r+1)*ppc) of the unit's page list. Each CTA
//  * stages the valid rows of its pages, K and V, global -> shared with
//    cp.async.bulk (one bulk copy per page and tensor) completing on one
//    mbarrier (bounded wait),
//  * computes scores for the G query heads of the group with 8 lanes per
//    token (16 dims per lane, 16-byte shared loads) and an fp32 online softmax,
//  * leaves its per-warp partials (running max, sum, weighted V) in shared
//    memory; CTA 0 merges the partials of all CTAs through distributed shared
//    memory and writes the output rows.
#include <cooperative_groups.h>

#include "ice_internal.cuh"

namespace cg = cooperative_groups;

namespace ice {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // bounded wait: 200 ms
constexpr unsigned long long kDebugWaitNs = 2ull * 1000 * 1000;  // forced-timeout test: 2 ms

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(unsigned dst, const void* src, unsigned bytes,
                                         unsigned bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Returns true once phase `parity` of the barrier has completed, false if it
// did not within `limit_ns` nanoseconds of wall time.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity,
                                          unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    for (int i = 0;; ++i) {
        unsigned done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 15) == 15 && global_ns() - t0 > limit_ns) return false;
        __nanosleep(i < 64 ? 20 : 200);
    }
}

// 16 consecutive elements as floats (two 16-byte loads for bf16, four for f32).
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float (&x)[16]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 w = q[h];
        const unsigned int a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[8 * h + 2 * k] = __uint_as_float(a[k] << 16);
            x[8 * h + 2 * k + 1] = __uint_as_float(a[k] & 0xFFFF0000u);
        }
    }
}
__device__ __forceinline__ void load16(const float* p, float (&x)[16]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float4 w = q[h];
        x[4 * h] = w.x;
        x[4 * h + 1] = w.y;
        x[4 * h + 2] = w.z;
        x[4 * h + 3] = w.w;
    }
}

template <typename T, int G>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(IndexView v, const T* __restrict__ q,
                                                           const int32_t* __restrict__ page_ids,
                                                           const int32_t* __restrict__ n_pages,
                                                           int page_stride, int ppc,
                                                           T* __restrict__ out) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bar_full;
    __shared__ __align__(8) unsigned long long bar_never;
    __shared__ int s_ntok;
    // partials: [warp][head] -> {m, l, acc[kD]}
    __shared__ float s_part[kAttnWarps][G][kD + 2];

    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int u = blockIdx.x / S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = v.P;
    constexpr int ROWB = kD * (int)sizeof(T);  // bytes per K or V row
    T* sk = reinterpret_cast<T*>(smem);
    T* sv = reinterpret_cast<T*>(smem + (size_t)ppc * P * ROWB);

    const unsigned bar = smem_addr(&bar_full);
    const unsigned bar_dbg = smem_addr(&bar_never);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_dbg, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ---- issue the page copies (thread 0): sizes first, then the copies ----------
    if (tid == 0) {
        int np = n_pages[u];
        if (np < 0 || np > page_stride) {
            set_status(v.status, ICE_ERR_BOUNDS);
            np = np < 0 ? 0 : page_stride;
        }
        const int first = rank * ppc, last = min(np, first + ppc);
        const int nalloc = v.next_id[v.ul(u, 0)];
        const int* cntp = v.list_cnt + v.leaf_base(u, 0);
        const int32_t* pl = page_ids + (long long)u * page_stride;
        const char* gk = reinterpret_cast<const char*>(v.page_k);
        const char* gv = reinterpret_cast<const char*>(v.page_v);
        unsigned rows = 0;
        for (int p = first; p < last; ++p) {
            const int pid = pl[p];
            if (pid < 0 || pid >= nalloc || pid >= v.C) {
                set_status(v.status, ICE_ERR_BOUNDS);
                continue;
            }
            const int c = cntp[pid];
            rows += (unsigned)(c < 0 ? 0 : (c > P ? P : c));
        }
        mbar_expect_tx(bar, 2u * rows * ROWB);  // also this phase's single arrival
        rows = 0;
        for (int p = first; p < last; ++p) {
            const int pid = pl[p];
            if (pid < 0 || pid >= nalloc || pid >= v.C) continue;
            int c = cntp[pid];
            c = c < 0 ? 0 : (c > P ? P : c);
            if (c == 0) continue;
            const long long row0 = v.page_row(u, pid, 0);
            bulk_g2s(smem_addr(sk) + rows * ROWB, gk + row0 * ROWB, (unsigned)c * ROWB, bar);
            bulk_g2s(smem_addr(sv) + rows * ROWB, gv + row0 * ROWB, (unsigned)c * ROWB, bar);
            rows += (unsigned)c;
        }
        s_ntok = (int)rows;
    }

    // ---- query registers: lane sub = lane & 7 owns dims [16 sub, 16 sub + 16) ----------
    const int sub = lane & 7, grp = lane >> 3;
    float qr[G][16];
    {
        const T* qu = q + (long long)u * G * kD;
        const float sc = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                float x[4];
                load4(qu + (long long)h * kD + 16 * sub + k, x);
#pragma unroll
                for (int z = 0; z < 4; ++z) qr[h][k + z] = x[z] * sc;
            }
    }
    __syncthreads();
    const int ntok = s_ntok;
    bool ok = true;
    if ((v.debug_flags & 1) && tid == 0) {
        // test hook: a barrier no one signals; the bounded wait must run out
        if (!mbar_wait(bar_dbg, 0, kDebugWaitNs)) set_status(v.status, ICE_ERR_TIMEOUT);
    }
    if (!mbar_wait(bar, 0, kWaitNs)) {
        ok = false;
        if (tid == 0) set_status(v.status, ICE_ERR_TIMEOUT);
        mbar_wait(bar, 0, kWaitNs);  // give copies still in flight one more bounded wait
    }

    // ---- scores + online softmax ----------------------------------------------------------
    float m[G], lsum[G], acc[G][16];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[h][k] = 0.0f;
    }
    if (ok) {
        // the trip count is uniform across the warp (full-mask shuffles inside);
        // a lane group whose token is past the end computes but does not update
        for (int t0 = warp * 4; t0 < ntok; t0 += kAttnWarps * 4) {
            const int t = t0 + grp;
            const bool valid = t < ntok;
            const int tr = valid ? t : t0;  // an in-range row for the idle groups
            float kv[16];
            load16(sk + (long long)tr * kD + 16 * sub, kv);
            float s[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float a = 0.0f;
#pragma unroll
                for (int k = 0; k < 16; ++k) a = fmaf(qr[h][k], kv[k], a);
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                a += __shfl_xor_sync(0xffffffffu, a, 4);
                s[h] = a;
            }
            if (valid) {
                float vv[16];
                load16(sv + (long long)t * kD + 16 * sub, vv);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float mn = fmaxf(m[h], s[h]);
                    const float corr = exp2f(m[h] - mn);
                    const float p = exp2f(s[h] - mn);
                    lsum[h] = lsum[h] * corr + p;
#pragma unroll
                    for (int k = 0; k < 16; ++k) acc[h][k] = fmaf(p, vv[k], acc[h][k] * corr);
                    m[h] = mn;
                }
            }
        }
    }
    // merge the 4 token groups of the warp (lanes sub, sub+8, sub+16, sub+24)
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[h], o);
            const float lo = __shfl_xor_sync(0xffffffffu, lsum[h], o);
            const float mn = fmaxf(m[h], mo);
            const float ca = mn == -INFINITY ? 0.0f : exp2f(m[h] - mn);
            const float cb = mn == -INFINITY ? 0.0f : exp2f(mo - mn);
            lsum[h] = lsum[h] * ca + lo * cb;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[h][k], o);
                acc[h][k] = acc[h][k] * ca + ao * cb;
            }
            m[h] = mn;
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int k = 0; k < 16; ++k) s_part[warp][h][16 * sub + k] = acc[h][k];
            if (sub == 0) {
                s_part[warp][h][kD] = m[h];
                s_part[warp][h][kD + 1] = lsum[h];
            }
        }
    }
    cluster.sync();
    // ---- CTA 0 merges all partials of the cluster ----------------------------------------
    if (rank == 0) {
        T* ou = out + (long long)u * G * kD;
        for (int e = tid; e < G * kD; e += kAttnThreads) {
            const int h = e / kD, dcol = e % kD;
            float M = -INFINITY;
            for (int r = 0; r < S; ++r) {
                const float* pr = cluster.map_shared_rank(&s_part[0][0][0], r);
                for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, pr[(w * G + h) * (kD + 2) + kD]);
            }
            float Lt = 0.0f, O = 0.0f;
            if (M != -INFINITY) {
                for (int r = 0; r < S; ++r) {
                    const float* pr = cluster.map_shared_rank(&s_part[0][0][0], r);
                    for (int w = 0; w < kAttnWarps; ++w) {
                        const float* pw = pr + (w * G + h) * (kD + 2);
                        const float mw = pw[kD];
                        if (mw == -INFINITY) continue;
                        const float c = exp2f(mw - M);
                        Lt = fmaf(pw[kD + 1], c, Lt);
                        O = fmaf(pw[dcol], c, O);
                    }
                }
            }
            ou[e] = from_f<T>(Lt > 0.0f ? O / Lt : 0.0f);
        }
    }
    cluster.sync();
}

template <typename T, int G>
static cudaError_t launch_attn_t(const IndexView& v, const void* q, const int32_t* page_ids,
                                 const int32_t* n_pages, int page_stride, void* out,
                                 cudaStream_t s) {
    // pages per CTA and CTAs per cluster (at most 8, the portable cluster size)
    int ppc = 4;
    if ((page_stride + ppc - 1) / ppc > 8) ppc = (page_stride + 7) / 8;
    const int S = max(1, (page_stride + ppc - 1) / ppc);
    const size_t bytes = (size_t)2 * ppc * v.P * kD * sizeof(T);
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<T, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(v.U * S), 1, 1);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<T, G>, v, (const T*)q, page_ids, n_pages,
                              page_stride, ppc, (T*)out);
}

template <typename T>
static cudaError_t launch_attn_dt(const IndexView& v, const void* q, const int32_t* page_ids,
                                  const int32_t* n_pages, int page_stride, void* out,
                                  cudaStream_t s) {
    switch (v.G) {
        case 1: return launch_attn_t<T, 1>(v, q, page_ids, n_pages, page_stride, out, s);
        case 2: return launch_attn_t<T, 2>(v, q, page_ids, n_pages, page_stride, out, s);
        case 4: return launch_attn_t<T, 4>(v, q, page_ids, n_pages, page_stride, out, s);
        case 8: return launch_attn_t<T, 8>(v, q, page_ids, n_pages, page_stride, out, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn(const IndexView& v, const void* q, const int32_t* page_ids,
                        const int32_t* n_pages, int page_stride, void* out, cudaStream_t s) {
    if (v.dtype == ICE_BF16)
        return launch_attn_dt<__nv_bfloat16>(v, q, page_ids, n_pages, page_stride, out, s);
    return launch_attn_dt<float>(v, q, page_ids, n_pages, page_stride, out, s);
}

// Pages per CTA the attention launch will use (host-side size checks).
int attn_pages_per_cta(int page_stride) {
    int ppc = 4;
    if ((page_stride + ppc - 1) / ppc > 8) ppc = (page_stride + 7) / 8;
    return ppc;
}

}  // namespace ice

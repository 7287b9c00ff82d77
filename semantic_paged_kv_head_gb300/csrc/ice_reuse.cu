// Reuse of a unit's page selection across decode steps ("IceCache" paper:
// the IceCache(r) variant, whose mechanism the paper does not describe).
//
// Reading taken here: a unit keeps the pages of its last selection for up to
// r further steps while the query codes (the 8-bit codes of the group query
// on every random direction of every composite, the same codes the selection
// computes first) stay exactly equal to the codes of the step that selected
// them. Any change of a code, r reuses in a row, or a unit with no selection
// yet, runs the selection again. This kernel takes that decision: one block
// per unit recomputes the query codes with the selection's fixed-order
// arithmetic, compares them with the stored codes, and updates the codes and
// the reuse age of the unit.
#include "ice_internal.cuh"

namespace ice {

namespace {

constexpr int kReuseThreads = kMaxL * kM * 32;  // one warp per direction

template <typename T, int G>
__global__ void __launch_bounds__(kReuseThreads) reuse_kernel(IndexView v, const T* __restrict__ q,
                                                              int r, unsigned char* __restrict__ codes,
                                                              int* __restrict__ age,
                                                              int32_t* __restrict__ reselect) {
    __shared__ int s_code[kMaxL * kM];
    const int u = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = v.L;
    // group query q_sel = ((q_0 + q_1) + q_2) + ..., lane holds elements 4 lane .. 4 lane + 3
    float qs[4];
    {
        const T* qu = q + (long long)u * G * kD;
        load4(qu + 4 * lane, qs);
#pragma unroll
        for (int h = 1; h < G; ++h) {
            float x[4];
            load4(qu + (long long)h * kD + 4 * lane, x);
#pragma unroll
            for (int k = 0; k < 4; ++k) qs[k] = __fadd_rn(qs[k], x[k]);
        }
    }
    // transformed query [q_sel / |q_sel|, 0] and its code on direction `warp`
    const float nq = warp_dot_fixed(qs, qs);
    float qt[4] = {0.f, 0.f, 0.f, 0.f};
    if (nq > 0.0f) {
        const float sn = __fsqrt_rn(nq);
#pragma unroll
        for (int k = 0; k < 4; ++k) qt[k] = __fdiv_rn(qs[k], sn);
    }
    if (warp < L * kM) {
        const float* ud = v.dirs + (long long)warp * kDirStride;
        float w[4];
        load4(ud + 4 * lane, w);
        const float p = __fmaf_rn(ud[kD], 0.0f, warp_dot_fixed(w, qt));
        if (lane == 0) s_code[warp] = quantise_code(p);
    }
    __syncthreads();
    if (tid == 0) {
        unsigned char* cu = codes + (long long)u * kMaxL * kM;
        bool same = true;
        for (int j = 0; j < L * kM; ++j) same = same && cu[j] == (unsigned char)s_code[j];
        const int a = age[u];  // < 0: no selection yet
        const bool keep = a >= 0 && a < r && same;
        if (keep) {
            age[u] = a + 1;
        } else {
            for (int j = 0; j < L * kM; ++j) cu[j] = (unsigned char)s_code[j];
            age[u] = 0;
        }
        reselect[u] = keep ? 0 : 1;
    }
}

template <typename T>
cudaError_t launch_reuse_dt(const IndexView& v, const void* q, int r, unsigned char* codes, int* age,
                            int32_t* reselect, cudaStream_t s) {
    const T* qq = static_cast<const T*>(q);
    switch (v.G) {
        case 1: reuse_kernel<T, 1><<<v.U, kReuseThreads, 0, s>>>(v, qq, r, codes, age, reselect); break;
        case 2: reuse_kernel<T, 2><<<v.U, kReuseThreads, 0, s>>>(v, qq, r, codes, age, reselect); break;
        case 4: reuse_kernel<T, 4><<<v.U, kReuseThreads, 0, s>>>(v, qq, r, codes, age, reselect); break;
        case 8: reuse_kernel<T, 8><<<v.U, kReuseThreads, 0, s>>>(v, qq, r, codes, age, reselect); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reuse(const IndexView& v, const void* q, int r, unsigned char* codes, int* age,
                         int32_t* reselect, cudaStream_t s) {
    if (v.dtype == ICE_BF16) return launch_reuse_dt<__nv_bfloat16>(v, q, r, codes, age, reselect, s);
    return launch_reuse_dt<float>(v, q, r, codes, age, reselect, s);
}

}  // namespace ice

// Union of the pages selected per query head (a variant of the selection:
// every query head of a group selects with its own query, and the group
// attends over the union of their pages). The union of unit u lists the pages
// of head 0 in its order, then the pages of head 1 not listed yet, and so on
// (first occurrence in head-major order).
#include "ice_internal.cuh"

namespace ice {

namespace {

constexpr int kUnionThreads = 128;

// One block per unit. head_ids [U][G][n_sel], head_n [U][G] -> ids [U][G*n_sel]
// (padded with -1), n [U]. G * n_sel <= 32 * kUnionThreads.
__global__ void __launch_bounds__(kUnionThreads) union_kernel(const int32_t* __restrict__ head_ids,
                                                             const int32_t* __restrict__ head_n,
                                                             int G, int n_sel,
                                                             int32_t* __restrict__ ids,
                                                             int32_t* __restrict__ n) {
    extern __shared__ int ent[];  // [G * n_sel] candidate entries, -1 = none
    __shared__ int s_part[kUnionThreads];
    const int u = blockIdx.x, tid = threadIdx.x;
    const int N = G * n_sel;
    for (int i = tid; i < N; i += kUnionThreads) {
        const int h = i / n_sel, k = i % n_sel;
        int c = head_n[(long long)u * G + h];
        c = c < 0 ? 0 : (c > n_sel ? n_sel : c);
        ent[i] = k < c ? head_ids[(long long)u * N + i] : -1;
    }
    __syncthreads();
    // thread t owns entries [t*per, (t+1)*per) (per <= 32): keeps those whose
    // page appears at no earlier index
    const int per = (N + kUnionThreads - 1) / kUnionThreads;
    const int lo = min(N, tid * per), hi = min(N, lo + per);
    unsigned keep = 0u;
    int mine = 0;
    for (int i = lo; i < hi; ++i) {
        const int p = ent[i];
        bool first = p >= 0;
        for (int j = 0; j < i && first; ++j) first = ent[j] != p;
        if (first) {
            keep |= 1u << (i - lo);
            ++mine;
        }
    }
    s_part[tid] = mine;
    __syncthreads();
    int base = 0;
    for (int t = 0; t < tid; ++t) base += s_part[t];
    int32_t* out = ids + (long long)u * N;
    for (int i = lo; i < hi; ++i)
        if ((keep >> (i - lo)) & 1u) out[base++] = ent[i];
    __syncthreads();
    if (tid == kUnionThreads - 1) {
        const int tot = base;
        n[u] = tot;
        s_part[0] = tot;
    }
    __syncthreads();
    for (int i = s_part[0] + tid; i < N; i += kUnionThreads) out[i] = -1;
}

}  // namespace

cudaError_t launch_union(int U, int G, int n_sel, const int32_t* head_ids, const int32_t* head_n,
                         int32_t* ids, int32_t* n, cudaStream_t s) {
    const size_t smem = (size_t)G * n_sel * sizeof(int);
    union_kernel<<<U, kUnionThreads, smem, s>>>(head_ids, head_n, G, n_sel, ids, n);
    return cudaGetLastError();
}

}  // namespace ice

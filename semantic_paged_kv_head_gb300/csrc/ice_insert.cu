// The insert kernel: one 128-thread block per unit inserts that unit's new
// token (see ice_insert.cuh).
#include "ice_insert.cuh"

namespace ice {

constexpr int kInsThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kInsThreads) insert_kernel(IndexView v, const T* __restrict__ knew,
                                                            const T* __restrict__ vnew) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_wait_then_release();
    const int u = blockIdx.x;
    insert_unit<T, kInsThreads>(v, u, knew + (long long)u * kD, vnew + (long long)u * kD, smem);
}

cudaError_t launch_insert(const IndexView& v, const void* k, const void* val, cudaStream_t s) {
    const size_t es = v.dtype == ICE_BF16 ? 2 : 4;
    const size_t bytes = (size_t)2 * (v.P + 1) * kD * es;
    if (v.dtype == ICE_BF16)
        return launch_pdl(insert_kernel<__nv_bfloat16>, dim3(v.U), dim3(kInsThreads), bytes, s, v,
                          (const __nv_bfloat16*)k, (const __nv_bfloat16*)val);
    return launch_pdl(insert_kernel<float>, dim3(v.U), dim3(kInsThreads), bytes, s, v, (const float*)k,
                      (const float*)val);
}

// Dynamic shared memory limit of the insert kernel (the staged rows of a
// split), set once at build so that inserts can be captured in CUDA graphs.
cudaError_t insert_prepare(int P, int dtype) {
    const size_t es = dtype == ICE_BF16 ? 2 : 4;
    const int bytes = (int)((size_t)2 * (P + 1) * kD * es);
    if (dtype == ICE_BF16)
        return cudaFuncSetAttribute(insert_kernel<__nv_bfloat16>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return cudaFuncSetAttribute(insert_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bytes);
}

}  // namespace ice

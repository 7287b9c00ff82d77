// Key codes without any allocation: the transform, projection and quantisation
// stage of the index build (squared norms, per-unit scale exponent, 8-bit codes
// of every key on every random direction, Morton keys), computed with scratch
// that lives in fixed-size device arrays of this file instead of memory
// obtained from cudaMalloc.
//
// Who needs this: code that must not allocate device memory while it runs, for
// example a serving loop that has handed all of the GPU's memory to its own
// pool allocator, or a latency-critical path where a cudaMalloc (which may
// synchronise the device) is not acceptable. Such callers pass only their
// inputs and outputs.
//
// The arrays below are created when the library is loaded and stay resident on
// every GPU that loads it until the process exits (about 4.1 MB). Every call
// uses the same arrays, so two calls that run on the GPU at the same time (for
// example on two streams) race and both give wrong results; calls on one
// stream are ordered and safe.
#include <mutex>

#include "ice_internal.cuh"

namespace ice {

constexpr long long kNoAllocMaxTokens = 1LL << 20;  // tokens per call, summed over units
constexpr int kNoAllocMaxUnits = 4096;

static __device__ __align__(256) float g_na_nrm2[kNoAllocMaxTokens];
static __device__ __align__(256) unsigned int g_na_umax[kNoAllocMaxUnits];
static __device__ __align__(256) float g_na_dirs[kMaxL * kM * kDirStride];

namespace {

// splitmix64 is a counter-based generator: draw k (from 0) of seed s is the
// mix of s + (k + 1) * golden-ratio increment, so each component of the
// directions can be computed on its own.
__device__ __forceinline__ unsigned long long sm64_draw(unsigned long long seed,
                                                        unsigned long long k) {
    unsigned long long z = seed + (k + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__global__ void na_dirs_kernel(float* __restrict__ dirs, unsigned long long seed, int L) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // over L * kM * (kD + 1)
    if (idx >= L * kM * (kD + 1)) return;
    const int row = idx / (kD + 1), i = idx % (kD + 1);
    dirs[row * kDirStride + i] = (sm64_draw(seed, (unsigned long long)idx) >> 63) ? -0.0625f : 0.0625f;
}

__global__ void na_clear_kernel(unsigned int* __restrict__ umax, int U) {
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < U) umax[u] = 0u;
}

// Squared norm with the fixed-order dot (one thread per key), per-unit maximum.
template <typename T>
__global__ void __launch_bounds__(256) na_norms_kernel(const T* __restrict__ keys, long long total,
                                                      long long n, float* __restrict__ nrm2,
                                                      unsigned int* __restrict__ umax) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const T* row = keys + i * kD;
    float acc[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        float v[4];
        load4_nc(row + 4 * l, v);
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) s = __fmaf_rn(v[k], v[k], s);
        acc[l] = s;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int l = 0; l < o; ++l) acc[l] = __fadd_rn(acc[l], acc[l + o]);
    nrm2[i] = acc[0];
    atomicMax(&umax[i / n], __float_as_uint(acc[0]));
}

__global__ void na_exponent_kernel(const unsigned int* __restrict__ umax, int* __restrict__ e_out,
                                   int U) {
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < U) e_out[u] = scale_exponent_dev(__uint_as_float(umax[u]));
}

// One thread per (key, composite): transformed key, 8 projections in the fixed
// order, codes, Morton key.
template <typename T>
__global__ void __launch_bounds__(128) na_codes_kernel(const T* __restrict__ keys,
                                                      const float* __restrict__ nrm2,
                                                      const int* __restrict__ e_unit,
                                                      const float* __restrict__ dirs, int U, int L,
                                                      long long n,
                                                      unsigned long long* __restrict__ mk) {
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= (long long)L * U * n) return;
    const int l = (int)(g / ((long long)U * n));
    const long long ut = g % ((long long)U * n);  // u * n + t
    const int u = (int)(ut / n);
    const int e = e_unit[u];
    const float sc = ldexpf(1.0f, -e), sc2 = ldexpf(1.0f, -2 * e);
    float r = __fsub_rn(1.0f, __fmul_rn(nrm2[ut], sc2));
    r = r > 0.0f ? r : 0.0f;
    const float tail = __fsqrt_rn(r);
    const T* row = keys + ut * kD;
    int code[kM];
#pragma unroll 1
    for (int j = 0; j < kM; ++j) {  // one direction at a time keeps the state in registers
        const float* ud = dirs + (l * kM + j) * kDirStride;
        float acc[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            float v[4];
            load4_nc(row + 4 * c, v);
            float s = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) s = __fmaf_rn(ud[4 * c + k], __fmul_rn(v[k], sc), s);
            acc[c] = s;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
            for (int c = 0; c < o; ++c) acc[c] = __fadd_rn(acc[c], acc[c + o]);
        code[j] = quantise_code(__fmaf_rn(ud[kD], tail, acc[0]));
    }
    mk[g] = morton8(code);
}

// Device address of the scratch arrays, looked up once per device (with that
// device current) under a lock, so that first calls from several host threads
// do not race on the table.
struct NoAllocPtrs {
    float* nrm2;
    unsigned int* umax;
    float* dirs;
    bool ready;
};
NoAllocPtrs g_na_ptrs[64];
std::mutex g_na_lock;

cudaError_t na_setup(int dev, NoAllocPtrs* out) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_na_lock);
    NoAllocPtrs& p = g_na_ptrs[dev];
    if (!p.ready) {
        NoAllocPtrs q{};
        cudaError_t e = cudaGetSymbolAddress((void**)&q.nrm2, g_na_nrm2);
        if (e == cudaSuccess) e = cudaGetSymbolAddress((void**)&q.umax, g_na_umax);
        if (e == cudaSuccess) e = cudaGetSymbolAddress((void**)&q.dirs, g_na_dirs);
        if (e != cudaSuccess) return e;
        q.ready = true;
        p = q;
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace ice

using namespace ice;

extern "C" int ice_key_codes_noalloc(const ice_params* params, const void* keys, int64_t n_tokens,
                                     uint64_t* morton_out, int32_t* e_out, void* stream) {
    if (!params || !keys || !morton_out || !e_out) return ICE_ERR_INVALID_ARG;
    if (params->d != kD || params->n_proj != kM) return ICE_ERR_UNSUPPORTED;
    if (params->n_composite < 1 || params->n_composite > kMaxL) return ICE_ERR_INVALID_ARG;
    if (params->dtype != ICE_F32 && params->dtype != ICE_BF16) return ICE_ERR_INVALID_ARG;
    if (params->dir_kind != ICE_DIR_RADEMACHER) return ICE_ERR_UNSUPPORTED;  // drawn on the device
    if (params->batch < 1 || params->n_layers < 1 || params->n_kv_heads < 1 || n_tokens < 1)
        return ICE_ERR_INVALID_ARG;
    if (((uintptr_t)keys & 15u) != 0) return ICE_ERR_INVALID_ARG;
    const long long U = (long long)params->batch * params->n_layers * params->n_kv_heads;
    if (U > kNoAllocMaxUnits || U * n_tokens > kNoAllocMaxTokens) return ICE_ERR_CAPACITY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ICE_ERR_CUDA;
    NoAllocPtrs p{};
    if (na_setup(dev, &p) != cudaSuccess) return ICE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    const int L = params->n_composite;
    const long long total = U * n_tokens;
    na_dirs_kernel<<<(L * kM * (kD + 1) + 255) / 256, 256, 0, st>>>(p.dirs, params->seed, L);
    na_clear_kernel<<<(int)((U + 255) / 256), 256, 0, st>>>(p.umax, (int)U);
    if (params->dtype == ICE_BF16)
        na_norms_kernel<__nv_bfloat16><<<(int)((total + 255) / 256), 256, 0, st>>>(
            (const __nv_bfloat16*)keys, total, n_tokens, p.nrm2, p.umax);
    else
        na_norms_kernel<float><<<(int)((total + 255) / 256), 256, 0, st>>>(
            (const float*)keys, total, n_tokens, p.nrm2, p.umax);
    na_exponent_kernel<<<(int)((U + 127) / 128), 128, 0, st>>>(p.umax, e_out, (int)U);
    const long long work = (long long)L * total;
    if (params->dtype == ICE_BF16)
        na_codes_kernel<__nv_bfloat16><<<(int)((work + 127) / 128), 128, 0, st>>>(
            (const __nv_bfloat16*)keys, p.nrm2, e_out, p.dirs, (int)U, L, n_tokens,
            (unsigned long long*)morton_out);
    else
        na_codes_kernel<float><<<(int)((work + 127) / 128), 128, 0, st>>>(
            (const float*)keys, p.nrm2, e_out, p.dirs, (int)U, L, n_tokens,
            (unsigned long long*)morton_out);
    return cudaGetLastError() == cudaSuccess ? ICE_OK : ICE_ERR_CUDA;
}

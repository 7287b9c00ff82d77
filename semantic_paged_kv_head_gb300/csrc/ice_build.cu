// Prefill build of the DCI-tree page index ("IceCache", Figure 2 step 1 and
// Figure 3): transform + projection + quantisation of every key, a segmented
// radix sort of the 96-bit keys, the trie leaves (split while a node holds
// more than P tokens), and the packing of K/V rows into the physical pages.
//
// Every unit (sequence, layer, KV head) is an independent segment; all units
// are processed by the same launches.
#include <algorithm>
#include <mutex>
#include <vector>

#include <cuda.h>  // the CUtensorMap type and its enums (the encoder is looked up at run time)

#include "ice_internal.cuh"
#include "ice_select_common.cuh"

namespace ice {

// ---------------------------------------------------------------------------
// K1a: squared norm of every key with the fixed-order dot, and the per-unit
// maximum (non-negative floats order like their bit patterns).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) norms_kernel(const T* __restrict__ keys, long long total,
                                                   long long n, float* __restrict__ nrm2,
                                                   unsigned int* __restrict__ umax) {
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    float r = 0.0f;
    if (i < total) {
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
        r = acc[0];
        nrm2[i] = r;
    }
    // one atomic per warp and unit: lanes of a warp may straddle two units
    long long u = i < total ? i / n : -1;
    long long u0 = __shfl_sync(0xffffffffu, u, 0);
    bool same = __all_sync(0xffffffffu, u == u0);
    if (same) {
        float m = r;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0 && u0 >= 0) atomicMax(&umax[u0], __float_as_uint(m));
    } else if (i < total) {
        atomicMax(&umax[u], __float_as_uint(r));
    }
}

__global__ void exponent_kernel(const unsigned int* __restrict__ umax, int* __restrict__ e_unit,
                                int U) {
    int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < U) e_unit[u] = scale_exponent_dev(__uint_as_float(umax[u]));
}

// ---------------------------------------------------------------------------
// K1b: transformed key k~ = [k 2^-e, sqrt(max(0, 1 - |k|^2 2^-2e))], its
// projections p = fma(u[d], tail, D(u[0:d], k~[0:d])) on the L*8 directions,
// 8-bit codes and the Morton key per composite. One thread per (token,
// direction); the token rows are staged in shared memory.
// ---------------------------------------------------------------------------
constexpr int kProjThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kProjThreads) project_kernel(
    const T* __restrict__ keys, const float* __restrict__ nrm2, const int* __restrict__ e_unit,
    const float* __restrict__ dirs, int L, long long n, int tiles_per_unit,
    unsigned long long* __restrict__ mk_out, int* __restrict__ tok_out, int U) {
    const int ndir = L * kM;
    const int tpb = kProjThreads / ndir;  // tokens per block
    __shared__ __align__(16) float kt[kProjThreads / kM][kD + 4];
    __shared__ float tail[kProjThreads / kM];
    __shared__ int codes[kProjThreads / kM][kMaxL * kM];
    const int u = blockIdx.x / tiles_per_unit;
    const long long t0 = (long long)(blockIdx.x % tiles_per_unit) * tpb;
    const int e = e_unit[u];
    const float sc = ldexpf(1.0f, -e);
    const float sc2 = ldexpf(1.0f, -2 * e);
    // stage k~ rows: 4 elements per thread per step
    for (int idx = threadIdx.x; idx < tpb * (kD / 4); idx += blockDim.x) {
        int r = idx / (kD / 4), c = (idx % (kD / 4)) * 4;
        long long t = t0 + r;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (t < n) load4_nc(keys + ((long long)u * n + t) * kD + c, v);
#pragma unroll
        for (int k = 0; k < 4; ++k) kt[r][c + k] = __fmul_rn(v[k], sc);
    }
    if (threadIdx.x < tpb) {
        long long t = t0 + threadIdx.x;
        float r = 0.0f;
        if (t < n) {
            r = __fsub_rn(1.0f, __fmul_rn(nrm2[(long long)u * n + t], sc2));
            r = r > 0.0f ? r : 0.0f;
        }
        tail[threadIdx.x] = __fsqrt_rn(r);
    }
    __syncthreads();
    const int r = threadIdx.x / ndir, dir = threadIdx.x % ndir;
    if (r < tpb) {
        const float* ud = dirs + (long long)dir * kDirStride;
        float acc[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            float4 x = *reinterpret_cast<const float4*>(&kt[r][4 * l]);
            float4 w = __ldg(reinterpret_cast<const float4*>(ud + 4 * l));
            float s = 0.0f;
            s = __fmaf_rn(w.x, x.x, s);
            s = __fmaf_rn(w.y, x.y, s);
            s = __fmaf_rn(w.z, x.z, s);
            s = __fmaf_rn(w.w, x.w, s);
            acc[l] = s;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
            for (int l = 0; l < o; ++l) acc[l] = __fadd_rn(acc[l], acc[l + o]);
        float p = __fmaf_rn(ud[kD], tail[r], acc[0]);
        codes[r][dir] = quantise_code(p);
    }
    __syncthreads();
    if (threadIdx.x < tpb * L) {
        int rr = threadIdx.x / L, l = threadIdx.x % L;
        long long t = t0 + rr;
        if (t < n) {
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = codes[rr][l * kM + j];
            long long o = ((long long)l * U + u) * n + t;
            mk_out[o] = morton8(c);
            tok_out[o] = (int)t;
        }
    }
}

// ---------------------------------------------------------------------------
// K1c: the same codes with the projection on tensor cores, for bf16 keys and
// +-1/16 directions (both exact in bf16; bf16 x bf16 products are exact in
// fp32). mma.sync m16n8k16 (bf16 in, fp32 accumulate) gives P = K U^T for 16
// tokens per warp; the tensor cores add the products in an order of their own,
// so a value whose (p + 1) * 128 lies within kCodeGuard of an integer (a code
// boundary) is recomputed with the fixed-order dot of K1b, and every code
// equals K1b's. The k index of each 16-wide step is permuted so that a lane's
// A and B fragments for two steps are one 16-byte load: logical k of step
// 2m + s maps to dimension 32m + 8(k mod 8 div 2) + 4s + 2(k div 8) + k mod 2,
// the same for keys and directions, which leaves the dot unchanged.
// ---------------------------------------------------------------------------
constexpr int kPmWarps = 8;
constexpr int kPmTok = kPmWarps * 16;  // tokens per block
constexpr float kCodeGuard = 1.0f / 256.0f;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], unsigned a0, unsigned a1, unsigned a2,
                                               unsigned a3, unsigned b0, unsigned b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The code of key row krow (bf16, scaled by sc) on direction ud with the
// fixed-order dot of K1b, evaluated by one warp: lane l forms the partial of
// elements 4l..4l+3 and the partials are added pairwise over lanes l and
// l + 16, 8, 4, 2, 1 (the order of K1b's per-thread tree). Every lane returns it.
__device__ __forceinline__ int exact_code_warp(const __nv_bfloat16* krow, float sc, const float* ud,
                                              float tail, int lane) {
    float x[4];
    load4_nc(krow + 4 * lane, x);
    const float4 w = __ldg(reinterpret_cast<const float4*>(ud + 4 * lane));
    float s = 0.0f;
    s = __fmaf_rn(w.x, __fmul_rn(x[0], sc), s);
    s = __fmaf_rn(w.y, __fmul_rn(x[1], sc), s);
    s = __fmaf_rn(w.z, __fmul_rn(x[2], sc), s);
    s = __fmaf_rn(w.w, __fmul_rn(x[3], sc), s);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    return quantise_code(__fmaf_rn(ud[kD], tail, s));
}

// bf16 pair (lo, hi) of two fp32 values that are exact in bf16.
__device__ __forceinline__ unsigned bf16_pair(float lo, float hi) {
    return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kPmWarps * 32) project_mma_kernel(
    const __nv_bfloat16* __restrict__ keys, const float* __restrict__ nrm2,
    const int* __restrict__ e_unit, const float* __restrict__ dirs, int L, long long n,
    int tiles_per_unit, unsigned long long* __restrict__ mk_out, int* __restrict__ tok_out, int U) {
    __shared__ float tail_s[kPmTok];
    __shared__ unsigned char codes[kPmTok][kMaxL * kM];
    __shared__ unsigned short queue[kPmTok * kMaxL * kM];  // (token << 4 | direction) to recompute
    __shared__ int qn;
    const int ndir = L * kM;
    const int u = blockIdx.x / tiles_per_unit;
    const long long t0 = (long long)(blockIdx.x % tiles_per_unit) * kPmTok;
    const int e = e_unit[u];
    const float sc = ldexpf(1.0f, -e), sc2 = ldexpf(1.0f, -2 * e);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16* ku = keys + (long long)u * n * kD;
    if (tid == 0) qn = 0;

    // warp w: tokens 16w .. 16w + 15 of the block; lane (r, q) = (lane / 4, lane % 4)
    const int r = lane >> 2, q = lane & 3;
    const int la = 16 * warp + r, lb = la + 8;  // the lane's two token rows (block-local)
    const long long ta = t0 + la, tb = t0 + lb;
    float tail[2];
#pragma unroll
    for (int z = 0; z < 2; ++z) {
        const long long t = z ? tb : ta;
        float rr = 0.0f;
        if (t < n) {
            rr = __fsub_rn(1.0f, __fmul_rn(nrm2[(long long)u * n + t], sc2));
            rr = rr > 0.0f ? rr : 0.0f;
        }
        tail[z] = __fsqrt_rn(rr);
    }
    if (q == 0) {
        tail_s[la] = tail[0];
        tail_s[lb] = tail[1];
    }
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
        if (ta < n) xa = __ldg(reinterpret_cast<const uint4*>(ku + ta * kD + 32 * m + 8 * q));
        if (tb < n) xb = __ldg(reinterpret_cast<const uint4*>(ku + tb * kD + 32 * m + 8 * q));
#pragma unroll
        for (int nt = 0; nt < kMaxL; ++nt) {
            if (nt * kM >= ndir) break;
            // direction nt * 8 + r, dimensions 32m + 8q .. + 7, as bf16 pairs
            const float* ud = dirs + (long long)(nt * kM + r) * kDirStride + 32 * m + 8 * q;
            const float4 w0 = __ldg(reinterpret_cast<const float4*>(ud));
            const float4 w1 = __ldg(reinterpret_cast<const float4*>(ud + 4));
            mma_bf16_16816(acc[nt], xa.x, xb.x, xa.y, xb.y, bf16_pair(w0.x, w0.y), bf16_pair(w0.z, w0.w));
            mma_bf16_16816(acc[nt], xa.z, xb.z, xa.w, xb.w, bf16_pair(w1.x, w1.y), bf16_pair(w1.z, w1.w));
        }
    }
    __syncthreads();  // qn is cleared
    // codes from the tensor-core values; values near a code boundary are queued
#pragma unroll
    for (int nt = 0; nt < kMaxL; ++nt) {
        if (nt * kM >= ndir) break;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int lt = i < 2 ? la : lb;
            const int dir = nt * kM + 2 * q + (i & 1);
            if (t0 + lt < n) {
                const float p = __fmaf_rn(dirs[(long long)dir * kDirStride + kD], tail[i >> 1],
                                          __fmul_rn(acc[nt][i], sc));
                const float y = __fmul_rn(__fadd_rn(p, 1.0f), 128.0f);
                const float fr = y - floorf(y);
                codes[lt][dir] = (unsigned char)quantise_code(p);
                if (fr < kCodeGuard || fr > 1.0f - kCodeGuard)
                    queue[atomicAdd(&qn, 1)] = (unsigned short)((lt << 4) | dir);
            }
        }
    }
    __syncthreads();
    for (int i = warp; i < qn; i += kPmWarps) {  // warp-uniform
        const int lt = queue[i] >> 4, dir = queue[i] & 15;
        const int c = exact_code_warp(ku + (t0 + lt) * kD, sc, dirs + (long long)dir * kDirStride,
                                      tail_s[lt], lane);
        if (lane == 0) codes[lt][dir] = (unsigned char)c;
    }
    __syncthreads();
    if (tid < kPmTok * L) {
        const int rr = tid / L, l = tid % L;
        const long long t = t0 + rr;
        if (t < n) {
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = codes[rr][l * kM + j];
            const long long o = ((long long)l * U + u) * n + t;
            mk_out[o] = morton8(c);
            tok_out[o] = (int)t;
        }
    }
}

// ---------------------------------------------------------------------------
// K1d: the key read of the build done once, on the fifth-generation tensor
// cores, for bf16 keys and +-1/16 directions: a tile of 128 tokens (128 x 128
// bf16, 32 KB) is staged by the tensor memory accelerator (two boxes of 64
// dimensions, 128-byte swizzle) and
//  * one thread issues 8 tcgen05.mma (kind::f16, M = 128, N = 16, K = 16) that
//    leave P_raw = K U^T (the unscaled projections, fp32) in tensor memory;
//  * meanwhile every thread forms its token's squared norm with the fixed-order
//    dot from the same shared-memory tile;
//  * each warp reads its 32 tokens' 16 projections back with tcgen05.ld and
//    stores them with the norm (68 bytes per token); the unit's largest norm is
//    kept with atomicMax.
// The next tile's copy is in flight while a tile is processed. The unit's
// exponent is known only after all its tokens are read, so the codes come from
// a second, light pass (K1e) over these 68 bytes: 2^-e is exact, so the scaled
// projection equals D(u, k) 2^-e of the fixed-order definition whenever the
// tensor cores' sum equals the fixed-order sum, and values within kCodeGuard of
// a code boundary are recomputed there in the fixed order.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 128;                 // tokens per tile (the MMA's M)
constexpr int kTcThreads = 128;              // one thread per token row, 4 warps
constexpr int kTcTileB = kTcRows * kD * 2;   // 32 KB
constexpr int kTcHalfB = kTcTileB / 2;       // one 64-dimension box
constexpr int kTcDirB = 16 * kD * 2;         // 16 directions x 128 bf16
constexpr int kTcStages = 2;                 // tiles in shared memory (one copy ahead)
constexpr int kTcSmem = 1024 + kTcStages * kTcTileB + kTcDirB;  // + alignment slack
constexpr int kTcBlocksPerSm = 3;            // 3 x 70.6 KB of shared memory, 3 x 32 tensor-memory columns
constexpr int kTcTmemCols = 32;
static_assert(kTcBlocksPerSm * (kTcSmem + 1024 + 64) <= 228 * 1024,
              "the blocks' shared memory (each with its 1 KB reserve and static part) fits one SM");
static_assert(kTcBlocksPerSm * kTcTmemCols <= 512, "the blocks' tensor-memory columns fit one SM");

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle: start address >> 4 (bits 0-13), leading offset 16 B (unused with
// this swizzle, bits 16-29), stride 1024 B between 8-row groups (bits 32-45),
// the fixed value 1 at bit 46, swizzle mode 2 (128 B) in bits 61-63.
__device__ __forceinline__ unsigned long long sdesc_k_sw128(unsigned saddr) {
    return (unsigned long long)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
constexpr unsigned kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void tc_mbar_init(unsigned bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(kTcThreads) project_tc_kernel(
    const __grid_constant__ CUtensorMap tmap, const float* __restrict__ dirs, int L, long long n,
    int tiles_per_unit, long long tiles_total, float* __restrict__ praw, float* __restrict__ nrm2,
    unsigned* __restrict__ umax, int* __restrict__ err) {
    extern __shared__ unsigned char tc_smem[];
    __shared__ __align__(8) unsigned long long bar_full[kTcStages], bar_mma;
    __shared__ unsigned tmem_slot;
    __shared__ int s_fail;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned raw0 = smem_u32(tc_smem);
    const unsigned base = (raw0 + 1023u) & ~1023u;  // the swizzle atoms need 1024-byte alignment
    const unsigned sB = base + kTcStages * kTcTileB;
    unsigned char* pB = tc_smem + (sB - raw0);
    // the directions in bf16 (exact for +-1/16): row j (direction), dimensions
    // 64h..64h+63 in half h; the 16-byte chunk c of row j sits at chunk c ^ (j mod 8)
    for (int idx = tid; idx < 16 * 16; idx += kTcThreads) {
        const int j = idx >> 4, chunk = idx & 15, h = chunk >> 3, c = chunk & 7;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (j < L * kM) {
            const float* ud = dirs + (long long)j * kDirStride + 64 * h + 8 * c;
            w.x = (__float_as_uint(ud[0]) >> 16) | (__float_as_uint(ud[1]) & 0xFFFF0000u);
            w.y = (__float_as_uint(ud[2]) >> 16) | (__float_as_uint(ud[3]) & 0xFFFF0000u);
            w.z = (__float_as_uint(ud[4]) >> 16) | (__float_as_uint(ud[5]) & 0xFFFF0000u);
            w.w = (__float_as_uint(ud[6]) >> 16) | (__float_as_uint(ud[7]) & 0xFFFF0000u);
        }
        *reinterpret_cast<uint4*>(pB + h * (kTcDirB / 2) + j * 128 + ((c ^ (j & 7)) << 4)) = w;
    }
    if (tid == 0) {
        s_fail = 0;
        for (int k = 0; k < kTcStages; ++k) tc_mbar_init(smem_u32(&bar_full[k]));
        tc_mbar_init(smem_u32(&bar_mma));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<unsigned long long>(&tmap)) : "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_slot)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the directions written by ordinary stores are read by the tensor cores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned tmem = tmem_slot;

    auto issue = [&](long long tile, int s) {  // thread 0
        const unsigned bar = smem_u32(&bar_full[s]);
        const unsigned dst = base + s * kTcTileB;
        const long long uu = tile / tiles_per_unit;
        const int y = (int)(uu * n + (tile % tiles_per_unit) * kTcRows);
        const unsigned long long tm = reinterpret_cast<unsigned long long>(&tmap);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kTcTileB)
                     : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                dst),
            "l"(tm), "r"(0), "r"(y), "r"(bar)
            : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                dst + kTcHalfB),
            "l"(tm), "r"(64), "r"(y), "r"(bar)
            : "memory");
    };

    long long tile = blockIdx.x;
    if (tid == 0)
        for (int k = 0; k + 1 < kTcStages; ++k)
            if (tile + (long long)k * gridDim.x < tiles_total) issue(tile + (long long)k * gridDim.x, k);
    int it = 0;
    // s_fail: 1 = the tile's copy did not land in time, 2 = its MMAs did not finish
    for (; tile < tiles_total; tile += gridDim.x, ++it) {  // block-uniform
        const int s = it % kTcStages;
        const unsigned ph = (unsigned)((it / kTcStages) & 1);
        const unsigned sA = base + s * kTcTileB;
        const long long ahead = tile + (long long)(kTcStages - 1) * gridDim.x;
        if (tid == 0 && ahead < tiles_total) issue(ahead, (it + kTcStages - 1) % kTcStages);
        if (!mbar_wait_bounded(smem_u32(&bar_full[s]), ph)) s_fail = 1;
        __syncthreads();
        if (s_fail) break;
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const unsigned off = (unsigned)((ks >> 2) * kTcHalfB + (ks & 3) * 32);
                const unsigned boff = (unsigned)((ks >> 2) * (kTcDirB / 2) + (ks & 3) * 32);
                const unsigned long long ad = sdesc_k_sw128(sA + off);
                const unsigned long long bd = sdesc_k_sw128(sB + boff);
                const unsigned acc = ks > 0 ? 1u : 0u;
                asm volatile(
                    "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                    " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                    "l"(ad), "l"(bd), "r"(kTcIdesc), "r"(acc)
                    : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&bar_mma))
                         : "memory");
        }
        // the token's squared norm in the fixed order, from the swizzled tile: lane
        // partial l covers dimensions 4l..4l+3, i.e. half l / 16, chunk (l mod 16) / 2
        float part[32];
        {
            const unsigned row = sA + tid * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 x;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                                 : "r"(row + h * kTcHalfB + ((c ^ (tid & 7)) << 4))
                                 : "memory");
                    const float e0 = __uint_as_float(x.x << 16), e1 = __uint_as_float(x.x & 0xFFFF0000u);
                    const float e2 = __uint_as_float(x.y << 16), e3 = __uint_as_float(x.y & 0xFFFF0000u);
                    const float e4 = __uint_as_float(x.z << 16), e5 = __uint_as_float(x.z & 0xFFFF0000u);
                    const float e6 = __uint_as_float(x.w << 16), e7 = __uint_as_float(x.w & 0xFFFF0000u);
                    float a = 0.0f, b = 0.0f;
                    a = __fmaf_rn(e0, e0, a);
                    a = __fmaf_rn(e1, e1, a);
                    a = __fmaf_rn(e2, e2, a);
                    a = __fmaf_rn(e3, e3, a);
                    b = __fmaf_rn(e4, e4, b);
                    b = __fmaf_rn(e5, e5, b);
                    b = __fmaf_rn(e6, e6, b);
                    b = __fmaf_rn(e7, e7, b);
                    part[16 * h + 2 * c] = a;
                    part[16 * h + 2 * c + 1] = b;
                }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                for (int l = 0; l < o; ++l) part[l] = __fadd_rn(part[l], part[l + o]);
        }
        const float nrm = part[0];
        // the projections of the warp's 32 tokens from tensor memory
        if (!mbar_wait_bounded(smem_u32(&bar_mma), (unsigned)(it & 1))) s_fail = 2;
        __syncthreads();
        if (s_fail) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        unsigned r[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
              "=r"(r[14]), "=r"(r[15])
            : "r"(tmem + ((unsigned)(32 * warp) << 16))
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const long long uu = tile / tiles_per_unit;
        const long long t = (tile % tiles_per_unit) * kTcRows + tid;
        const bool valid = t < n;
        if (valid) {
            const long long g = uu * n + t;
            float4* dst = reinterpret_cast<float4*>(praw + g * 16);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                     __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
            nrm2[g] = nrm;
        }
        float mx = valid ? nrm : 0.0f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) atomicMax(&umax[uu], __float_as_uint(mx));
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();  // the tile's buffer and tensor-memory columns are free again
    }
    if (s_fail) {
        // a wait ran out: report it, then let the copies and MMAs still in flight
        // finish (bounded) before the tensor memory is released
        if (tid == 0) {
            atomicExch(err, 1);
            if (s_fail == 1)
                mbar_wait_bounded(smem_u32(&bar_full[it % kTcStages]), (unsigned)((it / kTcStages) & 1));
            else
                mbar_wait_bounded(smem_u32(&bar_mma), (unsigned)(it & 1));
            for (int k = 1; k < kTcStages; ++k)  // the copies issued ahead
                if (tile + (long long)k * gridDim.x < tiles_total)
                    mbar_wait_bounded(smem_u32(&bar_full[(it + k) % kTcStages]),
                                      (unsigned)(((it + k) / kTcStages) & 1));
        }
        __syncthreads();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
}

// ---------------------------------------------------------------------------
// K1e: codes and Morton keys from the stored projections: p = fma(u[d], tail,
// P_raw 2^-e) with the unit's frozen exponent; a value whose (p + 1) * 128
// lies within kCodeGuard of an integer is recomputed from the key row with the
// fixed-order dot (one warp per queued value).
// ---------------------------------------------------------------------------
constexpr int kCodeTok = 256;

__global__ void __launch_bounds__(kCodeTok) codes_tc_kernel(
    const __nv_bfloat16* __restrict__ keys, const float* __restrict__ praw, const float* __restrict__ nrm2,
    const int* __restrict__ e_unit, const float* __restrict__ dirs, int L, long long n, int tiles_per_unit,
    unsigned long long* __restrict__ mk_out, int* __restrict__ tok_out, int U) {
    __shared__ unsigned char codes[kCodeTok][kMaxL * kM];
    __shared__ float tail_s[kCodeTok];
    __shared__ unsigned short queue[kCodeTok * kMaxL * kM];
    __shared__ int qn;
    const int ndir = L * kM;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = blockIdx.x / tiles_per_unit;
    const long long t0 = (long long)(blockIdx.x % tiles_per_unit) * kCodeTok;
    const long long t = t0 + tid;
    const int e = e_unit[u];
    const float sc = ldexpf(1.0f, -e), sc2 = ldexpf(1.0f, -2 * e);
    if (tid == 0) qn = 0;
    __syncthreads();
    if (t < n) {
        const long long g = (long long)u * n + t;
        float rr = __fsub_rn(1.0f, __fmul_rn(nrm2[g], sc2));
        rr = rr > 0.0f ? rr : 0.0f;
        const float tail = __fsqrt_rn(rr);
        tail_s[tid] = tail;
        const float4* src = reinterpret_cast<const float4*>(praw + g * 16);
        float raw[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 x = src[k];
            raw[4 * k] = x.x;
            raw[4 * k + 1] = x.y;
            raw[4 * k + 2] = x.z;
            raw[4 * k + 3] = x.w;
        }
#pragma unroll
        for (int dd = 0; dd < kMaxL * kM; ++dd) {
            if (dd >= ndir) break;
            const float p = __fmaf_rn(dirs[(long long)dd * kDirStride + kD], tail, __fmul_rn(raw[dd], sc));
            const float y = __fmul_rn(__fadd_rn(p, 1.0f), 128.0f);
            const float fr = y - floorf(y);
            codes[tid][dd] = (unsigned char)quantise_code(p);
            if (fr < kCodeGuard || fr > 1.0f - kCodeGuard)
                queue[atomicAdd(&qn, 1)] = (unsigned short)((tid << 4) | dd);
        }
    }
    __syncthreads();
    // the queued values, four per warp at a time: all their rows are requested
    // before any is reduced (one memory latency per round, not four)
    const __nv_bfloat16* ku = keys + (long long)u * n * kD;
    constexpr int kW = kCodeTok / 32, kB = 4;
    for (int i0 = warp; i0 < qn; i0 += kW * kB) {  // warp-uniform
        float x[kB][4];
        float4 w[kB];
        int lt[kB], dd[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int i = i0 + kW * b;
            lt[b] = i < qn ? queue[i] >> 4 : 0;
            dd[b] = i < qn ? queue[i] & 15 : 0;
            load4_nc(ku + (t0 + lt[b]) * kD + 4 * lane, x[b]);
            w[b] = __ldg(reinterpret_cast<const float4*>(dirs + (long long)dd[b] * kDirStride + 4 * lane));
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            float acc = 0.0f;  // the fixed-order dot of K1b: lane partial, then the pairwise tree
            acc = __fmaf_rn(w[b].x, __fmul_rn(x[b][0], sc), acc);
            acc = __fmaf_rn(w[b].y, __fmul_rn(x[b][1], sc), acc);
            acc = __fmaf_rn(w[b].z, __fmul_rn(x[b][2], sc), acc);
            acc = __fmaf_rn(w[b].w, __fmul_rn(x[b][3], sc), acc);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
            if (lane == 0 && i0 + kW * b < qn)
                codes[lt[b]][dd[b]] = (unsigned char)quantise_code(
                    __fmaf_rn(dirs[(long long)dd[b] * kDirStride + kD], tail_s[lt[b]], acc));
        }
    }
    __syncthreads();
    if (t < n) {
        for (int l = 0; l < L; ++l) {
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = codes[tid][l * kM + j];
            const long long o = ((long long)l * U + u) * n + t;
            mk_out[o] = morton8(c);
            tok_out[o] = (int)t;
        }
    }
}

// ---------------------------------------------------------------------------
// K2: stable LSD radix sort of (Morton key, token) within each segment
// (composite, unit), 8 bits per pass. Input order is ascending token, so equal
// Morton keys stay in token order and the result is sorted by the 96-bit key.
// ---------------------------------------------------------------------------
constexpr int kSortThreads = 256;
constexpr int kSortItems = 8;
constexpr int kSortTile = kSortThreads * kSortItems;

__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(
    const unsigned long long* __restrict__ keys, long long n, int tiles, int shift,
    int* __restrict__ hist) {
    __shared__ int h[256];
    const int seg = blockIdx.x / tiles, tile = blockIdx.x % tiles;
    h[threadIdx.x] = 0;
    __syncthreads();
    const long long base = (long long)seg * n + (long long)tile * kSortTile;
    const long long lim = min((long long)kSortTile, n - (long long)tile * kSortTile);
    for (int i = threadIdx.x; i < lim; i += kSortThreads)
        atomicAdd(&h[(int)((keys[base + i] >> shift) & 0xFF)], 1);
    __syncthreads();
    hist[((long long)seg * 256 + threadIdx.x) * tiles + tile] = h[threadIdx.x];
}

// Per segment: offsets[seg][digit][tile] = segment start + (all smaller
// digits) + (same digit in earlier tiles).
__global__ void __launch_bounds__(256) radix_scan_kernel(int* __restrict__ hist, long long n,
                                                         int tiles) {
    __shared__ int tot[256];
    const int seg = blockIdx.x, dgt = threadIdx.x;
    int* row = hist + ((long long)seg * 256 + dgt) * tiles;
    int s = 0;
    for (int t = 0; t < tiles; ++t) s += row[t];
    tot[dgt] = s;
    __syncthreads();
    if (dgt == 0) {
        int run = 0;
        for (int k = 0; k < 256; ++k) {
            int x = tot[k];
            tot[k] = run;
            run += x;
        }
    }
    __syncthreads();
    int run = tot[dgt];
    for (int t = 0; t < tiles; ++t) {
        int x = row[t];
        row[t] = run;
        run += x;
    }
}

__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(
    const unsigned long long* __restrict__ kin, const int* __restrict__ vin,
    unsigned long long* __restrict__ kout, int* __restrict__ vout, long long n, int tiles,
    int shift, const int* __restrict__ offs) {
    constexpr int W = kSortThreads / 32;
    __shared__ int running[256];
    __shared__ int base_off[256];
    __shared__ int wcnt[W][256];
    const int seg = blockIdx.x / tiles, tile = blockIdx.x % tiles;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    running[threadIdx.x] = 0;
    base_off[threadIdx.x] = offs[((long long)seg * 256 + threadIdx.x) * tiles + tile];
    const long long seg0 = (long long)seg * n;
    const long long base = seg0 + (long long)tile * kSortTile;
    const long long lim = min((long long)kSortTile, n - (long long)tile * kSortTile);
    const unsigned int lt = (1u << lane) - 1u;
    // Items are taken in tile order, one round of kSortThreads at a time; within
    // a round, warp w precedes warp w+1 and lane order is kept by match_any.
    for (int r = 0; r < kSortItems; ++r) {
        for (int w = 0; w < W; ++w) wcnt[w][threadIdx.x] = 0;
        __syncthreads();
        const int i = r * kSortThreads + threadIdx.x;
        const bool ok = i < lim;
        const unsigned long long k = ok ? kin[base + i] : 0ull;
        const int val = ok ? vin[base + i] : 0;
        const int dgt = ok ? (int)((k >> shift) & 0xFF) : 256;
        const unsigned int peers = __match_any_sync(0xffffffffu, dgt);
        const int rank = __popc(peers & lt);
        if (ok && rank == 0) wcnt[warp][dgt] = __popc(peers);
        __syncthreads();
        int round_total = 0;  // items of digit threadIdx.x in this round
        for (int w = 0; w < W; ++w) {
            int x = wcnt[w][threadIdx.x];
            wcnt[w][threadIdx.x] = round_total;
            round_total += x;
        }
        __syncthreads();
        if (ok) {
            long long pos = seg0 + base_off[dgt] + running[dgt] + wcnt[warp][dgt] + rank;
            kout[pos] = k;
            vout[pos] = val;
        }
        __syncthreads();
        running[threadIdx.x] += round_total;
    }
}

// ---------------------------------------------------------------------------
// K3a: trie leaves of each sorted segment. With a_j = lcp(key_j, key_{j+1}),
// the node of depth t around position i holds <= P keys iff every window of
// P+1 consecutive keys containing i has lcp < t, so the leaf depth of i is
// t_i = 1 + max over such windows of min(a_s .. a_{s+P-1}) (0 when n <= P),
// and i starts a leaf iff i == 0 or a_{i-1} < t_i.
// One block per segment walks it in chunks and numbers the leaves.
// ---------------------------------------------------------------------------
constexpr int kLeafThreads = 512;

__global__ void __launch_bounds__(kLeafThreads) leaf_scan_kernel(
    const unsigned long long* __restrict__ mk, const int* __restrict__ tok, long long n, int P,
    int* __restrict__ leaf_of, int* __restrict__ leaf_start, unsigned char* __restrict__ tdepth,
    int* __restrict__ nleaf_out) {
    constexpr int B = kLeafThreads;
    __shared__ unsigned char a[B + 2 * kMaxP + 2];   // adjacent lcps around the chunk
    __shared__ unsigned char wmin[B + kMaxP + 2];    // window minima
    __shared__ int scan[B / 32];
    __shared__ int carry;
    const int seg = blockIdx.x;
    const long long s0 = (long long)seg * n;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (long long c0 = 0; c0 < n; c0 += B) {
        // adjacent lcps a_j for j in [c0 - P - 1, c0 + B + P)
        const long long j0 = c0 - P - 1;
        const int na = B + 2 * P + 1;
        for (int x = threadIdx.x; x < na; x += B) {
            long long j = j0 + x;
            unsigned char v = 0;
            if (j >= 0 && j + 1 < n)
                v = (unsigned char)lcp96(mk[s0 + j], (unsigned)tok[s0 + j], mk[s0 + j + 1],
                                         (unsigned)tok[s0 + j + 1]);
            a[x] = v;
        }
        __syncthreads();
        // window minima W_s = min(a_s .. a_{s+P-1}) for s in [c0 - P, c0 + B)
        const long long w0 = c0 - P;
        for (int x = threadIdx.x; x < B + P; x += B) {
            long long s = w0 + x;
            unsigned char v = 0;
            if (s >= 0 && s + P <= n - 1) {
                v = 255;
                for (int k = 0; k < P; ++k) v = min(v, a[(int)(s + k - j0)]);
            } else {
                v = 0;  // window not inside the segment: contributes nothing
            }
            wmin[x] = v;
        }
        __syncthreads();
        const long long i = c0 + threadIdx.x;
        int flag = 0, t = 0;
        if (i < n) {
            if (n > P) {
                int best = -1;
                for (int k = 0; k <= P; ++k) {
                    long long s = i - k;
                    if (s >= 0 && s + P <= n - 1) best = max(best, (int)wmin[(int)(s - w0)]);
                }
                t = best + 1;
            }
            flag = (i == 0) || ((int)a[(int)(i - 1 - j0)] < t);
            tdepth[s0 + i] = (unsigned char)t;
        }
        // block-wide inclusive scan of flags
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int x = flag;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) scan[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int v = lane < B / 32 ? scan[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (lane < B / 32) scan[lane] = v;
        }
        __syncthreads();
        int incl = x + (warp > 0 ? scan[warp - 1] : 0) + carry;
        if (i < n) {
            int leaf = incl - 1;
            leaf_of[s0 + i] = leaf;
            if (flag) leaf_start[s0 + leaf] = (int)i;
        }
        __syncthreads();
        if (threadIdx.x == B - 1) carry = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) nleaf_out[seg] = carry;
}

// ---------------------------------------------------------------------------
// K3b: leaf records, slot lists and token locations, one thread per sorted
// position of every segment.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) leaf_write_kernel(
    IndexView v, const unsigned long long* __restrict__ mk, const int* __restrict__ tok,
    long long n, const int* __restrict__ leaf_of, const int* __restrict__ leaf_start,
    const unsigned char* __restrict__ tdepth, const int* __restrict__ nleaf) {
    long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    long long total = (long long)v.L * v.U * n;
    if (g >= total) return;
    const int seg = (int)(g / n);
    const long long i = g % n;
    const int l = seg / v.U, u = seg % v.U;
    const long long s0 = (long long)seg * n;
    const int leaf = leaf_of[g];
    const int nl = nleaf[seg];
    if (leaf >= v.C) {
        set_status(v.status, ICE_ERR_CAPACITY);
        return;
    }
    const int start = leaf_start[s0 + leaf];
    const int end = leaf + 1 < nl ? leaf_start[s0 + leaf + 1] : (int)n;
    const int slot = (int)i - start;
    if (slot < 0 || slot >= v.P || end - start > v.P) {  // a leaf never exceeds P tokens
        set_status(v.status, ICE_ERR_BOUNDS);
        return;
    }
    const unsigned long long m = mk[g];
    const int t = tok[g];
    const long long sb = v.slot_base(u, l) + (long long)leaf * v.P + slot;
    v.slot_tok[sb] = t;
    v.slot_key[sb] = m;
    if (l == 0) v.tok_loc[(long long)u * v.max_tokens + t] = leaf * v.P + slot;
    if (l == 1) v.tok_slot1[(long long)u * v.max_tokens + t] = leaf * v.P + slot;
    if (slot == 0) {
        const int depth = tdepth[g];
        unsigned long long pm;
        unsigned int pt;
        prefix96(m, (unsigned)t, depth, pm, pt);
        const long long lb = v.leaf_base(u, l) + leaf;
        LeafKey k;
        k.pm = pm;
        k.pt = pt;
        k.t = (unsigned)depth;
        v.leaf_key[lb] = k;
        put_leaf(v, lb, make_leaf_rec(pm, (unsigned)depth, leaf, end - start));
        v.list_cnt[v.leaf_base(u, l) + leaf] = end - start;
    }
    if (i == 0) {
        v.n_leaf[v.ul(u, l)] = nl;
        v.next_id[v.ul(u, l)] = nl;
    }
}

// ---------------------------------------------------------------------------
// K3b (L = 2): the composite-1 slot of every token gets the token's page row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) loc1_kernel(IndexView v, long long n) {
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // u * n + t
    if (g >= (long long)v.U * n) return;
    const int u = (int)(g / n);
    const long long t = g % n;
    const int s1 = v.tok_slot1[(long long)u * v.max_tokens + t];
    if (s1 < 0 || (long long)s1 >= v.C * v.P) return;  // not placed (reported earlier)
    v.slot_loc1[v.loc1_base(u) + s1] = v.tok_loc[(long long)u * v.max_tokens + t];
}

// ---------------------------------------------------------------------------
// K4: copy each token's K and V row into its page slot (16 B per thread).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) pack_kernel(IndexView v, const T* __restrict__ keys,
                                                   const T* __restrict__ values, long long n) {
    constexpr int VPR = kD * (int)sizeof(T) / 16;  // 16-byte vectors per row
    long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    long long total = (long long)v.U * n * VPR;
    if (g >= total) return;
    const int c = (int)(g % VPR);
    const long long row = g / VPR;  // u * n + t
    const int u = (int)(row / n);
    const long long t = row % n;
    const int loc = v.tok_loc[(long long)u * v.max_tokens + t];
    if (loc < 0 || (long long)loc >= v.C * v.P) return;  // token not placed (reported earlier)
    const long long dst = ((long long)u * v.C * v.P + loc) * VPR + c;
    reinterpret_cast<uint4*>(v.page_k)[dst] = __ldg(reinterpret_cast<const uint4*>(keys) + g);
    reinterpret_cast<uint4*>(v.page_v)[dst] = __ldg(reinterpret_cast<const uint4*>(values) + g);
}

// ---------------------------------------------------------------------------
// Host side of the build. Scratch is stream-ordered and released before return.
// ---------------------------------------------------------------------------

#define ICE_TRY(x)                          \
    do {                                    \
        cudaError_t e_ = (x);               \
        if (e_ != cudaSuccess) return e_;   \
    } while (0)

// The driver's tensor-map encoder, looked up once through the runtime (no link
// against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn key_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

// Tensor map of the keys as a [rows][128] bf16 matrix: boxes of 64 dimensions x
// 128 rows with the 128-byte swizzle (the layout the MMA descriptors expect);
// rows past the end read as zeros.
static bool encode_key_map(CUtensorMap* m, const void* keys, long long rows) {
    EncodeTiledFn enc = key_map_encoder();
    if (enc == nullptr || rows < 1 || rows > 0x7FFFFFFFLL) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTcRows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(keys), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Phase 1: keys -> sorted 96-bit keys and leaf numbering in scratch.
cudaError_t build_phase1(int dtype, const void* keys, int U, int L, int P, long long n,
                         const float* dirs, bool dirs_bf16_exact, int* e_unit, BuildScratch& s,
                         cudaStream_t st, int* final_buf) {
    const long long total = (long long)U * n;
    const int S = L * U;
    ICE_TRY(cudaMemsetAsync(s.umax, 0, sizeof(unsigned) * U, st));
    ICE_TRY(cudaMemsetAsync(s.err, 0, sizeof(int), st));
    // bf16 keys and +-1/16 directions: one read of the keys on the tensor cores
    // (K1d), when the tensor-map encoder of the driver is at hand
    CUtensorMap tmap;
    const bool tc_path = dtype == ICE_BF16 && dirs_bf16_exact && s.praw != nullptr &&
                         encode_key_map(&tmap, keys, total);
    if (tc_path) {
        static int nsm = 0;
        if (nsm == 0) {
            int dev = 0;
            ICE_TRY(cudaGetDevice(&dev));
            ICE_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
            ICE_TRY(cudaFuncSetAttribute(project_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTcSmem));
        }
        const int tpu = (int)((n + kTcRows - 1) / kTcRows);
        const long long tiles = (long long)U * tpu;
        const int grid = (int)std::min<long long>(tiles, (long long)kTcBlocksPerSm * nsm);
        project_tc_kernel<<<grid, kTcThreads, kTcSmem, st>>>(tmap, dirs, L, n, tpu, tiles, s.praw,
                                                             s.nrm2, s.umax, s.err);
    } else {
        const int nb = (int)((total + 255) / 256);
        if (dtype == ICE_BF16)
            norms_kernel<__nv_bfloat16><<<nb, 256, 0, st>>>((const __nv_bfloat16*)keys, total, n,
                                                             s.nrm2, s.umax);
        else
            norms_kernel<float><<<nb, 256, 0, st>>>((const float*)keys, total, n, s.nrm2, s.umax);
    }
    ICE_TRY(cudaGetLastError());
    exponent_kernel<<<(U + 127) / 128, 128, 0, st>>>(s.umax, e_unit, U);
    ICE_TRY(cudaGetLastError());
    const int tpb = kProjThreads / (L * kM);
    const int tiles_u = (int)((n + tpb - 1) / tpb);
    if (tc_path) {
        const int tiles_c = (int)((n + kCodeTok - 1) / kCodeTok);
        codes_tc_kernel<<<U * tiles_c, kCodeTok, 0, st>>>((const __nv_bfloat16*)keys, s.praw, s.nrm2,
                                                          e_unit, dirs, L, n, tiles_c, s.mk[0],
                                                          s.tk[0], U);
    } else if (dtype == ICE_BF16 && dirs_bf16_exact) {
        const int tiles_m = (int)((n + kPmTok - 1) / kPmTok);
        project_mma_kernel<<<U * tiles_m, kPmWarps * 32, 0, st>>>(
            (const __nv_bfloat16*)keys, s.nrm2, e_unit, dirs, L, n, tiles_m, s.mk[0], s.tk[0], U);
    } else if (dtype == ICE_BF16)
        project_kernel<__nv_bfloat16><<<U * tiles_u, kProjThreads, 0, st>>>(
            (const __nv_bfloat16*)keys, s.nrm2, e_unit, dirs, L, n, tiles_u, s.mk[0], s.tk[0], U);
    else
        project_kernel<float><<<U * tiles_u, kProjThreads, 0, st>>>(
            (const float*)keys, s.nrm2, e_unit, dirs, L, n, tiles_u, s.mk[0], s.tk[0], U);
    ICE_TRY(cudaGetLastError());
    const int tiles = (int)((n + kSortTile - 1) / kSortTile);
    int cur = 0;
    for (int shift = 0; shift < 64; shift += 8) {
        radix_hist_kernel<<<S * tiles, kSortThreads, 0, st>>>(s.mk[cur], n, tiles, shift, s.hist);
        ICE_TRY(cudaGetLastError());
        radix_scan_kernel<<<S, 256, 0, st>>>(s.hist, n, tiles);
        ICE_TRY(cudaGetLastError());
        radix_scatter_kernel<<<S * tiles, kSortThreads, 0, st>>>(s.mk[cur], s.tk[cur], s.mk[cur ^ 1],
                                                                 s.tk[cur ^ 1], n, tiles, shift,
                                                                 s.hist);
        ICE_TRY(cudaGetLastError());
        cur ^= 1;
    }
    *final_buf = cur;
    leaf_scan_kernel<<<S, kLeafThreads, 0, st>>>(s.mk[cur], s.tk[cur], n, P, s.leaf_of,
                                                 s.leaf_start, s.tdepth, s.nleaf);
    return cudaGetLastError();
}

cudaError_t build_phase2(const IndexView& v, const void* keys, const void* values, long long n,
                         BuildScratch& s, int cur, cudaStream_t st) {
    const long long total = (long long)v.L * v.U * n;
    leaf_write_kernel<<<(int)((total + 255) / 256), 256, 0, st>>>(
        v, s.mk[cur], s.tk[cur], n, s.leaf_of, s.leaf_start, s.tdepth, s.nleaf);
    ICE_TRY(cudaGetLastError());
    if (v.L > 1) {
        loc1_kernel<<<(int)(((long long)v.U * n + 255) / 256), 256, 0, st>>>(v, n);
        ICE_TRY(cudaGetLastError());
    }
    const int es = v.dtype == ICE_BF16 ? 2 : 4;
    const long long vec = (long long)v.U * n * (kD * es / 16);
    const int nb = (int)((vec + 255) / 256);
    if (v.dtype == ICE_BF16)
        pack_kernel<__nv_bfloat16><<<nb, 256, 0, st>>>(v, (const __nv_bfloat16*)keys,
                                                       (const __nv_bfloat16*)values, n);
    else
        pack_kernel<float><<<nb, 256, 0, st>>>(v, (const float*)keys, (const float*)values, n);
    return cudaGetLastError();
}

cudaError_t scratch_alloc(BuildScratch& s, int U, int L, long long n, bool with_praw,
                          cudaStream_t st) {
    const long long SN = (long long)L * U * n;
    const long long tiles = (n + kSortTile - 1) / kSortTile;
    ICE_TRY(cudaMallocAsync((void**)&s.nrm2, sizeof(float) * U * n, st));
    ICE_TRY(cudaMallocAsync((void**)&s.umax, sizeof(unsigned) * U, st));
    ICE_TRY(cudaMallocAsync((void**)&s.err, sizeof(int), st));
    if (with_praw) ICE_TRY(cudaMallocAsync((void**)&s.praw, sizeof(float) * 16 * U * n, st));
    for (int b = 0; b < 2; ++b) {
        ICE_TRY(cudaMallocAsync((void**)&s.mk[b], sizeof(unsigned long long) * SN, st));
        ICE_TRY(cudaMallocAsync((void**)&s.tk[b], sizeof(int) * SN, st));
    }
    ICE_TRY(cudaMallocAsync((void**)&s.hist, sizeof(int) * L * U * 256 * tiles, st));
    ICE_TRY(cudaMallocAsync((void**)&s.leaf_of, sizeof(int) * SN, st));
    ICE_TRY(cudaMallocAsync((void**)&s.leaf_start, sizeof(int) * SN, st));
    ICE_TRY(cudaMallocAsync((void**)&s.tdepth, SN, st));
    ICE_TRY(cudaMallocAsync((void**)&s.nleaf, sizeof(int) * L * U, st));
    return cudaSuccess;
}

void scratch_free(BuildScratch& s, cudaStream_t st) {
    void* ptrs[] = {s.nrm2, s.umax, s.mk[0], s.mk[1], s.tk[0], s.tk[1], s.hist, s.leaf_of,
                    s.leaf_start, s.tdepth, s.nleaf, s.praw, s.err};
    for (void* p : ptrs)
        if (p) cudaFreeAsync(p, st);
    s = BuildScratch();
}

}  // namespace ice

// Device helpers shared by the selection kernels (one block per unit, and one
// cluster of blocks per unit): wall-clock reads, bounded mbarrier waits, the
// leaf priority on fp16x2 code pairs, explicit shared-memory stores, warp-level
// bitonic sort and merge, and the 16-byte row pieces of the rescoring.
#pragma once

#include <cuda_fp16.h>

#include "ice_internal.cuh"

namespace ice {

constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // bounded barrier wait

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }
// Regions that asynchronous copies fill from global memory start on a 128-byte
// boundary: a 128-byte line then lands in one 128-byte piece of shared memory
// and travels as one request. A destination 16 bytes off splits every line
// into several requests; over the host link that doubled the bytes read
// (each partial request fetched more than it asked for).
__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }

// Bytes from p up to the next 128-byte boundary of the shared-memory window.
__device__ __forceinline__ int pad_to_128(const void* p) {
    return (int)((128u - ((unsigned)__cvta_generic_to_shared(p) & 127u)) & 127u);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

// Returns true once phase `parity` of the mbarrier has completed, false if it
// has not within kWaitNs of wall time (the caller then reports a timeout).
// try_wait suspends the thread until the phase completes or a hardware time
// limit passes, so a waiting warp resumes as soon as the copies have landed.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned bar, unsigned parity) {
    const unsigned long long t0 = global_ns();
    for (;;) {
        unsigned done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// Two bytes of x (selector s) as two fp16 values 1024 + byte (exact). The bit
// pattern is moved with memcpy: reading the word through a __half2 lvalue would
// break type-based aliasing rules.
__device__ __forceinline__ __half2 bytes_to_h2(unsigned x, unsigned s) {
    const unsigned w = __byte_perm(x, 0x64646464u, s);
    __half2 h;
    memcpy(&h, &w, sizeof(h));
    return h;
}

// 0xFF in byte k of the result where bit k of the 4-bit mask m is set.
__device__ __forceinline__ unsigned nibble_bytes(unsigned m) {
    return ((m * 0x00204081u) & 0x01010101u) * 0xFFu;
}

// Word k (0..7) of eight registers, without indexing local memory.
__device__ __forceinline__ unsigned byte_word(const unsigned (&w)[8], int k) {
    const unsigned a = (k & 1) ? w[1] : w[0], b = (k & 1) ? w[3] : w[2];
    const unsigned c = (k & 1) ? w[5] : w[4], d = (k & 1) ? w[7] : w[6];
    const unsigned ab = (k & 2) ? b : a, cd = (k & 2) ? d : c;
    return (k & 4) ? cd : ab;
}

// Widths hi - lo of the 8 code intervals of a prefix of length t, as fp16x2.
__device__ __forceinline__ void cell_widths(int t, __half2 (&w)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float a[2];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int j = 2 * k + z;
            int b = t >= 64 ? 8 : ((t + 7 - j) >> 3);
            b = b > 8 ? 8 : b;
            a[z] = (float)((1 << (8 - b)) - 1);
        }
        w[k] = __floats2half2_rn(a[0], a[1]);
    }
}

// L-infinity distance (code units) between the query codes q (biased fp16x2,
// directions 2k, 2k+1 in word k) and the cell of a leaf: lower corner codes 0-3
// in x and 4-7 in y (one byte each), prefix length t. Per direction, with
// d = q - lo and the cell's width w, the distance to [lo, lo + w] is the larger
// of lo - q = -d and q - (lo + w) = d - w (one of them is <= 0); every value is
// an integer of magnitude below 2048, exact in fp16.
__device__ __forceinline__ int leaf_priority(unsigned x, unsigned y, int t, const __half2 (&q)[4],
                                             const __half2* widths /* [97][4] */) {
    const __half2 lo[4] = {bytes_to_h2(x, 0x4140u), bytes_to_h2(x, 0x4342u),
                           bytes_to_h2(y, 0x4140u), bytes_to_h2(y, 0x4342u)};
    t = min(t, 96);
    __half2 m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __half2 d = __hsub2(q[k], lo[k]);
        m[k] = __hmax2(__hneg2(d), __hsub2(d, widths[t * 4 + k]));
    }
    const __half2 r = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
    const __half d = __hmax(__hmax(__low2half(r), __high2half(r)), __float2half(0.0f));
    const __half b = __hadd(d, __float2half(1024.0f));  // 1024 + d, d in [0, 255]
    return (int)(__half_as_ushort(b) & 0x3FFu);
}

// The ties taken from the boundary word of a tie walk: the one lane whose word
// holds the tokens where the running count reaches `need` (acc < need < acc +
// tot). Lane j looks at bit j of that word, a warp prefix sum of the tie counts
// gives the tokens taken before it, and the tie is taken while that count is
// below the need, as a walk over the word's bits in order would. Returns the
// taken bits in every lane, 0 when no lane's word holds the boundary. All lanes
// of the warp call it.
__device__ __forceinline__ unsigned boundary_take(unsigned bits, const unsigned (&cw)[8], int acc,
                                                  int tot, int need, int lane) {
    const unsigned bl = __ballot_sync(0xffffffffu, bits != 0u && acc < need && acc + tot > need);
    if (bl == 0u) return 0u;  // warp-uniform
    const int b = __ffs(bl) - 1;
    const unsigned wb = __shfl_sync(0xffffffffu, bits, b);
    const int accb = __shfl_sync(0xffffffffu, acc, b);
    unsigned cwb[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) cwb[q] = __shfl_sync(0xffffffffu, cw[q], b);
    const bool has = (wb >> lane) & 1u;
    const int c = has ? (int)((byte_word(cwb, lane >> 2) >> (8 * (lane & 3))) & 0xFFu) : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    return __ballot_sync(0xffffffffu, has && accb + inc - c < need);
}

// Byte store to shared memory through an explicit st.shared.u8. With a plain
// C++ byte store of the fp16-derived priority, the priority table did not
// receive the values in builds of this kernel for sm_103a with nvcc 13.0 (the
// bytes read back unchanged after the block barrier); the explicit store does.
__device__ __forceinline__ void st_shared_u8(unsigned char* p, int v) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"((unsigned)v & 0xFFu) : "memory");
}

// Two-byte store to shared memory (shared-window address a), explicit for the
// same reason as st_shared_u8.
__device__ __forceinline__ void st_shared_u16(unsigned a, int v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)(v & 0xFFFF)) : "memory");
}

// Ascending bitonic sort of one (key, value) per lane across the warp.
__device__ __forceinline__ void warp_sort32(unsigned long long& k, int& v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long ok = __shfl_xor_sync(0xffffffffu, k, stride);
            const int ov = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool up = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            const bool keep_min = lower == up;
            const bool take = keep_min ? (ok < k) : (ok > k);
            if (take) {
                k = ok;
                v = ov;
            }
        }
    }
}

// a (sorted ascending across lanes) := the 32 smallest of a and b (b sorted).
__device__ __forceinline__ void warp_merge32(unsigned long long& ka, int& va, unsigned long long kb,
                                             int vb, int lane) {
    const unsigned long long rk = __shfl_sync(0xffffffffu, kb, 31 - lane);
    const int rv = __shfl_sync(0xffffffffu, vb, 31 - lane);
    if (rk < ka) {
        ka = rk;
        va = rv;
    }
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const unsigned long long ok = __shfl_xor_sync(0xffffffffu, ka, stride);
        const int ov = __shfl_xor_sync(0xffffffffu, va, stride);
        const bool lower = (lane & stride) == 0;
        const bool take = lower ? (ok < ka) : (ok > ka);
        if (take) {
            ka = ok;
            va = ov;
        }
    }
}

// The 16-byte chunk at shared address p as fp32 values (8 bf16 or 4 f32).
template <typename T> __device__ __forceinline__ void load_chunk(const unsigned char* p, float (&x)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void load_chunk<__nv_bfloat16>(const unsigned char* p, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const unsigned u4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(u4[k] << 16);
        x[2 * k + 1] = __uint_as_float(u4[k] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void load_chunk<float>(const unsigned char* p, float (&x)[4]) {
    const float4 w = *reinterpret_cast<const float4*>(p);
    x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
}

}  // namespace ice

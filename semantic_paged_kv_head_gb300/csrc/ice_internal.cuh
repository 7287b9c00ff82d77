// Internal definitions shared by the kernels of libice.so.
//
// HBM layout of one index (U units, L composites, list capacity C per unit
// and composite, page size P, head dim D = 128, element type T):
//   dirs       [L][8][132] f32      random +-1/16 directions u[0..D] (splitmix64),
//                                   rows padded to 132 floats for 16-byte loads
//   e_unit     [U] i32              frozen scale exponent, c = 2^e
//   leaf_key   [U][L][C] LeafKey    96-bit prefix + length, sorted (left to right)
//   leaf_rec   [U][L][C] uint4      leaf record: x, y = lower cell corner lo[8]
//                                   (one byte per direction), z = list id << 8 |
//                                   token count, w = prefix length t (the upper
//                                   corner is lo | (2^(8 - known bits(t, j)) - 1))
//   n_leaf     [U][L] i32, next_id [U][L] i32
//   list_cnt   [U][L][C] i32        tokens held by list / page id
//   slot_tok   [U][L][C][P] i32     token of each slot
//   slot_key   [U][L][C][P] u64     Morton key of each slot's token
//   tok_loc    [U][max_tokens] i32  page * P + slot of each token (composite 0)
//   slot_loc1  [U][C][P] i32        tok_loc of the token of each composite-1 slot
//                                   (L = 2 only), so that the selection finds a
//                                   composite-1 candidate's row in one lookup
//   tok_slot1  [U][max_tokens] i32  composite-1 slot (list id * P + slot) of each
//                                   token, -1 if none: the insert updates
//                                   slot_loc1 through it when a page splits
//   page_k/v   [U][C][P][D] T       the physical pages (composite-0 lists)
// The select kernel streams leaf_rec (16 B per leaf); insert is the only
// reader of leaf_key and slot_key.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ice.h"

namespace ice {

constexpr int kD = 128;     // head dimension supported by the kernels
constexpr int kM = 8;       // projections per composite
constexpr int kMaxL = 2;    // composites
constexpr int kMaxG = 8;    // query heads per KV head
constexpr int kMaxP = 64;   // page size
constexpr int kDirStride = kD + 4;  // floats per direction row (u[0..D] + padding)

struct LeafKey {
    unsigned long long pm;  // Morton bits of the prefix (zero below t)
    unsigned int pt;        // token bits of the prefix (zero below t)
    unsigned int t;         // prefix length in bits, 0..96
};
static_assert(sizeof(LeafKey) == 16, "LeafKey must be 16 bytes");

// Device view of an index; passed by value to every kernel.
struct IndexView {
    int U, L, P, G, dtype;
    long long C;           // list capacity per unit and composite
    long long max_tokens;
    const float* dirs;
    int* e_unit;
    LeafKey* leaf_key;
    uint4* leaf_rec;
    // what the selection scan reads of each leaf record, 10 bytes instead of 16:
    // the lower cell corner (8 codes) and (prefix length | count << 7)
    unsigned long long* leaf_lo;
    unsigned short* leaf_tc;
    int* n_leaf;
    int* next_id;
    int* list_cnt;
    int* slot_tok;
    unsigned long long* slot_key;
    int* tok_loc;
    int* slot_loc1;  // nullptr when L = 1
    int* tok_slot1;  // nullptr when L = 1
    void* page_k;
    void* page_v;
    int* status;
    int* n_tok;  // [U] tokens in each unit (build + inserts), advanced by the insert kernel
    int debug;  // ICE_DEBUG_* flags (tests only), 0 in normal use
    int cluster_k;  // blocks per unit of the selection: 0 automatic, 1, 2, 4, 8 or 16
    // 1 when the previous kernel of the launch's stream wrote no index table: the cluster
    // selection then reads the index before it waits on that kernel (programmatic
    // dependent launch), so those reads overlap the previous kernel
    int early_index;

    __host__ __device__ long long ul(int u, int l) const { return (long long)u * L + l; }
    __host__ __device__ long long leaf_base(int u, int l) const { return ul(u, l) * C; }
    __host__ __device__ long long slot_base(int u, int l) const { return ul(u, l) * C * P; }
    __host__ __device__ long long loc1_base(int u) const { return (long long)u * C * P; }
    __host__ __device__ long long page_row(int u, long long page, int slot) const {
        return ((long long)u * C + page) * P + slot;
    }
};

// ---- programmatic dependent launch ---------------------------------------------
// The decode-path kernels are launched with the programmatic stream-serialization
// attribute, so that a kernel's launch (block scheduling, shared-memory setup)
// overlaps the previous kernel of the stream. Each kernel waits here, before its
// first global memory access, until the previous kernel has completed and its
// writes are visible, and then lets the next kernel of the stream be scheduled.
// Launched without the attribute, both instructions return at once.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename Kern, typename... Act>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Act&&>(args)...);
}

// 2^x by the hardware approximation (ex2.approx: a few ulp; results below the
// normal range flush to zero). The attention's softmax weights need far less
// accuracy than the tolerance of its result.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- status word -----------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
    atomicCAS(status, 0, code);
}

// ---- element access ----------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Load 4 consecutive elements (8 B for bf16, 16 B for f32) as floats.
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
    float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
    uint2 x = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(x.x << 16);
    v[1] = __uint_as_float(x.x & 0xFFFF0000u);
    v[2] = __uint_as_float(x.y << 16);
    v[3] = __uint_as_float(x.y & 0xFFFF0000u);
}
__device__ __forceinline__ void load4_nc(const float* p, float (&v)[4]) {
    float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void load4_nc(const __nv_bfloat16* p, float (&v)[4]) {
    uint2 x = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = __uint_as_float(x.x << 16);
    v[1] = __uint_as_float(x.x & 0xFFFF0000u);
    v[2] = __uint_as_float(x.y << 16);
    v[3] = __uint_as_float(x.y & 0xFFFF0000u);
}

// ---- the fixed-order fp32 dot ---------------------------------------------------
// Lane l holds a[4l..4l+3] and b[4l..4l+3]; it accumulates them in order with
// round-to-nearest fused multiply-adds from 0, and the warp then adds lane
// partials pairwise over xor distances 16, 8, 4, 2, 1. Every lane ends with the
// same value. The explicit _rn intrinsics keep the compiler from re-associating
// or contracting anything.
__device__ __forceinline__ float warp_dot_fixed(const float (&a)[4], const float (&b)[4]) {
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc = __fmaf_rn(a[i], b[i], acc);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    return acc;
}

// The same reduction order evaluated by one thread over a full row held in
// shared or global memory (used where one thread owns one key).
__device__ __forceinline__ float thread_dot_fixed_self(const float* x) {
    float acc[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) s = __fmaf_rn(x[4 * l + i], x[4 * l + i], s);
        acc[l] = s;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int l = 0; l < o; ++l) acc[l] = __fadd_rn(acc[l], acc[l + o]);
    return acc[0];
}

// Frozen scale exponent of a unit: the smallest e with 4^e >= maxn (the largest
// squared key norm), kept at e >= -60 so that 2^-2e stays a finite float; 0
// when maxn == 0.
__device__ __forceinline__ int scale_exponent_dev(float maxn) {
    if (!(maxn > 0.0f)) return 0;
    int x;
    float f = frexpf(maxn, &x);  // maxn = f * 2^x, f in [0.5, 1)
    int need = (f == 0.5f) ? x - 1 : x;  // 2e >= need
    int e = need >= 0 ? (need + 1) / 2 : -((-need) / 2);
    return e < -60 ? -60 : e;
}

// code = clamp(floor((p + 1) * 128), 0, 255) evaluated in fp32.
__device__ __forceinline__ int quantise_code(float p) {
    float y = __fmul_rn(__fadd_rn(p, 1.0f), 128.0f);
    float f = floorf(y);
    f = fminf(fmaxf(f, 0.0f), 255.0f);
    return (int)f;
}

// Morton interleave of 8 byte codes, MSB first: output bit 63 - (8*(7-b) + j)
// holds bit b of code j. Spread each code's bits 8 apart, then shift by j.
__device__ __forceinline__ unsigned long long spread8(unsigned int c) {
    unsigned long long x = c & 0xFFu;
    x = (x | (x << 28)) & 0x0000000F0000000FULL;
    x = (x | (x << 14)) & 0x0003000300030003ULL;
    x = (x | (x << 7)) & 0x0101010101010101ULL;
    return x;  // bit b of c moved to bit 8*b
}
__device__ __forceinline__ unsigned long long morton8(const int (&c)[8]) {
    unsigned long long m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m |= spread8((unsigned)c[j]) << (7 - j);
    return m;
}

// Code cell of a prefix of length t: known bits per direction, then lo/hi.
__device__ __forceinline__ uint4 cell_of_prefix(unsigned long long pm, unsigned int t) {
    unsigned char lo[8], hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int bj = t >= 64 ? 8 : (int)((t + 7 - j) >> 3);
        if (bj > 8) bj = 8;
        unsigned int v = 0;
#pragma unroll
        for (int b = 7; b >= 0; --b) {
            unsigned int bit = (unsigned int)(pm >> (8 * b + 7 - j)) & 1u;
            v |= bit << b;
        }
        unsigned int mask = bj == 0 ? 0u : (0xFFu << (8 - bj)) & 0xFFu;
        lo[j] = (unsigned char)(v & mask);
        hi[j] = (unsigned char)((v & mask) | (~mask & 0xFFu));
    }
    uint4 r;
    r.x = lo[0] | (lo[1] << 8) | (lo[2] << 16) | ((unsigned)lo[3] << 24);
    r.y = lo[4] | (lo[5] << 8) | (lo[6] << 16) | ((unsigned)lo[7] << 24);
    r.z = hi[0] | (hi[1] << 8) | (hi[2] << 16) | ((unsigned)hi[3] << 24);
    r.w = hi[4] | (hi[5] << 8) | (hi[6] << 16) | ((unsigned)hi[7] << 24);
    return r;
}

// Leaf record: lower cell corner of a prefix, list id, count, prefix length.
__device__ __forceinline__ uint4 make_leaf_rec(unsigned long long pm, unsigned t, int id, int cnt) {
    const uint4 cell = cell_of_prefix(pm, t);
    return make_uint4(cell.x, cell.y, ((unsigned)id << 8) | (unsigned)cnt, t);
}
__device__ __forceinline__ int rec_id(const uint4& r) { return (int)(r.z >> 8); }

// Writes leaf record r at position lb (leaf_base + index) and its scan copy.
__device__ __forceinline__ void put_leaf(const IndexView& v, long long lb, const uint4& r) {
    v.leaf_rec[lb] = r;
    v.leaf_lo[lb] = ((unsigned long long)r.y << 32) | r.x;
    v.leaf_tc[lb] = (unsigned short)(min(r.w, 127u) | ((r.z & 0xFFu) << 7));
}
// Scan-copy fields: prefix length and token count.
__device__ __forceinline__ int tc_t(unsigned tc) { return (int)(tc & 127u); }
__device__ __forceinline__ int tc_cnt(unsigned tc) { return (int)(tc >> 7); }
__device__ __forceinline__ int rec_cnt(const uint4& r) { return (int)(r.z & 0xFFu); }

// Length of the common prefix of two 96-bit keys.
__device__ __forceinline__ int lcp96(unsigned long long am, unsigned int at, unsigned long long bm,
                                     unsigned int bt) {
    unsigned long long x = am ^ bm;
    if (x) return __clzll((long long)x);
    unsigned int y = at ^ bt;
    if (y) return 64 + __clz((int)y);
    return 96;
}

// Prefix of length t of a 96-bit key.
__device__ __forceinline__ void prefix96(unsigned long long m, unsigned int tk, int t,
                                         unsigned long long& pm, unsigned int& pt) {
    if (t >= 64) {
        pm = m;
        int tb = t - 64;
        pt = tb == 0 ? 0u : (tb >= 32 ? tk : (tk & ~((1u << (32 - tb)) - 1u)));
    } else {
        pm = t == 0 ? 0ull : (m & ~((1ull << (64 - t)) - 1ull));
        pt = 0u;
    }
}

__device__ __forceinline__ bool key_less(unsigned long long am, unsigned int at,
                                         unsigned long long bm, unsigned int bt) {
    return am != bm ? am < bm : at < bt;
}

// Bit t (0 = most significant) of a 96-bit key.
__device__ __forceinline__ int key_bit96(unsigned long long m, unsigned int tk, int t) {
    return t < 64 ? (int)((m >> (63 - t)) & 1ull) : (int)((tk >> (95 - t)) & 1u);
}

// Order-preserving map of a float score to an unsigned key in which a HIGHER
// score gives a LOWER key (+0 and -0 map to the same key).
__device__ __forceinline__ unsigned int score_key_desc(float s) {
    s = __fadd_rn(s, 0.0f);  // -0 -> +0
    unsigned int b = __float_as_uint(s);
    unsigned int asc = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ~asc;
}

// ---- build scratch (stream-ordered, released at the end of ice_build) --------------
struct BuildScratch {
    float* nrm2 = nullptr;             // [U][n] squared key norms
    unsigned int* umax = nullptr;      // [U] max squared norm (float bits)
    unsigned long long* mk[2] = {nullptr, nullptr};  // [L][U][n] Morton keys (sort buffers)
    int* tk[2] = {nullptr, nullptr};   // [L][U][n] token ids (sort buffers)
    int* hist = nullptr;               // [L*U][256][tiles] radix counts / offsets
    int* leaf_of = nullptr;            // [L][U][n] leaf number of each sorted position
    int* leaf_start = nullptr;         // [L][U][n] first position of each leaf
    unsigned char* tdepth = nullptr;   // [L][U][n] leaf depth of each sorted position
    int* nleaf = nullptr;              // [L][U] leaves per segment
    float* praw = nullptr;             // [U][n][16] unscaled projections (tensor-core path)
    int* err = nullptr;                // set when a bounded wait of the build ran out
};
// dirs_bf16_exact: every direction component is exact in bf16 (the +-1/16
// directions); bf16 keys then take the tensor-core projection.
cudaError_t build_phase1(int dtype, const void* keys, int U, int L, int P, long long n,
                         const float* dirs, bool dirs_bf16_exact, int* e_unit, BuildScratch& s,
                         cudaStream_t st, int* final_buf);
cudaError_t build_phase2(const IndexView& v, const void* keys, const void* values, long long n,
                         BuildScratch& s, int cur, cudaStream_t st);
cudaError_t scratch_alloc(BuildScratch& s, int U, int L, long long n, bool with_praw,
                          cudaStream_t st);
void scratch_free(BuildScratch& s, cudaStream_t st);
int select_smem_bytes(long long C, int L, int P, int n_cand, int n_sel, int G, bool fused);
bool select_insert_fits(long long C, int L, int P, int n_cand, int n_sel, int es);
cudaError_t select_prepare();
// The selection spread over a thread-block cluster of K blocks per unit
// (ice_select_cluster.cu): the cluster size chosen for U units, the dynamic
// shared memory of a launch (-1 if the cluster path cannot take it: K not a
// power of two in [max(2, L), 16], n_sel > 32, or the tables too large), the
// per-device setup, and the launch (*launched false if clusters of that size
// cannot be resident; nothing is launched then).
int select_cluster_auto(int U, int L);
cudaError_t launch_select_heads_cluster(const IndexView& v, const void* q, int n_sel, int n_cand,
                                        int32_t* page_ids, int32_t* n_pages, cudaStream_t s,
                                        bool* launched);
int select_cluster_bytes(const IndexView& v, int K, int n_sel, int n_cand, bool fused);
cudaError_t select_cluster_prepare();
cudaError_t launch_select_cluster(const IndexView& v, int K, const void* q, int n_sel, int n_cand,
                                  int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                                  cudaStream_t s, bool* launched);

// ---- launchers (implemented in the .cu files) --------------------------------------
cudaError_t launch_insert(const IndexView& v, const void* k, const void* val, cudaStream_t s);
cudaError_t insert_prepare(int P, int dtype);
// out == nullptr: select only; otherwise select and attend over the selection.
// Largest dynamic shared memory of a select block: the opt-in maximum per block
// of the GPU (227 KB) less room for the kernel's static shared variables.
constexpr int kSelSmemMax = 220 * 1024;
// reselect: nullable [U]; a unit whose flag is 0 keeps its pages (page_ids,
// n_pages unchanged) and, in the fused call, attends over them
// knew, vnew: nullable; with the fused kernel, each block first inserts its
// unit's new token (the decode step in one launch)
cudaError_t launch_select(const IndexView& v, const void* q, int n_sel, int n_cand,
                          int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                          const int32_t* reselect, cudaStream_t s, const void* knew = nullptr,
                          const void* vnew = nullptr);
// Per-query-head selection (block = unit x head) and the union of each unit's
// per-head page lists in head-major first-occurrence order.
cudaError_t launch_select_heads(const IndexView& v, const void* q, int n_sel, int n_cand,
                                int32_t* page_ids, int32_t* n_pages, cudaStream_t s);
cudaError_t launch_union(int U, int G, int n_sel, const int32_t* head_ids, const int32_t* head_n,
                         int32_t* ids, int32_t* n, cudaStream_t s);
// Reuse decision per unit (query codes against the codes of the unit's last
// selection, and the reuse age); writes reselect[U] and updates codes/age.
cudaError_t launch_reuse(const IndexView& v, const void* q, int r, unsigned char* codes, int* age,
                         int32_t* reselect, cudaStream_t s);
// Plain-load attention (any pool; the path for a pool in pinned host memory).
cudaError_t launch_attn(const IndexView& v, const void* q, const int32_t* page_ids,
                        const int32_t* n_pages, int page_stride, void* out, cudaStream_t s);
// Attention with the pages staged by bulk copies (a pool in device memory). Up to
// one block per SM of the 152 it is faster than the plain-load kernel (8 units:
// 12.3 against 14.3 us per call); with more units the plain kernel, two blocks per
// SM with loads in flight during the arithmetic, is faster (256 units: 18.4 against
// 20.5 us).
constexpr int kAttnStagedMaxUnits = 152;
cudaError_t launch_attn_staged(const IndexView& v, const void* q, const int32_t* page_ids,
                               const int32_t* n_pages, int page_stride, void* out, cudaStream_t s);

}  // namespace ice

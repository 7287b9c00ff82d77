// C ABI of libice.so: argument checks, memory ownership and launch order.
// See include/ice.h for the contract of each call.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "ice_internal.cuh"

namespace {
// NVTX range over one API call (visible in Nsight timelines; free otherwise).
struct ApiRange {
    explicit ApiRange(const char* name) { nvtxRangePushA(name); }
    ~ApiRange() { nvtxRangePop(); }
};
}  // namespace

using namespace ice;

struct ice_index {
    ice_params p;
    int U = 0, G = 0;
    long long C = 0;
    long long n_tok = 0;
    size_t bytes = 0;
    size_t host_bytes = 0;
    int device = 0;
    std::vector<void*> owned;
    std::vector<void*> owned_host;  // pinned host page pool (ICE_KV_HOST)
    // selection reuse across steps (ice_select_attn_reuse), allocated on first use
    unsigned char* reuse_codes = nullptr;  // [U][kMaxL * kM] query codes of the last selection
    int* reuse_age = nullptr;              // [U] reuses since that selection; -1 = none
    int32_t* reuse_flag = nullptr;         // [U] 1 where this step selects
    int reuse_budget = -1;
    // the stream of the last launch that wrote index tables (an insert), until a selection
    // on that stream has waited for it; until then a selection on that stream reads the
    // index only after its wait on the previous kernel
    void* write_stream = nullptr;
    bool write_pending = false;
    IndexView v;
};

namespace {

// The view a selection launch on `stream` gets: the index may be read before the wait on
// the stream's previous kernel unless that kernel may have written it.
IndexView select_view(const ice_index* ix, void* stream) {
    IndexView vv = ix->v;
    vv.early_index = (ix->write_pending && ix->write_stream == stream) ? 0 : 1;
    return vv;
}

// A selection was launched on `stream`: it waits for the write pending there.
void select_issued(ice_index* ix, void* stream) {
    if (ix->write_pending && ix->write_stream == stream) ix->write_pending = false;
}

void index_written(ice_index* ix, void* stream) {
    ix->write_pending = true;
    ix->write_stream = stream;
}

// splitmix64 (Steele, Lea & Flood 2014), the generator of the directions.
uint64_t sm64(uint64_t& s) {
    s += 0x9E3779B97F4A7C15ULL;
    uint64_t z = s;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

int check_params(const ice_params* p) {
    if (!p) return ICE_ERR_INVALID_ARG;
    if (p->d != kD || p->n_proj != kM) return ICE_ERR_UNSUPPORTED;
    if (p->n_kv_heads < 1 || p->n_layers < 1 || p->batch < 1) return ICE_ERR_INVALID_ARG;
    if (p->n_q_heads < p->n_kv_heads || p->n_q_heads % p->n_kv_heads) return ICE_ERR_INVALID_ARG;
    const int G = p->n_q_heads / p->n_kv_heads;
    if (!(G == 1 || G == 2 || G == 4 || G == 8)) return ICE_ERR_UNSUPPORTED;
    if (p->page_size < 1 || p->page_size > kMaxP) return ICE_ERR_INVALID_ARG;
    if (p->n_composite < 1 || p->n_composite > kMaxL) return ICE_ERR_INVALID_ARG;
    if (p->n_cand < 0) return ICE_ERR_INVALID_ARG;
    if (p->dtype != ICE_F32 && p->dtype != ICE_BF16) return ICE_ERR_INVALID_ARG;
    if (p->kv_location != ICE_KV_DEVICE && p->kv_location != ICE_KV_HOST) return ICE_ERR_INVALID_ARG;
    if (p->dir_kind != ICE_DIR_RADEMACHER && p->dir_kind != ICE_DIR_GAUSSIAN) return ICE_ERR_INVALID_ARG;
    if (p->max_tokens < 0 || p->max_tokens > (1LL << 30)) return ICE_ERR_INVALID_ARG;
    const long long units = (long long)p->batch * p->n_layers * p->n_kv_heads;
    if (units > (1LL << 24)) return ICE_ERR_INVALID_ARG;
    return ICE_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The address a kernel dereferences for a caller's buffer: device memory of the
// index's GPU (or managed memory) as given, page-locked host memory through its
// device mapping (the kernels then read or write it over the CPU-GPU link).
// False for anything the GPU cannot address (pageable host memory, memory of
// another GPU, a bad pointer): the call is refused before any launch. While
// `stream` is being captured into a CUDA graph the pointer is taken as given
// (no driver query is made during a capture; the eager calls that precede a
// capture check the same buffers).
bool kernel_addr(const ice_index* ix, const void* p, void* stream, const void** out) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing((cudaStream_t)stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cs != cudaStreamCaptureStatusNone) {
        *out = p;
        return true;
    }
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if ((a.type == cudaMemoryTypeDevice && a.device == ix->device) || a.type == cudaMemoryTypeManaged) {
        *out = p;
        return true;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
        *out = a.devicePointer;
        return true;
    }
    return false;
}

template <typename T>
cudaError_t dev_alloc(ice_index* ix, T** out, size_t count) {
    void* p = nullptr;
    const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) return e;
    ix->owned.push_back(p);
    ix->bytes += bytes;
    *out = reinterpret_cast<T*>(p);
    return cudaSuccess;
}

// Pinned host memory mapped into the device's address space; *out is the
// device-side address of it.
cudaError_t host_alloc(ice_index* ix, unsigned char** out, size_t bytes) {
    void* h = nullptr;
    bytes = std::max<size_t>(bytes, 16);
    cudaError_t e = cudaHostAlloc(&h, bytes, cudaHostAllocMapped);
    if (e != cudaSuccess) return e;
    ix->owned_host.push_back(h);
    ix->host_bytes += bytes;
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, h, 0);
    if (e != cudaSuccess) return e;
    *out = reinterpret_cast<unsigned char*>(d);
    return cudaSuccess;
}

void free_all(ice_index* ix) {
    for (void* p : ix->owned) cudaFree(p);
    ix->owned.clear();
    for (void* p : ix->owned_host) cudaFreeHost(p);
    ix->owned_host.clear();
}

}  // namespace

// Replaces a non-null buffer argument by its kernel address, or refuses the call.
#define ICE_KERNEL_ADDR(ptr)                                                   \
    do {                                                                       \
        if ((ptr) != nullptr) {                                                \
            const void* d_ = nullptr;                                          \
            if (!kernel_addr(ix, (ptr), stream, &d_)) return ICE_ERR_INVALID_ARG; \
            (ptr) = (decltype(ptr))(d_);                                       \
        }                                                                      \
    } while (0)

extern "C" {

const char* ice_status_string(int s) {
    switch (s) {
        case ICE_OK: return "ok";
        case ICE_ERR_INVALID_ARG: return "invalid argument";
        case ICE_ERR_CAPACITY: return "capacity exhausted";
        case ICE_ERR_CUDA: return "CUDA runtime error";
        case ICE_ERR_TIMEOUT: return "bounded device wait timed out";
        case ICE_ERR_BOUNDS: return "page id or page count out of range";
        case ICE_ERR_UNSUPPORTED: return "unsupported parameters";
        default: return "unknown status";
    }
}

int ice_build(const ice_params* params, const void* keys, const void* values, int64_t n_tokens,
              void* stream, ice_index** out) {
    ApiRange range_("ice_build");
    if (!out) return ICE_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = check_params(params);
    if (rc) return rc;
    if (n_tokens < 0 || n_tokens > params->max_tokens || n_tokens > (1LL << 30))
        return ICE_ERR_INVALID_ARG;
    if (n_tokens > 0 && (!keys || !values || !aligned16(keys) || !aligned16(values)))
        return ICE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    ice_index* ix = new (std::nothrow) ice_index();
    if (!ix) return ICE_ERR_CUDA;
    ix->p = *params;
    if (ix->p.n_cand == 0) ix->p.n_cand = 0;  // resolved per select call (budget)
    ix->U = params->batch * params->n_layers * params->n_kv_heads;
    ix->G = params->n_q_heads / params->n_kv_heads;
    ix->n_tok = n_tokens;
    cudaGetDevice(&ix->device);
    const int U = ix->U, L = params->n_composite, P = params->page_size;
    const long long n = n_tokens;
    IndexView& v = ix->v;
    std::memset(&v, 0, sizeof(v));
    v.U = U;
    v.L = L;
    v.P = P;
    v.G = ix->G;
    v.dtype = params->dtype;
    v.max_tokens = std::max<long long>(1, params->max_tokens);

    // directions, on the host from splitmix64(seed) in the order (composite,
    // direction, component). Rademacher: sign bit -> -1/16, else +1/16.
    // Gaussian: z / 16 with z = sqrt(-2 ln u1) cos(2 pi u2) (Box-Muller) of the
    // next two draws, u1 = ((x1 >> 11) + 1) 2^-53, u2 = (x2 >> 11) 2^-53, in double.
    std::vector<float> dirs((size_t)L * kM * kDirStride, 0.0f);
    {
        uint64_t s = params->seed;
        const double two_pi = 2.0 * 3.14159265358979323846;
        for (int l = 0; l < L; ++l)
            for (int j = 0; j < kM; ++j)
                for (int i = 0; i <= kD; ++i) {
                    float& c = dirs[((size_t)l * kM + j) * kDirStride + i];
                    if (params->dir_kind == ICE_DIR_GAUSSIAN) {
                        const uint64_t x1 = sm64(s), x2 = sm64(s);
                        const double u1 = (double)((x1 >> 11) + 1) * 0x1.0p-53;
                        const double u2 = (double)(x2 >> 11) * 0x1.0p-53;
                        c = (float)(std::sqrt(-2.0 * std::log(u1)) * std::cos(two_pi * u2) / 16.0);
                    } else {
                        c = (sm64(s) >> 63) ? -0.0625f : 0.0625f;
                    }
                }
    }
    cudaError_t e = cudaSuccess;
    float* d_dirs = nullptr;
    int* d_status = nullptr;
    int* d_e = nullptr;
    int* d_ntok = nullptr;
    const std::vector<int> ntok0((size_t)U, (int)n);
    if ((e = dev_alloc(ix, &d_dirs, dirs.size())) != cudaSuccess) goto fail;
    if ((e = dev_alloc(ix, &d_ntok, (size_t)U)) != cudaSuccess) goto fail;
    if ((e = cudaMemcpyAsync(d_ntok, ntok0.data(), sizeof(int) * U, cudaMemcpyHostToDevice, st)) !=
        cudaSuccess)
        goto fail;
    if ((e = dev_alloc(ix, &d_status, 1)) != cudaSuccess) goto fail;
    if ((e = dev_alloc(ix, &d_e, (size_t)U)) != cudaSuccess) goto fail;
    if ((e = cudaMemcpyAsync(d_dirs, dirs.data(), dirs.size() * sizeof(float),
                             cudaMemcpyHostToDevice, st)) != cudaSuccess)
        goto fail;
    if ((e = cudaMemsetAsync(d_status, 0, sizeof(int), st)) != cudaSuccess) goto fail;
    if ((e = cudaMemsetAsync(d_e, 0, sizeof(int) * U, st)) != cudaSuccess) goto fail;
    v.dirs = d_dirs;
    v.status = d_status;
    v.e_unit = d_e;
    v.n_tok = d_ntok;
    {
        BuildScratch s;
        std::vector<int> nleaf((size_t)L * U, 0);
        int cur = 0;
        if (n > 0) {
            const bool tc = params->dtype == ICE_BF16 && params->dir_kind == ICE_DIR_RADEMACHER;
            if ((e = scratch_alloc(s, U, L, n, tc, st)) != cudaSuccess) {
                scratch_free(s, st);
                goto fail;
            }
            e = build_phase1(params->dtype, keys, U, L, P, n, d_dirs,
                             params->dir_kind == ICE_DIR_RADEMACHER, d_e, s, st, &cur);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(nleaf.data(), s.nleaf, sizeof(int) * L * U,
                                    cudaMemcpyDeviceToHost, st);
            if (e == cudaSuccess) e = cudaStreamSynchronize(st);
            int berr = 0;
            if (e == cudaSuccess) e = cudaMemcpy(&berr, s.err, sizeof(int), cudaMemcpyDeviceToHost);
            if (e == cudaSuccess && berr != 0) {  // a bounded wait of the key pass ran out
                scratch_free(s, st);
                cudaStreamSynchronize(st);
                free_all(ix);
                delete ix;
                return ICE_ERR_TIMEOUT;
            }
            if (e != cudaSuccess) {
                scratch_free(s, st);
                goto fail;
            }
        }
        // list capacity: the largest leaf count plus one new leaf per future insert
        long long mx = 0;
        for (int x : nleaf) mx = std::max<long long>(mx, x);
        // rounded up to 64 leaves: the selection scan copies leaf records in
        // aligned chunks of 64 that must stay inside the list
        ix->C = (std::max<long long>(1, mx + (v.max_tokens - n)) + 63) / 64 * 64;
        if (ix->C >= (1LL << 24) || ix->C * P > (1LL << 31) - 1) {
            scratch_free(s, st);
            free_all(ix);
            delete ix;
            return ICE_ERR_CAPACITY;
        }
        v.C = ix->C;
        const long long C = ix->C;
        const size_t es = params->dtype == ICE_BF16 ? 2 : 4;
        bool okc = true;
        okc = okc && dev_alloc(ix, &v.leaf_key, (size_t)U * L * C) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.leaf_rec, (size_t)U * L * C) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.leaf_lo, (size_t)U * L * C) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.leaf_tc, (size_t)U * L * C) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.n_leaf, (size_t)U * L) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.next_id, (size_t)U * L) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.list_cnt, (size_t)U * L * C) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.slot_tok, (size_t)U * L * C * P) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.slot_key, (size_t)U * L * C * P) == cudaSuccess;
        okc = okc && dev_alloc(ix, &v.tok_loc, (size_t)U * v.max_tokens) == cudaSuccess;
        if (L > 1) {
            okc = okc && dev_alloc(ix, &v.slot_loc1, (size_t)U * C * P) == cudaSuccess;
            okc = okc && dev_alloc(ix, &v.tok_slot1, (size_t)U * v.max_tokens) == cudaSuccess;
        }
        unsigned char* pk = nullptr;
        unsigned char* pv = nullptr;
        const size_t pool = (size_t)U * C * P * kD * es;
        if (params->kv_location == ICE_KV_HOST) {
            okc = okc && host_alloc(ix, &pk, pool) == cudaSuccess;
            okc = okc && host_alloc(ix, &pv, pool) == cudaSuccess;
        } else {
            okc = okc && dev_alloc(ix, &pk, pool) == cudaSuccess;
            okc = okc && dev_alloc(ix, &pv, pool) == cudaSuccess;
        }
        if (!okc) {
            scratch_free(s, st);
            cudaGetLastError();
            free_all(ix);
            delete ix;
            return ICE_ERR_CAPACITY;
        }
        v.page_k = pk;
        v.page_v = pv;
        if (select_prepare() != cudaSuccess || select_cluster_prepare() != cudaSuccess ||
            insert_prepare(P, params->dtype) != cudaSuccess) {
            scratch_free(s, st);
            cudaGetLastError();
            free_all(ix);
            delete ix;
            return ICE_ERR_CUDA;
        }
        e = cudaMemsetAsync(v.n_leaf, 0, sizeof(int) * U * L, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(v.next_id, 0, sizeof(int) * U * L, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(v.list_cnt, 0, sizeof(int) * U * L * C, st);
        if (e == cudaSuccess)  // -1: token not placed yet
            e = cudaMemsetAsync(v.tok_loc, 0xFF, sizeof(int) * U * v.max_tokens, st);
        if (e == cudaSuccess && L > 1)
            e = cudaMemsetAsync(v.slot_loc1, 0xFF, sizeof(int) * U * C * P, st);
        if (e == cudaSuccess && L > 1)  // -1: token in no composite-1 list yet
            e = cudaMemsetAsync(v.tok_slot1, 0xFF, sizeof(int) * U * v.max_tokens, st);
        if (e == cudaSuccess && n > 0) e = build_phase2(v, keys, values, n, s, cur, st);
        scratch_free(s, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) goto fail;
    }
    *out = ix;
    return ICE_OK;
fail:
    cudaGetLastError();
    free_all(ix);
    delete ix;
    return ICE_ERR_CUDA;
}

int ice_insert(ice_index* ix, const void* k, const void* v, void* stream) {
    ApiRange range_("ice_insert");
    if (!ix || !k || !v || !aligned16(k) || !aligned16(v)) return ICE_ERR_INVALID_ARG;
    ICE_KERNEL_ADDR(k);
    ICE_KERNEL_ADDR(v);
    if (ix->n_tok >= ix->v.max_tokens) return ICE_ERR_CAPACITY;
    cudaError_t e = launch_insert(ix->v, k, v, (cudaStream_t)stream);
    if (e != cudaSuccess) return ICE_ERR_CUDA;
    index_written(ix, stream);
    ix->n_tok += 1;
    return ICE_OK;
}

// cluster_ok: the call may run on the cluster selection kernel (plain select
// and select + attention), which holds larger per-unit tables than one block.
static int select_args(const ice_index* ix, const void* q, int32_t token_budget,
                       const int32_t* page_ids, const int32_t* n_pages, const void* out,
                       bool cluster_ok = false) {
    if (!ix || !q || !page_ids || !n_pages || !aligned16(q)) return ICE_ERR_INVALID_ARG;
    if (out && !aligned16(out)) return ICE_ERR_INVALID_ARG;
    const int P = ix->p.page_size;
    if (token_budget < P || token_budget % P) return ICE_ERR_INVALID_ARG;
    const int n_sel = token_budget / P;
    if (n_sel > 512) return ICE_ERR_UNSUPPORTED;
    const int n_cand = ix->p.n_cand > 0 ? ix->p.n_cand : token_budget;
    if (n_cand > (1 << 16)) return ICE_ERR_UNSUPPORTED;
    const bool one_fits =
        select_smem_bytes(ix->C, ix->p.n_composite, P, n_cand, n_sel, ix->G, out != nullptr) <= kSelSmemMax;
    if (cluster_ok) {
        const int forced = ix->v.cluster_k;
        if (forced >= 2)
            return select_cluster_bytes(ix->v, forced, n_sel, n_cand, out != nullptr) >= 0
                       ? ICE_OK
                       : ICE_ERR_UNSUPPORTED;
        if (forced == 1) return one_fits ? ICE_OK : ICE_ERR_UNSUPPORTED;
        if (one_fits) return ICE_OK;
        const int K = std::max(2, select_cluster_auto(ix->U, ix->p.n_composite));
        return select_cluster_bytes(ix->v, K, n_sel, n_cand, out != nullptr) >= 0 ? ICE_OK
                                                                                  : ICE_ERR_UNSUPPORTED;
    }
    if (!one_fits) return ICE_ERR_UNSUPPORTED;
    return ICE_OK;
}

static int select_common(ice_index* ix, const void* q, int32_t token_budget, int32_t* page_ids,
                         int32_t* n_pages, int32_t* stats, void* out, void* stream,
                         const int32_t* reselect = nullptr) {
    const int a = select_args(ix, q, token_budget, page_ids, n_pages, out, reselect == nullptr);
    if (a != ICE_OK) return a;
    ICE_KERNEL_ADDR(q);
    ICE_KERNEL_ADDR(page_ids);
    ICE_KERNEL_ADDR(n_pages);
    ICE_KERNEL_ADDR(stats);
    ICE_KERNEL_ADDR(out);
    const int P = ix->p.page_size;
    const int n_sel = token_budget / P;
    const int n_cand = ix->p.n_cand > 0 ? ix->p.n_cand : token_budget;
    cudaError_t e = launch_select(select_view(ix, stream), q, n_sel, n_cand, page_ids, n_pages, stats,
                                  out, reselect, (cudaStream_t)stream);
    if (e != cudaSuccess) return ICE_ERR_CUDA;
    select_issued(ix, stream);
    return ICE_OK;
}

int ice_select(ice_index* ix, const void* q, int32_t token_budget, int32_t* page_ids,
               int32_t* n_pages, int32_t* stats, void* stream) {
    ApiRange range_("ice_select");
    return select_common(ix, q, token_budget, page_ids, n_pages, stats, nullptr, stream);
}

int ice_select_attn(ice_index* ix, const void* q, int32_t token_budget, int32_t* page_ids,
                    int32_t* n_pages, int32_t* stats, void* out, void* stream) {
    ApiRange range_("ice_select_attn");
    if (!ix || !out) return ICE_ERR_INVALID_ARG;
    if (ix->p.kv_location == ICE_KV_HOST) {
        // the fused kernel stages pages with bulk tensor-memory copies; a host pool
        // is read by the two plain-load kernels instead
        if (!aligned16(out)) return ICE_ERR_INVALID_ARG;
        int r = select_common(ix, q, token_budget, page_ids, n_pages, stats, nullptr, stream);
        if (r != ICE_OK) return r;
        return ice_sparse_attn(ix, q, page_ids, n_pages, token_budget / ix->p.page_size, out, stream);
    }
    return select_common(ix, q, token_budget, page_ids, n_pages, stats, out, stream);
}

int ice_select_attn_reuse(ice_index* ix, const void* q, int32_t token_budget, int32_t r,
                          int32_t* page_ids, int32_t* n_pages, int32_t* reselected, void* out,
                          void* stream) {
    ApiRange range_("ice_select_attn_reuse");
    if (!ix || !out || r < 0) return ICE_ERR_INVALID_ARG;
    const int a = select_args(ix, q, token_budget, page_ids, n_pages, out);
    if (a != ICE_OK) return a;
    ICE_KERNEL_ADDR(q);
    ICE_KERNEL_ADDR(page_ids);
    ICE_KERNEL_ADDR(n_pages);
    ICE_KERNEL_ADDR(reselected);
    ICE_KERNEL_ADDR(out);
    cudaStream_t st = (cudaStream_t)stream;
    const int U = ix->U;
    if (!ix->reuse_age) {
        bool ok = dev_alloc(ix, &ix->reuse_codes, (size_t)U * kMaxL * kM) == cudaSuccess;
        ok = ok && dev_alloc(ix, &ix->reuse_age, (size_t)U) == cudaSuccess;
        ok = ok && dev_alloc(ix, &ix->reuse_flag, (size_t)U) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            return ICE_ERR_CAPACITY;
        }
        ix->reuse_budget = -1;
    }
    if (token_budget != ix->reuse_budget) {  // kept pages were chosen for another budget
        if (cudaMemsetAsync(ix->reuse_age, 0xFF, sizeof(int) * U, st) != cudaSuccess) return ICE_ERR_CUDA;
        ix->reuse_budget = token_budget;
    }
    if (launch_reuse(ix->v, q, r, ix->reuse_codes, ix->reuse_age, ix->reuse_flag, st) != cudaSuccess)
        return ICE_ERR_CUDA;
    int res;
    if (ix->p.kv_location == ICE_KV_HOST) {
        res = select_common(ix, q, token_budget, page_ids, n_pages, nullptr, nullptr, stream,
                            ix->reuse_flag);
        if (res == ICE_OK)
            res = ice_sparse_attn(ix, q, page_ids, n_pages, token_budget / ix->p.page_size, out, stream);
    } else {
        res = select_common(ix, q, token_budget, page_ids, n_pages, nullptr, out, stream,
                            ix->reuse_flag);
    }
    if (res == ICE_OK && reselected &&
        cudaMemcpyAsync(reselected, ix->reuse_flag, sizeof(int32_t) * U, cudaMemcpyDefault, st) !=
            cudaSuccess)
        return ICE_ERR_CUDA;
    return res;
}

int ice_decode_step(ice_index* ix, const void* k, const void* v, const void* q,
                    int32_t token_budget, int32_t* page_ids, int32_t* n_pages, void* out,
                    void* stream) {
    ApiRange range_("ice_decode_step");
    if (!ix || !out) return ICE_ERR_INVALID_ARG;
    const int a = select_args(ix, q, token_budget, page_ids, n_pages, out);
    if (a != ICE_OK) return a;
    if (!k || !v || !aligned16(k) || !aligned16(v)) return ICE_ERR_INVALID_ARG;
    if (ix->n_tok >= ix->v.max_tokens) return ICE_ERR_CAPACITY;
    ICE_KERNEL_ADDR(k);
    ICE_KERNEL_ADDR(v);
    ICE_KERNEL_ADDR(q);
    ICE_KERNEL_ADDR(page_ids);
    ICE_KERNEL_ADDR(n_pages);
    ICE_KERNEL_ADDR(out);
    const int P = ix->p.page_size;
    const int n_sel = token_budget / P;
    const int n_cand = ix->p.n_cand > 0 ? ix->p.n_cand : token_budget;
    const int es = ix->p.dtype == ICE_BF16 ? 2 : 4;
    // few units: the insert kernel, then the selection over a cluster of blocks per unit
    // (two launches, both capturable); many units: one launch in which every block
    // inserts its unit's token and then selects and attends
    const int Kc = ix->v.cluster_k > 0 ? ix->v.cluster_k : select_cluster_auto(ix->U, ix->p.n_composite);
    if (ix->p.kv_location == ICE_KV_DEVICE && Kc >= 2 &&
        select_cluster_bytes(ix->v, Kc, n_sel, n_cand, true) >= 0) {
        if (launch_insert(ix->v, k, v, (cudaStream_t)stream) != cudaSuccess) return ICE_ERR_CUDA;
        index_written(ix, stream);
        ix->n_tok += 1;
        cudaError_t e = launch_select(select_view(ix, stream), q, n_sel, n_cand, page_ids, n_pages,
                                      nullptr, out, nullptr, (cudaStream_t)stream);
        if (e != cudaSuccess) return ICE_ERR_CUDA;
        select_issued(ix, stream);
        return ICE_OK;
    }
    if (ix->p.kv_location == ICE_KV_DEVICE &&
        select_insert_fits(ix->C, ix->p.n_composite, P, n_cand, n_sel, es)) {
        // one launch: every block inserts its unit's token, then selects and attends
        cudaError_t e = launch_select(select_view(ix, stream), q, n_sel, n_cand, page_ids, n_pages,
                                      nullptr, out, nullptr, (cudaStream_t)stream, k, v);
        if (e != cudaSuccess) return ICE_ERR_CUDA;
        index_written(ix, stream);  // its blocks insert before they select
        ix->n_tok += 1;
        return ICE_OK;
    }
    const int r = ice_insert(ix, k, v, stream);
    if (r != ICE_OK) return r;
    return ice_select_attn(ix, q, token_budget, page_ids, n_pages, nullptr, out, stream);
}

int ice_select_heads(ice_index* ix, const void* q, int32_t token_budget, int32_t* head_page_ids,
                     int32_t* head_n_pages, int32_t* page_ids, int32_t* n_pages, void* stream) {
    ApiRange range_("ice_select_heads");
    const int a = select_args(ix, q, token_budget, page_ids, n_pages, nullptr);
    if (a != ICE_OK) return a;
    if (!head_page_ids || !head_n_pages) return ICE_ERR_INVALID_ARG;
    ICE_KERNEL_ADDR(q);
    ICE_KERNEL_ADDR(head_page_ids);
    ICE_KERNEL_ADDR(head_n_pages);
    ICE_KERNEL_ADDR(page_ids);
    ICE_KERNEL_ADDR(n_pages);
    const int n_sel = token_budget / ix->p.page_size;
    if (ix->G * n_sel > 512) return ICE_ERR_UNSUPPORTED;  // the attention's page-list bound
    const int n_cand = ix->p.n_cand > 0 ? ix->p.n_cand : token_budget;
    cudaStream_t st = (cudaStream_t)stream;
    if (launch_select_heads(select_view(ix, stream), q, n_sel, n_cand, head_page_ids, head_n_pages,
                            st) != cudaSuccess)
        return ICE_ERR_CUDA;
    select_issued(ix, stream);
    if (launch_union(ix->U, ix->G, n_sel, head_page_ids, head_n_pages, page_ids, n_pages, st) !=
        cudaSuccess)
        return ICE_ERR_CUDA;
    return ICE_OK;
}

int ice_reuse_reset(ice_index* ix, void* stream) {
    if (!ix) return ICE_ERR_INVALID_ARG;
    if (!ix->reuse_age) return ICE_OK;
    return cudaMemsetAsync(ix->reuse_age, 0xFF, sizeof(int) * ix->U, (cudaStream_t)stream) == cudaSuccess
               ? ICE_OK
               : ICE_ERR_CUDA;
}

int ice_sparse_attn(ice_index* ix, const void* q, const int32_t* page_ids, const int32_t* n_pages,
                    int32_t page_stride, void* out, void* stream) {
    ApiRange range_("ice_sparse_attn");
    if (!ix || !q || !page_ids || !n_pages || !out || !aligned16(q) || !aligned16(out))
        return ICE_ERR_INVALID_ARG;
    if (page_stride < 1 || page_stride > 512) return ICE_ERR_INVALID_ARG;
    ICE_KERNEL_ADDR(q);
    ICE_KERNEL_ADDR(page_ids);
    ICE_KERNEL_ADDR(n_pages);
    ICE_KERNEL_ADDR(out);
    // pages in device memory are staged by bulk copies while the units fit one block per
    // SM; a host pool, and launches of more units, take the plain-load kernel
    cudaError_t e = ix->p.kv_location == ICE_KV_DEVICE && ix->U <= kAttnStagedMaxUnits
                        ? launch_attn_staged(ix->v, q, page_ids, n_pages, page_stride, out, (cudaStream_t)stream)
                        : launch_attn(ix->v, q, page_ids, n_pages, page_stride, out, (cudaStream_t)stream);
    return e == cudaSuccess ? ICE_OK : ICE_ERR_CUDA;
}

int ice_get_error(ice_index* ix, void* stream) {
    if (!ix) return ICE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ICE_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, ix->v.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ICE_ERR_CUDA;
    if (h != 0 && cudaMemset(ix->v.status, 0, sizeof(int)) != cudaSuccess) return ICE_ERR_CUDA;
    return h;
}

void ice_destroy(ice_index* ix) {
    if (!ix) return;
    cudaDeviceSynchronize();
    free_all(ix);
    delete ix;
}

int ice_debug_set_flags(ice_index* ix, int32_t flags) {
    if (!ix || (flags & ~ICE_DEBUG_STALL_ATTN)) return ICE_ERR_INVALID_ARG;
    ix->v.debug = flags;
    return ICE_OK;
}

int ice_set_cluster_size(ice_index* ix, int32_t k) {
    if (!ix || !(k == 0 || k == 1 || k == 2 || k == 4 || k == 8 || k == 16)) return ICE_ERR_INVALID_ARG;
    if (k >= 2 && k < ix->p.n_composite) return ICE_ERR_INVALID_ARG;
    ix->v.cluster_k = k;
    return ICE_OK;
}

int ice_get_info(const ice_index* ix, ice_info* info) {
    if (!ix || !info) return ICE_ERR_INVALID_ARG;
    info->n_units = ix->U;
    int nt = 0;  // the device count (inserts replayed from CUDA graphs included)
    if (cudaMemcpy(&nt, ix->v.n_tok, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ICE_ERR_CUDA;
    info->n_tokens = nt;
    info->max_tokens = ix->v.max_tokens;
    info->list_capacity = ix->C;
    info->pool_bytes = (int64_t)ix->bytes;
    info->group = ix->G;
    info->n_composite = ix->p.n_composite;
    info->page_size = ix->p.page_size;
    info->dtype = ix->p.dtype;
    info->host_bytes = (int64_t)ix->host_bytes;
    info->kv_location = ix->p.kv_location;
    info->reserved = 0;
    return ICE_OK;
}

int64_t ice_debug_dump(ice_index* ix, int32_t unit, void* host_buf, int64_t cap, void* stream) {
    if (!ix || unit < 0 || unit >= ix->U) return ICE_ERR_INVALID_ARG;
    const int L = ix->p.n_composite, P = ix->p.page_size;
    const long long C = ix->C;
    const int64_t per_l = C * 16 + C * 16 + C * 4 + C * P * 4 + C * P * 8;
    const int64_t loc1 = L > 1 ? C * P * 4 + ix->v.max_tokens * 4 : 0;
    const int64_t need = 16 * 8 + L * per_l + ix->v.max_tokens * 4 + loc1;
    if (!host_buf || cap < need) return need;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ICE_ERR_CUDA;
    const IndexView& v = ix->v;
    int64_t hdr[16] = {0};
    hdr[0] = L;
    hdr[1] = P;
    hdr[2] = C;
    int nt = 0;
    bool okn = cudaMemcpy(&nt, v.n_tok + unit, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    if (!okn) return ICE_ERR_CUDA;
    hdr[3] = nt;
    int e = 0, nl[kMaxL] = {0, 0}, ni[kMaxL] = {0, 0};
    bool ok = cudaMemcpy(&e, v.e_unit + unit, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    ok = ok && cudaMemcpy(nl, v.n_leaf + (long long)unit * L, sizeof(int) * L,
                          cudaMemcpyDeviceToHost) == cudaSuccess;
    ok = ok && cudaMemcpy(ni, v.next_id + (long long)unit * L, sizeof(int) * L,
                          cudaMemcpyDeviceToHost) == cudaSuccess;
    hdr[4] = e;
    for (int l = 0; l < L; ++l) {
        hdr[5 + l] = nl[l];
        hdr[9 + l] = ni[l];
    }
    char* o = (char*)host_buf;
    std::memcpy(o, hdr, sizeof(hdr));
    o += sizeof(hdr);
    for (int l = 0; l < L && ok; ++l) {
        const long long lb = v.leaf_base(unit, l), sb = v.slot_base(unit, l);
        ok = ok && cudaMemcpy(o, v.leaf_key + lb, C * 16, cudaMemcpyDeviceToHost) == cudaSuccess;
        o += C * 16;
        ok = ok && cudaMemcpy(o, v.leaf_rec + lb, C * 16, cudaMemcpyDeviceToHost) == cudaSuccess;
        o += C * 16;
        ok = ok && cudaMemcpy(o, v.list_cnt + lb, C * 4, cudaMemcpyDeviceToHost) == cudaSuccess;
        o += C * 4;
        ok = ok && cudaMemcpy(o, v.slot_tok + sb, C * P * 4, cudaMemcpyDeviceToHost) == cudaSuccess;
        o += C * P * 4;
        ok = ok && cudaMemcpy(o, v.slot_key + sb, C * P * 8, cudaMemcpyDeviceToHost) == cudaSuccess;
        o += C * P * 8;
    }
    ok = ok && cudaMemcpy(o, v.tok_loc + (long long)unit * v.max_tokens, v.max_tokens * 4,
                          cudaMemcpyDeviceToHost) == cudaSuccess;
    o += v.max_tokens * 4;
    if (L > 1) {
        ok = ok && cudaMemcpy(o, v.slot_loc1 + v.loc1_base(unit), C * P * 4, cudaMemcpyDeviceToHost) ==
                       cudaSuccess;
        o += C * P * 4;
        ok = ok && cudaMemcpy(o, v.tok_slot1 + (long long)unit * v.max_tokens, v.max_tokens * 4,
                              cudaMemcpyDeviceToHost) == cudaSuccess;
    }
    return ok ? ICE_OK : ICE_ERR_CUDA;
}

int ice_debug_page(ice_index* ix, int32_t unit, int32_t page_id, void* host_k, void* host_v,
                   void* stream) {
    if (!ix || unit < 0 || unit >= ix->U || page_id < 0 || page_id >= ix->C || !host_k || !host_v)
        return ICE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ICE_ERR_CUDA;
    const size_t es = ix->p.dtype == ICE_BF16 ? 2 : 4;
    const size_t bytes = (size_t)ix->p.page_size * kD * es;
    const size_t off = (size_t)ix->v.page_row(unit, page_id, 0) * kD * es;
    bool ok = cudaMemcpy(host_k, (char*)ix->v.page_k + off, bytes, cudaMemcpyDefault) == cudaSuccess;
    ok = ok && cudaMemcpy(host_v, (char*)ix->v.page_v + off, bytes, cudaMemcpyDefault) == cudaSuccess;
    return ok ? ICE_OK : ICE_ERR_CUDA;
}


}  // extern "C"

// Decode-time page selection ("IceCache", Figure 2 steps 2-3; the blog's
// mechanism section: P-DCI, the prioritised DCI search, picks the pages most
// relevant to the current query).
//
// One 512-thread block per unit, organised for memory-level parallelism (the
// work per unit is a chain of dependent phases, so the latency of each phase
// is what the block must hide):
//  1. the first batch of leaf records is requested before the query prep:
//     q_sel = sum of the group's heads (fp32, head order), its normalisation
//     and the 8-bit codes of its projections per composite;
//  2. all composites are scanned in one pass: priority of every leaf = the
//     L-infinity distance in code units between the query codes and the leaf's
//     cell, and token counts by priority go to sub-histograms shared by two
//     warps each;
//  3. per composite, the threshold priority pi* is the smallest with
//     cumulative count >= n_cand; leaves with priority < pi* are taken, and
//     those at pi* in left-to-right order while the tokens taken before them at
//     pi* are fewer than needed (the order a best-first tree search visits
//     leaves in);
//  4. every slot of every taken leaf is expanded in one parallel round into a
//     candidate (token, row); a composite-1 token whose page was taken in
//     composite 0 is a duplicate and dropped;
//  5. every candidate is rescored with the fixed-order fp32 dot q_sel . k, four
//     rows per warp instruction (8 lanes per row, each lane evaluating four of
//     the 32 lane partials of the fixed order);
//  6. candidates are sorted by (score desc, token asc) and walked; the page of
//     each is taken on first occurrence until n_sel pages are taken.
#include "ice_internal.cuh"

namespace ice {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSubH = 8;     // sub-histograms per composite (two warps each)
constexpr int kScanUnr = 8;  // leaf records in flight per thread
constexpr int kRowUnr = 2;   // candidate rows per lane group per round

struct SelSmem {
    int prio, cnt, hist, chosen, cmeta, coff, bm0, bm_taken, keys, vals, end;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline SelSmem sel_layout(long long C, int L, int n_cand, int sort_cap) {
    SelSmem s;
    int o = 0;
    s.prio = o; o = align16(o + L * (int)C);
    s.cnt = o; o = align16(o + L * (int)C);
    s.hist = o; o = align16(o + L * kSubH * 256 * 4);
    s.chosen = o; o = align16(o + L * n_cand * 4);
    s.cmeta = o; o = align16(o + L * n_cand * 4);
    s.coff = o; o = align16(o + L * (n_cand + 1) * 4);
    s.bm0 = o; o = align16(o + (int)((C + 31) / 32) * 4);
    s.bm_taken = o; o = align16(o + (int)((C + 31) / 32) * 4);
    s.keys = o; o = align16(o + sort_cap * 8);
    s.vals = o; o = align16(o + sort_cap * 4);
    s.end = o;
    return s;
}

__device__ __forceinline__ int cell_dist(uint4 cell, const int (&qc)[8]) {
    const unsigned lo[2] = {cell.x, cell.y}, hi[2] = {cell.z, cell.w};
    int best = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int l = (int)((lo[j >> 2] >> (8 * (j & 3))) & 0xFF);
        const int h = (int)((hi[j >> 2] >> (8 * (j & 3))) & 0xFF);
        const int c = qc[j];
        const int dj = c < l ? l - c : (c > h ? c - h : 0);
        best = max(best, dj);
    }
    return best;
}

// Raw row chunk of 4 elements (8 B for bf16, 16 B for f32) and its widening.
template <typename T> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
    uint2 r;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { r = __ldg(reinterpret_cast<const uint2*>(p)); }
    __device__ __forceinline__ void get(float (&x)[4]) const {
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xFFFF0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xFFFF0000u);
    }
};
template <> struct Chunk<float> {
    float4 r;
    __device__ __forceinline__ void load(const float* p) { r = __ldg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ void get(float (&x)[4]) const {
        x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
    }
};

template <typename T>
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(
    IndexView v, const T* __restrict__ q, int n_sel, int n_cand, int sort_cap,
    int32_t* __restrict__ page_ids, int32_t* __restrict__ n_pages_out, int32_t* __restrict__ stats) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float s_qsel[kD];
    __shared__ int s_qcode[kMaxL][kM];
    __shared__ int s_pstar[kMaxL], s_need[kMaxL], s_nch[kMaxL], s_tot[kMaxL];
    __shared__ int s_ncand, s_nraw;
    __shared__ int s_wsum[kMaxL][kSelWarps];

    const int u = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = v.L, P = v.P;
    const long long C = v.C;
    const SelSmem lay = sel_layout(C, L, n_cand, sort_cap);
    unsigned char* prio = smem + lay.prio;                            // [L][C]
    unsigned char* cnts = smem + lay.cnt;                             // [L][C]
    int* hist = reinterpret_cast<int*>(smem + lay.hist);              // [L][kSubH][256]
    int* chosen = reinterpret_cast<int*>(smem + lay.chosen);          // [L][n_cand] leaf index
    unsigned* cmeta = reinterpret_cast<unsigned*>(smem + lay.cmeta);  // [L][n_cand] leaf meta
    int* coff = reinterpret_cast<int*>(smem + lay.coff);              // [L][n_cand + 1]
    unsigned* bm0 = reinterpret_cast<unsigned*>(smem + lay.bm0);
    unsigned* bm_taken = reinterpret_cast<unsigned*>(smem + lay.bm_taken);
    unsigned long long* skey = reinterpret_cast<unsigned long long*>(smem + lay.keys);
    int* sval = reinterpret_cast<int*>(smem + lay.vals);
    const int nwords = (int)((C + 31) / 32);

    int N[kMaxL] = {0, 0};
    for (int l = 0; l < L; ++l) {
        const int x = v.n_leaf[v.ul(u, l)];
        N[l] = x < 0 ? 0 : (x > C ? (int)C : x);
    }
    const int Ntot = N[0] + N[1];

    // ---- 1a. request the first batch of leaf records --------------------------------
    uint4 c4[kScanUnr];
    unsigned m4[kScanUnr];
    auto load_batch = [&](int base) {
#pragma unroll
        for (int k = 0; k < kScanUnr; ++k) {
            const int i = base + k * kSelThreads + tid;
            if (i < Ntot) {
                const int l = i < N[0] ? 0 : 1;
                const long long o = v.leaf_base(u, l) + (i - (l ? N[0] : 0));
                c4[k] = __ldg(v.leaf_cell + o);
                m4[k] = __ldg(v.leaf_meta + o);
            }
        }
    };
    load_batch(0);

    // ---- 1b. query prep ---------------------------------------------------------------
    {
        float qs[4];
        const T* qu = q + (long long)u * v.G * kD;
        load4(qu + 4 * lane, qs);
        for (int h = 1; h < v.G; ++h) {
            float x[4];
            load4(qu + (long long)h * kD + 4 * lane, x);
#pragma unroll
            for (int k = 0; k < 4; ++k) qs[k] = __fadd_rn(qs[k], x[k]);
        }
        const float nq = warp_dot_fixed(qs, qs);
        float qt[4] = {0.f, 0.f, 0.f, 0.f};
        if (nq > 0.0f) {
            const float sn = __fsqrt_rn(nq);
#pragma unroll
            for (int k = 0; k < 4; ++k) qt[k] = __fdiv_rn(qs[k], sn);
        }
        for (int dir = warp; dir < L * kM; dir += kSelWarps) {
            const float* ud = v.dirs + (long long)dir * kDirStride;
            float w[4];
            load4(ud + 4 * lane, w);
            const float p = __fmaf_rn(ud[kD], 0.0f, warp_dot_fixed(w, qt));
            if (lane == 0) s_qcode[dir / kM][dir % kM] = quantise_code(p);
        }
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) s_qsel[4 * lane + k] = qs[k];
        }
    }
    for (int i = tid; i < L * kSubH * 256; i += kSelThreads) hist[i] = 0;
    for (int i = tid; i < nwords; i += kSelThreads) {
        bm0[i] = 0u;
        bm_taken[i] = 0u;
    }
    if (tid < kMaxL) {
        s_nch[tid] = 0;
        s_tot[tid] = 0;
    }
    if (tid == 0) {
        s_ncand = 0;
        s_nraw = 0;
    }
    __syncthreads();

    // ---- 2. priorities + sub-histograms of token counts, all composites ------------------
    {
        int qc[kMaxL][8];
#pragma unroll
        for (int l = 0; l < kMaxL; ++l)
#pragma unroll
            for (int j = 0; j < 8; ++j) qc[l][j] = l < L ? s_qcode[l][j] : 0;
        const int sub = warp >> 1;
        for (int base = 0; base < Ntot; base += kScanUnr * kSelThreads) {
            if (base > 0) load_batch(base);
#pragma unroll
            for (int k = 0; k < kScanUnr; ++k) {
                const int i = base + k * kSelThreads + tid;
                if (i < Ntot) {
                    const int l = i < N[0] ? 0 : 1;
                    const int li = i - (l ? N[0] : 0);
                    const int pr = cell_dist(c4[k], l ? qc[1] : qc[0]);
                    const int cn = (int)(m4[k] & 0xFFu);
                    prio[l * C + li] = (unsigned char)pr;
                    cnts[l * C + li] = (unsigned char)cn;
                    atomicAdd(&hist[(l * kSubH + sub) * 256 + pr], cn);
                }
            }
        }
    }
    __syncthreads();

    // ---- 3a. threshold priority per composite (warp l) -----------------------------------
    if (warp < L) {
        const int l = warp;
        int loc[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            int x = 0;
#pragma unroll
            for (int s = 0; s < kSubH; ++s) x += hist[(l * kSubH + s) * 256 + lane * 8 + k];
            loc[k] = x;
            sum += x;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int excl = incl - sum;
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= n_cand);
        if (hit == 0u) {
            if (lane == 0) {
                s_pstar[l] = 256;  // fewer than n_cand tokens in total: take all leaves
                s_need[l] = 0;
            }
        } else if (lane == __ffs(hit) - 1) {
            int run = excl, k = 0;
            while (run + loc[k] < n_cand) {
                run += loc[k];
                ++k;
            }
            s_pstar[l] = lane * 8 + k;
            s_need[l] = n_cand - run;
        }
    }
    __syncthreads();

    // ---- 3b. leaves taken at pi*, in position order (contiguous range per thread) ------
    {
        int lo_i[kMaxL], hi_i[kMaxL], mine[kMaxL], incl[kMaxL];
#pragma unroll
        for (int l = 0; l < kMaxL; ++l) {
            const int per = (N[l] + kSelThreads - 1) / kSelThreads;
            lo_i[l] = min(N[l], tid * per);
            hi_i[l] = min(N[l], lo_i[l] + per);
            mine[l] = 0;
            if (l < L && s_pstar[l] < 256) {
                const int ps = s_pstar[l];
                for (int i = lo_i[l]; i < hi_i[l]; ++i)
                    if (prio[l * C + i] == ps) mine[l] += cnts[l * C + i];
            }
            incl[l] = mine[l];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl[l], o);
                if (lane >= o) incl[l] += y;
            }
            if (lane == 31) s_wsum[l][warp] = incl[l];
        }
        __syncthreads();
#pragma unroll
        for (int l = 0; l < kMaxL; ++l) {
            if (l >= L) break;
            int run = incl[l] - mine[l];
            for (int w = 0; w < warp; ++w) run += s_wsum[l][w];
            const int ps = s_pstar[l], need = s_need[l];
            int* ch = chosen + l * n_cand;
            for (int i = lo_i[l]; i < hi_i[l]; ++i) {
                const int pr = prio[l * C + i];
                bool take = pr < ps;
                if (pr == ps) {
                    take = run < need;
                    run += cnts[l * C + i];
                }
                if (take) {
                    const int slot = atomicAdd(&s_nch[l], 1);
                    if (slot < n_cand) ch[slot] = i;
                }
            }
        }
    }
    __syncthreads();

    // ---- 3c. metadata of the taken leaves (one parallel round) -------------------------
    for (int l = 0; l < L; ++l) {
        const int nch = min(s_nch[l], n_cand);
        for (int k = tid; k < nch; k += kSelThreads)
            cmeta[l * n_cand + k] = __ldg(v.leaf_meta + v.leaf_base(u, l) + chosen[l * n_cand + k]);
    }
    __syncthreads();
    // exclusive offsets of the taken leaves' slots (warp l), composite-0 page bitmap
    if (warp < L) {
        const int l = warp;
        const int nch = min(s_nch[l], n_cand);
        int carry = 0;
        for (int k0 = 0; k0 < nch; k0 += 32) {
            const int k = k0 + lane;
            const int c = k < nch ? (int)(cmeta[l * n_cand + k] & 0xFFu) : 0;
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (k < nch) coff[l * (n_cand + 1) + k] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            coff[l * (n_cand + 1) + nch] = carry;
            s_tot[l] = carry;
        }
    }
    {
        const int nch0 = min(s_nch[0], n_cand);
        for (int k = tid; k < nch0; k += kSelThreads) {
            const int id = (int)(cmeta[k] >> 8);
            if (id < C) atomicOr(&bm0[id >> 5], 1u << (id & 31));
        }
    }
    __syncthreads();

    // ---- 4. candidate expansion: every (leaf, slot) at once ------------------------------
    {
        const int tot0 = s_tot[0], total = tot0 + (L > 1 ? s_tot[1] : 0);
        if (tid == 0) s_nraw = total;
        for (int j0 = warp * 32; j0 < total; j0 += kSelThreads) {
            const int j = j0 + lane;
            bool keep = false;
            int tok = 0, loc = 0;
            if (j < total) {
                const int l = j < tot0 ? 0 : 1;
                const int jj = j - (l ? tot0 : 0);
                const int nch = min(s_nch[l], n_cand);
                const int* off = coff + l * (n_cand + 1);
                int lo = 0, hi = nch;  // last k with off[k] <= jj
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (off[mid] <= jj) lo = mid; else hi = mid;
                }
                const int slot = jj - off[lo];
                const int id = (int)(cmeta[l * n_cand + lo] >> 8);
                if (id < C && slot < P) {
                    tok = __ldg(v.slot_tok + v.slot_base(u, l) + (long long)id * P + slot);
                    if (l == 0) {
                        loc = id * P + slot;
                        keep = true;
                    } else if (tok >= 0 && tok < v.max_tokens) {
                        loc = __ldg(v.tok_loc + (long long)u * v.max_tokens + tok);
                        const int pg = loc / P;
                        keep = loc >= 0 && pg < C && !((bm0[pg >> 5] >> (pg & 31)) & 1u);
                    }
                }
            }
            const unsigned km = __ballot_sync(0xffffffffu, keep);
            int pos0 = 0;
            if (lane == 0 && km) pos0 = atomicAdd(&s_ncand, __popc(km));
            pos0 = __shfl_sync(0xffffffffu, pos0, 0);
            if (keep) {
                const int pos = pos0 + __popc(km & ((1u << lane) - 1u));
                if (pos < sort_cap) {
                    skey[pos] = (unsigned long long)(unsigned)tok;
                    sval[pos] = loc;
                }
            }
        }
    }
    __syncthreads();
    const int ncand = min(s_ncand, sort_cap);

    // ---- 5. exact rescoring, 4 rows per warp instruction ---------------------------------
    {
        const int g8 = lane >> 3, p = lane & 7;
        // lane p evaluates lane partials p, p+8, p+16, p+24 of the fixed order:
        // elements 4p + 32j .. 4p + 32j + 3 for j = 0..3
        float qv[16];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[4 * j + i] = s_qsel[4 * p + 32 * j + i];
        const T* pk = reinterpret_cast<const T*>(v.page_k) + (long long)u * C * P * kD;
        for (int r0 = warp * 4 * kRowUnr; r0 < ncand; r0 += kSelWarps * 4 * kRowUnr) {
            Chunk<T> ch[kRowUnr][4];
            int tk[kRowUnr], lc[kRowUnr];
#pragma unroll
            for (int k = 0; k < kRowUnr; ++k) {
                const int r = r0 + 4 * k + g8;
                tk[k] = -1;
                lc[k] = 0;
                if (r < ncand) {
                    tk[k] = (int)skey[r];
                    lc[k] = sval[r];
                    const T* row = pk + (long long)lc[k] * kD + 4 * p;
#pragma unroll
                    for (int j = 0; j < 4; ++j) ch[k][j].load(row + 32 * j);
                }
            }
#pragma unroll
            for (int k = 0; k < kRowUnr; ++k) {
                float part[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x[4] = {0.f, 0.f, 0.f, 0.f};
                    if (tk[k] >= 0) ch[k][j].get(x);
                    float a = 0.0f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) a = __fmaf_rn(qv[4 * j + i], x[i], a);
                    part[j] = a;
                }
                // levels 16 and 8 of the pairwise sum inside the lane, 4, 2, 1 across lanes
                float b = __fadd_rn(__fadd_rn(part[0], part[2]), __fadd_rn(part[1], part[3]));
                b = __fadd_rn(b, __shfl_xor_sync(0xffffffffu, b, 4));
                b = __fadd_rn(b, __shfl_xor_sync(0xffffffffu, b, 2));
                b = __fadd_rn(b, __shfl_xor_sync(0xffffffffu, b, 1));
                const int r = r0 + 4 * k + g8;
                if (p == 0 && tk[k] >= 0) {
                    skey[r] = ((unsigned long long)score_key_desc(b) << 32) | (unsigned)tk[k];
                    sval[r] = lc[k] / P;
                }
            }
        }
    }
    int npow = 1;
    while (npow < ncand) npow <<= 1;
    for (int c = ncand + tid; c < npow; c += kSelThreads) {
        skey[c] = ~0ull;
        sval[c] = -1;
    }
    __syncthreads();

    // ---- 6a. bitonic sort by (score desc, token asc) -----------------------------------
    for (int k = 2; k <= npow; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow; i += kSelThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = skey[i], b = skey[ixj];
                    if ((a > b) == ((i & k) == 0)) {
                        skey[i] = b;
                        skey[ixj] = a;
                        const int t = sval[i];
                        sval[i] = sval[ixj];
                        sval[ixj] = t;
                    }
                }
            }
            __syncthreads();
        }
    }

    // ---- 6b. walk: first occurrences of pages in rank order -----------------------------
    if (warp == 0) {
        int taken = 0;
        int32_t* out = page_ids + (long long)u * n_sel;
        for (int c0 = 0; c0 < ncand && taken < n_sel; c0 += 32) {
            const int c = c0 + lane;
            const int pg = c < ncand ? sval[c] : -1;
            bool fresh = pg >= 0 && pg < C && !((bm_taken[pg >> 5] >> (pg & 31)) & 1u);
            const unsigned peers = __match_any_sync(0xffffffffu, pg);
            fresh = fresh && (lane == __ffs(peers) - 1);
            const unsigned fm = __ballot_sync(0xffffffffu, fresh);
            if (fresh) {
                const int r = taken + __popc(fm & ((1u << lane) - 1u));
                if (r < n_sel) {
                    out[r] = pg;
                    atomicOr(&bm_taken[pg >> 5], 1u << (pg & 31));  // lanes may share a word
                }
            }
            taken = min(n_sel, taken + __popc(fm));
            __syncwarp();
        }
        for (int r = taken + lane; r < n_sel; r += 32) out[r] = -1;
        if (lane == 0) n_pages_out[u] = taken;
        if (stats) {
            __syncwarp();
            int tok_sel = 0;
            for (int r = lane; r < taken; r += 32) tok_sel += v.list_cnt[v.leaf_base(u, 0) + out[r]];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) tok_sel += __shfl_xor_sync(0xffffffffu, tok_sel, o);
            if (lane == 0) {
                stats[4 * u + 0] = Ntot;
                stats[4 * u + 1] = ncand;
                stats[4 * u + 2] = tok_sel;
                stats[4 * u + 3] = s_nraw;
            }
        }
    }
    if (tid == 0 && s_ncand > sort_cap) set_status(v.status, ICE_ERR_CAPACITY);
}

static int sort_capacity(int L, int P, int n_cand) {
    const int cand_cap = L * (n_cand + P - 1);
    int sort_cap = 1;
    while (sort_cap < cand_cap) sort_cap <<= 1;
    return sort_cap;
}

cudaError_t launch_select(const IndexView& v, const void* q, int n_sel, int n_cand,
                          int32_t* page_ids, int32_t* n_pages, int32_t* stats, cudaStream_t s) {
    const int sort_cap = sort_capacity(v.L, v.P, n_cand);
    const int bytes = sel_layout(v.C, v.L, n_cand, sort_cap).end;
    cudaError_t e;
    if (v.dtype == ICE_BF16) {
        e = cudaFuncSetAttribute(select_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        select_kernel<__nv_bfloat16><<<v.U, kSelThreads, bytes, s>>>(
            v, (const __nv_bfloat16*)q, n_sel, n_cand, sort_cap, page_ids, n_pages, stats);
    } else {
        e = cudaFuncSetAttribute(select_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bytes);
        if (e != cudaSuccess) return e;
        select_kernel<float><<<v.U, kSelThreads, bytes, s>>>(v, (const float*)q, n_sel, n_cand,
                                                            sort_cap, page_ids, n_pages, stats);
    }
    return cudaGetLastError();
}

// Dynamic shared memory the select kernel needs (host check before launch).
int select_smem_bytes(long long C, int L, int P, int n_cand) {
    return sel_layout(C, L, n_cand, sort_capacity(L, P, n_cand)).end;
}

}  // namespace ice

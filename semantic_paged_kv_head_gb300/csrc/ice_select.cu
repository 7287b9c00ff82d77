// Decode-time page selection ("IceCache", Figure 2 steps 2-3; the blog's
// mechanism section: P-DCI, the prioritised DCI search, picks the pages most
// relevant to the current query).
//
// One thread block per unit:
//  1. query prep: q_sel = sum of the group's heads (fp32, head order), its
//     normalisation and the 8-bit codes of its projections per composite;
//  2. per composite: priority of every leaf = L-infinity distance in code units
//     between the query codes and the leaf's cell; a histogram of token counts
//     by priority gives the threshold priority pi*; leaves with priority < pi*
//     are taken, and those at pi* in left-to-right order until n_cand tokens
//     are reached (the order a best-first tree search visits them in);
//  3. the tokens of the taken leaves are the candidates; a composite-1 token
//     whose page is already taken in composite 0 is a duplicate and skipped;
//  4. every candidate is rescored with the fixed-order fp32 dot q_sel . k
//     (one warp per key, 16-byte coalesced row loads);
//  5. candidates are sorted by (score desc, token asc) and walked; the page of
//     each is taken on first occurrence until n_sel pages are taken.
#include "ice_internal.cuh"

namespace ice {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

struct SelSmem {
    // offsets (bytes) into dynamic shared memory
    int prio, cnt, bm0, bm_taken, chosen, keys, vals, end;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline SelSmem sel_layout(long long C, int L, int n_cand, int sort_cap) {
    SelSmem s;
    int o = 0;
    s.prio = o; o = align16(o + (int)C);
    s.cnt = o; o = align16(o + (int)C);
    s.bm0 = o; o = align16(o + (int)((C + 31) / 32) * 4);
    s.bm_taken = o; o = align16(o + (int)((C + 31) / 32) * 4);
    s.chosen = o; o = align16(o + L * n_cand * 4);
    s.keys = o; o = align16(o + sort_cap * 8);
    s.vals = o; o = align16(o + sort_cap * 4);
    s.end = o;
    return s;
}

__device__ __forceinline__ int cell_dist(uint4 cell, const int (&qc)[8]) {
    unsigned lo[2] = {cell.x, cell.y}, hi[2] = {cell.z, cell.w};
    int best = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int l = (int)((lo[j >> 2] >> (8 * (j & 3))) & 0xFF);
        int h = (int)((hi[j >> 2] >> (8 * (j & 3))) & 0xFF);
        int c = qc[j];
        int dj = c < l ? l - c : (c > h ? c - h : 0);
        best = max(best, dj);
    }
    return best;
}

template <typename T>
__global__ void __launch_bounds__(kSelThreads) select_kernel(IndexView v, const T* __restrict__ q,
                                                             int n_sel, int n_cand, int sort_cap,
                                                             int32_t* __restrict__ page_ids,
                                                             int32_t* __restrict__ n_pages_out,
                                                             int32_t* __restrict__ stats) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float s_qsel[kD];
    __shared__ float s_qt[kD];
    __shared__ int s_qcode[kMaxL][kM];
    __shared__ int s_hist[256];
    __shared__ int s_pstar, s_need, s_nchosen[kMaxL], s_ncand, s_nraw, s_scanned;
    __shared__ int s_wsum[kSelWarps];

    const int u = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const SelSmem L_ = sel_layout(v.C, v.L, n_cand, sort_cap);
    unsigned char* prio = smem + L_.prio;
    unsigned char* cnts = smem + L_.cnt;
    unsigned int* bm0 = reinterpret_cast<unsigned int*>(smem + L_.bm0);
    unsigned int* bm_taken = reinterpret_cast<unsigned int*>(smem + L_.bm_taken);
    int* chosen = reinterpret_cast<int*>(smem + L_.chosen);
    unsigned long long* skey = reinterpret_cast<unsigned long long*>(smem + L_.keys);
    int* sval = reinterpret_cast<int*>(smem + L_.vals);
    const int nwords = (int)((v.C + 31) / 32);

    // ---- 1. query prep ------------------------------------------------------
    float qs[4];
    {
        const T* qu = q + (long long)u * v.G * kD;
        load4(qu + 4 * lane, qs);
        for (int h = 1; h < v.G; ++h) {
            float x[4];
            load4(qu + (long long)h * kD + 4 * lane, x);
#pragma unroll
            for (int k = 0; k < 4; ++k) qs[k] = __fadd_rn(qs[k], x[k]);
        }
    }
    {
        const float nq = warp_dot_fixed(qs, qs);
        float qt[4] = {0.f, 0.f, 0.f, 0.f};
        if (nq > 0.0f) {
            const float sn = __fsqrt_rn(nq);
#pragma unroll
            for (int k = 0; k < 4; ++k) qt[k] = __fdiv_rn(qs[k], sn);
        }
        const int ndir = v.L * kM;
        for (int dir = warp; dir < ndir; dir += kSelWarps) {
            const float* ud = v.dirs + (long long)dir * kDirStride;
            float w[4];
            load4(ud + 4 * lane, w);
            float p = warp_dot_fixed(w, qt);
            p = __fmaf_rn(ud[kD], 0.0f, p);
            if (lane == 0) s_qcode[dir / kM][dir % kM] = quantise_code(p);
        }
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) s_qsel[4 * lane + k] = qs[k];
        }
    }
    for (int i = tid; i < nwords; i += kSelThreads) {
        bm0[i] = 0u;
        bm_taken[i] = 0u;
    }
    if (tid == 0) {
        s_ncand = 0;
        s_nraw = 0;
        s_scanned = 0;
    }
    __syncthreads();

    // ---- 2. prioritised leaf search per composite -------------------------------
    for (int l = 0; l < v.L; ++l) {
        int N = v.n_leaf[v.ul(u, l)];
        N = N < 0 ? 0 : (N > v.C ? (int)v.C : N);
        const uint4* cell = v.leaf_cell + v.leaf_base(u, l);
        const unsigned int* meta = v.leaf_meta + v.leaf_base(u, l);
        int qc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) qc[j] = s_qcode[l][j];
        if (tid < 256) s_hist[tid] = 0;
        __syncthreads();
        // 2a: priorities + histogram of token counts (4 leaves in flight per thread)
        for (int base = 0; base < N; base += 4 * kSelThreads) {
            uint4 c4[4];
            unsigned int m4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int i = base + k * kSelThreads + tid;
                if (i < N) {
                    c4[k] = __ldg(cell + i);
                    m4[k] = __ldg(meta + i);
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int i = base + k * kSelThreads + tid;
                if (i < N) {
                    int pr = cell_dist(c4[k], qc);
                    int cn = (int)(m4[k] & 0xFFu);
                    prio[i] = (unsigned char)pr;
                    cnts[i] = (unsigned char)cn;
                    atomicAdd(&s_hist[pr], cn);
                }
            }
        }
        __syncthreads();
        // 2b: threshold priority pi* (smallest with cumulative count >= n_cand)
        if (warp == 0) {
            int loc[8], sum = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                loc[k] = s_hist[lane * 8 + k];
                sum += loc[k];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - sum;
            const unsigned int hit = __ballot_sync(0xffffffffu, incl >= n_cand);
            if (hit == 0u) {
                if (lane == 0) {
                    s_pstar = 256;  // fewer than n_cand tokens in total: take all leaves
                    s_need = 0;
                }
            } else if (lane == __ffs(hit) - 1) {
                int run = excl, k = 0;
                while (run + loc[k] < n_cand) {
                    run += loc[k];
                    ++k;
                }
                s_pstar = lane * 8 + k;
                s_need = n_cand - run;
            }
        }
        __syncthreads();
        const int pstar = s_pstar, need = s_need;
        // 2c: leaves at pi* are taken in position order while the tokens taken
        // at pi* so far are fewer than `need`. Each thread owns a contiguous
        // range of leaves; a block scan orders the ranges.
        const int per = (N + kSelThreads - 1) / kSelThreads;
        const int lo_i = tid * per, hi_i = min(N, lo_i + per);
        int mine = 0;
        if (pstar < 256)
            for (int i = lo_i; i < hi_i; ++i)
                if (prio[i] == pstar) mine += cnts[i];
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        if (tid == 0) s_nchosen[l] = 0;
        __syncthreads();
        int woff = 0;
        for (int w = 0; w < warp; ++w) woff += s_wsum[w];
        int run = woff + incl - mine;  // tokens at pi* in earlier leaves
        int* ch = chosen + l * n_cand;
        for (int i = lo_i; i < hi_i; ++i) {
            const int pr = prio[i];
            bool take = pr < pstar;
            if (pr == pstar) {
                take = run < need;
                run += cnts[i];
            }
            if (take) {
                int slot = atomicAdd(&s_nchosen[l], 1);
                if (slot < n_cand) ch[slot] = i;
            }
        }
        if (tid == 0) s_scanned += N;
        __syncthreads();
    }

    // ---- 3. candidates -------------------------------------------------------------
    // composite-0 taken pages into the membership bitmap
    {
        const int nc0 = min(s_nchosen[0], n_cand);
        const unsigned int* meta0 = v.leaf_meta + v.leaf_base(u, 0);
        for (int c = tid; c < nc0; c += kSelThreads) {
            const int id = (int)(meta0[chosen[c]] >> 8);
            if (id >= 0 && id < v.C) atomicOr(&bm0[id >> 5], 1u << (id & 31));
        }
    }
    __syncthreads();
    for (int l = 0; l < v.L; ++l) {
        const int ncl = min(s_nchosen[l], n_cand);
        const unsigned int* metal = v.leaf_meta + v.leaf_base(u, l);
        const int* ch = chosen + l * n_cand;
        const long long sb = v.slot_base(u, l);
        for (int c = warp; c < ncl; c += kSelWarps) {
            const unsigned int m = metal[ch[c]];
            const int id = (int)(m >> 8), cn = (int)(m & 0xFFu);
            bool keep = false;
            int tok = 0, loc = 0;
            if (lane < cn && id < v.C) {
                tok = v.slot_tok[sb + (long long)id * v.P + lane];
                if (l == 0) {
                    loc = id * v.P + lane;
                    keep = true;
                } else if (tok >= 0 && tok < v.max_tokens) {
                    loc = v.tok_loc[(long long)u * v.max_tokens + tok];
                    const int pg = loc / v.P;
                    keep = loc >= 0 && pg < v.C && !((bm0[pg >> 5] >> (pg & 31)) & 1u);
                }
            }
            if (lane < cn && lane == 0) atomicAdd(&s_nraw, cn);
            const unsigned int km = __ballot_sync(0xffffffffu, keep);
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

    // ---- 4. exact rescoring: one warp per candidate key -----------------------------
    {
        const T* pk = reinterpret_cast<const T*>(v.page_k) + (long long)u * v.C * v.P * kD;
        float qv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) qv[k] = s_qsel[4 * lane + k];
        constexpr int UNR = 4;
        for (int c0 = warp * UNR; c0 < ncand; c0 += kSelWarps * UNR) {
            float kr[UNR][4];
            int tk[UNR], lc[UNR];
#pragma unroll
            for (int k = 0; k < UNR; ++k) {
                const int c = c0 + k;
                if (c < ncand) {
                    tk[k] = (int)skey[c];
                    lc[k] = sval[c];
                    load4_nc(pk + (long long)lc[k] * kD + 4 * lane, kr[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < UNR; ++k) {
                const int c = c0 + k;
                if (c < ncand) {  // uniform across the warp
                    const float s = warp_dot_fixed(qv, kr[k]);
                    if (lane == 0) {
                        skey[c] = ((unsigned long long)score_key_desc(s) << 32) | (unsigned)tk[k];
                        sval[c] = lc[k] / v.P;
                    }
                }
            }
        }
    }
    // pad to a power of two for the bitonic sort
    int npow = 1;
    while (npow < ncand) npow <<= 1;
    for (int c = ncand + tid; c < npow; c += kSelThreads) {
        skey[c] = ~0ull;
        sval[c] = -1;
    }
    __syncthreads();

    // ---- 5a. bitonic sort by (score desc, token asc) ------------------------------
    for (int k = 2; k <= npow; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow; i += kSelThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = skey[i], b = skey[ixj];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) {
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

    // ---- 5b. walk: first occurrences of pages, in rank order ------------------------
    if (warp == 0) {
        int taken = 0;
        int32_t* out = page_ids + (long long)u * n_sel;
        for (int c0 = 0; c0 < ncand && taken < n_sel; c0 += 32) {
            const int c = c0 + lane;
            const int pg = c < ncand ? sval[c] : -1;
            bool fresh = pg >= 0 && pg < v.C && !((bm_taken[pg >> 5] >> (pg & 31)) & 1u);
            const unsigned int peers = __match_any_sync(0xffffffffu, pg);
            fresh = fresh && (lane == __ffs(peers) - 1);
            const unsigned int fm = __ballot_sync(0xffffffffu, fresh);
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
            // tokens in the selected pages
            int tok_sel = 0;
            for (int r = lane; r < taken; r += 32) tok_sel += v.list_cnt[v.leaf_base(u, 0) + out[r]];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) tok_sel += __shfl_xor_sync(0xffffffffu, tok_sel, o);
            if (lane == 0) {
                stats[4 * u + 0] = s_scanned;
                stats[4 * u + 1] = ncand;
                stats[4 * u + 2] = tok_sel;
                stats[4 * u + 3] = s_nraw;
            }
        }
    }
    if (tid == 0 && s_ncand > sort_cap) set_status(v.status, ICE_ERR_CAPACITY);
}

cudaError_t launch_select(const IndexView& v, const void* q, int n_sel, int n_cand,
                          int32_t* page_ids, int32_t* n_pages, int32_t* stats, cudaStream_t s) {
    const int cand_cap = v.L * (n_cand + v.P - 1);
    int sort_cap = 1;
    while (sort_cap < cand_cap) sort_cap <<= 1;
    const SelSmem lay = sel_layout(v.C, v.L, n_cand, sort_cap);
    const int bytes = lay.end;
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
    const int cand_cap = L * (n_cand + P - 1);
    int sort_cap = 1;
    while (sort_cap < cand_cap) sort_cap <<= 1;
    return sel_layout(C, L, n_cand, sort_cap).end;
}

}  // namespace ice

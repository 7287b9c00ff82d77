// Decode-time page selection and attention of one unit spread over a cluster
// of K thread blocks ("IceCache", Figure 2 steps 2-3; the blog's mechanism
// section: P-DCI, the prioritised DCI search, picks the pages for the current
// query, and attention runs over every token of those pages).
//
// The selection of a unit is a chain of dependent phases. One block per unit
// leaves most of the GPU idle when a decode step launches few units (one layer
// at a time), and its chain sets the step time. Here the K blocks of a cluster
// share a unit, and the phases that touch many bytes are split between them:
//  * composites: blocks [0, K/L) serve composite 0, the others composite 1;
//  * leaf scan: the Kc = K/L blocks of a composite scan contiguous ranges of its
//    leaves (64-leaf chunks), so that position order is block order;
//  * threshold: the blocks' priority histograms are added over distributed
//    shared memory (DSMEM), and every block of the composite derives the same
//    pi* and need;
//  * ties at pi*: each block publishes the tokens of its own ties; a block takes
//    its ties in position order while the ties of the blocks before it plus its
//    own taken so far stay below the need (the flat (priority, position) order);
//  * duplicates: composite-0 blocks set the pages they took in a bitmap of
//    block 0; a composite-1 candidate whose page is set there is dropped;
//  * rescoring: every block rescores its own candidates (fixed-order fp32 dot)
//    and keeps the minimum (score desc, token asc) key of every page it saw;
//  * ranking: each block publishes its n_sel best pages to block 0. A page in
//    the global top n_sel reaches there with its true minimum, because the block
//    that holds that minimum has fewer than n_sel pages above it; every other
//    page arrives with a key no smaller than its true minimum. So the n_sel
//    smallest of the published keys, taken per page, are the selection. Every
//    block computes it from block 0's lists;
//  * attention: block r attends selected pages r, r + K, ... (fp32 online
//    softmax over pages staged with bulk copies), and the blocks' partial
//    (max, sum, accumulator) triples are merged in block order over DSMEM, each
//    block writing a slice of the output.
// Every block of a cluster passes the same sequence of cluster barriers, and
// no block leaves while another may still read its shared memory.
#include <cooperative_groups.h>

#include <map>
#include <mutex>
#include <tuple>

#include "ice_internal.cuh"
#include "ice_select_common.cuh"

namespace cg = cooperative_groups;

namespace ice {

constexpr int kCT = 256;           // threads per block
constexpr int kCW = kCT / 32;      // warps per block
constexpr int kCSubH = 8;          // sub-histograms (lane groups)
constexpr int kCHistRow = 257;     // words per sub-histogram row
constexpr int kCRing = 3;          // scan chunks in flight per warp
constexpr int kCSlotB = 1024;      // one chunk: 64 leaf records of 16 B
constexpr int kCRingB = kCW * kCRing * kCSlotB;
constexpr int kCTop = 32;          // largest n_sel of the cluster path (warp top-32 ranking)
constexpr int kCluSmemMax = 220 * 1024;

struct CluSmem {
    // live through the kernel; the hub fields are written by every block into
    // block 0 and read there
    int sel, scnt, toff, lhist, hubx, hub_leaf, hub_pe, hub_part, qf, bm0;
    int X;  // phase region: scan tables, then candidates, then ranking, then attention staging
    int ring, prio, cnt, lid, tieb, hist, ghist, gpre, chosen, cmeta;  // scan
    int tl, toffc, skey, sval, hpage, hkey, hcnt, top, stage;     // candidates (stage: rows)
    int g_page, g_key, gk, gp;                                    // ranking
    int end;
};

struct CluDims {
    int rcap;       // leaves of a block's scan range (multiple of 64)
    int n_cand;     // candidates per composite
    int s_tot;      // candidate slots of a unit, all composites: L (n_cand + P - 1)
    int share_cap;  // candidate slots of one block: ceil(s_tot / K)
    int hcap_l;     // a block's page table (power of two > share_cap)
    int gcap;       // the ranking's page table (power of two > 2 K n_sel)
};

__host__ __device__ inline CluSmem clu_layout(long long C, const CluDims& d, int L, int n_sel,
                                              int K, int G, bool fused, int min_total) {
    CluSmem s;
    int o = 0;
    s.sel = o; o = align16(o + kCTop * 4);
    s.scnt = o; o = align16(o + kCTop * 4);
    s.toff = o; o = align16(o + (kCTop + 1) * 4);
    s.lhist = o; o = align16(o + 256 * 4);
    s.hubx = o; o = align16(o + 32 * 4);
    s.hub_leaf = o; o = align16(o + L * d.n_cand * 4);
    s.hub_pe = o; o = align16(o + K * n_sel * 16);
    s.hub_part = o; o = align16(o + (fused ? K * (G * (kD + 2) + 4) * 4 : 0));
    s.qf = o; o = align16(o + (fused ? G * kD * 4 : 0));
    s.bm0 = o; o = align16(o + (L > 1 ? (int)((C + 31) / 32) * 4 : 0));
    o = align128(o);  // the scan's copy ring starts here
    s.X = o;
    int a = o;  // scan
    s.ring = a; a = align16(a + kCRingB);
    s.prio = a; a = align16(a + d.rcap);
    s.cnt = a; a = align16(a + d.rcap);
    s.lid = a; a = align16(a + d.rcap * 4);
    s.tieb = a; a = align16(a + (d.rcap / 32) * 4);
    s.hist = a; a = align16(a + kCSubH * kCHistRow * 4);
    s.ghist = a; a = align16(a + 256 * 4);
    s.gpre = a; a = align16(a + 256 * 4);
    s.chosen = a; a = align16(a + d.n_cand * 4);
    s.cmeta = a; a = align16(a + d.n_cand * 4);
    int b = o;  // candidates
    s.tl = b; b = align16(b + L * d.n_cand * 4);
    s.toffc = b; b = align16(b + (L * d.n_cand + 1) * 4);
    s.skey = b; b = align16(b + d.share_cap * 8);
    s.sval = b; b = align16(b + d.share_cap * 4);
    s.hpage = b; b = align16(b + d.hcap_l * 4);
    s.hkey = b; b = align16(b + d.hcap_l * 8);
    s.hcnt = b; b = align16(b + d.hcap_l * 4);
    s.top = b; b = align16(b + kCW * 32 * 12);
    b = align128(b);
    s.stage = b;
    int g = o;  // ranking
    s.g_page = g; g = align16(g + d.gcap * 4);
    s.g_key = g; g = align16(g + d.gcap * 8);
    s.gk = g; g = align16(g + K * n_sel * 8);
    s.gp = g; g = align16(g + K * n_sel * 4);
    int e = a > b ? a : b;
    e = g > e ? g : e;
    s.end = e > min_total ? e : min_total;
    return s;
}

// The .aligned cluster barrier expects every thread of a warp to execute it together:
// the warp is reconverged first.
__device__ __forceinline__ void clu_arrive() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void clu_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The 32 smallest (key, index) pairs of keys[0..cnt), ascending, in lane order of
// every warp's (tk, tv) on return (empty places: key ~0, index -1): each warp
// sorts batches of 32 and keeps a running top 32, then the warps' lists are
// merged pairwise. topk/topv: [kCW][32] scratch. Every thread of the block calls it.
__device__ __forceinline__ void block_top32(const unsigned long long* keys, const int* idx, int cnt,
                                            unsigned long long* topk, int* topv,
                                            unsigned long long& tk, int& tv) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = (cnt + 31) / 32;
    tk = ~0ull;
    tv = -1;
    for (int bt = warp; bt < nb; bt += kCW) {  // warp-uniform
        const int j = bt * 32 + lane;
        unsigned long long k = j < cnt ? keys[j] : ~0ull;
        int vv = j < cnt ? idx[j] : -1;
        warp_sort32(k, vv, lane);
        warp_merge32(tk, tv, k, vv, lane);
    }
    const int nw = min(kCW, max(nb, 1));
    if (warp < nw) {
        topk[warp * 32 + lane] = tk;
        topv[warp * 32 + lane] = tv;
    }
    __syncthreads();
    for (int st = 1; st < nw; st <<= 1) {
        if ((warp & (2 * st - 1)) == 0 && warp + st < nw) {
            unsigned long long a = topk[warp * 32 + lane];
            int av = topv[warp * 32 + lane];
            warp_merge32(a, av, topk[(warp + st) * 32 + lane], topv[(warp + st) * 32 + lane], lane);
            topk[warp * 32 + lane] = a;
            topv[warp * 32 + lane] = av;
        }
        __syncthreads();
    }
    tk = topk[lane];
    tv = topv[lane];
}

// Partial attention of the G query heads over this block's share of the
// selected pages (s_sel[r], s_sel[r + K], ...): the pages' K and V rows are
// staged with one bulk copy per page and tensor onto an mbarrier, in rounds
// that fit the staging region; warp w takes tokens w, w + kCW, ... of a round
// (lane = (head, group of 4G dimensions)); the warps' (max, sum, accumulator)
// triples are merged in warp order and stored to dst[h][kD + 2] (block 0's
// shared memory), with this block's timeout flag after them.
template <typename T, int G>
__device__ __forceinline__ void attend_partial(const IndexView& v, int u, const float* s_q,
                                               const int* s_sel, const int* s_scnt, int taken,
                                               int r, int K, int* s_toff, unsigned char* stage,
                                               int stage_bytes, unsigned bar, int* s_fail,
                                               float* dst) {
    constexpr int LG = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;  // log2 G
    constexpr int HS = 5 - LG;  // lane l holds the score of head l >> HS
    constexpr int ROWB = kD * (int)sizeof(T);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = v.P;
    const long long C = v.C;
    const int hl = lane >> HS;
    const int npg = taken > r ? (taken - r + K - 1) / K : 0;
    if (warp == 0) {
        int carry = 0;
        for (int i0 = 0; i0 < npg; i0 += 32) {
            const int i = i0 + lane;
            int c = 0;
            if (i < npg) {
                const int pg = s_sel[r + K * i];
                c = (pg >= 0 && pg < C) ? s_scnt[r + K * i] : 0;
                c = c < 0 ? 0 : (c > P ? P : c);
            }
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (i < npg) s_toff[i] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_toff[npg] = carry;
    }
    float qa[G][4];  // dimensions 4 lane .. 4 lane + 3 of every head
    {
        const float sc = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int k = 0; k < 4; ++k) qa[hh][k] = s_q[hh * kD + 4 * lane + k] * sc;
    }
    __syncthreads();
    const int rows_cap = stage_bytes / (2 * ROWB);
    const T* sk = reinterpret_cast<const T*>(stage);
    const T* sv = reinterpret_cast<const T*>(stage + (size_t)rows_cap * ROWB);
    float m = -INFINITY, lsum = 0.0f, acc[G][4];  // m, lsum: head hl
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[hh][k] = 0.0f;
    int p0 = 0, round = 0;
    while (p0 < npg) {  // block-uniform rounds
        int p1 = p0 + 1;
        while (p1 < npg && s_toff[p1 + 1] - s_toff[p0] <= rows_cap) ++p1;
        const int t0 = s_toff[p0], nrow = s_toff[p1] - t0;
        if (warp == 0) {
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                // ICE_DEBUG_STALL_ATTN: expect 16 bytes that no copy delivers (tests of
                // the bounded wait)
                const unsigned extra = (v.debug & ICE_DEBUG_STALL_ATTN) ? 16u : 0u;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                             "r"((unsigned)(2 * nrow * ROWB) + extra)
                             : "memory");
            }
            __syncwarp();
            for (int i = p0 + lane; i < p1; i += 32) {
                const int c = s_toff[i + 1] - s_toff[i];
                if (c > 0) {
                    const long long row0 = v.page_row(u, s_sel[r + K * i], 0);
                    const unsigned off = (unsigned)(s_toff[i] - t0) * ROWB;
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            smem_u32(sk) + off),
                        "l"(reinterpret_cast<const char*>(v.page_k) + row0 * ROWB), "r"((unsigned)c * ROWB),
                        "r"(bar)
                        : "memory");
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            smem_u32(sv) + off),
                        "l"(reinterpret_cast<const char*>(v.page_v) + row0 * ROWB), "r"((unsigned)c * ROWB),
                        "r"(bar)
                        : "memory");
                }
            }
        }
        const bool ok = mbar_wait_bounded(bar, (unsigned)(round & 1));
        if (!ok) {
            *s_fail = 1;
            set_status(v.status, ICE_ERR_TIMEOUT);
            mbar_wait_bounded(bar, (unsigned)(round & 1));  // copies possibly still in flight
        }
        if (ok) {
            for (int j = warp; j < nrow; j += kCW) {  // warp-uniform
                float kx[4];
                load4(sk + (size_t)j * kD + 4 * lane, kx);
                float sv4[G];  // this lane's part of every head's score
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float2 s2 = __fmul2_rn(make_float2(qa[hh][0], qa[hh][1]), make_float2(kx[0], kx[1]));
                    s2 = __ffma2_rn(make_float2(qa[hh][2], qa[hh][3]), make_float2(kx[2], kx[3]), s2);
                    sv4[hh] = s2.x + s2.y;
                }
                // halving exchanges: lanes with bit b set keep the upper half of their heads
#pragma unroll
                for (int lv = 0; lv < LG; ++lv) {
                    const int b = 4 - lv, half = G >> (lv + 1);
                    const bool up = (lane >> b) & 1;
#pragma unroll
                    for (int k = 0; k < half; ++k) {
                        const float keep = up ? sv4[k + half] : sv4[k];
                        const float send = up ? sv4[k] : sv4[k + half];
                        sv4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << b);
                    }
                }
                float sc = sv4[0];
#pragma unroll
                for (int b = HS - 1; b >= 0; --b) sc += __shfl_xor_sync(0xffffffffu, sc, 1 << b);
                const float mn = fmaxf(m, sc);
                const float corr = exp2_approx(m - mn);
                const float p = exp2_approx(sc - mn);
                lsum = lsum * corr + p;
                m = mn;
                float vx[4];
                load4(sv + (size_t)j * kD + 4 * lane, vx);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float ch = __shfl_sync(0xffffffffu, corr, hh << HS);
                    const float ph = __shfl_sync(0xffffffffu, p, hh << HS);
                    const float2 c2 = make_float2(ch, ch), p2 = make_float2(ph, ph);
#pragma unroll
                    for (int k = 0; k < 4; k += 2) {
                        const float2 a2 = __ffma2_rn(p2, make_float2(vx[k], vx[k + 1]),
                                                     __fmul2_rn(make_float2(acc[hh][k], acc[hh][k + 1]), c2));
                        acc[hh][k] = a2.x;
                        acc[hh][k + 1] = a2.y;
                    }
                }
            }
        }
        __syncthreads();  // the round's rows are consumed before the next copies land
        if (*s_fail) break;  // no further copies on a barrier whose phase may never complete
        p0 = p1;
        ++round;
    }
    // rows [warp][head] of PR floats (accumulator, m, sum): one 16-byte store per lane and
    // head, where scalar stores 16 bytes apart would conflict four ways in the banks
    constexpr int PR = kD + 4;
    float* part = reinterpret_cast<float*>(stage);
    {
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
            *reinterpret_cast<float4*>(part + (warp * G + hh) * PR + 4 * lane) =
                make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
        if ((lane & ((1 << HS) - 1)) == 0)
            *reinterpret_cast<float2*>(part + (warp * G + hl) * PR + kD) = make_float2(m, lsum);
    }
    __syncthreads();
    for (int e = tid; e < G * kD; e += kCT) {
        const int hh = e / kD, dcol = e % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCW; ++w) M = fmaxf(M, part[(w * G + hh) * PR + kD]);
        float Lt = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kCW; ++w) {
                const float* pw = part + (w * G + hh) * PR;
                if (pw[kD] == -INFINITY) continue;
                const float cf = exp2_approx(pw[kD] - M);
                Lt = fmaf(pw[kD + 1], cf, Lt);
                O = fmaf(pw[dcol], cf, O);
            }
        }
        dst[hh * (kD + 2) + dcol] = O;
        if (dcol == 0) {
            dst[hh * (kD + 2) + kD] = M;
            dst[hh * (kD + 2) + kD + 1] = Lt;
        }
    }
    if (tid == 0) reinterpret_cast<int*>(dst)[G * (kD + 2)] = *s_fail;
}

template <typename T, int G, bool FUSED>
__global__ void __launch_bounds__(kCT, 2) select_cluster_kernel(
    IndexView v, const T* __restrict__ q, int n_sel, CluDims dm, int smem_total,
    int32_t* __restrict__ page_ids, int32_t* __restrict__ n_pages_out,
    int32_t* __restrict__ stats, T* __restrict__ attn_out, int head_div) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(16) float2 s_qp[kD / 2];  // (q_sel[e], q_sel[e + 64]), e < 64
    __shared__ int s_qcode[kM];
    __shared__ __align__(16) __half2 s_width[97 * 4];
    __shared__ int s_pstar, s_need, s_nch, s_base, s_ncand, s_cmp, s_fail, s_gn, s_taken, s_nl[kMaxL];
    __shared__ __align__(8) unsigned long long s_bar;

    cg::cluster_group cluster = cg::this_cluster();
    const int K = (int)cluster.num_blocks();
    const int r = (int)cluster.block_rank();
    // head_div > 1: per-query-head selection, row = (unit, head) with the unit's tables
    const int row = blockIdx.x / K, u = row / head_div;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = v.L, P = v.P;
    const int pshift = (P & (P - 1)) == 0 ? __ffs(P) - 1 : -1;  // page of a slot by a shift
    const long long C = v.C;
    const int Kc = K / L, l = r / Kc, rc = r % Kc;
    const int n_cand = dm.n_cand;
    const CluSmem lay = clu_layout(C, dm, L, n_sel, K, G, FUSED, 0);
    int* s_sel = reinterpret_cast<int*>(smem + lay.sel);
    int* s_scnt = reinterpret_cast<int*>(smem + lay.scnt);
    int* s_toff = reinterpret_cast<int*>(smem + lay.toff);
    int* lhist = reinterpret_cast<int*>(smem + lay.lhist);
    // [0..L) taken leaves per composite, 3 candidates, 4 expanded slots, 8 + r pages of block r
    int* hubx = reinterpret_cast<int*>(smem + lay.hubx);
    unsigned* hub_leaf = reinterpret_cast<unsigned*>(smem + lay.hub_leaf);  // [L][n_cand] id << 8 | count
    uint4* hub_pe = reinterpret_cast<uint4*>(smem + lay.hub_pe);  // [K][n_sel] (key lo, key hi, page, count)
    float* hub_part = reinterpret_cast<float*>(smem + lay.hub_part);  // [K][G (kD + 2) + 4]
    float* qf = reinterpret_cast<float*>(smem + lay.qf);
    unsigned* bm0 = reinterpret_cast<unsigned*>(smem + lay.bm0);
    const int nwords0 = (int)((C + 31) / 32);
    int* hubx0 = cluster.map_shared_rank(hubx, 0);

    // ---- 1. leaf count, query heads and directions requested together ------------------
    // The query may be the previous kernel's output: it is read after the wait on that
    // kernel (programmatic dependent launch). The index tables are read before the wait
    // when that kernel wrote none of them (early): the leaf counts, the directions and the
    // scan's first copies then overlap the previous kernel.
    const bool early = v.early_index != 0;
    float qh[G][4];
    const T* qu = q + (long long)row * G * kD;
    auto load_query = [&]() {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) load4(qu + (long long)hh * kD + 4 * lane, qh[hh]);
    };
    if (!early) {
        pdl_wait_then_release();
        load_query();
    }
    int Nl = v.n_leaf[v.ul(u, l)];
    int Nall = 0;
    if (r == 0)
        for (int ll = 0; ll < L; ++ll) Nall += max(0, min(v.n_leaf[v.ul(u, ll)], (int)C));
    float wdir[4] = {0.f, 0.f, 0.f, 0.f};
    float wlast = 0.f;
    if (warp < kM) {
        const float* ud = v.dirs + (long long)(l * kM + warp) * kDirStride;
        load4(ud + 4 * lane, wdir);
        wlast = ud[kD];
    }
    int* hist = reinterpret_cast<int*>(smem + lay.hist);
    unsigned* tieb = reinterpret_cast<unsigned*>(smem + lay.tieb);
    if (tid < 97) {
        __half2 w[4];
        cell_widths(tid, w);
#pragma unroll
        for (int k = 0; k < 4; ++k) s_width[tid * 4 + k] = w[k];
    }
    for (int i = tid; i < kCSubH * kCHistRow; i += kCT) hist[i] = 0;
    for (int i = tid; i < dm.rcap / 32; i += kCT) tieb[i] = 0u;
    if (L > 1)
        for (int i = tid; i < nwords0; i += kCT) bm0[i] = 0u;
    if (r == 0 && tid < 32) hubx[tid] = 0;
    if (tid == 0) {
        s_nch = 0;
        s_ncand = 0;
        s_fail = 0;
        if (FUSED) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    // a block of a composite that is not split starts the cluster barrier now: its
    // histogram is the composite's, and the barrier only has to order block 0's
    // cleared counters before the first remote update
    if (Kc == 1) clu_arrive();
    Nl = Nl < 0 ? 0 : (Nl > C ? (int)C : Nl);
    // this block's leaves: 64-leaf chunks [c0, c1) of the composite, in position order
    const int chunks = (Nl + 63) >> 6;
    const int c0 = rc * chunks / Kc, c1 = (rc + 1) * chunks / Kc;
    const int nck = c1 - c0;
    const int lo_leaf = 64 * c0;
    const int nloc = max(0, min(Nl, 64 * c1) - lo_leaf);
    // the scan reads whole leaf records (lower corner, list id | count, prefix length),
    // so the ids of the taken leaves are at hand without a second round trip
    const uint4* lrec = v.leaf_rec + v.leaf_base(u, l) + lo_leaf;
    const unsigned ring = smem_u32(smem + lay.ring + warp * (kCRing * kCSlotB));
    auto ring_issue = [&](int k, int slot) {
        const unsigned d = ring + slot * kCSlotB + lane * 32;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(lrec + 64 * k + 2 * lane)
                     : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + 16),
                     "l"(lrec + 64 * k + 2 * lane + 1)
                     : "memory");
    };
#pragma unroll
    for (int sidx = 0; sidx < kCRing; ++sidx) {
        const int k = warp + sidx * kCW;
        if (k < nck) ring_issue(k, sidx);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (early) {
        pdl_wait_then_release();
        load_query();
    }
    // query prep: q_sel = sum of the heads in head order, q~ = q_sel / |q_sel|,
    // codes of this block's composite (warp j: direction j)
    {
        float qs[4] = {qh[0][0], qh[0][1], qh[0][2], qh[0][3]};
#pragma unroll
        for (int hh = 1; hh < G; ++hh)
#pragma unroll
            for (int k = 0; k < 4; ++k) qs[k] = __fadd_rn(qs[k], qh[hh][k]);
        const float nq = warp_dot_fixed(qs, qs);
        float qt[4] = {0.f, 0.f, 0.f, 0.f};
        if (nq > 0.0f) {
            const float sn = __fsqrt_rn(nq);
#pragma unroll
            for (int k = 0; k < 4; ++k) qt[k] = __fdiv_rn(qs[k], sn);
        }
        if (warp < kM) {
            const float p = __fmaf_rn(wlast, 0.0f, warp_dot_fixed(wdir, qt));
            if (lane == 0) s_qcode[warp] = quantise_code(p);
        }
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = 4 * lane + k;
                if (e < kD / 2) s_qp[e].x = qs[k];
                else s_qp[e - kD / 2].y = qs[k];
            }
            if (FUSED) {
#pragma unroll
                for (int hh = 0; hh < G; ++hh)
#pragma unroll
                    for (int k = 0; k < 4; ++k) qf[hh * kD + 4 * lane + k] = qh[hh][k];
            }
        }
    }
    __syncthreads();

    // ---- 2. priorities, counts and sub-histograms of this block's leaves ----------------
    unsigned char* prio = smem + lay.prio;
    unsigned char* cnts = smem + lay.cnt;
    unsigned* lid = reinterpret_cast<unsigned*>(smem + lay.lid);  // list id << 8 | count
    {
        __half2 qc[4];
        {
            unsigned lo4 = 0, hi4 = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo4 |= (unsigned)s_qcode[j] << (8 * j);
                hi4 |= (unsigned)s_qcode[4 + j] << (8 * j);
            }
            qc[0] = bytes_to_h2(lo4, 0x4140u);
            qc[1] = bytes_to_h2(lo4, 0x4342u);
            qc[2] = bytes_to_h2(hi4, 0x4140u);
            qc[3] = bytes_to_h2(hi4, 0x4342u);
        }
        int* hl = hist + (lane & (kCSubH - 1)) * kCHistRow;
        const unsigned pr_base = smem_u32(prio);
        const unsigned cn_base = smem_u32(cnts);
        int slot = 0;
        for (int k = warp; k < nck; k += kCW) {  // warp-uniform
            asm volatile("cp.async.wait_group %0;" ::"n"(kCRing - 1) : "memory");
            const unsigned d = ring + slot * kCSlotB + lane * 32;
            uint4 ra, rb;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(ra.x), "=r"(ra.y), "=r"(ra.z), "=r"(ra.w)
                         : "r"(d)
                         : "memory");
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(rb.x), "=r"(rb.y), "=r"(rb.z), "=r"(rb.w)
                         : "r"(d + 16)
                         : "memory");
            const int i0 = 64 * k + 2 * lane;
            const int p0 = leaf_priority(ra.x, ra.y, (int)min(ra.w, 127u), qc, s_width);
            const int p1 = leaf_priority(rb.x, rb.y, (int)min(rb.w, 127u), qc, s_width);
            const int cA = (int)(ra.z & 0xFFu), cB = (int)(rb.z & 0xFFu);
            if (i0 < nloc) {
                st_shared_u16(pr_base + i0, p0 | (p1 << 8));
                st_shared_u16(cn_base + i0, cA | (cB << 8));
                *reinterpret_cast<uint2*>(lid + i0) = make_uint2(ra.z, rb.z);
                atomicAdd(&hl[p0], cA);
                if (i0 + 1 < nloc) atomicAdd(&hl[p1], cB);
            }
            const int kn = k + kCRing * kCW;
            if (kn < nck) ring_issue(kn, slot);
            asm volatile("cp.async.commit_group;" ::: "memory");
            slot = slot + 1 == kCRing ? 0 : slot + 1;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncthreads();

    // ---- 3. the composite's histogram (pulled over DSMEM when it is split), pi*, and the
    //         tokens at pi* in the composite's blocks before this one -------------------------
    int* ghist = reinterpret_cast<int*>(smem + lay.ghist);
    int* gpre = reinterpret_cast<int*>(smem + lay.gpre);
    {
        int hsum = 0;
#pragma unroll
        for (int sh = 0; sh < kCSubH; ++sh) hsum += hist[sh * kCHistRow + tid];
        if (Kc > 1) {
            lhist[tid] = hsum;
            clu_arrive();
            clu_wait();
            int x[16];  // Kc <= 16 blocks per composite
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                x[rr] = rr < Kc ? cluster.map_shared_rank(lhist, l * Kc + rr)[tid] : 0;
            int tot = 0, pre = 0;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                tot += x[rr];
                pre += rr < rc ? x[rr] : 0;
            }
            ghist[tid] = tot;
            gpre[tid] = pre;
        } else {
            ghist[tid] = hsum;
            gpre[tid] = 0;
        }
    }
    __syncthreads();
    if (warp == 0) {
        int loc[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            loc[k] = ghist[lane * 8 + k];
            sum += loc[k];
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
                s_pstar = 256;  // fewer than n_cand tokens in the composite: take every leaf
                s_need = 0;
            }
        } else if (lane == __ffs(hit) - 1) {
            int run = excl, k = 0;
            while (run + loc[k] < n_cand) {
                run += loc[k];
                ++k;
            }
            const int ps = lane * 8 + k;
            s_pstar = ps;
            // the ties of the blocks before this one come first in position order
            s_need = max(0, n_cand - run - gpre[ps]);
        }
    }
    __syncthreads();

    // ---- 4. leaves below pi* are taken; leaves at pi* are marked in a bitmap ---------------
    int* chosen = reinterpret_cast<int*>(smem + lay.chosen);
    unsigned* cmeta = reinterpret_cast<unsigned*>(smem + lay.cmeta);
    {
        const int ps = s_pstar;
        const unsigned* p32 = reinterpret_cast<const unsigned*>(prio);
        const int nw = (nloc + 3) >> 2;
        // a word with no priority <= ps holds nothing to take or mark: for ps < 128 the
        // test is the borrow of a bytewise subtraction of ps + 1
        const unsigned lim = 0x01010101u * (unsigned)(ps + 1);
        for (int w4 = tid; w4 < nw; w4 += kCT) {
            const unsigned word = p32[w4];
            if (ps < 128 && ((word - lim) & ~word & 0x80808080u) == 0u) continue;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = 4 * w4 + b;
                if (i >= nloc) break;
                const int pr = (int)((word >> (8 * b)) & 0xFFu);
                if (pr < ps) {
                    const int slot = atomicAdd(&s_nch, 1);
                    if (slot < n_cand) {
                        chosen[slot] = i;
                        cmeta[slot] = lid[i];
                    }
                } else if (pr == ps) {
                    atomicOr(&tieb[i >> 5], 1u << (i & 31));
                }
            }
        }
    }
    __syncthreads();
    // this block's ties in position order while the tokens taken before them < need
    if (warp == 0) {
        const int need = s_need;
        const int nwords = (nloc + 31) >> 5;
        const int nbelow = min(s_nch, n_cand);
        int run = 0, ntaken = 0;
        for (int w0 = 0; w0 < nwords && run < need; w0 += 32) {
            const int wi = w0 + lane;
            const unsigned bits = wi < nwords ? tieb[wi] : 0u;
            uint4 ca = make_uint4(0u, 0u, 0u, 0u), cb = ca;
            if (bits) {
                ca = *reinterpret_cast<const uint4*>(cnts + wi * 32);
                cb = *reinterpret_cast<const uint4*>(cnts + wi * 32 + 16);
            }
            const unsigned cw[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
            unsigned tsum = 0u;
#pragma unroll
            for (int qd = 0; qd < 8; ++qd)
                tsum = __dp4a(cw[qd] & nibble_bytes((bits >> (4 * qd)) & 0xFu), 0x01010101u, tsum);
            const int tot = (int)tsum;
            int inc = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const int acc = run + inc - tot;
            const unsigned bt = boundary_take(bits, cw, acc, tot, need, lane);
            const unsigned take = acc + tot <= need ? bits : (acc < need ? bt : 0u);
            const int mine = __popc(take);
            int tinc = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, tinc, o);
                if (lane >= o) tinc += y;
            }
            const int sbase = nbelow + ntaken + tinc - mine;
            // one pass per word with ties taken (each lane one bit), or one pass per tie of
            // the busiest lane, whichever is fewer
            const unsigned nz = __ballot_sync(0xffffffffu, take != 0u);
            if (__popc(nz) < __reduce_max_sync(0xffffffffu, (unsigned)mine)) {  // warp-uniform
                for (unsigned z = nz; z; z &= z - 1u) {
                    const int w = __ffs(z) - 1;
                    const unsigned t = __shfl_sync(0xffffffffu, take, w);
                    const int sb = __shfl_sync(0xffffffffu, sbase, w);
                    const int slot = sb + __popc(t & ((1u << lane) - 1u));
                    if (((t >> lane) & 1u) && slot < n_cand) {
                        const int i = (w0 + w) * 32 + lane;
                        chosen[slot] = i;
                        cmeta[slot] = lid[i];
                    }
                }
            } else {
                int slot = sbase;
                for (unsigned bb = take; bb; bb &= bb - 1u, ++slot)
                    if (slot < n_cand) {
                        const int i = wi * 32 + __ffs(bb) - 1;
                        chosen[slot] = i;
                        cmeta[slot] = lid[i];
                    }
            }
            ntaken += __shfl_sync(0xffffffffu, tinc, 31);
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_nch = min(nbelow + ntaken, n_cand);
    }
    if (Kc == 1) clu_wait();  // block 0's counters are cleared (the barrier started at the top)
    __syncthreads();
    // the taken leaves (list id | count) go to block 0's table of the composite
    const int nch = s_nch;
    if (tid == 0) s_base = nch > 0 ? atomicAdd(&hubx0[l], nch) : 0;
    __syncthreads();
    {
        unsigned* hl0 = cluster.map_shared_rank(hub_leaf, 0) + l * n_cand;
        const int base = s_base;
        for (int k = tid; k < nch; k += kCT)
            if (base + k < n_cand) hl0[base + k] = cmeta[k];
    }
    clu_arrive();
    clu_wait();

    // ---- 5. every block expands an equal share of the unit's candidate slots --------------
    unsigned* tl = reinterpret_cast<unsigned*>(smem + lay.tl);
    int* toffc = reinterpret_cast<int*>(smem + lay.toffc);
    unsigned long long* skey = reinterpret_cast<unsigned long long*>(smem + lay.skey);
    int* sval = reinterpret_cast<int*>(smem + lay.sval);
    if (tid < L) s_nl[tid] = min(hubx0[tid], n_cand);
    __syncthreads();
    const int nl0 = s_nl[0], nt = nl0 + (L > 1 ? s_nl[1] : 0);
    {
        const unsigned* hl0 = cluster.map_shared_rank(hub_leaf, 0);
        for (int k = tid; k < nt; k += kCT) {
            const unsigned e = k < nl0 ? hl0[k] : hl0[n_cand + (k - nl0)];
            tl[k] = e;
            if (L > 1 && k < nl0) {
                const int id = (int)(e >> 8);
                if (id < C) atomicOr(&bm0[id >> 5], 1u << (id & 31));
            }
        }
    }
    __syncthreads();
    if (warp == 0) {  // slot offsets of the taken leaves
        int carry = 0;
        for (int k0 = 0; k0 < nt; k0 += 32) {
            const int k = k0 + lane;
            const int c = k < nt ? (int)(tl[k] & 0xFFu) : 0;
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (k < nt) toffc[k] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) toffc[nt] = carry;
    }
    __syncthreads();
    const int total = toffc[nt];
    const int j0 = (int)((long long)r * total / K), j1 = (int)((long long)(r + 1) * total / K);
    for (int jb = j0 + warp * 32; jb < j1; jb += kCT) {
        const int j = jb + lane;
        bool keep = false;
        int tok = 0, loc = 0;
        if (j < j1) {
            int lo = 0, hi = nt;  // last k with toffc[k] <= j
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (toffc[mid] <= j) lo = mid; else hi = mid;
            }
            const int slot = j - toffc[lo];
            const int cl = lo < nl0 ? 0 : 1;
            const int id = (int)(tl[lo] >> 8);
            if (id < C && slot < P) {
                tok = v.slot_tok[v.slot_base(u, cl) + (long long)id * P + slot];
                if (cl == 0) {
                    loc = id * P + slot;
                    keep = true;
                } else {
                    // a composite-1 token whose page composite 0 took whole is a duplicate
                    loc = v.slot_loc1[v.loc1_base(u) + (long long)id * P + slot];
                    const int pg = loc >= 0 ? (pshift >= 0 ? loc >> pshift : loc / P) : 0;
                    keep = tok >= 0 && loc >= 0 && pg < C && !((bm0[pg >> 5] >> (pg & 31)) & 1u);
                }
            }
        }
        const unsigned km = __ballot_sync(0xffffffffu, keep);
        int pos0 = 0;
        if (lane == 0 && km) pos0 = atomicAdd(&s_ncand, __popc(km));
        pos0 = __shfl_sync(0xffffffffu, pos0, 0);
        if (keep) {
            const int pos = pos0 + __popc(km & ((1u << lane) - 1u));
            if (pos < dm.share_cap) {
                skey[pos] = (unsigned long long)(unsigned)tok;
                sval[pos] = loc;
            }
        }
    }
    // page table of this block's candidates
    int* hpage = reinterpret_cast<int*>(smem + lay.hpage);
    unsigned long long* hkey = reinterpret_cast<unsigned long long*>(smem + lay.hkey);
    int* hcnt = reinterpret_cast<int*>(smem + lay.hcnt);
    for (int i = tid; i < dm.hcap_l; i += kCT) {
        hpage[i] = -1;
        hkey[i] = ~0ull;
    }
    __syncthreads();
    const int ncand = min(s_ncand, dm.share_cap);

    // ---- 6. exact rescoring of this block's candidates; per-page minimum key ---------------
    {
        constexpr int EPC = 16 / (int)sizeof(T);
        constexpr int CPR = kD / EPC;
        constexpr int ROWB = kD * (int)sizeof(T);
        const int pad = pad_to_128(smem + lay.stage);  // 0 when the window starts aligned
        unsigned char* stg = smem + lay.stage + pad;
        const int half = min((smem_total - lay.stage - pad) / (2 * ROWB), kCT / 2);
        const int nchunk = (ncand + half - 1) / half;
        const char* pk = reinterpret_cast<const char*>(v.page_k) + (long long)u * C * P * ROWB;
        const int hmask = dm.hcap_l - 1;
        // thread tid copies piece c = tid mod CPR of rows tid / CPR, + RSTEP, ...; when
        // the swizzle repeats within RSTEP rows the piece's position stays fixed
        constexpr int RSTEP = kCT / CPR;
        constexpr bool kFixedPos = RSTEP % (CPR / 2) == 0;
        const int cpc = tid % CPR, r_first = tid / CPR;
        auto issue = [&](int ch) {
            if (ch < nchunk) {
                const int rb = ch * half, nr = min(half, ncand - rb);
                const unsigned buf = smem_u32(stg + (ch & 1) * half * ROWB);
                const char* src = pk + 16 * cpc;
                for (int rr = r_first; rr < nr; rr += RSTEP) {
                    const int pos = kFixedPos ? (cpc ^ ((r_first & (CPR / 2 - 1)) << 1))
                                              : (cpc ^ ((rr & (CPR / 2 - 1)) << 1));
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                     buf + rr * ROWB + 16 * pos),
                                 "l"(src + (long long)sval[rb + rr] * ROWB)
                                 : "memory");
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        issue(0);
        issue(1);
        for (int ch = 0; ch < nchunk; ++ch) {  // block-uniform
            const int rb0 = ch * half, nr = min(half, ncand - rb0);
            const unsigned char* stgc = stg + (ch & 1) * half * ROWB;
            asm volatile("cp.async.wait_group 1;" ::: "memory");
            __syncthreads();
            const int rr = tid >> 1, t = tid & 1;
            const bool ok = rr < nr;
            const int sw = (rr & (CPR / 2 - 1)) << 1;
            int pg = -1;
            unsigned long long key = ~0ull;
            float s4[2] = {0.0f, 0.0f};
            if (ok) {
                const unsigned char* rowp = stgc + rr * ROWB;
                float s16[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int ln = ((j >> 1) << 2) | (t << 1) | (j & 1);
                    const int e0 = 4 * ln, e1 = 4 * (ln + 16);
                    const int cc0 = e0 / EPC, cc1 = e1 / EPC;
                    float x0[EPC], x1[EPC];
                    load_chunk<T>(rowp + 16 * (cc0 ^ sw), x0);
                    load_chunk<T>(rowp + 16 * (cc1 ^ sw), x1);
                    const int o0 = e0 % EPC, o1 = e1 % EPC;
                    float2 ab = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        ab = __ffma2_rn(s_qp[e0 + i], make_float2(x0[o0 + i], x1[o1 + i]), ab);
                    s16[j] = __fadd_rn(ab.x, ab.y);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) s16[j] = __fadd_rn(s16[j], s16[j + 4]);
                s4[0] = __fadd_rn(s16[0], s16[2]);
                s4[1] = __fadd_rn(s16[1], s16[3]);
            }
            {
                const float p0 = __shfl_xor_sync(0xffffffffu, s4[0], 1);
                const float p1 = __shfl_xor_sync(0xffffffffu, s4[1], 1);
                const float a0 = t ? p0 : s4[0], a2 = t ? s4[0] : p0;
                const float a1 = t ? p1 : s4[1], a3 = t ? s4[1] : p1;
                const float sc = __fadd_rn(__fadd_rn(a0, a2), __fadd_rn(a1, a3));
                if (ok) {
                    pg = pshift >= 0 ? sval[rb0 + rr] >> pshift : sval[rb0 + rr] / P;
                    key = ((unsigned long long)score_key_desc(sc) << 32) | (unsigned)skey[rb0 + rr];
                }
            }
#pragma unroll
            for (int o = 2; o < 32; o <<= 1) {
                const int opg = __shfl_up_sync(0xffffffffu, pg, o);
                const unsigned long long okey = __shfl_up_sync(0xffffffffu, key, o);
                if (lane >= o && opg == pg && okey < key) key = okey;
            }
            const int next_pg = __shfl_down_sync(0xffffffffu, pg, 2);
            if (ok && t == 0 && (lane >= 30 || next_pg != pg)) {
                unsigned hh = ((unsigned)pg * 2654435761u) & (unsigned)hmask;
                for (int probe = 0; probe < dm.hcap_l; ++probe) {
                    const int old = atomicCAS(&hpage[hh], -1, pg);
                    if (old == -1 || old == pg) {
                        if (old == -1)  // the page's token count travels with it to the attention
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(hcnt + hh)),
                                         "l"(v.list_cnt + v.leaf_base(u, 0) + pg)
                                         : "memory");
                        atomicMin(&hkey[hh], key);
                        break;
                    }
                    hh = (hh + 1) & (unsigned)hmask;
                }
            }
            __syncthreads();
            issue(ch + 2);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    if (tid == 0) s_cmp = 0;
    __syncthreads();
    // this block's n_sel best pages (minimum key, count) go to block 0's table: a page
    // of the unit's selection is among the best pages of the block that holds its
    // minimum (fewer than n_sel of that block's pages rank before it there)
    {
        unsigned long long* ck = skey;  // compacted in place of the candidates
        int* cpg = sval;
        for (int h0 = warp * 32; h0 < dm.hcap_l; h0 += kCT) {  // warp-uniform
            const int hh = h0 + lane;
            const int pg = hh < dm.hcap_l ? hpage[hh] : -1;
            const unsigned km = __ballot_sync(0xffffffffu, pg >= 0);
            int base = 0;
            if (lane == 0 && km) base = atomicAdd(&s_cmp, __popc(km));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (pg >= 0) {
                const int pos = base + __popc(km & ((1u << lane) - 1u));
                ck[pos] = hkey[hh];
                cpg[pos] = hh;
            }
        }
        __syncthreads();
        const int npl = s_cmp;
        if (tid == 0) {
            hubx0[8 + r] = min(npl, n_sel);
            atomicAdd(&hubx0[3], ncand);
            atomicAdd(&hubx0[4], j1 - j0);
        }
        uint4* pe0 = cluster.map_shared_rank(hub_pe, 0) + r * n_sel;
        if (npl <= kCT) {
            // a page's place among this block's pages: the number with a smaller key
            if (tid < npl) {
                const unsigned long long key = ck[tid];
                int rank = 0;
                for (int j = 0; j < npl; ++j) rank += ck[j] < key ? 1 : 0;
                if (rank < n_sel) {
                    const int hh = cpg[tid];
                    pe0[rank] = make_uint4((unsigned)key, (unsigned)(key >> 32), (unsigned)hpage[hh],
                                           (unsigned)hcnt[hh]);
                }
            }
        } else {
            unsigned long long tk;
            int tv;
            block_top32(ck, cpg, npl, reinterpret_cast<unsigned long long*>(smem + lay.top),
                        reinterpret_cast<int*>(smem + lay.top + kCW * 32 * 8), tk, tv);
            if (warp == 0 && lane < min(npl, n_sel))
                pe0[lane] = make_uint4((unsigned)tk, (unsigned)(tk >> 32), (unsigned)hpage[tv],
                                       (unsigned)hcnt[tv]);
        }
    }
    clu_arrive();
    clu_wait();

    // ---- 7. the selection (block 0): per page the minimum key over the blocks' lists, the
    //         n_sel smallest; sent to every block of the cluster -----------------------------
    if (r == 0) {
        int* g_page = reinterpret_cast<int*>(smem + lay.g_page);
        unsigned long long* g_key = reinterpret_cast<unsigned long long*>(smem + lay.g_key);
        unsigned long long* gk = reinterpret_cast<unsigned long long*>(smem + lay.gk);  // [K n_sel]
        int* gslot = reinterpret_cast<int*>(smem + lay.gp);                            // [K n_sel]
        for (int i2 = tid; i2 < dm.gcap; i2 += kCT) {
            g_page[i2] = -1;
            g_key[i2] = ~0ull;
        }
        if (tid == 0) s_gn = 0;
        __syncthreads();
        const int gmask = dm.gcap - 1;
        const int NE = K * n_sel;
        // each entry takes its page's slot in the table and lowers the page's minimum
        for (int e = tid; e < NE; e += kCT) {
            const int rr = e / n_sel;
            int slot = -1;
            if (e - rr * n_sel < min(hubx[8 + rr], n_sel)) {
                const uint4 x = hub_pe[e];
                const unsigned long long key = ((unsigned long long)x.y << 32) | x.x;
                const int pg = (int)x.z;
                unsigned hh = ((unsigned)pg * 2654435761u) & (unsigned)gmask;
                for (int probe = 0; probe < dm.gcap; ++probe) {
                    const int old = atomicCAS(&g_page[hh], -1, pg);
                    if (old == -1 || old == pg) {
                        atomicMin(&g_key[hh], key);
                        slot = (int)hh;
                        break;
                    }
                    hh = (hh + 1) & (unsigned)gmask;
                }
            }
            gslot[e] = slot;
        }
        __syncthreads();
        // an entry that holds its page's minimum keeps its key, every other entry ~0
        for (int e = tid; e < NE; e += kCT) {
            unsigned long long w = ~0ull;
            if (gslot[e] >= 0) {
                const uint4 x = hub_pe[e];
                const unsigned long long key = ((unsigned long long)x.y << 32) | x.x;
                if (g_key[gslot[e]] == key) w = key;
            }
            gk[e] = w;
        }
        __syncthreads();
        // the rank of a page is the number of kept keys below its own (keys are unique);
        // tpe adjacent threads share an entry's count and add their parts
        const int tpe = NE <= kCT / 8 ? 8 : NE <= kCT / 4 ? 4 : NE <= kCT / 2 ? 2 : 1;
        for (int base = 0; base < NE * tpe; base += kCT) {  // block-uniform
            const int idx = base + tid;
            const int e = idx / tpe, part = idx % tpe;
            const bool live = idx < NE * tpe;
            const unsigned long long key = live ? gk[e] : ~0ull;
            int rank = 0;
            if (key != ~0ull) {
                const int jlo = part * NE / tpe, jhi = (part + 1) * NE / tpe;
#pragma unroll 8
                for (int j2 = jlo; j2 < jhi; ++j2) rank += gk[j2] < key ? 1 : 0;
            }
            for (int o = 1; o < tpe; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
            if (key != ~0ull && part == 0) {
                atomicAdd(&s_gn, 1);
                if (rank < n_sel) {
                    const uint4 x = hub_pe[e];
                    s_sel[rank] = (int)x.z;
                    s_scnt[rank] = (int)x.w;
                }
            }
        }
        __syncthreads();
        const int taken = min(n_sel, s_gn);
        if (tid >= taken && tid < n_sel) {
            s_sel[tid] = -1;
            s_scnt[tid] = 0;
        }
        if (tid == 0) s_taken = taken;
        __syncthreads();
        if (FUSED) {  // the selection to the other blocks
            for (int e = tid; e < (K - 1) * n_sel; e += kCT) {
                const int rr = 1 + e / n_sel, i2 = e % n_sel;
                cluster.map_shared_rank(s_sel, rr)[i2] = s_sel[i2];
                cluster.map_shared_rank(s_scnt, rr)[i2] = s_scnt[i2];
            }
            if (tid > 0 && tid < K) *cluster.map_shared_rank(&s_taken, tid) = taken;
        }
    }
    if (tid == 0 && ncand < s_ncand) set_status(v.status, ICE_ERR_CAPACITY);
    clu_arrive();
    // block 0 writes the selection out while the barrier completes (block 0 keeps its
    // tables until every block has passed it)
    if (r == 0 && warp == 0) {
        const int taken = s_taken;
        if (lane < n_sel) page_ids[(long long)row * n_sel + lane] = s_sel[lane];
        int tok_sel = lane < taken ? s_scnt[lane] : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) tok_sel += __shfl_xor_sync(0xffffffffu, tok_sel, o);
        if (lane == 0) {
            n_pages_out[row] = taken;
            if (stats) {
                stats[4 * row + 0] = Nall;
                stats[4 * row + 1] = hubx[3];
                stats[4 * row + 2] = tok_sel;
                stats[4 * row + 3] = hubx[4];
            }
        }
    }
    clu_wait();
    if (!FUSED) return;
    const int taken = s_taken;

    // ---- 8. attention over this block's pages; the partials are merged in block 0 -----------
    if constexpr (FUSED) {
        const int PW = G * (kD + 2) + 4;
        attend_partial<T, G>(v, u, qf, s_sel, s_scnt, taken, r, K, s_toff, smem + lay.X,
                             smem_total - lay.X, smem_u32(&s_bar), &s_fail,
                             cluster.map_shared_rank(hub_part, 0) + r * PW);
        clu_arrive();
        clu_wait();
        if (r == 0) {
            T* ou = attn_out + (long long)row * G * kD;
            for (int e = tid; e < G * kD; e += kCT) {
                const int hh = e / kD, dcol = e % kD;
                float M = -INFINITY;
                int fail = 0;
                for (int rr = 0; rr < K; ++rr) {
                    const float* cp = hub_part + rr * PW;
                    M = fmaxf(M, cp[hh * (kD + 2) + kD]);
                    fail |= reinterpret_cast<const int*>(cp)[G * (kD + 2)];
                }
                float Lt = 0.0f, O = 0.0f;
                if (M != -INFINITY && !fail) {
                    for (int rr = 0; rr < K; ++rr) {
                        const float* cp = hub_part + rr * PW;
                        const float mr = cp[hh * (kD + 2) + kD];
                        if (mr == -INFINITY) continue;
                        const float cf = exp2_approx(mr - M);
                        Lt = fmaf(cp[hh * (kD + 2) + kD + 1], cf, Lt);
                        O = fmaf(cp[hh * (kD + 2) + dcol], cf, O);
                    }
                }
                ou[e] = from_f<T>(Lt > 0.0f ? O / Lt : 0.0f);
            }
        }
    }
}

// ---- host side -------------------------------------------------------------------------

namespace {

struct CluPlan {
    int K = 1, bytes = 0;
    CluDims d{};
};

int pow2_at_least(int x) {
    int c = 1;
    while (c < x) c <<= 1;
    return c;
}

CluPlan clu_plan(const IndexView& v, int K, int n_sel, int n_cand, bool fused, int target_bytes) {
    CluPlan p;
    p.K = K;
    const int L = v.L, P = v.P;
    const int Kc = K / L;
    const long long ch = (v.C + 63) / 64;
    p.d.rcap = (int)(64 * ((ch + Kc - 1) / Kc));
    p.d.n_cand = n_cand;
    p.d.s_tot = L * (n_cand + P - 1);
    p.d.share_cap = (p.d.s_tot + K - 1) / K;
    p.d.hcap_l = pow2_at_least(p.d.share_cap + 1);
    p.d.gcap = pow2_at_least(2 * K * n_sel + 1);
    const int es = v.dtype == ICE_BF16 ? 2 : 4;
    const CluSmem lay = clu_layout(v.C, p.d, L, n_sel, K, v.G, fused, 0);
    int need = lay.end;
    // the rescoring stages at least two rows a half, the attention at least one
    // page's K and V rows and then the warps' partials
    need = std::max(need, lay.stage + 2 * 2 * kD * es);
    if (fused) {
        need = std::max(need, lay.X + 2 * P * kD * es);
        need = std::max(need, lay.X + kCW * v.G * (kD + 4) * 4);  // partial rows of kD + 4
    }
    p.bytes = need > kCluSmemMax ? need : std::min(std::max(need, target_bytes), kCluSmemMax);
    return p;
}

template <typename T, int G, bool F>
cudaError_t clu_launch(const IndexView& v, const CluPlan& p, const void* q, int n_sel,
                       int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                       cudaStream_t s, int head_div = 1) {
    auto kern = select_cluster_kernel<T, G, F>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(v.U * head_div * p.K));
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = (size_t)p.bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)p.K;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait_then_release
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, v, (const T*)q, n_sel, p.d, p.bytes, page_ids, n_pages,
                              stats, (T*)out, head_div);
}

template <typename T, int G, bool F>
cudaError_t clu_prepare_one() {
    auto kern = select_cluster_kernel<T, G, F>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCluSmemMax);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

// Whether clusters of p.K blocks with p.bytes of shared memory can be resident
// at all (cached per configuration).
template <typename T, int G, bool F>
bool clu_fits(const IndexView& v, const CluPlan& p) {
    static std::mutex mu;
    static std::map<std::tuple<int, int>, bool> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(p.K, p.bytes);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(v.U * p.K));
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = (size_t)p.bytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)p.K;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, select_cluster_kernel<T, G, F>, &cfg);
    if (e != cudaSuccess) cudaGetLastError();
    const bool ok = e == cudaSuccess && n > 0;
    cache[key] = ok;
    return ok;
}

template <typename T, bool F>
cudaError_t clu_dispatch_g(const IndexView& v, const CluPlan& p, const void* q, int n_sel,
                           int n_cand, int32_t* page_ids, int32_t* n_pages, int32_t* stats,
                           void* out, cudaStream_t s, bool check_only, bool* fits) {
    switch (v.G) {
#define ICE_CLU_G(GG)                                                                              \
    case GG:                                                                                       \
        if (check_only) {                                                                          \
            *fits = clu_fits<T, GG, F>(v, p);                                                      \
            return cudaSuccess;                                                                    \
        }                                                                                          \
        return clu_launch<T, GG, F>(v, p, q, n_sel, page_ids, n_pages, stats, out, s);
        ICE_CLU_G(1) ICE_CLU_G(2) ICE_CLU_G(4) ICE_CLU_G(8)
#undef ICE_CLU_G
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t clu_dispatch(const IndexView& v, const CluPlan& p, const void* q, int n_sel, int n_cand,
                         int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                         cudaStream_t s, bool check_only, bool* fits) {
    const bool fused = out != nullptr;
    if (v.dtype == ICE_BF16)
        return fused ? clu_dispatch_g<__nv_bfloat16, true>(v, p, q, n_sel, n_cand, page_ids, n_pages,
                                                            stats, out, s, check_only, fits)
                     : clu_dispatch_g<__nv_bfloat16, false>(v, p, q, n_sel, n_cand, page_ids, n_pages,
                                                             stats, out, s, check_only, fits);
    return fused ? clu_dispatch_g<float, true>(v, p, q, n_sel, n_cand, page_ids, n_pages, stats, out,
                                               s, check_only, fits)
                 : clu_dispatch_g<float, false>(v, p, q, n_sel, n_cand, page_ids, n_pages, stats, out,
                                                s, check_only, fits);
}

}  // namespace

cudaError_t select_cluster_prepare() {
    cudaError_t e = cudaSuccess;
#define ICE_CLU_PREP(T, G)                                        \
    if (e == cudaSuccess) e = clu_prepare_one<T, G, true>();      \
    if (e == cudaSuccess) e = clu_prepare_one<T, G, false>();
    ICE_CLU_PREP(__nv_bfloat16, 1) ICE_CLU_PREP(__nv_bfloat16, 2) ICE_CLU_PREP(__nv_bfloat16, 4)
    ICE_CLU_PREP(__nv_bfloat16, 8) ICE_CLU_PREP(float, 1) ICE_CLU_PREP(float, 2)
    ICE_CLU_PREP(float, 4) ICE_CLU_PREP(float, 8)
#undef ICE_CLU_PREP
    return e;
}

// Shared memory a block is given beyond its tables (room to stage candidate rows
// and pages): two blocks per SM for launches of up to two blocks per SM, four
// blocks per SM above that.
int clu_target_bytes(int blocks) { return blocks <= 304 ? 100 * 1024 : 54 * 1024; }

// Cluster size for U units: 8 blocks per unit up to 19 units (one layer of
// 8 KV heads: 64 blocks; 16 blocks per unit measured slower there, the block
// that ranks gathers twice the lists), 4 up to 38, 2 up to 76; the one-block
// kernel for large launches, whose blocks already fill the SMs.
int select_cluster_auto(int U, int L) {
    int K = 1;
    if (U <= 19) K = 8;
    else if (U <= 38) K = 4;
    else if (U <= 76) K = 2;
    if (K < L) K = 1;
    return K;
}

int select_cluster_bytes(const IndexView& v, int K, int n_sel, int n_cand, bool fused) {
    if (K < 2 || K > 16 || (K & (K - 1)) || K < v.L || n_sel > kCTop) return -1;
    const CluPlan p = clu_plan(v, K, n_sel, n_cand, fused, clu_target_bytes(v.U * K));
    return p.bytes > kCluSmemMax ? -1 : p.bytes;
}

cudaError_t launch_select_cluster(const IndexView& v, int K, const void* q, int n_sel, int n_cand,
                                  int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                                  cudaStream_t s, bool* launched) {
    *launched = false;
    const bool fused = out != nullptr;
    if (select_cluster_bytes(v, K, n_sel, n_cand, fused) < 0) return cudaSuccess;
    const CluPlan p = clu_plan(v, K, n_sel, n_cand, fused, clu_target_bytes(v.U * K));
    bool fits = false;
    cudaError_t e = clu_dispatch(v, p, q, n_sel, n_cand, page_ids, n_pages, stats, out, s, true, &fits);
    if (e != cudaSuccess || !fits) return e;
    e = clu_dispatch(v, p, q, n_sel, n_cand, page_ids, n_pages, stats, out, s, false, &fits);
    if (e == cudaSuccess) *launched = true;
    return e;
}

// Per-query-head selection (one row per (unit, query head), the head's query alone)
// with a cluster of blocks per row. Sets *launched when it ran; leaves the launch to
// the one-block kernel when the rows are many or a cluster cannot hold them.
cudaError_t launch_select_heads_cluster(const IndexView& v, const void* q, int n_sel, int n_cand,
                                        int32_t* page_ids, int32_t* n_pages, cudaStream_t s,
                                        bool* launched) {
    *launched = false;
    const int rows = v.U * v.G;
    const int K = v.cluster_k > 0 ? v.cluster_k : select_cluster_auto(rows, v.L);
    if (K < 2 || select_cluster_bytes(v, K, n_sel, n_cand, false) < 0) return cudaSuccess;
    const CluPlan p = clu_plan(v, K, n_sel, n_cand, false, clu_target_bytes(rows * K));
    const bool fits = v.dtype == ICE_BF16 ? clu_fits<__nv_bfloat16, 1, false>(v, p)
                                          : clu_fits<float, 1, false>(v, p);
    if (!fits) return cudaSuccess;
    const cudaError_t e =
        v.dtype == ICE_BF16
            ? clu_launch<__nv_bfloat16, 1, false>(v, p, q, n_sel, page_ids, n_pages, nullptr, nullptr, s, v.G)
            : clu_launch<float, 1, false>(v, p, q, n_sel, page_ids, n_pages, nullptr, nullptr, s, v.G);
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace ice

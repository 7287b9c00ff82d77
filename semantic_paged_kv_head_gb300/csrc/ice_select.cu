// Decode-time page selection ("IceCache", Figure 2 steps 2-3; the blog's
// mechanism section: P-DCI, the prioritised DCI search, picks the pages most
// relevant to the current query), and optionally the attention over the
// selected pages in the same block (Figure 2 step 3).
//
// One 512-thread block per unit. The work of a unit is a chain of dependent
// phases, so each phase is organised to keep many requests in flight and to
// spend few instructions per element:
//  1. the unit's leaf counts, the group's query heads and the projection
//     directions are requested together; the first batch of leaf records is
//     requested before the query prep (q_sel = sum of the heads in head order,
//     normalised, projected and quantised per composite) is computed;
//  2. all composites are scanned: the priority of a leaf is the L-infinity
//     distance in code units between the query codes and the leaf's cell,
//     evaluated two directions per instruction on fp16x2 (codes are exact
//     small integers there); priority and token count of every leaf go to
//     shared memory, token counts by priority to sub-histograms;
//  3. per composite, pi* is the smallest priority whose cumulative count
//     reaches n_cand; leaves below pi* are taken (their records requested in
//     the same pass), and leaves at pi* in left-to-right order while the tokens
//     taken before them at pi* are fewer than needed (the order a best-first
//     tree search visits leaves in);
//  4. every slot of every taken leaf becomes a candidate (token, row) in one
//     parallel round; a composite-1 token whose page composite 0 already took
//     is a duplicate and dropped;
//  5. every candidate is rescored with the fixed-order fp32 dot q_sel . k
//     (8 lanes per row, each lane evaluating four of the 32 lane partials of
//     the fixed order), and its (score desc, token asc) key is min-reduced
//     into its page's slot of a shared-memory hash table: a page's first
//     occurrence in the ranked candidate list is its smallest key;
//  6. the n_sel pages with the smallest keys, in key order, are the selection
//     (warp-level bitonic top-32 and a merge tree over the warps' lists; a
//     block-wide bitonic sort when n_sel > 32);
//  7. (fused) the K and V rows of the selected pages are staged in shared
//     memory with bulk asynchronous copies (cp.async.bulk, one per page and
//     tensor, completing on one mbarrier) into the space the selection no
//     longer needs, and the G query heads attend over them: lane = (head, 32/G
//     dimensions' group), one token per warp instruction, fp32 online softmax
//     per warp, warps merged in a fixed order.
#include "ice_internal.cuh"
#include "ice_insert.cuh"
#include "ice_select_common.cuh"

namespace ice {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSubH = 8;      // sub-histograms per composite (lane groups)
constexpr int kHistRow = 257;  // words per sub-histogram row (256 priorities + 1 pad)
constexpr int kRing = 3;      // scan chunks of 64 leaves in flight per warp
constexpr int kSlotB = 640;   // one chunk: 64 corners (8 B) + 64 (t | count << 7) (2 B)
constexpr int kRingB = kSelWarps * kRing * kSlotB;
constexpr int kTopK = 32;     // warp top-k width
constexpr int kFusedSmem = 108 * 1024;  // fused blocks grow to this (two blocks per SM)

// Shared-memory layout. sel/toff live through the whole kernel; keys .. top
// hold the leaf-record copy ring during the scan, then the page hash (from
// phase 3b on) and the candidates (from phase 4 on). Everything from `free`
// on is dead once the candidates are expanded: rescoring stages candidate rows
// there, and the fused attention stages pages there (from `keys` on, after the
// ranking) and finally the warps' partial results.
struct SelSmem {
    int sel, toff, qf;
    int keys, vals, hpage, hkey, hcnt, top, ring;
    int free;
    int prio, cnt, chosen, cmeta, coff, tieb, bm0, hist;
    int end;
};

__host__ __device__ inline SelSmem sel_layout(long long C, int L, int n_cand, int sort_cap,
                                              int hcap, int n_sel, int min_total) {
    SelSmem s;
    int o = 0;
    s.sel = o; o = align16(o + n_sel * 4);
    s.toff = o; o = align16(o + (n_sel + 1) * 4);
    s.qf = o; o = align128(o + kMaxG * kD * 4);
    s.keys = o; o = align16(o + sort_cap * 8);
    s.vals = o; o = align16(o + sort_cap * 4);
    s.hpage = o; o = align16(o + hcap * 4);
    s.hkey = o; o = align16(o + hcap * 8);
    s.hcnt = o; o = align16(o + hcap * 4);
    s.top = o; o = align16(o + kSelWarps * kTopK * 12);
    s.ring = s.keys;  // the scan's copy ring, dead before the candidates are written
    if (o < s.ring + kRingB) o = s.ring + kRingB;
    o = align128(o);
    s.free = o;
    const int Cp = align16((int)C);
    s.prio = o; o = align16(o + L * Cp);
    s.cnt = o; o = align16(o + L * Cp);
    s.chosen = o; o = align16(o + L * n_cand * 4);
    s.cmeta = o; o = align16(o + L * n_cand * 4);
    s.coff = o; o = align16(o + L * (n_cand + 1) * 4);
    s.tieb = o; o = align16(o + L * (int)((C + 31) / 32) * 4);
    s.bm0 = o; o = align16(o + (int)((C + 31) / 32) * 4);
    s.hist = o; o = align16(o + L * kSubH * kHistRow * 4);
    s.end = o > min_total ? o : min_total;
    return s;
}

// Attention of the G query heads of unit u over every token of the selected
// pages (the fused tail). Pages are staged in rounds that fit the staging
// region: lanes of warp 0 issue one bulk copy per page for K and one for V onto
// one mbarrier; then every warp takes tokens w, w + 16, ... of the round. Lane
// l holds dimensions 4l..4l+3 of every head: a token's row is read once per
// warp. The heads' partial scores are summed across the lanes by halving: at
// each of the first log2 G exchange levels a lane keeps half of the heads it
// holds and sends the other half, so that after the last level lane l holds
// the score of head (l >> (5 - log2 G)). That lane keeps the head's softmax
// state, and every lane takes the G (correction, weight) pairs by shuffles.
template <typename T, int G>
__device__ __forceinline__ void attend_staged(const IndexView& v, int u, const T* __restrict__ q,
                                              const float* s_q, const int* hpage, const int* hcnt,
                                              int hcap, int npg, const int* s_sel, int* s_toff,
                                              int* s_ntok, unsigned char* stage,
                                              int stage_bytes, unsigned bar, int* s_fail,
                                              T* __restrict__ out) {
    constexpr int LG = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;  // log2 G
    constexpr int HS = 5 - LG;  // lane l holds the score of head l >> HS
    constexpr int ROWB = kD * (int)sizeof(T);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = v.P;
    const int hl = lane >> HS;
    // token offsets of the selected pages (warp 0), counts read in parallel
    if (warp == 0) {
        int carry = 0;
        for (int r0 = 0; r0 < npg; r0 += 32) {
            const int r = r0 + lane;
            int c = 0;
            if (r < npg) {
                const int pg = s_sel[r];
                if (hcnt != nullptr) {  // the count copied into the page table with the page
                    unsigned hh = ((unsigned)pg * 2654435761u) & (unsigned)(hcap - 1);
                    for (int probe = 0; probe < hcap; ++probe) {
                        const int hp = hpage[hh];
                        if (hp == pg) {
                            c = hcnt[hh];
                            break;
                        }
                        if (hp == -1) break;
                        hh = (hh + 1) & (unsigned)(hcap - 1);
                    }
                } else if (pg >= 0 && pg < v.C) {
                    c = v.list_cnt[v.leaf_base(u, 0) + pg];
                }
                c = c < 0 ? 0 : (c > P ? P : c);
            }
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (r < npg) s_toff[r] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            s_toff[npg] = carry;
            *s_ntok = carry;
        }
    }
    float qa[G][4];
    {
        const float sc = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            if (s_q != nullptr) {  // the query rows kept in shared memory since the start
#pragma unroll
                for (int k = 0; k < 4; ++k) qa[hh][k] = s_q[hh * kD + 4 * lane + k] * sc;
            } else {
                float x[4];
                load4(q + ((long long)u * G + hh) * kD + 4 * lane, x);
#pragma unroll
                for (int k = 0; k < 4; ++k) qa[hh][k] = x[k] * sc;
            }
        }
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
    while (p0 < npg) {  // every thread computes the same rounds
        int p1 = p0 + 1;
        while (p1 < npg && s_toff[p1 + 1] - s_toff[p0] <= rows_cap) ++p1;
        const int t0 = s_toff[p0], nrow = s_toff[p1] - t0;
        if (warp == 0) {
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                // ICE_DEBUG_STALL_ATTN: expect 16 bytes that no copy delivers, so the
                // bounded wait below runs out (tests of the timeout path)
                const unsigned extra = (v.debug & ICE_DEBUG_STALL_ATTN) ? 16u : 0u;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                             "r"((unsigned)(2 * nrow * ROWB) + extra)
                             : "memory");
            }
            __syncwarp();
            for (int r = p0 + lane; r < p1; r += 32) {
                const int c = s_toff[r + 1] - s_toff[r];
                if (c > 0) {
                    const long long row0 = v.page_row(u, s_sel[r], 0);
                    const unsigned off = (unsigned)(s_toff[r] - t0) * ROWB;
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
            // any thread whose wait ran out marks the block; the copies may still
            // be in flight, so wait for them once more (bounded) before leaving
            *s_fail = 1;
            set_status(v.status, ICE_ERR_TIMEOUT);
            mbar_wait_bounded(bar, (unsigned)(round & 1));
        }
        if (ok) {
            for (int j = warp; j < nrow; j += kSelWarps) {  // warp-uniform
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
                const float p = exp2_approx(sc - mn);
                float vx[4];
                load4(sv + (size_t)j * kD + 4 * lane, vx);
                if (__any_sync(0xffffffffu, mn != m)) {  // a head's maximum rose: rescale
                    const float corr = exp2_approx(m - mn);
                    lsum = lsum * corr + p;
                    m = mn;
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
                } else {  // every maximum held: the correction is 2^0 = 1
                    lsum += p;
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float ph = __shfl_sync(0xffffffffu, p, hh << HS);
                        const float2 p2 = make_float2(ph, ph);
#pragma unroll
                        for (int k = 0; k < 4; k += 2) {
                            const float2 a2 = __ffma2_rn(p2, make_float2(vx[k], vx[k + 1]),
                                                         make_float2(acc[hh][k], acc[hh][k + 1]));
                            acc[hh][k] = a2.x;
                            acc[hh][k + 1] = a2.y;
                        }
                    }
                }
            }
        }
        __syncthreads();  // the round's rows are consumed before the next copies land
        // after a timeout the barrier's phase may never complete: issue no further
        // expect_tx or copies on it (block-uniform: s_fail is read after the barrier)
        if (*s_fail) break;
        p0 = p1;
        ++round;
    }
    // partials into the (now free) staging region: rows [warp][head] of PR floats, the
    // accumulator, then m and the sum. Rows of 16-byte multiples take one 16-byte store per
    // lane and head, where scalar stores 16 bytes apart would conflict four ways in the banks
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
    // the warps' weights 2^(m_w - M) per head and the head's softmax sum, once: warp hh,
    // lane w holds warp w's (max, sum) of head hh
    float* cfs = part + kSelWarps * G * PR;  // [G][kSelWarps] weights, then [G] sums
    if (warp < G) {
        const int hh = warp;
        const float mw = lane < kSelWarps ? part[(lane * G + hh) * PR + kD] : -INFINITY;
        float M = mw;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float cf = (M == -INFINITY || mw == -INFINITY) ? 0.0f : exp2_approx(mw - M);
        float Lt = lane < kSelWarps ? part[(lane * G + hh) * PR + kD + 1] * cf : 0.0f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) Lt += __shfl_xor_sync(0xffffffffu, Lt, o);
        if (lane < kSelWarps) cfs[hh * kSelWarps + lane] = cf;
        if (lane == 0) cfs[G * kSelWarps + hh] = *s_fail ? 0.0f : Lt;
    }
    __syncthreads();
    T* ou = out + (long long)u * G * kD;
    for (int e = tid; e < G * kD; e += kSelThreads) {
        const int hh = e / kD, dcol = e % kD;
        const float Lt = cfs[G * kSelWarps + hh];
        float O = 0.0f;
        if (Lt > 0.0f) {
#pragma unroll
            for (int w = 0; w < kSelWarps; ++w)
                O = fmaf(part[(w * G + hh) * PR + dcol], cfs[hh * kSelWarps + w], O);
        }
        ou[e] = from_f<T>(Lt > 0.0f ? O / Lt : 0.0f);
    }
}

// The decode step's insert, kept out of line so that the select path's code and
// register allocation stay those of the plain fused call.
template <typename T>
__device__ __noinline__ void insert_unit_call(const IndexView& v, int u, const T* kin, const T* vin,
                                              unsigned char* rows) {
    insert_unit<T, kSelThreads>(v, u, kin, vin, rows);
}

// More than kTopK pages to select: a block-wide bitonic sort of the compacted
// (key, page) pairs, the first n_sel in order. Out of line (rarely taken), so that
// the selection's own code path stays contiguous.
__device__ __noinline__ void block_sort_select(unsigned long long* skey, int* sval, int npg, int n_sel,
                                               int taken, int32_t* out, int* s_sel) {
    const int tid = threadIdx.x;
    int npow = 1;
    while (npow < npg) npow <<= 1;
    for (int c = npg + tid; c < npow; c += kSelThreads) {
        skey[c] = ~0ull;
        sval[c] = -1;
    }
    __syncthreads();
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
    for (int r = tid; r < n_sel; r += kSelThreads) {
        const int pg = r < taken ? sval[r] : -1;
        out[r] = pg;
        s_sel[r] = pg;
    }
}

// INSERT: the one-launch decode step, whose blocks insert their unit's token first.
// KEEP: selection reuse, where a unit may keep its pages and only attend. Both are
// separate instantiations: the out-of-line insert call in the kernel slowed the plain
// fused selection, which never takes it, by 1.3 us on the 32-layer step.
template <typename T, int G, bool FUSED, bool INSERT = false, bool KEEP = false>
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(
    IndexView v, const T* __restrict__ q, int n_sel, int n_cand, int sort_cap, int hcap,
    int smem_total, int32_t* __restrict__ page_ids, int32_t* __restrict__ n_pages_out,
    int32_t* __restrict__ stats, T* __restrict__ attn_out, const int32_t* __restrict__ reselect,
    int head_div, const T* __restrict__ knew, const T* __restrict__ vnew) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(16) float2 s_qp[kD / 2];  // (q_sel[e], q_sel[e + 64]), e < 64
    __shared__ __align__(16) float s_qt[kD];        // q~, the normalised q_sel
    __shared__ int s_qcode[kMaxL][kM];
    __shared__ __align__(16) __half2 s_width[97 * 4];
    __shared__ int s_pstar[kMaxL], s_need[kMaxL], s_nch[kMaxL], s_tot[kMaxL];
    __shared__ int s_ncand, s_nraw, s_npg, s_ntok, s_fail, s_cmp;
    __shared__ __align__(8) unsigned long long s_bar;

    pdl_wait_then_release();
    // head_div > 1: per-query-head selection, block = (unit, head), row = block
    const int u = blockIdx.x / head_div, row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = v.L, P = v.P;
    const int pshift = (P & (P - 1)) == 0 ? __ffs(P) - 1 : -1;  // page of a slot by a shift
    const long long C = v.C;
    const int Cp = align16((int)C);
    const SelSmem lay = sel_layout(C, L, n_cand, sort_cap, hcap, n_sel, 0);
    int* s_sel = reinterpret_cast<int*>(smem + lay.sel);              // [n_sel] selected pages
    int* s_toff = reinterpret_cast<int*>(smem + lay.toff);            // [n_sel + 1] token offsets
    unsigned char* prio = smem + lay.prio;                            // [L][Cp]
    unsigned char* cnts = smem + lay.cnt;                             // [L][Cp]
    int* hist = reinterpret_cast<int*>(smem + lay.hist);              // [L][kSubH][kHistRow]
    int* chosen = reinterpret_cast<int*>(smem + lay.chosen);          // [L][n_cand] leaf index
    unsigned* cmeta = reinterpret_cast<unsigned*>(smem + lay.cmeta);  // [L][n_cand] id|count
    int* coff = reinterpret_cast<int*>(smem + lay.coff);              // [L][n_cand + 1]
    unsigned* tieb = reinterpret_cast<unsigned*>(smem + lay.tieb);    // [L][nwords] leaves at pi*
    unsigned* bm0 = reinterpret_cast<unsigned*>(smem + lay.bm0);
    unsigned long long* skey = reinterpret_cast<unsigned long long*>(smem + lay.keys);
    int* sval = reinterpret_cast<int*>(smem + lay.vals);
    int* hpage = reinterpret_cast<int*>(smem + lay.hpage);
    int* hcnt = reinterpret_cast<int*>(smem + lay.hcnt);
    unsigned long long* hkey = reinterpret_cast<unsigned long long*>(smem + lay.hkey);
    unsigned long long* topk = reinterpret_cast<unsigned long long*>(smem + lay.top);
    int* topv = reinterpret_cast<int*>(smem + lay.top + kSelWarps * kTopK * 8);
    const int nwords = (int)((C + 31) / 32);
    const uint4* recs = v.leaf_rec;

    // the fused decode step: this block first inserts its unit's new token
    if constexpr (FUSED && INSERT) {
        if (knew != nullptr) {  // block-uniform
            insert_unit_call<T>(v, u, knew + (long long)u * kD, vnew + (long long)u * kD,
                                smem + lay.free);
            // the new rows reach the bulk copies of the attention (async proxy)
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncthreads();
        }
    }

    // the unit keeps the pages it selected before (reuse across steps): no
    // selection, and the fused call attends over the pages in page_ids
    if (KEEP && reselect != nullptr && reselect[u] == 0) {  // block-uniform
        if (FUSED) {
            const int taken = min(max(n_pages_out[u], 0), n_sel);
            for (int i = tid; i < taken; i += kSelThreads) s_sel[i] = page_ids[(long long)u * n_sel + i];
            if (tid == 0) {
                s_fail = 0;
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar)) : "memory");
                asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            }
            __syncthreads();
            attend_staged<T, G>(v, u, q, nullptr, nullptr, nullptr, 0, taken, s_sel, s_toff, &s_ntok,
                                smem + lay.keys, smem_total - lay.keys, smem_u32(&s_bar), &s_fail,
                                attn_out);
        }
        return;
    }

    // ---- 1. leaf counts, query heads and directions requested together -------------------
    int N[kMaxL] = {0, 0};
    for (int l = 0; l < L; ++l) N[l] = v.n_leaf[v.ul(u, l)];
    float qh[G][4];  // warp 0 only
    const T* qu = q + (long long)row * G * kD;
    if (warp == 0)
#pragma unroll
        for (int h = 0; h < G; ++h) load4(qu + (long long)h * kD + 4 * lane, qh[h]);
    float wdir[4] = {0.f, 0.f, 0.f, 0.f};
    float wlast = 0.f;
    if (warp < L * kM) {
        const float* ud = v.dirs + (long long)warp * kDirStride;
        load4(ud + 4 * lane, wdir);
        wlast = ud[kD];
    }
    // The scan streams the leaves' 10-byte scan copies through a per-warp ring of
    // cp.async copies: warp w reads composite sl = w / wpc, chunks of 64 leaves
    // wg, wg + wpc, ...; lane t copies (and later reads) leaves 2t and 2t+1 of a
    // chunk, so each lane consumes only its own copies and no barrier is needed.
    // The first kRing chunks are requested now, before the leaf count arrives
    // (chunks past the count are copied but never read; the capacity, a multiple
    // of 64, bounds the reads).
    const int wpc = kSelWarps / L;
    const int sl = warp / wpc, wg = warp % wpc;
    const unsigned long long* slo = v.leaf_lo + v.leaf_base(u, sl);
    const unsigned short* stc = v.leaf_tc + v.leaf_base(u, sl);
    const unsigned ring = smem_u32(smem + lay.ring + warp * (kRing * kSlotB));
    auto ring_issue = [&](int k, int slot) {
        const unsigned d = ring + slot * kSlotB;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + lane * 16),
                     "l"(slo + 64 * k + 2 * lane)
                     : "memory");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d + 512 + lane * 4),
                     "l"(stc + 64 * k + 2 * lane)
                     : "memory");
    };
#pragma unroll
    for (int sidx = 0; sidx < kRing; ++sidx) {
        const int k = wg + sidx * wpc;
        if (64LL * k < C) ring_issue(k, sidx);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    // tables and counters that need nothing from memory, while the loads are in flight
    if (tid < 97) {
        __half2 w[4];
        cell_widths(tid, w);
#pragma unroll
        for (int k = 0; k < 4; ++k) s_width[tid * 4 + k] = w[k];
    }
    for (int i = tid; i < L * kSubH * kHistRow; i += kSelThreads) hist[i] = 0;
    for (int i = tid; i < nwords; i += kSelThreads) bm0[i] = 0u;
    for (int i = tid; i < L * nwords; i += kSelThreads) tieb[i] = 0u;
    if (tid < kMaxL) {
        s_nch[tid] = 0;
        s_tot[tid] = 0;
    }
    if (tid == 0) {
        s_ncand = 0;
        s_nraw = 0;
        s_npg = 0;
        s_fail = 0;
        if (FUSED) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    for (int l = 0; l < L; ++l) N[l] = N[l] < 0 ? 0 : (N[l] > C ? (int)C : N[l]);
    const int Ntot = N[0] + N[1];

    // query prep: q_sel = the heads' sum in head order and q~ = q_sel / |q_sel| once
    // (warp 0, into shared memory), then the codes (warp j: direction j)
    {
        if (warp == 0) {
            float qs[4] = {qh[0][0], qh[0][1], qh[0][2], qh[0][3]};
#pragma unroll
            for (int h = 1; h < G; ++h)
#pragma unroll
                for (int k = 0; k < 4; ++k) qs[k] = __fadd_rn(qs[k], qh[h][k]);
            const float nq = warp_dot_fixed(qs, qs);
            float qt[4] = {0.f, 0.f, 0.f, 0.f};
            if (nq > 0.0f) {
                const float sn = __fsqrt_rn(nq);
#pragma unroll
                for (int k = 0; k < 4; ++k) qt[k] = __fdiv_rn(qs[k], sn);
            }
            *reinterpret_cast<float4*>(s_qt + 4 * lane) = make_float4(qt[0], qt[1], qt[2], qt[3]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = 4 * lane + k;
                if (e < kD / 2) s_qp[e].x = qs[k];
                else s_qp[e - kD / 2].y = qs[k];
            }
            if (FUSED) {  // the query rows, for the attention tail
                float* qf = reinterpret_cast<float*>(smem + lay.qf);
#pragma unroll
                for (int hh = 0; hh < G; ++hh)
#pragma unroll
                    for (int k = 0; k < 4; ++k) qf[hh * kD + 4 * lane + k] = qh[hh][k];
            }
        }
        __syncthreads();
        if (warp < L * kM) {
            const float4 t4 = *reinterpret_cast<const float4*>(s_qt + 4 * lane);
            const float qt[4] = {t4.x, t4.y, t4.z, t4.w};
            const float p = __fmaf_rn(wlast, 0.0f, warp_dot_fixed(wdir, qt));
            if (lane == 0) s_qcode[warp / kM][warp % kM] = quantise_code(p);
        }
    }
    __syncthreads();

    // ---- 2. priorities, counts and sub-histograms of token counts --------------------
    {
        __half2 qc[4];
        {
            unsigned lo4 = 0, hi4 = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo4 |= (unsigned)s_qcode[sl][j] << (8 * j);
                hi4 |= (unsigned)s_qcode[sl][4 + j] << (8 * j);
            }
            qc[0] = bytes_to_h2(lo4, 0x4140u);
            qc[1] = bytes_to_h2(lo4, 0x4342u);
            qc[2] = bytes_to_h2(hi4, 0x4140u);
            qc[3] = bytes_to_h2(hi4, 0x4342u);
        }
        // neighbouring leaves share few priorities (a handful per 32 leaves):
        // lanes t, t+8, t+16, t+24 share a sub-histogram, so at most four lanes of
        // an instruction add to one counter, and the 257-word row stride puts
        // equal priorities of different sub-histograms in different banks
        const int Nl = N[sl];
        int* hl = hist + (sl * kSubH + (lane & (kSubH - 1))) * kHistRow;
        const unsigned pr_base = smem_u32(prio + sl * Cp);
        const unsigned cn_base = smem_u32(cnts + sl * Cp);
        int slot = 0;
        for (int k = wg; 64 * k < Nl; k += wpc) {  // warp-uniform
            asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
            const unsigned d = ring + slot * kSlotB;
            uint4 lo2;
            unsigned tc2;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(lo2.x), "=r"(lo2.y), "=r"(lo2.z), "=r"(lo2.w)
                         : "r"(d + lane * 16)
                         : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tc2) : "r"(d + 512 + lane * 4) : "memory");
            const int i0 = 64 * k + 2 * lane;
            const unsigned tca = tc2 & 0xFFFFu, tcb = tc2 >> 16;
            const int p0 = leaf_priority(lo2.x, lo2.y, tc_t(tca), qc, s_width);
            const int p1 = leaf_priority(lo2.z, lo2.w, tc_t(tcb), qc, s_width);
            const int c0 = tc_cnt(tca), c1 = tc_cnt(tcb);
            if (i0 < Nl) {
                st_shared_u16(pr_base + i0, p0 | (p1 << 8));
                st_shared_u16(cn_base + i0, c0 | (c1 << 8));
                atomicAdd(&hl[p0], c0);
                if (i0 + 1 < Nl) atomicAdd(&hl[p1], c1);
            }
            // the slot's values are in registers: refill it with the chunk kRing ahead
            const int kn = k + kRing * wpc;
            if (64 * kn < Nl) ring_issue(kn, slot);
            asm volatile("cp.async.commit_group;" ::: "memory");
            slot = slot + 1 == kRing ? 0 : slot + 1;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
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
            for (int s = 0; s < kSubH; ++s) x += hist[(l * kSubH + s) * kHistRow + lane * 8 + k];
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

    // ---- 3b. leaves below pi* are taken; leaves at pi* are marked in a bitmap ------------
    // (the page table takes over the scan ring's memory)
    for (int i = tid; i < hcap; i += kSelThreads) {
        hpage[i] = -1;
        hkey[i] = ~0ull;
    }
#pragma unroll
    for (int l = 0; l < kMaxL; ++l) {
        if (l >= L) break;
        const int ps = s_pstar[l];
        const unsigned* p32 = reinterpret_cast<const unsigned*>(prio + l * Cp);
        const uint4* lrec = recs + v.leaf_base(u, l);
        const int nw = (N[l] + 3) >> 2;
        // a word with no priority <= ps holds nothing to take or mark: for ps < 128 the
        // test is the borrow of a bytewise subtraction of ps + 1 (a byte below ps + 1
        // borrows into its top bit, which its own value does not set)
        const unsigned lim = 0x01010101u * (unsigned)(ps + 1);
        for (int w4 = tid; w4 < nw; w4 += kSelThreads) {
            const unsigned word = p32[w4];
            if (ps < 128 && ((word - lim) & ~word & 0x80808080u) == 0u) continue;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = 4 * w4 + b;
                if (i >= N[l]) break;
                const int pr = (int)((word >> (8 * b)) & 0xFFu);
                if (pr < ps) {
                    const int slot = atomicAdd(&s_nch[l], 1);
                    if (slot < n_cand) {
                        chosen[l * n_cand + slot] = i;
                        // the leaf's id | count, copied while the ties are walked
                        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                                         smem_u32(cmeta + l * n_cand + slot)),
                                     "l"(&lrec[i].z)
                                     : "memory");
                    }
                } else if (pr == ps) {
                    atomicOr(&tieb[l * nwords + (i >> 5)], 1u << (i & 31));
                }
            }
        }
    }
    __syncthreads();
    // ---- 3c. leaves at pi*, in position order, while tokens taken before them < need ------
    // Warp l walks composite l's tie bitmap 32 words (1024 leaves) at a time, in
    // position order: each lane sums the tokens of its word's ties, a warp scan
    // gives every lane the tokens taken before it, and the lane takes its ties
    // while that running count is below the need. The same warp then computes the
    // slot offsets of all taken leaves (3d) from the count bytes of the scan, while
    // the taken leaves' records (list ids) are still being copied.
    if (warp < L) {
        const int l = warp;
        const int need = s_need[l];
        const unsigned* tb = tieb + l * nwords;
        const unsigned char* cl = cnts + l * Cp;
        const uint4* lrec = recs + v.leaf_base(u, l);
        const int nbelow = min(s_nch[l], n_cand);
        int run = 0, ntaken = 0;  // tie tokens and tie leaves taken so far (warp-uniform)
        for (int w0 = 0; w0 < nwords && run < need; w0 += 32) {
            const int wi = w0 + lane;
            const unsigned bits = wi < nwords ? tb[wi] : 0u;
            // the count bytes of the word's 32 leaves, in registers
            uint4 ca = make_uint4(0u, 0u, 0u, 0u), cb = ca;
            if (bits) {
                ca = *reinterpret_cast<const uint4*>(cl + wi * 32);
                cb = *reinterpret_cast<const uint4*>(cl + wi * 32 + 16);
            }
            const unsigned cw[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
            unsigned tsum = 0u;  // tokens of the word's ties: count bytes under the tie mask
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
            int acc = run + inc - tot, mine = 0;
            unsigned take = 0u;
            if (acc + tot <= need) {  // every tie of the word is taken (counts are >= 1)
                take = bits;
                mine = __popc(bits);
            } else {  // the word where the need is reached (or none is taken)
                for (unsigned b = bits; b && acc < need; b &= b - 1u) {
                    const int bit = __ffs(b) - 1;
                    take |= 1u << bit;
                    acc += (int)((byte_word(cw, bit >> 2) >> (8 * (bit & 3))) & 0xFFu);
                    ++mine;
                }
            }
            int tinc = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, tinc, o);
                if (lane >= o) tinc += y;
            }
            int slot = nbelow + ntaken + tinc - mine;
            for (unsigned b = take; b; b &= b - 1u, ++slot)
                if (slot < n_cand) {
                    const int i = wi * 32 + __ffs(b) - 1;
                    chosen[l * n_cand + slot] = i;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                                     smem_u32(cmeta + l * n_cand + slot)),
                                 "l"(&lrec[i].z)
                                 : "memory");
                }
            ntaken += __shfl_sync(0xffffffffu, tinc, 31);
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        __syncwarp();
        // ---- 3d. slot offsets of the taken leaves (counts from the scan's bytes) -----------
        const int nch = min(nbelow + ntaken, n_cand);
        int carry = 0;
        for (int k0 = 0; k0 < nch; k0 += 32) {
            const int k = k0 + lane;
            const int c = k < nch ? (int)cl[chosen[l * n_cand + k]] : 0;
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
            s_nch[l] = nbelow + ntaken;
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // the taken leaves' records
    __syncthreads();
    {  // composite-0 pages already taken whole
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
                    // plain loads: a fused decode step has just written these lists.
                    // A composite-1 slot carries its token's page row, requested
                    // together with the token.
                    tok = v.slot_tok[v.slot_base(u, l) + (long long)id * P + slot];
                    if (l == 0) {
                        loc = id * P + slot;
                        keep = true;
                    } else {
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
                if (pos < sort_cap) {
                    skey[pos] = (unsigned long long)(unsigned)tok;
                    sval[pos] = loc;
                }
            }
        }
    }
    __syncthreads();
    const int ncand = min(s_ncand, sort_cap);

    // ---- 5. exact rescoring, one candidate row per thread; per-page minimum key ------------
    // Candidate rows are staged in the free region with cp.async, in chunks that
    // alternate between two halves of it: the next chunk is in flight while the
    // current one is scored. Consecutive lanes request consecutive 16-byte pieces
    // of a row (coalesced); piece c of row r is stored at piece position
    // c ^ 2 (r mod pieces-per-row/2), so that the pieces the threads of one
    // shared-memory wavefront read (four rows, two threads per row) fall in
    // distinct banks. The fixed-order dot of a row is split over two threads:
    // virtual lane l accumulates elements 4l..4l+3, and the pairwise tree adds
    // lanes l and l+16 first, then l+8, l+4, l+2, l+1.
    {
        constexpr int EPC = 16 / (int)sizeof(T);  // elements per piece
        constexpr int CPR = kD / EPC;             // pieces per row
        constexpr int ROWB = kD * (int)sizeof(T);
        const int pad = pad_to_128(smem + lay.free);  // 0 when the window starts aligned
        unsigned char* stg = smem + lay.free + pad;
        const int half = min((smem_total - lay.free - pad) / (2 * ROWB), kSelThreads / 2);  // rows per half (two threads a row)
        const int nchunk = (ncand + half - 1) / half;
        const char* pk = reinterpret_cast<const char*>(v.page_k) + (long long)u * C * P * ROWB;
        const int hmask = hcap - 1;
        // thread tid copies piece c = tid mod CPR of rows tid / CPR, + RSTEP, ...: the
        // swizzled position of the piece is the same in all of them (the swizzle
        // repeats every CPR / 2 rows), so only the row's source address changes per copy
        constexpr int RSTEP = kSelThreads / CPR;
        static_assert(RSTEP % (CPR / 2) == 0, "the swizzle must repeat every RSTEP rows");
        const int cpc = tid % CPR, r_first = tid / CPR;
        const int cpos = cpc ^ ((r_first & (CPR / 2 - 1)) << 1);
        auto issue = [&](int ch) {  // chunk ch into half ch & 1; every thread commits a group
            if (ch < nchunk) {
                const int rb = ch * half, nr = min(half, ncand - rb);
                unsigned dst = smem_u32(stg + (ch & 1) * half * ROWB + r_first * ROWB + 16 * cpos);
                const char* src = pk + 16 * cpc;
                for (int r = r_first; r < nr; r += RSTEP, dst += RSTEP * ROWB)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                                 "l"(src + (long long)sval[rb + r] * ROWB)
                                 : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        issue(0);
        issue(1);
        for (int ch = 0; ch < nchunk; ++ch) {  // block-uniform
            const int rb0 = ch * half, nr = min(half, ncand - rb0);
            const unsigned char* stgc = stg + (ch & 1) * half * ROWB;
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // chunk ch has landed
            __syncthreads();
            if (16 * warp < nr) {  // warp-uniform: warp w holds rows 16w .. 16w + 15
                // two threads per row: thread t of the pair owns the virtual lanes l with
                // bit 1 of l equal to t, so the tree's levels 16, 8 and 4 stay inside
                // the thread and level 2 is one exchange with the partner
                const int r = tid >> 1, t = tid & 1;
                const bool ok = r < nr;
                const int sw = (r & (CPR / 2 - 1)) << 1;
                int pg = -1;
                unsigned long long key = ~0ull;
                float s4[2] = {0.0f, 0.0f};
                if (ok) {
                    const unsigned char* rowp = stgc + r * ROWB;
                    float s16[8];  // s16 of the owned lanes l < 16, in increasing order
    #pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int l = ((j >> 1) << 2) | (t << 1) | (j & 1);  // 4(j/2) + 2t + (j mod 2)
                        const int e0 = 4 * l, e1 = 4 * (l + 16);
                        const int c0 = e0 / EPC, c1 = e1 / EPC;  // pieces holding the two groups
                        float x0[EPC], x1[EPC];
                        load_chunk<T>(rowp + 16 * (c0 ^ sw), x0);
                        load_chunk<T>(rowp + 16 * (c1 ^ sw), x1);
                        const int o0 = e0 % EPC, o1 = e1 % EPC;
                        // the partials of lanes l and l + 16 (elements e0 + i and
                        // e1 + i = e0 + 64 + i) as the two halves of a packed pair
                        float2 ab = make_float2(0.0f, 0.0f);
    #pragma unroll
                        for (int i = 0; i < 4; ++i)
                            ab = __ffma2_rn(s_qp[e0 + i], make_float2(x0[o0 + i], x1[o1 + i]), ab);
                        s16[j] = __fadd_rn(ab.x, ab.y);
                    }
                    // level 8: l + 8 is owned entry j + 4; level 4: l + 4 is entry j + 2
    #pragma unroll
                    for (int j = 0; j < 4; ++j) s16[j] = __fadd_rn(s16[j], s16[j + 4]);
                    s4[0] = __fadd_rn(s16[0], s16[2]);  // lane 2t
                    s4[1] = __fadd_rn(s16[1], s16[3]);  // lane 2t + 1
                }
                {
                    const float p0 = __shfl_xor_sync(0xffffffffu, s4[0], 1);
                    const float p1 = __shfl_xor_sync(0xffffffffu, s4[1], 1);
                    // level 2: lane 0 + lane 2, lane 1 + lane 3; level 1: their sum
                    const float a0 = t ? p0 : s4[0], a2 = t ? s4[0] : p0;
                    const float a1 = t ? p1 : s4[1], a3 = t ? s4[1] : p1;
                    const float sc = __fadd_rn(__fadd_rn(a0, a2), __fadd_rn(a1, a3));
                    if (ok) {
                        pg = pshift >= 0 ? sval[rb0 + r] >> pshift : sval[rb0 + r] / P;
                        key = ((unsigned long long)score_key_desc(sc) << 32) | (unsigned)skey[rb0 + r];
                    }
                }
                // rows of one page are adjacent in the candidate list: a segmented
                // minimum over runs of equal pages (rows two lanes apart) leaves each
                // run's minimum in its last row, which alone updates the table
    #pragma unroll
                for (int o = 2; o < 32; o <<= 1) {
                    const int opg = __shfl_up_sync(0xffffffffu, pg, o);
                    const unsigned long long okey = __shfl_up_sync(0xffffffffu, key, o);
                    if (lane >= o && opg == pg && okey < key) key = okey;
                }
                const int next_pg = __shfl_down_sync(0xffffffffu, pg, 2);
                bool fresh = false;
                if (ok && t == 0 && (lane >= 30 || next_pg != pg)) {
                    unsigned h = ((unsigned)pg * 2654435761u) & (unsigned)hmask;
                    for (int probe = 0; probe < hcap; ++probe) {
                        const int old = atomicCAS(&hpage[h], -1, pg);
                        if (old == -1 || old == pg) {
                            fresh = old == -1;
                            if (FUSED && fresh)  // the page's token count, for the attention tail
                                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                                                 smem_u32(hcnt + h)),
                                             "l"(v.list_cnt + v.leaf_base(u, 0) + pg)
                                             : "memory");
                            atomicMin(&hkey[h], key);
                            break;
                        }
                        h = (h + 1) & (unsigned)hmask;
                    }
                }
                {
                    const unsigned nf = __ballot_sync(0xffffffffu, fresh);
                    if (lane == 0 && nf) atomicAdd(&s_npg, __popc(nf));
                }
            }
            __syncthreads();  // the chunk's rows are read before the next chunk lands there
            issue(ch + 2);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncthreads();
    const int npg = s_npg;  // distinct pages among the candidates
    const int taken = min(n_sel, npg);
    int32_t* out = page_ids + (long long)row * n_sel;

    // ---- 6. the n_sel smallest page keys in order ------------------------------------------
    // compact the occupied hash slots into (key, page) pairs
    if (tid == 0) s_cmp = 0;
    __syncthreads();
    for (int h0 = warp * 32; h0 < hcap; h0 += kSelThreads) {  // warp-uniform
        const int h = h0 + lane;
        const int pg = h < hcap ? hpage[h] : -1;
        const unsigned km = __ballot_sync(0xffffffffu, pg >= 0);
        int base = 0;
        if (lane == 0 && km) base = atomicAdd(&s_cmp, __popc(km));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (pg >= 0) {
            const int pos = base + __popc(km & ((1u << lane) - 1u));
            skey[pos] = hkey[h];
            sval[pos] = pg;
        }
    }
    __syncthreads();
    if (n_sel <= kTopK) {
        const int nb = (npg + 31) / 32;  // batches of 32 entries
        unsigned long long tk = ~0ull;
        int tv = -1;
        for (int bt = warp; bt < nb; bt += kSelWarps) {  // warp-uniform
            const int j = bt * 32 + lane;
            unsigned long long k = j < npg ? skey[j] : ~0ull;
            int vv = j < npg ? sval[j] : -1;
            warp_sort32(k, vv, lane);
            warp_merge32(tk, tv, k, vv, lane);
        }
        const int nw = min(kSelWarps, max(nb, 1));  // warps holding a list
        if (warp < nw) {
            topk[warp * kTopK + lane] = tk;
            topv[warp * kTopK + lane] = tv;
        }
        __syncthreads();
        // pairwise merge tree over the warps' lists: warp w takes in w + st
        for (int st = 1; st < nw; st <<= 1) {
            if ((warp & (2 * st - 1)) == 0 && warp + st < nw) {
                unsigned long long a = topk[warp * kTopK + lane];
                int av = topv[warp * kTopK + lane];
                warp_merge32(a, av, topk[(warp + st) * kTopK + lane],
                             topv[(warp + st) * kTopK + lane], lane);
                topk[warp * kTopK + lane] = a;
                topv[warp * kTopK + lane] = av;
            }
            __syncthreads();
        }
        if (warp == 0 && lane < n_sel) {
            const int pg = lane < taken ? topv[lane] : -1;
            out[lane] = pg;
            s_sel[lane] = pg;
        }
    } else {
        block_sort_select(skey, sval, npg, n_sel, taken, out, s_sel);
    }
    __syncthreads();
    if (tid == 0) n_pages_out[row] = taken;
    if (stats && warp == 0) {
        int tok_sel = 0;
        for (int r = lane; r < taken; r += 32) tok_sel += v.list_cnt[v.leaf_base(u, 0) + s_sel[r]];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) tok_sel += __shfl_xor_sync(0xffffffffu, tok_sel, o);
        if (lane == 0) {
            stats[4 * row + 0] = Ntot;
            stats[4 * row + 1] = ncand;
            stats[4 * row + 2] = tok_sel;
            stats[4 * row + 3] = s_nraw;
        }
    }
    if (tid == 0 && ncand < s_ncand) set_status(v.status, ICE_ERR_CAPACITY);
    if constexpr (FUSED)
        attend_staged<T, G>(v, u, q, reinterpret_cast<const float*>(smem + lay.qf), hpage, hcnt,
                            hcap, taken, s_sel, s_toff, &s_ntok, smem + lay.keys,
                            smem_total - lay.keys, smem_u32(&s_bar), &s_fail, attn_out);
}

// Sparse attention over a given page list ("IceCache", Figure 2 step 3), for a
// page pool in device memory: the fused kernel's attention tail on its own. One
// 512-thread block per unit stages the pages' K and V rows with one bulk copy
// per page and row kind, so a round of pages costs one memory latency. A page id
// that is negative, not allocated or past the list capacity marks the status
// ICE_ERR_BOUNDS and contributes nothing, as does a list length outside
// [0, page_stride].
constexpr int kAttnStagedSmem = 104 * 1024;  // two blocks per SM with the static arrays
constexpr int kAttnMaxPages = 512;
static_assert(kAttnMaxPages <= kSelThreads, "one list slot per thread");
static_assert(kAttnStagedSmem - 128 >= 2 * kMaxP * kD * 4, "a page's f32 K and V rows fit one round");
static_assert(kAttnStagedSmem - 128 >= kSelWarps * 4 * (kD + 4) * 4 + 4 * (kSelWarps + 1) * 4,
              "the partials of four heads fit the staging region");

template <typename T, int G>
__global__ void __launch_bounds__(kSelThreads, 2) attn_staged_kernel(
    IndexView v, const T* __restrict__ q, const int32_t* __restrict__ page_ids,
    const int32_t* __restrict__ n_pages, int page_stride, T* __restrict__ out) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_sel[kAttnMaxPages];
    __shared__ int s_toff[kAttnMaxPages + 1];
    __shared__ int s_ntok, s_fail;
    __shared__ __align__(8) unsigned long long s_bar;
    pdl_wait_then_release();
    const int u = blockIdx.x, tid = threadIdx.x;
    // the list length, the allocated page count and every slot of the list's row are read
    // together (page_stride <= kSelThreads): one memory latency
    int np = n_pages[u];
    const int nalloc = v.next_id[v.ul(u, 0)];
    int pid = tid < page_stride ? page_ids[(long long)u * page_stride + tid] : -1;
    if (np < 0 || np > page_stride) {
        if (tid == 0) set_status(v.status, ICE_ERR_BOUNDS);
        np = np < 0 ? 0 : page_stride;
    }
    if (tid < np) {
        if (pid < 0 || pid >= nalloc || pid >= v.C) {
            set_status(v.status, ICE_ERR_BOUNDS);
            pid = -1;  // no rows
        }
        s_sel[tid] = pid;
    }
    if (tid == 0) {
        s_fail = 0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int pad = pad_to_128(smem);
    attend_staged<T, G>(v, u, q, nullptr, nullptr, nullptr, 0, np, s_sel, s_toff, &s_ntok, smem + pad,
                        kAttnStagedSmem - pad, smem_u32(&s_bar), &s_fail, out);
}

template <typename T>
static cudaError_t launch_attn_staged_dt(const IndexView& v, const void* q, const int32_t* page_ids,
                                         const int32_t* n_pages, int page_stride, void* out,
                                         cudaStream_t s) {
    const T* qq = (const T*)q;
    T* oo = (T*)out;
    const size_t b = kAttnStagedSmem;
    switch (v.G) {
        case 1: return launch_pdl(attn_staged_kernel<T, 1>, dim3(v.U), dim3(kSelThreads), b, s, v, qq, page_ids, n_pages, page_stride, oo);
        case 2: return launch_pdl(attn_staged_kernel<T, 2>, dim3(v.U), dim3(kSelThreads), b, s, v, qq, page_ids, n_pages, page_stride, oo);
        case 4: return launch_pdl(attn_staged_kernel<T, 4>, dim3(v.U), dim3(kSelThreads), b, s, v, qq, page_ids, n_pages, page_stride, oo);
        // eight heads hold 64 registers of query and output per lane, the whole bound of
        // two 512-thread blocks per SM: the plain-load kernel, without that bound
        case 8: return launch_attn(v, q, page_ids, n_pages, page_stride, out, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn_staged(const IndexView& v, const void* q, const int32_t* page_ids,
                               const int32_t* n_pages, int page_stride, void* out, cudaStream_t s) {
    if (page_stride < 1 || page_stride > kAttnMaxPages) return cudaErrorInvalidValue;
    if (v.dtype == ICE_BF16)
        return launch_attn_staged_dt<__nv_bfloat16>(v, q, page_ids, n_pages, page_stride, out, s);
    return launch_attn_staged_dt<float>(v, q, page_ids, n_pages, page_stride, out, s);
}

static void select_caps(int L, int P, int n_cand, int* sort_cap, int* hcap) {
    const int cand_cap = L * (n_cand + P - 1);
    int c = 1;
    while (c < cand_cap) c <<= 1;
    *sort_cap = c;
    *hcap = c;  // at least one slot per candidate: probing always ends
}

// Dynamic shared memory of a launch (fused blocks are padded up to kFusedSmem so
// that the page staging region is as large as two blocks per SM allow).
// Whether the fused kernel's free region holds the rows a decode-step insert
// stages for a split (2 (P + 1) rows of es bytes per element).
bool select_insert_fits(long long C, int L, int P, int n_cand, int n_sel, int es) {
    int sc, hc;
    select_caps(L, P, n_cand, &sc, &hc);
    const SelSmem lay = sel_layout(C, L, n_cand, sc, hc, n_sel, kFusedSmem);
    return (long long)2 * (P + 1) * kD * es <= (long long)(lay.end - lay.free);
}

int select_smem_bytes(long long C, int L, int P, int n_cand, int n_sel, int G, bool fused) {
    (void)G;
    int sc, hc;
    select_caps(L, P, n_cand, &sc, &hc);
    (void)fused;
    return sel_layout(C, L, n_cand, sc, hc, n_sel, kFusedSmem).end;
}

template <typename T, int G>
static cudaError_t launch_select_g(const IndexView& v, const void* q, int n_sel, int n_cand,
                                   int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                                   const int32_t* reselect, const void* knew, const void* vnew,
                                   cudaStream_t s) {
    int sort_cap, hcap;
    select_caps(v.L, v.P, n_cand, &sort_cap, &hcap);
    const bool fused = out != nullptr;
    const int bytes = select_smem_bytes(v.C, v.L, v.P, n_cand, n_sel, G, fused);
    if (fused && knew != nullptr)
        return launch_pdl(select_kernel<T, G, true, true>, dim3(v.U), dim3(kSelThreads), (size_t)bytes, s,
                          v, (const T*)q, n_sel, n_cand, sort_cap, hcap, bytes, page_ids, n_pages, stats,
                          (T*)out, reselect, 1, (const T*)knew, (const T*)vnew);
    if (reselect != nullptr) {
        if (fused)
            return launch_pdl(select_kernel<T, G, true, false, true>, dim3(v.U), dim3(kSelThreads),
                              (size_t)bytes, s, v, (const T*)q, n_sel, n_cand, sort_cap, hcap, bytes,
                              page_ids, n_pages, stats, (T*)out, reselect, 1, (const T*)nullptr,
                              (const T*)nullptr);
        return launch_pdl(select_kernel<T, G, false, false, true>, dim3(v.U), dim3(kSelThreads),
                          (size_t)bytes, s, v, (const T*)q, n_sel, n_cand, sort_cap, hcap, bytes, page_ids,
                          n_pages, stats, (T*)nullptr, reselect, 1, (const T*)nullptr, (const T*)nullptr);
    }
    if (fused)
        return launch_pdl(select_kernel<T, G, true>, dim3(v.U), dim3(kSelThreads), (size_t)bytes, s, v,
                          (const T*)q, n_sel, n_cand, sort_cap, hcap, bytes, page_ids, n_pages, stats,
                          (T*)out, reselect, 1, (const T*)knew, (const T*)vnew);
    return launch_pdl(select_kernel<T, G, false>, dim3(v.U), dim3(kSelThreads), (size_t)bytes, s, v,
                      (const T*)q, n_sel, n_cand, sort_cap, hcap, bytes, page_ids, n_pages, stats,
                      (T*)nullptr, reselect, 1, (const T*)nullptr, (const T*)nullptr);
}

template <typename T>
static cudaError_t launch_select_dt(const IndexView& v, const void* q, int n_sel, int n_cand,
                                    int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                                    const int32_t* reselect, const void* knew, const void* vnew,
                                    cudaStream_t s) {
    switch (v.G) {
        case 1: return launch_select_g<T, 1>(v, q, n_sel, n_cand, page_ids, n_pages, stats, out, reselect, knew, vnew, s);
        case 2: return launch_select_g<T, 2>(v, q, n_sel, n_cand, page_ids, n_pages, stats, out, reselect, knew, vnew, s);
        case 4: return launch_select_g<T, 4>(v, q, n_sel, n_cand, page_ids, n_pages, stats, out, reselect, knew, vnew, s);
        case 8: return launch_select_g<T, 8>(v, q, n_sel, n_cand, page_ids, n_pages, stats, out, reselect, knew, vnew, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_select(const IndexView& v, const void* q, int n_sel, int n_cand,
                          int32_t* page_ids, int32_t* n_pages, int32_t* stats, void* out,
                          const int32_t* reselect, cudaStream_t s, const void* knew,
                          const void* vnew) {
    if (reselect == nullptr && knew == nullptr) {
        // plain select (+ attention): a cluster of blocks per unit when the launch
        // has few units, or when one block cannot hold the unit's tables
        const bool one_fits = select_smem_bytes(v.C, v.L, v.P, n_cand, n_sel, v.G, out != nullptr) <=
                              kSelSmemMax;
        int K = v.cluster_k > 0 ? v.cluster_k : select_cluster_auto(v.U, v.L);
        if (K == 1 && !one_fits) K = v.L > 2 ? v.L : 2;
        if (K >= 2) {
            bool launched = false;
            const cudaError_t e = launch_select_cluster(v, K, q, n_sel, n_cand, page_ids, n_pages,
                                                        stats, out, s, &launched);
            if (e != cudaSuccess || launched) return e;
            if (v.cluster_k > 0 || !one_fits) return cudaErrorInvalidConfiguration;
        }
    }
    if (v.dtype == ICE_BF16)
        return launch_select_dt<__nv_bfloat16>(v, q, n_sel, n_cand, page_ids, n_pages, stats, out,
                                               reselect, knew, vnew, s);
    return launch_select_dt<float>(v, q, n_sel, n_cand, page_ids, n_pages, stats, out, reselect,
                                   knew, vnew, s);
}

// Per-query-head selection: every (unit, query head) selects with that head's query
// alone (q_sel = q_h), through the single-head instantiations: a cluster of blocks per
// row when the rows are few, else one block per row.
cudaError_t launch_select_heads(const IndexView& v, const void* q, int n_sel, int n_cand,
                                int32_t* page_ids, int32_t* n_pages, cudaStream_t s) {
    {  // few rows: a cluster of blocks per (unit, head)
        bool launched = false;
        const cudaError_t e = launch_select_heads_cluster(v, q, n_sel, n_cand, page_ids, n_pages, s,
                                                          &launched);
        if (e != cudaSuccess || launched) return e;
    }
    int sort_cap, hcap;
    select_caps(v.L, v.P, n_cand, &sort_cap, &hcap);
    const int bytes = select_smem_bytes(v.C, v.L, v.P, n_cand, n_sel, 1, false);
    if (v.dtype == ICE_BF16)
        select_kernel<__nv_bfloat16, 1, false><<<v.U * v.G, kSelThreads, bytes, s>>>(
            v, (const __nv_bfloat16*)q, n_sel, n_cand, sort_cap, hcap, bytes, page_ids, n_pages,
            nullptr, nullptr, nullptr, v.G, nullptr, nullptr);
    else
        select_kernel<float, 1, false><<<v.U * v.G, kSelThreads, bytes, s>>>(
            v, (const float*)q, n_sel, n_cand, sort_cap, hcap, bytes, page_ids, n_pages, nullptr,
            nullptr, nullptr, v.G, nullptr, nullptr);
    return cudaGetLastError();
}

// Raise the dynamic shared memory limit of the select kernels once per device.
cudaError_t select_prepare() {
    const int lim = kSelSmemMax;
    cudaError_t e = cudaSuccess;
#define ICE_SET_SMEM(T, G)                                                                        \
    if (e == cudaSuccess)                                                                         \
        e = cudaFuncSetAttribute(select_kernel<T, G, false>,                                      \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);               \
    if (e == cudaSuccess)                                                                         \
        e = cudaFuncSetAttribute(select_kernel<T, G, true>,                                       \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);               \
    if (e == cudaSuccess)                                                                         \
        e = cudaFuncSetAttribute(select_kernel<T, G, true, true>,                                 \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);               \
    if (e == cudaSuccess)                                                                         \
        e = cudaFuncSetAttribute(select_kernel<T, G, true, false, true>,                          \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);               \
    if (e == cudaSuccess)                                                                         \
        e = cudaFuncSetAttribute(select_kernel<T, G, false, false, true>,                         \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);               \
    if (e == cudaSuccess && G < 8)                                                                \
        e = cudaFuncSetAttribute(attn_staged_kernel<T, (G < 8 ? G : 4)>,                          \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnStagedSmem);
    ICE_SET_SMEM(__nv_bfloat16, 1) ICE_SET_SMEM(__nv_bfloat16, 2) ICE_SET_SMEM(__nv_bfloat16, 4)
    ICE_SET_SMEM(__nv_bfloat16, 8) ICE_SET_SMEM(float, 1) ICE_SET_SMEM(float, 2)
    ICE_SET_SMEM(float, 4) ICE_SET_SMEM(float, 8)
#undef ICE_SET_SMEM
    return e;
}

}  // namespace ice

// Dynamic insertion of one generated token into one unit, by a block of NT
// threads ("IceCache" abstract: a hierarchical, dynamically updatable
// structure; the blog: no rebuild when a new token appears). Used by the
// insert kernel (one 128-thread block per unit) and by the fused decode step
// (the select kernel's block inserts its unit's token before it selects).
//
// The trie over 96-bit keys is history independent: a node is a leaf iff its
// parent holds more than P keys. Adding key x therefore changes only the leaf
// on x's path:
//  * x carries the prefix of an existing leaf holding < P tokens: append;
//  * that leaf holds P tokens: its P+1 keys share exactly lambda = lcp(min, max)
//    bits, so it splits into the two children at bit lambda (left keeps the
//    page id, right takes the next free id);
//  * x carries no leaf prefix: x opens a new leaf one bit below its longest
//    common prefix with any existing key (its neighbours in key order).
// Composites are handled one after the other.
#pragma once
#include "ice_internal.cuh"

namespace ice {

// Token tok now sits in composite-1 slot s1 (list id * P + slot): record the
// slot and copy the token's page row (composite 0 is updated first) into it.
__device__ __forceinline__ void place_loc1(const IndexView& v, int u, int tok, int s1) {
    v.tok_slot1[(long long)u * v.max_tokens + tok] = s1;
    v.slot_loc1[v.loc1_base(u) + s1] = v.tok_loc[(long long)u * v.max_tokens + tok];
}

// Shift leaf keys, records and the records' scan copies [from, N) one place to
// the right, backwards, in rounds of 1024 elements (1024 / NT per thread of the
// NT-thread block): all loads of a round are in flight together, then the
// stores (the next round reads only indices below the ones this round wrote).
template <int NT>
__device__ void shift_right(LeafKey* key, uint4* rec, unsigned long long* lo, unsigned short* tc,
                            int from, int N) {
    constexpr int kShiftUnr = NT >= 1024 ? 1 : 1024 / NT;
    for (int end = N; end > from; end -= NT * kShiftUnr) {
        const int start = max(from, end - NT * kShiftUnr);
        LeafKey k[kShiftUnr];
        uint4 r[kShiftUnr];
        unsigned long long a[kShiftUnr];
        unsigned short c[kShiftUnr];
#pragma unroll
        for (int j = 0; j < kShiftUnr; ++j) {
            const int i = start + (int)threadIdx.x + j * NT;
            if (i < end) {
                k[j] = key[i];
                r[j] = rec[i];
                a[j] = lo[i];
                c[j] = tc[i];
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kShiftUnr; ++j) {
            const int i = start + (int)threadIdx.x + j * NT;
            if (i < end) {
                key[i + 1] = k[j];
                rec[i + 1] = r[j];
                lo[i + 1] = a[j];
                tc[i + 1] = c[j];
            }
        }
        __syncthreads();
    }
}

// The new token of unit u: key kin, value vin (device rows of kD elements);
// rows: shared memory for 2 (P + 1) rows of T (the staged K and V of a split).
// Every thread of the block calls it; the token index is the unit's count.
template <typename T, int NT>
__device__ void insert_unit(const IndexView& v, int u, const T* __restrict__ kin,
                            const T* __restrict__ vin, unsigned char* rows) {
    constexpr int ROW = kD;  // elements per row
    T* rows_k = reinterpret_cast<T*>(rows);                      // [P+1][D]
    T* rows_v = rows_k + (size_t)(v.P + 1) * ROW;                // [P+1][D]
    __shared__ unsigned long long s_mk[kMaxL];
    __shared__ unsigned long long e_m[kMaxP + 1];
    __shared__ unsigned int e_t[kMaxP + 1];
    __shared__ int e_slot[kMaxP + 1];  // original slot (P = the new token)
    __shared__ int s_sorted[kMaxP + 1];
    __shared__ int s_ts1[kMaxP + 1];  // composite-1 slots of a splitting leaf's tokens
    __shared__ int s_cnt, s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = v.P;
    // Every request that depends on nothing else goes out first, together: the token
    // count, the leaf counts and next list ids, the new token's rows, its key for the
    // projections, the unit's exponent and the directions of this warp's projections
    // (the L * kM direction dots are spread over the warps; each warp forms the scaled
    // key itself, in the same fixed order). The addresses are valid whatever the count.
    static_assert(NT >= kD, "one element of the new rows per thread");
    constexpr int NW = NT / 32;
    constexpr int kPerWarp = (kMaxL * kM + NW - 1) / NW;
    // the new token's index is the unit's count, kept on the device (so that a
    // captured CUDA graph of inserts advances it on every replay)
    const int tok = v.n_tok[u];
    const int Lc = v.L;
    int n_l = 0, nid_l = 0;
    if (tid < Lc) {
        n_l = v.n_leaf[v.ul(u, tid)];
        nid_l = v.next_id[v.ul(u, tid)];
    }
    T kin_i{}, vin_i{};
    if (tid < kD) {
        kin_i = kin[tid];
        vin_i = vin[tid];
    }
    float k4[4];
    load4(kin + 4 * lane, k4);
    const int e = v.e_unit[u];
    float w[kPerWarp][4], wl[kPerWarp];  // this warp's directions
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int dj = warp + i * NW;
        if (dj < v.L * kM) {
            const float* ud = v.dirs + (long long)dj * kDirStride;
            load4(ud + 4 * lane, w[i]);
            wl[i] = ud[kD];
        }
    }
    if (tok < 0 || tok >= v.max_tokens) {  // block-uniform
        if (tid == 0) set_status(v.status, ICE_ERR_CAPACITY);
        return;
    }

    // the new token's K and V rows, staged as row P of the split's staging: the append,
    // the split and the new leaf copy them from there, with no memory latency of their own
    if (tid < kD) {
        rows_k[(size_t)P * kD + tid] = kin_i;
        rows_v[(size_t)P * kD + tid] = vin_i;
    }

    // ---- the search for the new key's leaf runs for all composites at once: thread
    //      group l (NT / L threads) searches composite l. The first probes are requested
    //      while the warps form the new key's codes.
    __shared__ int s_N[kMaxL], s_nid[kMaxL], s_lo2[kMaxL], s_hi2[kMaxL], s_a[kMaxL], s_fin[kMaxL];
    __shared__ LeafKey s_pk[kMaxL];
    __shared__ uint4 s_pr[kMaxL];
    if (tid < Lc) {
        s_N[tid] = n_l;
        s_nid[tid] = nid_l;
        s_lo2[tid] = 0;
        s_a[tid] = -1;
        s_fin[tid] = 0;
        s_pr[tid] = make_uint4(0u, 0u, 0u, 0u);
        s_pk[tid] = LeafKey{0ull, 0u, 0u};
    }
    if (tid == 0) s_abort = 0;
    __syncthreads();
    if (tid < Lc) s_hi2[tid] = s_N[tid];
    const int gsz = NT / Lc, gl = tid / gsz, gi = tid - gl * gsz;
    const bool in_group = gl < Lc;
    // probe of this thread in the current round: leaf key and record (the record of
    // the last probe at or below the key is the leaf's, without another round trip)
    auto probe = [&](int lo, int hi, int& i, LeafKey& k, uint4& r) {
        const int span = hi - lo;
        const int step = span <= gsz ? 1 : (span + gsz - 1) / gsz;
        i = lo + gi * step;
        if (in_group && i < hi) {
            const long long lb = v.leaf_base(u, gl);
            k = v.leaf_key[lb + i];
            r = v.leaf_rec[lb + i];
        }
        return step;
    };
    int pi = 0, pstep = 0;
    LeafKey pk{0ull, 0u, 0u};
    uint4 pr = make_uint4(0u, 0u, 0u, 0u);
    if (in_group) pstep = probe(0, s_N[gl], pi, pk, pr);

    // ---- key of the new token: frozen scale, projections, codes; one thread per
    //      composite interleaves the codes ------------------------------------------------
    {
        __shared__ int s_code[kMaxL * kM];
        const float nrm2 = warp_dot_fixed(k4, k4);
        const float sc = ldexpf(1.0f, -e), sc2 = ldexpf(1.0f, -2 * e);
        float kt[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) kt[i] = __fmul_rn(k4[i], sc);
        float r = __fsub_rn(1.0f, __fmul_rn(nrm2, sc2));
        r = r > 0.0f ? r : 0.0f;
        const float tail = __fsqrt_rn(r);
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            const int dj = warp + i * NW;
            if (dj < v.L * kM) {  // warp-uniform
                const float p = __fmaf_rn(wl[i], tail, warp_dot_fixed(w[i], kt));
                if (lane == 0) s_code[dj] = quantise_code(p);
            }
        }
        __syncthreads();
        if (tid < v.L) {
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = s_code[tid * kM + j];
            s_mk[tid] = morton8(c);
        }
    }
    __syncthreads();
    // k-ary rounds: a = number of leaves whose prefix <= x, per composite
    __shared__ int s_cntp[kMaxL];
    for (int round = 0; round < 64; ++round) {  // block-uniform; ends when every composite is done
        if (tid < Lc) s_cntp[tid] = 0;
        __syncthreads();
        bool le = false;
        if (in_group && !s_fin[gl] && pi < s_hi2[gl])
            le = !key_less(s_mk[gl], (unsigned)tok, pk.pm, pk.pt);
        if (le) atomicAdd(&s_cntp[gl], 1);
        __syncthreads();
        if (in_group && !s_fin[gl]) {
            const int c = s_cntp[gl];
            const int lo = s_lo2[gl], hi = s_hi2[gl];
            // the last probe at or below the key publishes its leaf (keys are sorted)
            if (c > 0 && gi == c - 1) {
                s_pk[gl] = pk;
                s_pr[gl] = pr;
            }
            if (pstep == 1) {  // every leaf of [lo, hi) was probed: done
                if (gi == 0) {
                    s_a[gl] = lo + c;
                    s_fin[gl] = 1;
                }
            } else if (c == 0) {
                if (gi == 0) {
                    s_a[gl] = lo;
                    s_fin[gl] = 1;
                }
            } else if (gi == 0) {
                const int pc = lo + (c - 1) * pstep;
                s_lo2[gl] = pc + 1;
                s_hi2[gl] = min(hi, pc + pstep);
            }
        }
        __syncthreads();
        bool all = true;
        for (int l = 0; l < Lc; ++l) all = all && s_fin[l];
        if (all) break;
        if (in_group && !s_fin[gl]) pstep = probe(s_lo2[gl], s_hi2[gl], pi, pk, pr);
    }

    for (int l = 0; l < v.L; ++l) {
        const unsigned long long xm = s_mk[l];
        const unsigned int xt = (unsigned)tok;
        LeafKey* lk = v.leaf_key + v.leaf_base(u, l);
        const long long lb0 = v.leaf_base(u, l);
        uint4* lr = v.leaf_rec + lb0;
        unsigned long long* llo = v.leaf_lo + lb0;
        unsigned short* ltc = v.leaf_tc + lb0;
        int* cntl = v.list_cnt + v.leaf_base(u, l);
        int* stok = v.slot_tok + v.slot_base(u, l);
        unsigned long long* skey = v.slot_key + v.slot_base(u, l);
        const int N = s_N[l];
        const int nid = s_nid[l];
        const int pos = s_a[l] - 1;  // last leaf with prefix <= x, or -1
        bool member = false;
        uint4 rc = make_uint4(0u, 0u, 0u, 0u);
        if (pos >= 0) {
            const LeafKey k = s_pk[l];
            unsigned long long pm;
            unsigned int pt;
            prefix96(xm, xt, (int)k.t, pm, pt);
            member = pm == k.pm && pt == k.pt;
            rc = s_pr[l];
        }
        const int id = rec_id(rc), cnt = rec_cnt(rc);
        const bool split = member && cnt >= P;
        __syncthreads();  // every thread has read the leaf before any thread updates it
        // capacity: a split or a new leaf needs one more leaf record and list id
        if (!(member && !split) && (N + 1 > v.C || nid + 1 > v.C)) {
            if (tid == 0) set_status(v.status, ICE_ERR_CAPACITY);
            __syncthreads();
            break;
        }

        if (member && !split) {
            // ---- append to the leaf ---------------------------------------------------
            if (tid == 0) {
                const long long sb = (long long)id * P + cnt;
                stok[sb] = tok;
                skey[sb] = xm;
                cntl[id] = cnt + 1;
                uint4 r2 = rc;
                r2.z = ((unsigned)id << 8) | (unsigned)(cnt + 1);
                put_leaf(v, lb0 + pos, r2);
                if (l == 0) v.tok_loc[(long long)u * v.max_tokens + tok] = id * P + cnt;
                if (l == 1) place_loc1(v, u, tok, (int)sb);
            }
            if (l == 0) {
                T* pk = reinterpret_cast<T*>(v.page_k) + v.page_row(u, id, cnt) * kD;
                T* pv = reinterpret_cast<T*>(v.page_v) + v.page_row(u, id, cnt) * kD;
                for (int i = tid; i < kD; i += NT) {
                    pk[i] = rows_k[(size_t)P * kD + i];
                    pv[i] = rows_v[(size_t)P * kD + i];
                }
            }
            __syncthreads();
            continue;
        }

        if (split) {
            // ---- split the full leaf in two ---------------------------------------------
            for (int j = tid; j <= P; j += NT) {
                if (j < P) {
                    e_m[j] = skey[(long long)id * P + j];
                    e_t[j] = (unsigned)stok[(long long)id * P + j];
                } else {
                    e_m[j] = xm;
                    e_t[j] = xt;
                }
                e_slot[j] = j;
            }
            if (l == 0) {  // stage the P old rows, K and V (row P holds the new token's)
                const T* pk = reinterpret_cast<const T*>(v.page_k) + v.page_row(u, id, 0) * kD;
                const T* pv = reinterpret_cast<const T*>(v.page_v) + v.page_row(u, id, 0) * kD;
                for (int i = tid; i < P * kD; i += NT) {
                    const int r = i / kD, c = i % kD;
                    rows_k[i] = pk[(long long)r * kD + c];
                    rows_v[i] = pv[(long long)r * kD + c];
                }
            }
            __syncthreads();
            // rank of each key among the P+1 (keys are distinct); meanwhile the upper half of
            // the block requests the composite-1 slots of the leaf's tokens, which follow
            // them to their new rows below (stored to shared memory in the next step)
            for (int j = tid; j <= P; j += NT) {
                int r = 0;
                for (int k = 0; k <= P; ++k) r += key_less(e_m[k], e_t[k], e_m[j], e_t[j]);
                s_sorted[r] = j;
            }
            const bool fetch_s1 = l == 0 && v.tok_slot1 != nullptr && tid >= NT / 2;
            int ts1[(kMaxP + 1 + NT / 2 - 1) / (NT / 2)];
            if (fetch_s1) {
#pragma unroll
                for (int q2 = 0; q2 < (kMaxP + 1 + NT / 2 - 1) / (NT / 2); ++q2) {
                    const int j = tid - NT / 2 + q2 * (NT / 2);
                    ts1[q2] = j <= P ? v.tok_slot1[(long long)u * v.max_tokens + e_t[j]] : -1;
                }
            }
            __syncthreads();
            const int f = s_sorted[0], g = s_sorted[P];
            const int lam = lcp96(e_m[f], e_t[f], e_m[g], e_t[g]);
            if (tid == 0) {
                int nl = 0;
                for (int r = 0; r <= P; ++r) nl += key_bit96(e_m[s_sorted[r]], e_t[s_sorted[r]], lam) == 0;
                s_cnt = nl;
            }
            if (fetch_s1) {
#pragma unroll
                for (int q2 = 0; q2 < (kMaxP + 1 + NT / 2 - 1) / (NT / 2); ++q2) {
                    const int j = tid - NT / 2 + q2 * (NT / 2);
                    if (j <= P) s_ts1[j] = ts1[q2];
                }
            }
            __syncthreads();
            const int nl = s_cnt, nr = P + 1 - nl;
            const int rid = nid;  // right child takes the next free id
            for (int r = tid; r <= P; r += NT) {
                const int j = s_sorted[r];
                const int dst = r < nl ? id : rid;
                const int slot = r < nl ? r : r - nl;
                stok[(long long)dst * P + slot] = (int)e_t[j];
                skey[(long long)dst * P + slot] = e_m[j];
                if (l == 0) {
                    v.tok_loc[(long long)u * v.max_tokens + e_t[j]] = dst * P + slot;
                    // the token's composite-1 slot follows it to its new row
                    if (v.tok_slot1 != nullptr) {
                        const int s1 = s_ts1[j];
                        if (s1 >= 0) v.slot_loc1[v.loc1_base(u) + s1] = dst * P + slot;
                    }
                }
                if (l == 1) place_loc1(v, u, (int)e_t[j], dst * P + slot);
            }
            if (l == 0) {
                for (int i = tid; i < (P + 1) * kD; i += NT) {
                    const int r = i / kD, c = i % kD;
                    const int j = s_sorted[r];
                    const int dst = r < nl ? id : rid;
                    const int slot = r < nl ? r : r - nl;
                    const long long o = v.page_row(u, dst, slot) * kD + c;
                    reinterpret_cast<T*>(v.page_k)[o] = rows_k[(long long)j * kD + c];
                    reinterpret_cast<T*>(v.page_v)[o] = rows_v[(long long)j * kD + c];
                }
            }
            __syncthreads();
            shift_right<NT>(lk, lr, llo, ltc, pos + 1, N);
            if (tid == 0) {
                cntl[id] = nl;
                cntl[rid] = nr;
                const int t = lam + 1;
                LeafKey kl, kr;
                prefix96(e_m[f], e_t[f], t, kl.pm, kl.pt);
                prefix96(e_m[g], e_t[g], t, kr.pm, kr.pt);
                kl.t = kr.t = (unsigned)t;
                lk[pos] = kl;
                put_leaf(v, lb0 + pos, make_leaf_rec(kl.pm, (unsigned)t, id, nl));
                lk[pos + 1] = kr;
                put_leaf(v, lb0 + pos + 1, make_leaf_rec(kr.pm, (unsigned)t, rid, nr));
                v.n_leaf[v.ul(u, l)] = N + 1;
                v.next_id[v.ul(u, l)] = nid + 1;
            }
            __syncthreads();
            continue;
        }

        // ---- x lies where no leaf exists: a new leaf below its longest common
        //      prefix with the neighbouring keys -------------------------------------------
        {
            int best = -1;
            // predecessor leaf `pos` and successor leaf `pos + 1`: all their keys
            for (int side = 0; side < 2; ++side) {
                const int li = pos + side;
                if (li < 0 || li >= N) continue;
                const uint4 r2 = lr[li];
                const int id2 = rec_id(r2), c2 = rec_cnt(r2);
                int bl = -1;
                if (tid < c2) {
                    const unsigned long long km = skey[(long long)id2 * P + tid];
                    const unsigned int kt = (unsigned)stok[(long long)id2 * P + tid];
                    bl = lcp96(xm, xt, km, kt);
                }
                for (int o = 16; o >= 1; o >>= 1) bl = max(bl, __shfl_xor_sync(0xffffffffu, bl, o));
                best = max(best, bl);
            }
            // combine the warps (P <= 64 keys live in warps 0 and 1)
            __shared__ int s_best[NT / 32];
            if (lane == 0) s_best[warp] = best;
            __syncthreads();
            if (tid == 0) {
                int b = -1;
                for (int w = 0; w < NT / 32; ++w) b = max(b, s_best[w]);
                s_cnt = b + 1;  // depth of the new leaf
            }
            __syncthreads();
            const int t = s_cnt;
            const int nidl = nid;
            if (l == 0) {
                T* pk = reinterpret_cast<T*>(v.page_k) + v.page_row(u, nidl, 0) * kD;
                T* pv = reinterpret_cast<T*>(v.page_v) + v.page_row(u, nidl, 0) * kD;
                for (int i = tid; i < kD; i += NT) {
                    pk[i] = rows_k[(size_t)P * kD + i];
                    pv[i] = rows_v[(size_t)P * kD + i];
                }
            }
            shift_right<NT>(lk, lr, llo, ltc, pos + 1, N);
            if (tid == 0) {
                stok[(long long)nidl * P] = tok;
                skey[(long long)nidl * P] = xm;
                cntl[nidl] = 1;
                if (l == 0) v.tok_loc[(long long)u * v.max_tokens + tok] = nidl * P;
                if (l == 1) place_loc1(v, u, tok, nidl * P);
                LeafKey k;
                prefix96(xm, xt, t, k.pm, k.pt);
                k.t = (unsigned)t;
                lk[pos + 1] = k;
                put_leaf(v, lb0 + pos + 1, make_leaf_rec(k.pm, (unsigned)t, nidl, 1));
                v.n_leaf[v.ul(u, l)] = N + 1;
                v.next_id[v.ul(u, l)] = nid + 1;
            }
            __syncthreads();
        }
    }
    if (tid == 0) v.n_tok[u] = tok + 1;  // every thread read the count at the start
}

}  // namespace ice

// IceCache decode-time path: CPU ORACLE (test infrastructure only).
//
// A plain, slow, single-threaded statement of what the GPU library computes,
// written from the IceCache paper ("IceCache", arXiv 2604.10539) and its blog
// post: the DCI-tree page index built at prefill (Figure 2 step 1, Figure 3),
// dynamic insertion of generated tokens without a rebuild (the abstract's
// hierarchical structure that is updated in place), the P-DCI prioritised
// query that finds the pages
// holding the query's top keys (Figure 2 steps 2-3), and sparse GQA attention
// over every token of the selected pages (Figure 2 step 3).
//
// Only tests, the smoke check and the benchmark's CPU-baseline leg use this
// file. It shares no code, header or table with the CUDA library. Build it
// with -O2 -ffp-contract=off so that every float operation written here is the
// one that runs (no fused multiply-add except where std::fma is spelled out).
//
// Readings where the paper and the blog are silent (each one is listed with its
// reason in the design notes of the repository):
//  * transformed key space: keys are scaled by 2^-e, c = 2^e the smallest power
//    of two with c^2 >= max ||k||^2 (frozen at build), and augmented with
//    sqrt(1 - ||k||^2 / c^2), so that the nearest neighbour of the normalised
//    query is the key with the largest inner product (the IceFormer lineage);
//  * DCI projections: L composite indices of m Rademacher directions +-1/16 in
//    R^{d+1}, drawn from splitmix64(seed);
//  * the DCI-tree: a binary trie over the 96-bit key (Morton interleave of the
//    m 8-bit projection codes, then the token index) that splits a node while it
//    holds more than page_size tokens; each non-empty leaf of composite 0 is one
//    physical page;
//  * the prioritised search: leaves in increasing (L-infinity cell distance in
//    code units, left-to-right position) order until n_cand tokens are taken,
//    which is the order a best-first tree search pops them in (both are
//    implemented here and compared);
//  * page selection: candidates of all composites are rescored with a
//    fixed-order fp32 dot, ranked by (score desc, token asc), and the pages of
//    the ranked tokens are taken in first-occurrence order up to budget/page.
//
// Parity pins live in tests/test_oracle_*.py; see the header of each test.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <queue>
#include <set>
#include <vector>

namespace {

constexpr int kCodeBits = 8;  // B: bits per projection code

// ---------------------------------------------------------------------------
// Fixed-order fp32 dot product D(a, b).
// Lane l of 32 owns elements [l*w, (l+1)*w), w = d/32, and accumulates them in
// increasing order with fused multiply-adds from 0; the 32 lane sums are then
// added pairwise, lane l with lane l+o for o = 16, 8, 4, 2, 1.
// ---------------------------------------------------------------------------
float dot_fixed(const float* a, const float* b, int d) {
    const int w = d / 32;
    float acc[32];
    for (int l = 0; l < 32; ++l) {
        float s = 0.0f;
        for (int i = 0; i < w; ++i) s = std::fma(a[l * w + i], b[l * w + i], s);
        acc[l] = s;
    }
    for (int o = 16; o >= 1; o >>= 1)
        for (int l = 0; l < o; ++l) acc[l] = acc[l] + acc[l + o];
    return acc[0];
}

// splitmix64 (Steele, Lea & Flood 2014): add the golden-ratio increment, then
// two xor-shift-multiply rounds and a final xor-shift.
uint64_t splitmix64_next(uint64_t& state) {
    state += 0x9E3779B97F4A7C15ULL;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

int ceil_half(int a) { return a >= 0 ? (a + 1) / 2 : -((-a) / 2); }

// Smallest e with (2^e)^2 >= maxn, kept within [-60, 64] so that 2^-e and
// 2^-2e stay finite floats. maxn == 0 gives e = 0.
int scale_exponent(float maxn) {
    if (!(maxn > 0.0f)) return 0;
    int x = 0;
    float f = std::frexp(maxn, &x);  // maxn = f * 2^x, f in [0.5, 1)
    int e = (f == 0.5f) ? ceil_half(x - 1) : ceil_half(x);
    if (e < -60) e = -60;
    return e;
}

// code = clamp(floor((p + 1) * 2^(B-1)), 0, 2^B - 1), all in fp32.
int quantise(float p) {
    float y = (p + 1.0f) * 128.0f;
    float f = std::floor(y);
    if (f < 0.0f) return 0;
    if (f > 255.0f) return 255;
    return (int)f;
}

// 96-bit key: Morton interleave of the codes (bits above), token index below.
struct Key {
    uint64_t hi;
    uint32_t lo;
    bool operator<(const Key& o) const { return hi != o.hi ? hi < o.hi : lo < o.lo; }
    bool operator==(const Key& o) const { return hi == o.hi && lo == o.lo; }
};

// Bit t (0 = most significant) of the 96-bit key.
int key_bit(const Key& k, int t) {
    if (t < 64) return (int)((k.hi >> (63 - t)) & 1ULL);
    return (int)((k.lo >> (95 - t)) & 1U);
}

// Key with all bits from position t on cleared.
Key key_prefix(const Key& k, int t) {
    Key p{0, 0};
    if (t >= 64) {
        p.hi = k.hi;
        int tb = t - 64;  // token bits kept
        p.lo = tb == 0 ? 0u : (tb >= 32 ? k.lo : (k.lo & ~((1u << (32 - tb)) - 1u)));
    } else {
        p.hi = t == 0 ? 0ULL : (k.hi & ~((1ULL << (64 - t)) - 1ULL));
        p.lo = 0;
    }
    return p;
}

// Morton interleave of m codes, most significant bit first: for bit b from 7
// down to 0, for direction j from 0 to m-1, bit b of code j. Left-aligned.
uint64_t morton(const int* codes, int m) {
    uint64_t out = 0;
    int pos = 0;
    for (int b = kCodeBits - 1; b >= 0; --b)
        for (int j = 0; j < m; ++j) {
            uint64_t bit = (uint64_t)((codes[j] >> b) & 1);
            out |= bit << (63 - pos);
            ++pos;
        }
    return out;
}

struct Leaf {
    int t;                  // prefix length in bits (0..96)
    Key prefix;             // key bits [0, t), zero below
    int id;                 // page id (composite 0) or list id (composite > 0)
    std::vector<int> toks;  // token indices in this leaf
};

struct Composite {
    std::vector<Leaf> leaves;  // left-to-right (ascending prefix)
    int next_id = 0;
    std::vector<Key> keys;     // per token
    std::vector<int> codes;    // per token, m codes
};

struct Index {
    int d, m, L, P;
    uint64_t seed;
    int e = 0;
    std::vector<float> dirs;  // [L][m][d+1]
    int n = 0;
    std::vector<float> K, V;  // [n][d], values as given (bf16 widened or f32)
    std::vector<Composite> comp;
};

// Number of known bits of direction j in a prefix of length t.
int known_bits(int t, int j, int m) {
    if (t >= m * kCodeBits) return kCodeBits;
    int b = (t - j + m - 1) / m;
    if (b < 0) b = 0;
    if (b > kCodeBits) b = kCodeBits;
    return b;
}

// Cell of a prefix: for each direction the code interval [lo, hi] the prefix
// allows. The known bits of code j are read back from the prefix bits.
void prefix_cell(const Key& prefix, int t, int m, int* lo, int* hi) {
    for (int j = 0; j < m; ++j) {
        int bj = known_bits(t, j, m);
        int v = 0;
        for (int b = kCodeBits - 1; b >= kCodeBits - bj; --b) {
            int pos = (kCodeBits - 1 - b) * m + j;  // position from the MSB
            v |= key_bit(prefix, pos) << b;
        }
        lo[j] = v;
        hi[j] = v | ((1 << (kCodeBits - bj)) - 1);
    }
}

// L-infinity distance in code units between a query code vector and a cell.
int cell_distance(const int* qc, const int* lo, const int* hi, int m) {
    int best = 0;
    for (int j = 0; j < m; ++j) {
        int dj = 0;
        if (qc[j] < lo[j]) dj = lo[j] - qc[j];
        else if (qc[j] > hi[j]) dj = qc[j] - hi[j];
        best = std::max(best, dj);
    }
    return best;
}

// Recursive partition of a node: tokens `toks` (sorted by key) all share the
// first t bits. A node holding at most P tokens is a leaf (kept only when it
// holds at least one); a larger node splits by bit t into its 0- and 1-child.
void split_node(const std::vector<Key>& keys, std::vector<int> toks, int t, int P,
                std::vector<Leaf>& out) {
    if ((int)toks.size() <= P) {
        if (!toks.empty()) {
            Leaf lf;
            lf.t = t;
            lf.prefix = key_prefix(keys[toks[0]], t);
            lf.id = -1;
            lf.toks = std::move(toks);
            out.push_back(std::move(lf));
        }
        return;
    }
    std::vector<int> left, right;
    for (int tk : toks) (key_bit(keys[tk], t) ? right : left).push_back(tk);
    split_node(keys, std::move(left), t + 1, P, out);
    split_node(keys, std::move(right), t + 1, P, out);
}

// Transform one key (given its squared norm) and project it on the directions
// of composite l; write the m codes.
void key_codes(const Index& ix, int l, const float* k, float nrm2, int* codes) {
    const int d = ix.d;
    const float sc = std::ldexp(1.0f, -ix.e);
    const float sc2 = std::ldexp(1.0f, -2 * ix.e);
    std::vector<float> kt(d);
    for (int i = 0; i < d; ++i) kt[i] = k[i] * sc;
    float r = 1.0f - nrm2 * sc2;
    if (!(r > 0.0f)) r = 0.0f;
    const float tail = std::sqrt(r);
    for (int j = 0; j < ix.m; ++j) {
        const float* u = &ix.dirs[((size_t)l * ix.m + j) * (d + 1)];
        float p = std::fma(u[d], tail, dot_fixed(u, kt.data(), d));
        codes[j] = quantise(p);
    }
}

Key make_key(const int* codes, int m, int tok) { return Key{morton(codes, m), (uint32_t)tok}; }

// ---------------------------------------------------------------------------
// Query side.
// ---------------------------------------------------------------------------
struct Query {
    std::vector<float> qsel;  // sum of the group's query heads
    std::vector<std::vector<int>> codes;  // [L][m]
};

Query prepare_query(const Index& ix, const float* q, int G) {
    const int d = ix.d;
    Query Q;
    Q.qsel.assign(q, q + d);
    for (int h = 1; h < G; ++h)
        for (int i = 0; i < d; ++i) Q.qsel[i] = Q.qsel[i] + q[(size_t)h * d + i];
    float nq = dot_fixed(Q.qsel.data(), Q.qsel.data(), d);
    std::vector<float> qt(d, 0.0f);
    if (nq > 0.0f) {
        float s = std::sqrt(nq);
        for (int i = 0; i < d; ++i) qt[i] = Q.qsel[i] / s;
    }
    Q.codes.assign(ix.L, std::vector<int>(ix.m));
    for (int l = 0; l < ix.L; ++l)
        for (int j = 0; j < ix.m; ++j) {
            const float* u = &ix.dirs[((size_t)l * ix.m + j) * (d + 1)];
            float p = std::fma(u[d], 0.0f, dot_fixed(u, qt.data(), d));
            Q.codes[l][j] = quantise(p);
        }
    return Q;
}

// Flat statement of the search: leaves sorted by (priority, position), taken
// whole until at least n_cand tokens are collected.
std::vector<int> leaf_order_flat(const Index& ix, int l, const std::vector<int>& qc, int n_cand,
                                 std::vector<int>* prio_out) {
    const Composite& C = ix.comp[l];
    const int N = (int)C.leaves.size();
    std::vector<int> prio(N);
    std::vector<int> lo(ix.m), hi(ix.m);
    for (int i = 0; i < N; ++i) {
        prefix_cell(C.leaves[i].prefix, C.leaves[i].t, ix.m, lo.data(), hi.data());
        prio[i] = cell_distance(qc.data(), lo.data(), hi.data(), ix.m);
    }
    std::vector<int> ord(N);
    for (int i = 0; i < N; ++i) ord[i] = i;
    std::sort(ord.begin(), ord.end(), [&](int a, int b) {
        return prio[a] != prio[b] ? prio[a] < prio[b] : a < b;
    });
    std::vector<int> taken;
    long cum = 0;
    for (int i : ord) {
        if (cum >= n_cand) break;
        taken.push_back(i);
        cum += (long)C.leaves[i].toks.size();
    }
    if (prio_out) *prio_out = prio;
    return taken;
}

// Best-first statement of the same search over the explicit trie: a priority
// queue of nodes keyed by (cell distance, prefix); a popped internal node
// pushes its children, a popped leaf is emitted. Nodes are the prefixes of the
// leaves; a child's cell lies inside its parent's, so keys never decrease.
std::vector<int> leaf_order_tree(const Index& ix, int l, const std::vector<int>& qc, int n_cand) {
    const Composite& C = ix.comp[l];
    const int N = (int)C.leaves.size();
    std::vector<int> taken;
    if (N == 0) return taken;
    struct Node {
        int dist;
        Key prefix;
        int t;
        int leaf;  // leaf index, or -1 for an internal node
    };
    auto cmp = [](const Node& a, const Node& b) {  // max-heap comparator -> min order
        if (a.dist != b.dist) return a.dist > b.dist;
        if (!(a.prefix == b.prefix)) return b.prefix < a.prefix;
        return a.t > b.t;
    };
    std::priority_queue<Node, std::vector<Node>, decltype(cmp)> pq(cmp);
    std::vector<int> lo(ix.m), hi(ix.m);
    auto make = [&](const Key& pre, int t) {
        Node nd;
        nd.prefix = pre;
        nd.t = t;
        prefix_cell(pre, t, ix.m, lo.data(), hi.data());
        nd.dist = cell_distance(qc.data(), lo.data(), hi.data(), ix.m);
        nd.leaf = -1;
        for (int i = 0; i < N; ++i)
            if (C.leaves[i].t == t && C.leaves[i].prefix == pre) nd.leaf = i;
        return nd;
    };
    // a node exists if it is a prefix of some leaf
    auto exists = [&](const Key& pre, int t) {
        for (const Leaf& lf : C.leaves)
            if (lf.t >= t && key_prefix(lf.prefix, t) == pre) return true;
        return false;
    };
    pq.push(make(Key{0, 0}, 0));
    long cum = 0;
    while (!pq.empty() && cum < n_cand) {
        Node nd = pq.top();
        pq.pop();
        if (nd.leaf >= 0) {
            taken.push_back(nd.leaf);
            cum += (long)C.leaves[nd.leaf].toks.size();
            continue;
        }
        for (int bit = 0; bit < 2; ++bit) {
            Key ch = nd.prefix;
            int t = nd.t;
            if (t < 64) ch.hi |= (uint64_t)bit << (63 - t);
            else ch.lo |= (uint32_t)bit << (95 - t);
            if (exists(ch, t + 1)) pq.push(make(ch, t + 1));
        }
    }
    return taken;
}

}  // namespace

// ===========================================================================
// C interface used by the Python wrapper (oracle/oracle.py).
// ===========================================================================
extern "C" {

uint64_t orc_splitmix64(uint64_t* state) { return splitmix64_next(*state); }

float orc_dot(const float* a, const float* b, int d) { return dot_fixed(a, b, d); }

int orc_scale_exponent(float maxn) { return scale_exponent(maxn); }

int orc_quantise(float p) { return quantise(p); }

uint64_t orc_morton(const int32_t* codes, int m) {
    int c[8];
    for (int j = 0; j < m; ++j) c[j] = codes[j];
    return morton(c, m);
}

// Directions u_{l,j} in R^{d+1}: one splitmix64 draw per component, in the
// order l, j, i; the sign bit (bit 63) picks -1/16, otherwise +1/16.
void orc_directions(uint64_t seed, int L, int m, int d, float* out) {
    uint64_t st = seed;
    for (int l = 0; l < L; ++l)
        for (int j = 0; j < m; ++j)
            for (int i = 0; i <= d; ++i) {
                uint64_t x = splitmix64_next(st);
                out[((size_t)l * m + j) * (d + 1) + i] = (x >> 63) ? -0.0625f : 0.0625f;
            }
}

// Gaussian directions (a variant of the search): each component is z / 16 with
// z standard normal from the Box-Muller transform (Box & Muller, 1958) of two
// splitmix64 draws x1, x2 taken in the order l, j, i:
//   u1 = ((x1 >> 11) + 1) * 2^-53 in (0, 1],  u2 = (x2 >> 11) * 2^-53 in [0, 1),
//   z = sqrt(-2 ln u1) * cos(2 pi u2), in double, rounded to float after / 16.
// The variance of a component is that of the Rademacher +-1/16 directions.
void orc_directions_gauss(uint64_t seed, int L, int m, int d, float* out) {
    uint64_t st = seed;
    const double two_pi = 2.0 * 3.14159265358979323846;
    for (int l = 0; l < L; ++l)
        for (int j = 0; j < m; ++j)
            for (int i = 0; i <= d; ++i) {
                const uint64_t x1 = splitmix64_next(st);
                const uint64_t x2 = splitmix64_next(st);
                const double u1 = (double)((x1 >> 11) + 1) * 0x1.0p-53;
                const double u2 = (double)(x2 >> 11) * 0x1.0p-53;
                const double z = std::sqrt(-2.0 * std::log(u1)) * std::cos(two_pi * u2);
                out[((size_t)l * m + j) * (d + 1) + i] = (float)(z / 16.0);
            }
}

// kind 0: Rademacher +-1/16 (the default reading); kind 1: Gaussian.
void* orc_create_kind(int d, int m, int L, int P, uint64_t seed, int kind) {
    if (d <= 0 || d % 32 != 0 || m < 1 || m > 8 || L < 1 || P < 1) return nullptr;
    if (kind != 0 && kind != 1) return nullptr;
    Index* ix = new Index();
    ix->d = d;
    ix->m = m;
    ix->L = L;
    ix->P = P;
    ix->seed = seed;
    ix->dirs.resize((size_t)L * m * (d + 1));
    if (kind == 0)
        orc_directions(seed, L, m, d, ix->dirs.data());
    else
        orc_directions_gauss(seed, L, m, d, ix->dirs.data());
    ix->comp.resize(L);
    return ix;
}

void* orc_create(int d, int m, int L, int P, uint64_t seed) { return orc_create_kind(d, m, L, P, seed, 0); }

void orc_destroy(void* h) { delete (Index*)h; }

// Prefill build. forced_e < -1000 computes e from the keys; otherwise it is
// used as given (a fresh build with the exponent of an earlier index).
int orc_build(void* h, const float* K, const float* V, int n, int forced_e) {
    Index& ix = *(Index*)h;
    const int d = ix.d;
    ix.n = n;
    ix.K.assign(K, K + (size_t)n * d);
    ix.V.assign(V, V + (size_t)n * d);
    std::vector<float> nrm2(n);
    float maxn = 0.0f;
    for (int t = 0; t < n; ++t) {
        nrm2[t] = dot_fixed(&ix.K[(size_t)t * d], &ix.K[(size_t)t * d], d);
        if (nrm2[t] > maxn) maxn = nrm2[t];
    }
    ix.e = forced_e < -1000 ? scale_exponent(maxn) : forced_e;
    for (int l = 0; l < ix.L; ++l) {
        Composite& C = ix.comp[l];
        C.keys.assign(n, Key{0, 0});
        C.codes.assign((size_t)n * ix.m, 0);
        for (int t = 0; t < n; ++t) {
            key_codes(ix, l, &ix.K[(size_t)t * d], nrm2[t], &C.codes[(size_t)t * ix.m]);
            C.keys[t] = make_key(&C.codes[(size_t)t * ix.m], ix.m, t);
        }
        std::vector<int> ord(n);
        for (int t = 0; t < n; ++t) ord[t] = t;
        std::sort(ord.begin(), ord.end(), [&](int a, int b) { return C.keys[a] < C.keys[b]; });
        C.leaves.clear();
        split_node(C.keys, ord, 0, ix.P, C.leaves);
        for (size_t i = 0; i < C.leaves.size(); ++i) C.leaves[i].id = (int)i;
        C.next_id = (int)C.leaves.size();
    }
    return 0;
}

// Insert one generated token (index = current token count) into every
// composite. Returns 0.
int orc_insert(void* h, const float* k, const float* v) {
    Index& ix = *(Index*)h;
    const int d = ix.d;
    const int tok = ix.n;
    ix.K.insert(ix.K.end(), k, k + d);
    ix.V.insert(ix.V.end(), v, v + d);
    ix.n += 1;
    const float nrm2 = dot_fixed(k, k, d);
    for (int l = 0; l < ix.L; ++l) {
        Composite& C = ix.comp[l];
        std::vector<int> codes(ix.m);
        key_codes(ix, l, k, nrm2, codes.data());
        C.codes.insert(C.codes.end(), codes.begin(), codes.end());
        Key x = make_key(codes.data(), ix.m, tok);
        C.keys.push_back(x);
        // 1. the leaf whose prefix x carries
        int found = -1;
        for (size_t i = 0; i < C.leaves.size(); ++i)
            if (key_prefix(x, C.leaves[i].t) == C.leaves[i].prefix) { found = (int)i; break; }
        if (found >= 0) {
            Leaf& lf = C.leaves[found];
            lf.toks.push_back(tok);
            if ((int)lf.toks.size() <= ix.P) continue;
            // overflow: re-partition this node's tokens below its prefix
            std::vector<int> toks = lf.toks;
            std::sort(toks.begin(), toks.end(), [&](int a, int b) { return C.keys[a] < C.keys[b]; });
            std::vector<Leaf> sub;
            split_node(C.keys, toks, lf.t, ix.P, sub);
            const int old_id = lf.id;
            for (size_t s = 0; s < sub.size(); ++s) sub[s].id = s == 0 ? old_id : C.next_id++;
            C.leaves.erase(C.leaves.begin() + found);
            C.leaves.insert(C.leaves.begin() + found, sub.begin(), sub.end());
            continue;
        }
        // 2. x lies in an empty part of the trie: its leaf is the shortest
        //    prefix of x that at most P keys (x included) carry.
        int lo_t = 0, hi_t = 96;  // count(prefix_t) is non-increasing in t
        auto count = [&](int t) {
            Key px = key_prefix(x, t);
            int c = 0;
            for (const Key& y : C.keys) c += key_prefix(y, t) == px;
            return c;
        };
        while (lo_t < hi_t) {
            int mid = (lo_t + hi_t) / 2;
            if (count(mid) <= ix.P) hi_t = mid; else lo_t = mid + 1;
        }
        Leaf nl;
        nl.t = lo_t;
        nl.prefix = key_prefix(x, lo_t);
        nl.id = C.next_id++;
        nl.toks = {tok};
        size_t pos = 0;
        while (pos < C.leaves.size() && C.leaves[pos].prefix < nl.prefix) ++pos;
        C.leaves.insert(C.leaves.begin() + pos, nl);
    }
    return 0;
}

int orc_e(void* h) { return ((Index*)h)->e; }
int orc_n(void* h) { return ((Index*)h)->n; }
int orc_n_leaves(void* h, int l) { return (int)((Index*)h)->comp[l].leaves.size(); }
int orc_next_id(void* h, int l) { return ((Index*)h)->comp[l].next_id; }

// Per-token Morton keys and codes of composite l.
void orc_token_keys(void* h, int l, uint64_t* mk, int32_t* codes) {
    Index& ix = *(Index*)h;
    const Composite& C = ix.comp[l];
    for (int t = 0; t < ix.n; ++t) {
        mk[t] = C.keys[t].hi;
        for (int j = 0; j < ix.m; ++j) codes[(size_t)t * ix.m + j] = C.codes[(size_t)t * ix.m + j];
    }
}

// Raw projections p_{l,j} of every token (for range checks).
void orc_projections(void* h, float* out) {
    Index& ix = *(Index*)h;
    const int d = ix.d;
    const float sc = std::ldexp(1.0f, -ix.e);
    const float sc2 = std::ldexp(1.0f, -2 * ix.e);
    std::vector<float> kt(d);
    for (int t = 0; t < ix.n; ++t) {
        const float* k = &ix.K[(size_t)t * d];
        float nrm2 = dot_fixed(k, k, d);
        for (int i = 0; i < d; ++i) kt[i] = k[i] * sc;
        float r = 1.0f - nrm2 * sc2;
        if (!(r > 0.0f)) r = 0.0f;
        float tail = std::sqrt(r);
        for (int l = 0; l < ix.L; ++l)
            for (int j = 0; j < ix.m; ++j) {
                const float* u = &ix.dirs[((size_t)l * ix.m + j) * (d + 1)];
                out[((size_t)t * ix.L + l) * ix.m + j] = std::fma(u[d], tail, dot_fixed(u, kt.data(), d));
            }
    }
}

// Transformed key k~ = [k * 2^-e, sqrt(max(0, 1 - ||k||^2 2^-2e))] of token t.
void orc_transformed_key(void* h, int t, float* out) {
    Index& ix = *(Index*)h;
    const int d = ix.d;
    const float* k = &ix.K[(size_t)t * d];
    const float sc = std::ldexp(1.0f, -ix.e);
    const float sc2 = std::ldexp(1.0f, -2 * ix.e);
    float nrm2 = dot_fixed(k, k, d);
    for (int i = 0; i < d; ++i) out[i] = k[i] * sc;
    float r = 1.0f - nrm2 * sc2;
    if (!(r > 0.0f)) r = 0.0f;
    out[d] = std::sqrt(r);
}

// Canonical dump of composite l, leaves left to right. Per leaf: prefix length,
// prefix (Morton part, token part), id, count, cell lo/hi (m each); the tokens
// of each leaf sorted ascending are written to toks at offsets off[i]..off[i+1].
void orc_dump(void* h, int l, int32_t* t_out, uint64_t* pm_out, uint32_t* pt_out, int32_t* id_out,
              int32_t* cnt_out, int32_t* lo_out, int32_t* hi_out, int64_t* off, int32_t* toks) {
    Index& ix = *(Index*)h;
    const Composite& C = ix.comp[l];
    int64_t o = 0;
    for (size_t i = 0; i < C.leaves.size(); ++i) {
        const Leaf& lf = C.leaves[i];
        t_out[i] = lf.t;
        pm_out[i] = lf.prefix.hi;
        pt_out[i] = lf.prefix.lo;
        id_out[i] = lf.id;
        cnt_out[i] = (int)lf.toks.size();
        prefix_cell(lf.prefix, lf.t, ix.m, &lo_out[i * ix.m], &hi_out[i * ix.m]);
        off[i] = o;
        std::vector<int> s = lf.toks;
        std::sort(s.begin(), s.end());
        for (int tk : s) toks[o++] = tk;
    }
    off[C.leaves.size()] = o;
}

// Query codes of every composite ([L][m]) and the fp32 sum of the group.
void orc_query(void* h, const float* q, int G, int32_t* codes, float* qsel) {
    Index& ix = *(Index*)h;
    Query Q = prepare_query(ix, q, G);
    for (int l = 0; l < ix.L; ++l)
        for (int j = 0; j < ix.m; ++j) codes[l * ix.m + j] = Q.codes[l][j];
    for (int i = 0; i < ix.d; ++i) qsel[i] = Q.qsel[i];
}

// Leaves taken by the search in composite l, in the order taken. mode 0: flat
// (priority, position) sort; mode 1: best-first tree search. prio (optional)
// receives every leaf's priority. Returns the number of leaves taken.
int orc_leaf_order(void* h, const float* q, int G, int l, int n_cand, int mode, int32_t* out,
                   int32_t* prio) {
    Index& ix = *(Index*)h;
    Query Q = prepare_query(ix, q, G);
    std::vector<int> pr;
    std::vector<int> ord = mode == 0 ? leaf_order_flat(ix, l, Q.codes[l], n_cand, &pr)
                                     : leaf_order_tree(ix, l, Q.codes[l], n_cand);
    for (size_t i = 0; i < ord.size(); ++i) out[i] = ord[i];
    if (prio && mode == 0)
        for (size_t i = 0; i < pr.size(); ++i) prio[i] = pr[i];
    return (int)ord.size();
}

// Page selection for one unit. page_ids receives n_sel = budget / P entries
// (-1 past the end); *n_pages the number selected. trace[0] = leaves scanned
// (all composites), trace[1] = |C| distinct candidates rescored, trace[2] =
// tokens in the selected pages, trace[3] = 1 if the best-first search agreed
// with the flat search in every composite (when check_tree), else 0.
int orc_select(void* h, const float* q, int G, int budget, int n_cand, int32_t* page_ids,
               int32_t* n_pages, int64_t* trace, int check_tree) {
    Index& ix = *(Index*)h;
    const int d = ix.d;
    const int n_sel = budget / ix.P;
    Query Q = prepare_query(ix, q, G);
    std::set<int> cand;
    long scanned = 0;
    int tree_ok = 1;
    for (int l = 0; l < ix.L; ++l) {
        const Composite& C = ix.comp[l];
        scanned += (long)C.leaves.size();
        std::vector<int> ord = leaf_order_flat(ix, l, Q.codes[l], n_cand, nullptr);
        if (check_tree) {
            std::vector<int> tr = leaf_order_tree(ix, l, Q.codes[l], n_cand);
            if (tr != ord) tree_ok = 0;
        }
        for (int li : ord)
            for (int tk : C.leaves[li].toks) cand.insert(tk);
    }
    // token -> page (composite 0 leaf id)
    std::vector<int> page_of(ix.n, -1);
    std::vector<int> page_cnt;
    for (const Leaf& lf : ix.comp[0].leaves)
        for (int tk : lf.toks) page_of[tk] = lf.id;
    struct Scored {
        float s;
        int t;
    };
    std::vector<Scored> sc;
    for (int tk : cand) sc.push_back({dot_fixed(Q.qsel.data(), &ix.K[(size_t)tk * d], d), tk});
    std::sort(sc.begin(), sc.end(), [](const Scored& a, const Scored& b) {
        if (a.s > b.s) return true;
        if (a.s < b.s) return false;
        return a.t < b.t;
    });
    std::vector<int> sel;
    for (const Scored& x : sc) {
        if ((int)sel.size() >= n_sel) break;
        int p = page_of[x.t];
        if (std::find(sel.begin(), sel.end(), p) == sel.end()) sel.push_back(p);
    }
    for (int i = 0; i < n_sel; ++i) page_ids[i] = i < (int)sel.size() ? sel[i] : -1;
    *n_pages = (int)sel.size();
    long sel_tokens = 0;
    for (const Leaf& lf : ix.comp[0].leaves)
        if (std::find(sel.begin(), sel.end(), lf.id) != sel.end()) sel_tokens += (long)lf.toks.size();
    if (trace) {
        trace[0] = scanned;
        trace[1] = (int64_t)cand.size();
        trace[2] = sel_tokens;
        trace[3] = tree_ok;
    }
    return 0;
}

// Attention over the tokens S of the given pages, in fp64, for each of the G
// query heads: o_h = sum_t softmax_t(q_h . k_t / sqrt(d)) v_t.
void orc_attn(void* h, const float* q, int G, const int32_t* page_ids, int n_pages, double* out) {
    Index& ix = *(Index*)h;
    const int d = ix.d;
    std::vector<int> S;
    for (int i = 0; i < n_pages; ++i)
        for (const Leaf& lf : ix.comp[0].leaves)
            if (lf.id == page_ids[i]) S.insert(S.end(), lf.toks.begin(), lf.toks.end());
    const double scale = 1.0 / std::sqrt((double)d);
    for (int g = 0; g < G; ++g) {
        double* o = out + (size_t)g * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (S.empty()) continue;
        std::vector<double> s(S.size());
        double mx = -INFINITY;
        for (size_t a = 0; a < S.size(); ++a) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += (double)q[(size_t)g * d + i] * (double)ix.K[(size_t)S[a] * d + i];
            s[a] = acc * scale;
            mx = std::max(mx, s[a]);
        }
        double z = 0.0;
        for (size_t a = 0; a < S.size(); ++a) {
            double w = std::exp(s[a] - mx);
            z += w;
            for (int i = 0; i < d; ++i) o[i] += w * (double)ix.V[(size_t)S[a] * d + i];
        }
        for (int i = 0; i < d; ++i) o[i] /= z;
    }
}

// Dense attention over all n tokens (the full-KV special case), fp64.
void orc_dense_attn(const float* q, int G, const float* K, const float* V, int n, int d, double* out) {
    const double scale = 1.0 / std::sqrt((double)d);
    std::vector<double> s(n);
    for (int g = 0; g < G; ++g) {
        double* o = out + (size_t)g * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (n == 0) continue;
        double mx = -INFINITY;
        for (int t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += (double)q[(size_t)g * d + i] * (double)K[(size_t)t * d + i];
            s[t] = acc * scale;
            mx = std::max(mx, s[t]);
        }
        double z = 0.0;
        for (int t = 0; t < n; ++t) {
            double w = std::exp(s[t] - mx);
            z += w;
            for (int i = 0; i < d; ++i) o[i] += w * (double)V[(size_t)t * d + i];
        }
        for (int i = 0; i < d; ++i) o[i] /= z;
    }
}

// Brute-force ranking of all tokens by the fixed-order fp32 score D(qsel, k)
// (ties: lower token first). Writes the token order.
void orc_brute_rank(void* h, const float* q, int G, int32_t* order) {
    Index& ix = *(Index*)h;
    Query Q = prepare_query(ix, q, G);
    std::vector<float> s(ix.n);
    for (int t = 0; t < ix.n; ++t) s[t] = dot_fixed(Q.qsel.data(), &ix.K[(size_t)t * ix.d], ix.d);
    std::vector<int> ord(ix.n);
    for (int t = 0; t < ix.n; ++t) ord[t] = t;
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return s[a] > s[b]; });
    for (int t = 0; t < ix.n; ++t) order[t] = ord[t];
}

// Exact top-k by the fp64 inner product with the fp32 group sum (ties: lower
// token first), the "TOP-k" reference used for recall.
void orc_exact_topk(void* h, const float* q, int G, int k, int32_t* out) {
    Index& ix = *(Index*)h;
    Query Q = prepare_query(ix, q, G);
    std::vector<double> s(ix.n);
    for (int t = 0; t < ix.n; ++t) {
        double acc = 0.0;
        for (int i = 0; i < ix.d; ++i) acc += (double)Q.qsel[i] * (double)ix.K[(size_t)t * ix.d + i];
        s[t] = acc;
    }
    std::vector<int> ord(ix.n);
    for (int t = 0; t < ix.n; ++t) ord[t] = t;
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return s[a] > s[b]; });
    for (int i = 0; i < k && i < ix.n; ++i) out[i] = ord[i];
}

// Page id of every token (composite 0).
void orc_page_of(void* h, int32_t* out) {
    Index& ix = *(Index*)h;
    for (int t = 0; t < ix.n; ++t) out[t] = -1;
    for (const Leaf& lf : ix.comp[0].leaves)
        for (int tk : lf.toks) out[tk] = lf.id;
}

}  // extern "C"

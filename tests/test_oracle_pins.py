"""Pins of the CPU oracle against facts other than itself.

Each test ties one oracle function to a published value, a closed form, a
hand-derived example, brute force on tiny inputs, or an invariant that the
IceCache pages state ("IceCache", Figure 2: every token indexed into one leaf =
one physical page of fixed size; abstract: the structure is updatable without
a rebuild; Table 1 rows FULL and TOP-k: dense attention and exact top-k are the
limiting cases of the selection).
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

U = 2.0 ** -24  # unit roundoff of float32


def _golden_ints(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(x) for x in f.read().split("\n") if x and not x.startswith("#")]


# --------------------------------------------------------------------------
# Direction generator
# --------------------------------------------------------------------------
def test_splitmix64_published_vector(oracle_mod):
    assert oracle_mod.splitmix64_stream(1234567, 5) == _golden_ints("splitmix64_seed1234567.txt")


def test_directions_are_rademacher_from_stream(oracle_mod):
    L, m, d, seed = 2, 8, 128, 7
    u = oracle_mod.directions(seed, L, m, d)
    assert set(np.unique(u).tolist()) == {-0.0625, 0.0625}
    stream = oracle_mod.splitmix64_stream(seed, L * m * (d + 1))
    signs = np.array([-1.0 if (x >> 63) else 1.0 for x in stream]).reshape(L, m, d + 1)
    assert np.array_equal(np.sign(u), signs)


# --------------------------------------------------------------------------
# Fixed-order dot D(a, b)
# --------------------------------------------------------------------------
def test_dot_hand_derived_order():
    # d = 128: lane l owns a[4l..4l+3]. Put 2^24, 1, 1 in lane 0 and 1 in lanes
    # 8 and 24, b = ones. Lane 0: fma chain 2^24 -> 2^24+1 rounds to 2^24 (tie
    # to even) -> 2^24. Level o=16 adds lane 24 into lane 8: 1+1 = 2. Level o=8
    # adds lane 8 into lane 0: 2^24 + 2 (exact). Result 2^24 + 2, while the
    # exact sum is 2^24 + 4 and a left-to-right sum gives 2^24.
    from oracle import oracle as O
    a = np.zeros(128, np.float32)
    a[0], a[1], a[2], a[32], a[96] = 2.0 ** 24, 1, 1, 1, 1
    b = np.ones(128, np.float32)
    assert O.dot(a, b) == 2.0 ** 24 + 2


def test_dot_within_rounding_bound(oracle_mod):
    rng = np.random.default_rng(1)
    gamma = 9 * U / (1 - 9 * U)  # 4 fma + 5 additions on any path
    for _ in range(200):
        a = rng.standard_normal(128).astype(np.float32)
        b = rng.standard_normal(128).astype(np.float32) * rng.choice([1e-3, 1.0, 1e3])
        exact = float(np.dot(a.astype(np.float64), b.astype(np.float64)))
        bound = gamma * float(np.sum(np.abs(a.astype(np.float64) * b)))
        assert abs(oracle_mod.dot(a, b) - exact) <= bound


def test_dot_exact_on_small_integers(oracle_mod):
    rng = np.random.default_rng(2)
    for d in (32, 64, 128, 256):
        a = rng.integers(-100, 100, d).astype(np.float32)
        b = rng.integers(-100, 100, d).astype(np.float32)
        assert oracle_mod.dot(a, b) == float(np.dot(a.astype(np.int64), b.astype(np.int64)))


# --------------------------------------------------------------------------
# Transform: scale exponent, quantiser, Morton layout
# --------------------------------------------------------------------------
def test_scale_exponent_is_smallest_power(oracle_mod):
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(1e-6, 1e6, 500), 4.0 ** np.arange(-10, 11),
                           4.0 ** np.arange(-10, 11) * 1.0000001, [2.0, 0.5, 3.0]])
    for v in vals.astype(np.float32):
        e = oracle_mod.scale_exponent(v)
        c2 = 4.0 ** e
        assert c2 >= v and c2 / 4 < v, (v, e)
    assert oracle_mod.scale_exponent(0.0) == 0
    assert oracle_mod.scale_exponent(16.0) == 2 and oracle_mod.scale_exponent(16.000002) == 3


def test_quantiser_closed_form(oracle_mod):
    q = oracle_mod.quantise
    assert q(-1.0) == 0 and q(-2.0) == 0 and q(0.0) == 128 and q(1.0) == 255 and q(5.0) == 255
    assert q(1.0 - 2.0 ** -8) == 255 and q(1.0 - 2.0 ** -7 - 2.0 ** -20) == 254
    for k in range(256):  # cell k is [k/128 - 1, (k+1)/128 - 1)
        lo = k / 128.0 - 1.0
        assert q(lo) == k
        assert q(lo + 0.5 / 128.0) == k


def test_morton_layout(oracle_mod):
    mo = oracle_mod.morton
    assert mo([0x80, 0, 0, 0, 0, 0, 0, 0]) == 1 << 63
    assert mo([0, 0x80, 0, 0, 0, 0, 0, 0]) == 1 << 62
    assert mo([1, 0, 0, 0, 0, 0, 0, 0]) == 1 << 7
    assert mo([0, 0, 0, 0, 0, 0, 0, 1]) == 1
    assert mo([0xFF] * 8) == (1 << 64) - 1
    # m = 2: 16 bits left-aligned, code0 bit 7, code1 bit 7, code0 bit 6, ...;
    # bit b of code j sits at position (7 - b) * 2 + j from the top: code0 bits
    # 7, 0 -> positions 0, 14; code1 bits 1, 0 -> positions 13, 15.
    assert mo([0b10000001, 0b00000011]) == (1 << 63) | (1 << 50) | (1 << 49) | (1 << 48)


def test_transform_closed_form_mips_to_nn(oracle_mod):
    """||q~ - k~||^2 = 2 - 2 q.k / (||q|| c): nearest neighbour = max inner product."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(4)
    n, d = 64, 128
    K = (rng.standard_normal((n, d)) * rng.uniform(0.2, 3.0, (n, 1))).astype(np.float32)
    ix = OracleIndex(d, 8, 1, 16, 0).build(K, K)
    c = 2.0 ** ix.e
    kt = np.stack([ix.transformed_key(t) for t in range(n)]).astype(np.float64)
    assert np.allclose(np.sum(kt ** 2, axis=1), 1.0, atol=1e-5)  # every k~ on the unit sphere
    assert np.all(np.linalg.norm(K.astype(np.float64), axis=1) <= c)
    assert np.max(np.linalg.norm(K.astype(np.float64), axis=1)) > c / 2
    for _ in range(20):
        q = rng.standard_normal(d)
        qt = np.concatenate([q / np.linalg.norm(q), [0.0]])
        dist = np.sum((kt - qt) ** 2, axis=1)
        ip = K.astype(np.float64) @ q
        assert np.allclose(dist, 2 - 2 * ip / (np.linalg.norm(q) * c), atol=1e-5)
        order_ip = np.argsort(-ip, kind="stable")
        gaps = np.abs(np.diff(ip[order_ip]))
        if gaps.min() > 1e-3:
            assert np.array_equal(np.argsort(dist, kind="stable"), order_ip)


def test_projection_range_and_value(oracle_mod):
    """|p| <= ||u|| ||k~|| = sqrt(d+1)/16, and p matches the fp64 projection."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(5)
    n, d, L, m = 200, 128, 2, 8
    K = (rng.standard_normal((n, d)) * 2).astype(np.float32)
    ix = OracleIndex(d, m, L, 16, 11).build(K, K)
    p = ix.projections()
    assert np.max(np.abs(p)) <= math.sqrt(d + 1) / 16
    u = oracle_mod.directions(11, L, m, d).astype(np.float64)
    for t in range(0, n, 17):
        kt = ix.transformed_key(t).astype(np.float64)
        ref = u @ kt  # [L, m]
        assert np.allclose(p[t], ref, atol=1e-6)
    mk, codes = ix.token_keys(1)
    assert np.array_equal(codes, np.clip(np.floor((p[:, 1, :].astype(np.float32) + np.float32(1))
                                                  * np.float32(128)), 0, 255).astype(np.int32))
    for t in range(0, n, 13):
        assert mk[t] == oracle_mod.morton(codes[t])


# --------------------------------------------------------------------------
# Partition invariants
# --------------------------------------------------------------------------
def _key96(mk, t):
    return (int(mk) << 32) | int(t)


def _check_partition(ix, l, P):
    n = ix.n
    dmp = ix.dump(l)
    mk, codes = ix.token_keys(l)
    keys = [_key96(mk[t], t) for t in range(n)]
    N = len(dmp["t"])
    seen = np.zeros(n, np.int32)
    prev_max = -1
    for i in range(N):
        toks = dmp["toks"][dmp["off"][i]:dmp["off"][i + 1]]
        assert 1 <= len(toks) <= P
        assert len(toks) == dmp["cnt"][i]
        seen[toks] += 1
        t = int(dmp["t"][i])
        prefix = (int(dmp["pm"][i]) << 32) | int(dmp["pt"][i])
        mask = ((1 << 96) - 1) ^ ((1 << (96 - t)) - 1)
        # every token of the leaf carries its prefix, and only those tokens do
        carriers = [tk for tk in range(n) if keys[tk] & mask == prefix]
        assert sorted(carriers) == sorted(toks.tolist())
        # minimality: the parent node holds more than P tokens
        if t > 0:
            pmask = ((1 << 96) - 1) ^ ((1 << (97 - t)) - 1)
            assert sum(1 for k in keys if k & pmask == prefix & pmask) > P
        else:
            assert n <= P
        # leaves are contiguous runs of the sorted key order
        kk = sorted(keys[tk] for tk in toks)
        assert kk[0] > prev_max
        prev_max = kk[-1]
        # cell: every token's codes lie in [lo, hi], cell width 2^(8 - known bits)
        for tk in toks:
            assert np.all(codes[tk] >= dmp["lo"][i]) and np.all(codes[tk] <= dmp["hi"][i])
        m = codes.shape[1]
        for j in range(m):
            bj = 8 if t >= 8 * m else min(8, max(0, (t - j + m - 1) // m))
            assert dmp["hi"][i][j] - dmp["lo"][i][j] + 1 == 1 << (8 - bj)
    assert np.all(seen == 1)  # every token in exactly one leaf / page
    return dmp


def _clustered(rng, n, d, centers, spread=0.3):
    mu = rng.standard_normal((centers, d))
    return (mu[rng.integers(0, centers, n)] + spread * rng.standard_normal((n, d))).astype(np.float32)


@pytest.mark.parametrize("n,P,L", [(1, 16, 1), (16, 16, 1), (17, 16, 2), (300, 16, 2),
                                   (500, 32, 2), (257, 4, 1)])
def test_partition_invariants(oracle_mod, n, P, L):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(n * 7 + P)
    K = _clustered(rng, n, 128, 8)
    ix = OracleIndex(128, 8, L, P, 3).build(K, K)
    for l in range(L):
        dmp = _check_partition(ix, l, P)
        assert np.array_equal(dmp["id"], np.arange(len(dmp["id"])))  # build: left to right
    if n <= P:
        assert ix.n_leaves(0) == 1 and ix.dump(0)["t"][0] == 0


def test_partition_all_keys_equal(oracle_mod):
    # 40 equal keys, P = 16: the Morton parts tie, so the node splits on token
    # bits. Tokens < 64 share bits 31..6; bit 5 separates 0..31 from 32..39;
    # 0..31 (32 > 16) splits on bit 4. Leaves: [0..15] and [16..31] at prefix
    # length 64 + 28 = 92, [32..39] at 64 + 27 = 91.
    from oracle.oracle import OracleIndex
    K = np.tile(np.linspace(-1, 1, 128, dtype=np.float32), (40, 1))
    ix = OracleIndex(128, 8, 1, 16, 0).build(K, K)
    dmp = _check_partition(ix, 0, 16)
    assert dmp["t"].tolist() == [92, 92, 91]
    assert dmp["cnt"].tolist() == [16, 16, 8]
    assert dmp["toks"].tolist() == list(range(40))


def test_partition_duplicate_keys(oracle_mod):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(9)
    base = _clustered(rng, 20, 128, 4)
    K = base[rng.integers(0, 20, 400)]
    ix = OracleIndex(128, 8, 2, 16, 5).build(K, K)
    for l in range(2):
        _check_partition(ix, l, 16)


# --------------------------------------------------------------------------
# Search
# --------------------------------------------------------------------------
def test_cell_distance_brute_force_m2(oracle_mod):
    """L-infinity distance to a cell equals the minimum over the cell's points (m = 2)."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(10)
    K = _clustered(rng, 600, 128, 6, 0.5)
    ix = OracleIndex(128, 2, 1, 8, 21).build(K, K)
    dmp = ix.dump(0)
    for trial in range(6):
        q = rng.standard_normal((2, 128)).astype(np.float32)
        codes, _ = ix.query(q)
        _, prio = ix.leaf_order(q, 0, 10)
        qc = codes[0]
        for i in range(0, len(dmp["t"]), 7):
            lo, hi = dmp["lo"][i], dmp["hi"][i]
            xs = np.arange(lo[0], hi[0] + 1)
            ys = np.arange(lo[1], hi[1] + 1)
            gx, gy = np.meshgrid(xs, ys)
            brute = np.min(np.maximum(np.abs(gx - qc[0]), np.abs(gy - qc[1])))
            assert prio[i] == brute


@pytest.mark.parametrize("seed", range(6))
def test_best_first_tree_search_equals_flat_order(oracle_mod, seed):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(50, 1500))
    P = int(rng.choice([4, 16, 32]))
    K = _clustered(rng, n, 128, int(rng.integers(1, 40)))
    ix = OracleIndex(128, 8, 2, P, seed).build(K, K)
    for _ in range(3):
        q = (K[rng.integers(0, n)] + 0.3 * rng.standard_normal(128)).astype(np.float32)[None].repeat(
            int(rng.integers(1, 5)), 0)
        n_cand = int(rng.integers(1, n + 50))
        for l in range(2):
            flat, _ = ix.leaf_order(q, l, n_cand)
            tree, _ = ix.leaf_order(q, l, n_cand, tree=True)
            assert np.array_equal(flat, tree)
        _, _, tr = ix.select(q, P * 4, n_cand, check_tree=True)
        assert tr["tree_ok"]


# --------------------------------------------------------------------------
# Selection special cases
# --------------------------------------------------------------------------
def _first_distinct_pages(order, page_of, n_sel):
    out = []
    for t in order:
        p = page_of[t]
        if p not in out:
            out.append(p)
        if len(out) == n_sel:
            break
    return out


@pytest.mark.parametrize("seed", range(4))
def test_exhaustive_selection_is_brute_force_ranking(oracle_mod, seed):
    """With n_cand >= n every token is rescored: the pages are the first
    distinct pages of the brute-force ranking of all tokens (ties: lower token)."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(200 + seed)
    n, P = int(rng.integers(100, 900)), 16
    K = _clustered(rng, n, 128, 16)
    ix = OracleIndex(128, 8, 2, P, seed).build(K, K)
    q = (K[0] + 0.3 * rng.standard_normal((4, 128))).astype(np.float32)
    budget = 128
    ids, npg, tr = ix.select(q, budget, n_cand=n + 1)
    assert tr["cands"] == n
    # brute force in fp64 of the same fp32 group sum, checked against the
    # oracle's fixed-order ranking wherever fp64 separates the scores clearly
    _, qsel = ix.query(q)
    s64 = K.astype(np.float64) @ qsel.astype(np.float64)
    order = ix.brute_rank(q)
    assert np.all(np.diff(s64[order]) <= 1e-3)
    exp = _first_distinct_pages(order, ix.page_of(), budget // P)
    assert ids[:npg].tolist() == exp


def test_selection_ties_break_by_token_index(oracle_mod):
    """Equal keys tie exactly in fp32: the lowest token index ranks first."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(7)
    base = _clustered(rng, 40, 128, 4)
    K = np.concatenate([base, base, base])  # token t, t+40, t+80 share a key
    ix = OracleIndex(128, 8, 1, 4, 2).build(K, K)
    q = (base[3] + 0.1 * rng.standard_normal((2, 128))).astype(np.float32)
    order = ix.brute_rank(q)
    pos = np.argsort(order)
    for t in range(40):
        assert pos[t] < pos[t + 40] < pos[t + 80]
    ids, npg, _ = ix.select(q, 16, n_cand=1000)
    assert ids[:npg].tolist() == _first_distinct_pages(order, ix.page_of(), 4)


def test_full_budget_equals_dense_attention(oracle_mod):
    """Budget and candidates covering the whole context select every page, and
    sparse attention equals full-KV attention (Table 1, FULL row)."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(11)
    n, P = 300, 16
    K = _clustered(rng, n, 128, 8)
    V = rng.standard_normal((n, 128)).astype(np.float32)
    ix = OracleIndex(128, 8, 2, P, 1).build(K, V)
    q = (K[5] + 0.3 * rng.standard_normal((4, 128))).astype(np.float32)
    budget = P * ix.n_leaves(0)
    ids, npg, _ = ix.select(q, budget, n_cand=n)
    assert npg == ix.n_leaves(0)
    assert sorted(ids.tolist()) == list(range(npg))
    np.testing.assert_allclose(ix.attn(q, ids, npg), oracle_mod.dense_attn(q, K, V), atol=1e-12)


# --------------------------------------------------------------------------
# Dense attention closed forms
# --------------------------------------------------------------------------
def test_dense_attention_closed_forms(oracle_mod):
    rng = np.random.default_rng(12)
    n, d = 37, 128
    K = rng.standard_normal((n, d)).astype(np.float32)
    V = rng.standard_normal((n, d)).astype(np.float32)
    # zero query: uniform weights
    np.testing.assert_allclose(oracle_mod.dense_attn(np.zeros((2, d), np.float32), K, V)[0],
                               V.astype(np.float64).mean(0), atol=1e-12)
    # identical keys: uniform weights
    Kc = np.tile(K[:1], (n, 1))
    np.testing.assert_allclose(oracle_mod.dense_attn(K[:2], Kc, V)[1], V.astype(np.float64).mean(0),
                               atol=1e-12)
    # one token: its value
    np.testing.assert_allclose(oracle_mod.dense_attn(K[:1], K[:1], V[:1])[0], V[0], atol=1e-12)
    # two tokens: weights sigma(delta), delta = (s1 - s0) / sqrt(d)
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 3.0
    K2 = np.zeros((2, d), np.float32)
    K2[1, 0] = 2.0
    V2 = np.stack([np.full(d, 1.0), np.full(d, -1.0)]).astype(np.float32)
    w1 = 1.0 / (1.0 + math.exp(-6.0 / math.sqrt(d)))
    np.testing.assert_allclose(oracle_mod.dense_attn(q, K2, V2)[0], np.full(d, (1 - w1) - w1),
                               atol=1e-12)


# --------------------------------------------------------------------------
# Insertion without rebuild == fresh build (spec invariant)
# --------------------------------------------------------------------------
def _canonical(ix, l):
    d = ix.dump(l)
    return [(int(d["t"][i]), int(d["pm"][i]), int(d["pt"][i]),
             tuple(d["toks"][d["off"][i]:d["off"][i + 1]].tolist())) for i in range(len(d["t"]))]


@pytest.mark.parametrize("seed,n0,steps,P", [(0, 0, 40, 4), (1, 5, 60, 16), (2, 300, 200, 16),
                                            (3, 200, 150, 32), (4, 64, 120, 8)])
def test_insert_equals_fresh_build(oracle_mod, seed, n0, steps, P):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(300 + seed)
    K = _clustered(rng, n0 + steps, 128, 12)
    K[n0 + steps // 2] *= 3.0  # a generated key beyond the frozen norm bound (tail clamps to 0)
    V = rng.standard_normal((n0 + steps, 128)).astype(np.float32)
    dyn = OracleIndex(128, 8, 2, P, seed).build(K[:n0], V[:n0])
    e = dyn.e
    for s in range(steps):
        dyn.insert(K[n0 + s], V[n0 + s])
        if s % 37 == 0 or s == steps - 1:
            fresh = OracleIndex(128, 8, 2, P, seed).build(K[:n0 + s + 1], V[:n0 + s + 1], forced_e=e)
            for l in range(2):
                assert _canonical(dyn, l) == _canonical(fresh, l)
                _check_partition(dyn, l, P)
                ids = dyn.dump(l)["id"]
                assert sorted(ids.tolist()) == list(range(dyn.next_id(l)))  # ids stay dense
    # and the inserted index still answers like the fresh one
    q = (K[1] + 0.3 * rng.standard_normal((4, 128))).astype(np.float32)
    fresh = OracleIndex(128, 8, 2, P, seed).build(K, V, forced_e=e)
    a_ids, a_n, _ = dyn.select(q, 8 * P)
    b_ids, b_n, _ = fresh.select(q, 8 * P)
    pa, pb = dyn.page_of(), fresh.page_of()
    assert a_n == b_n
    for x, y in zip(a_ids[:a_n], b_ids[:b_n]):  # same pages up to their ids
        assert sorted(np.nonzero(pa == x)[0].tolist()) == sorted(np.nonzero(pb == y)[0].tolist())


def test_insert_split_keeps_old_id_for_left_child(oracle_mod):
    """A full leaf that overflows splits in two: the left child keeps the page
    id, the right child takes the next free id."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(13)
    K = _clustered(rng, 200, 128, 3)
    ix = OracleIndex(128, 8, 1, 8, 4).build(K[:120], K[:120])
    for s in range(120, 200):
        before = ix.dump(0)
        nid = ix.next_id(0)
        ix.insert(K[s], K[s])
        after = ix.dump(0)
        if len(after["t"]) == len(before["t"]) + 1 and ix.next_id(0) == nid + 1:
            new = int(np.nonzero(after["id"] == nid)[0][0])
            # either a split (left neighbour holds the old id of the full leaf) or a new leaf
            tok_leaf_new = set(after["toks"][after["off"][new]:after["off"][new + 1]].tolist())
            if len(tok_leaf_new) > 1 or s not in tok_leaf_new:
                left = new - 1
                old = [i for i in range(len(before["t"])) if before["id"][i] == after["id"][left]][0]
                assert before["cnt"][old] == 8
                assert after["cnt"][left] + after["cnt"][new] == 9


def test_gaussian_directions_follow_box_muller():
    """Gaussian directions: component (l, j, i) is z / 16 with z the Box-Muller
    normal of the next two splitmix64 draws (recomputed here with Python's math
    module from the generator's stream), and their spread matches the
    Rademacher +-1/16 directions."""
    import math
    from oracle import oracle as O
    seed, L, m, d = 99, 2, 8, 128
    g = O.directions(seed, L, m, d, kind=1)
    draws = O.splitmix64_stream(seed, 2 * 12)
    for c in range(12):
        x1, x2 = draws[2 * c], draws[2 * c + 1]
        u1 = ((x1 >> 11) + 1) * 2.0 ** -53
        u2 = (x2 >> 11) * 2.0 ** -53
        z = math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
        assert g.reshape(-1)[c] == np.float32(z / 16.0), c
    flat = g.reshape(-1).astype(np.float64)
    assert abs(flat.mean()) < 0.01 and abs(flat.std() - 1 / 16) < 0.005
    r = O.directions(seed, L, m, d, kind=0)
    assert set(np.unique(r).tolist()) == {-0.0625, 0.0625}


# --------------------------------------------------------------------------
# Query preparation (Figure 2 step 2: the query is mapped into the same
# projected code space as the keys). q_sel is the fp32 sum of the group's heads
# taken in head order, q~ = [q_sel / ||q_sel||, 0] (the query side of the
# MIPS-to-NN transform has tail 0), and its codes quantise u . q~.
# --------------------------------------------------------------------------
def _codes_fp64(u, qsel):
    """Codes of the query from the definition, in fp64: q~ = q_sel / ||q_sel||
    with tail 0, p = u[:d] . q~, code = clamp(floor((p + 1) 128), 0, 255).
    Also returns the distance of (p + 1) 128 to the nearest integer."""
    q64 = np.asarray(qsel, np.float64)
    qt = q64 / np.linalg.norm(q64)
    p = u[..., :-1].astype(np.float64) @ qt
    y = (p + 1.0) * 128.0
    return np.clip(np.floor(y), 0, 255).astype(np.int32), np.abs(y - np.round(y))


def _index_for_query(seed, L=2, m=8):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(seed)
    K = _clustered(rng, 50, 128, 4)
    return OracleIndex(128, m, L, 16, seed).build(K, K)


def test_query_codes_one_axis_closed_form(oracle_mod):
    """q_sel = 3 e_5: q~ = e_5 exactly, so p_j = u_j[5] = +-1/16 and the code is
    (1 +- 1/16) 128 = 136 or 120 exactly. Without the normalisation the codes
    would be 152 / 104; with a tail of 1 instead of 0 they would move by
    u_j[d] 128 = +-8."""
    ix = _index_for_query(31)
    u = oracle_mod.directions(31, 2, 8, 128)
    q = np.zeros((4, 128), np.float32)
    q[2, 5] = 3.0
    codes, qsel = ix.query(q)
    assert qsel[5] == 3.0 and np.count_nonzero(qsel) == 1
    expect = np.where(u[:, :, 5] > 0, 136, 120)
    assert np.array_equal(codes, expect)


def test_query_heads_summed_in_head_order(oracle_mod):
    """q_sel = ((q_0 + q_1) + q_2) + q_3 in fp32: with 2^24, 1, 1 in one
    component, each addition rounds back to 2^24 (ties to even), whereas any
    order that adds the two ones first gives 2^24 + 2."""
    ix = _index_for_query(32)
    q = np.zeros((4, 128), np.float32)
    q[0, 7], q[1, 7], q[2, 7] = 2.0 ** 24, 1.0, 1.0
    q[3, 9] = -5.0
    _, qsel = ix.query(q)
    assert qsel[7] == 2.0 ** 24 and qsel[9] == -5.0
    assert np.count_nonzero(qsel) == 2


def test_query_heads_cancel_to_known_vector(oracle_mod):
    """Heads a, b - a, 0, 0 (small integers, so every fp32 sum is exact) give
    q_sel = b, and the codes are those of b / ||b|| from the definition."""
    rng = np.random.default_rng(33)
    ix = _index_for_query(33)
    u = oracle_mod.directions(33, 2, 8, 128)
    checked = 0
    for _ in range(20):
        a = rng.integers(-50, 50, 128).astype(np.float32)
        b = rng.integers(-50, 50, 128).astype(np.float32)
        q = np.stack([a, b - a, np.zeros(128), np.zeros(128)]).astype(np.float32)
        codes, qsel = ix.query(q)
        assert np.array_equal(qsel, b)
        ref, gap = _codes_fp64(u, b)
        safe = gap > 1e-3  # away from a code boundary, fp32 and fp64 agree
        assert np.array_equal(codes[safe], ref[safe])
        checked += int(safe.sum())
    assert checked >= 300


def test_query_codes_match_definition_random(oracle_mod):
    """Random group queries (G = 1, 2, 4, 8): q_sel is the sequential fp32 sum
    of the heads, and every code away from a boundary is the fp64 definition's.
    Checked against a reading that skips the normalisation and one that puts 1
    in the query's tail: both disagree with the oracle on these inputs."""
    rng = np.random.default_rng(34)
    ix = _index_for_query(34)
    u = oracle_mod.directions(34, 2, 8, 128)
    for G in (1, 2, 4, 8):
        for _ in range(8):
            q = (rng.standard_normal((G, 128)) * rng.uniform(0.1, 4.0)).astype(np.float32)
            codes, qsel = ix.query(q)
            acc = q[0].copy()
            for h in range(1, G):
                acc = (acc + q[h]).astype(np.float32)
            assert np.array_equal(qsel, acc)
            ref, gap = _codes_fp64(u, acc)
            safe = gap > 1e-3
            assert safe.sum() >= 12
            assert np.array_equal(codes[safe], ref[safe])
            # the two wrong readings give other codes on these queries
            raw = np.clip(np.floor((u[..., :-1].astype(np.float64) @ acc.astype(np.float64) + 1)
                                   * 128), 0, 255)
            tail1 = np.clip(np.floor((u[..., :-1].astype(np.float64)
                                      @ (acc / np.linalg.norm(acc.astype(np.float64)))
                                      + u[..., -1] + 1) * 128), 0, 255)
            assert not np.array_equal(codes, raw) or np.linalg.norm(acc) == 1.0
            assert not np.array_equal(codes, tail1)


def test_zero_query_has_centre_codes(oracle_mod):
    """A group whose heads sum to zero has no direction: q~ = 0, every
    projection is 0 and every code is the centre code 128."""
    ix = _index_for_query(35)
    q = np.zeros((4, 128), np.float32)
    q[0, 3], q[1, 3] = 2.5, -2.5
    codes, qsel = ix.query(q)
    assert not np.any(qsel)
    assert np.all(codes == 128)


# --------------------------------------------------------------------------
# Stop rule of the prioritised search (Figure 2 step 2, the P-DCI query):
# leaves are taken whole, in increasing (priority, position) order, and the
# search stops after the first leaf at which the running token count reaches
# n_cand. Expected sets are derived here from the leaf table (counts and cells
# of the dump, pinned by the partition tests) and the query codes (pinned
# above); the priority is the L-infinity cell distance (pinned by brute force).
# --------------------------------------------------------------------------
def _expected_order(dmp, qc):
    lo, hi = dmp["lo"], dmp["hi"]
    below = np.maximum(lo - qc[None, :], 0)
    above = np.maximum(qc[None, :] - hi, 0)
    prio = np.max(np.maximum(below, above), axis=1)
    order = np.lexsort((np.arange(len(prio)), prio))
    return order, prio


@pytest.mark.parametrize("m,P,seed", [(8, 4, 41), (2, 4, 42), (8, 16, 43), (2, 8, 44)])
def test_stop_rule_takes_whole_leaves_until_n_cand(oracle_mod, m, P, seed):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(seed)
    n = 700
    K = _clustered(rng, n, 128, 10, 0.5)
    ix = OracleIndex(128, m, 2, P, seed).build(K, K)
    boundary_hits = 0
    for trial in range(3):
        q = (K[rng.integers(0, n)] + 0.3 * rng.standard_normal((4, 128))).astype(np.float32)
        codes, _ = ix.query(q)
        for l in range(2):
            dmp = ix.dump(l)
            order, prio = _expected_order(dmp, codes[l])
            cum = np.cumsum(dmp["cnt"][order])
            _, oprio = ix.leaf_order(q, l, 1)
            assert np.array_equal(oprio, prio)
            ks = sorted({0, 1, 2, 3, len(cum) // 4, len(cum) // 2, len(cum) - 2, len(cum) - 1})
            for k in ks:
                for n_cand in (int(cum[k]) - 1, int(cum[k]), int(cum[k]) + 1):
                    if n_cand < 1:
                        continue
                    # the first position whose running count reaches n_cand
                    stop = int(np.searchsorted(cum, n_cand, side="left"))
                    expect = order[:min(stop + 1, len(order))]
                    flat, _ = ix.leaf_order(q, l, n_cand)
                    tree, _ = ix.leaf_order(q, l, n_cand, tree=True)
                    assert np.array_equal(flat, expect), (l, k, n_cand)
                    assert np.array_equal(tree, expect), (l, k, n_cand)
                    if n_cand == int(cum[k]):
                        boundary_hits += 1
                        assert len(flat) == k + 1  # landing on a leaf end: no leaf more
    assert boundary_hits >= 20


def test_stop_rule_through_selection_trace(oracle_mod):
    """With one composite the candidates are exactly the taken leaves' tokens:
    for n_cand on a leaf boundary the selection rescores cum[k] tokens, one
    past it cum[k + 1]."""
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(45)
    K = _clustered(rng, 500, 128, 8, 0.5)
    ix = OracleIndex(128, 8, 1, 8, 45).build(K, K)
    q = (K[17] + 0.3 * rng.standard_normal((2, 128))).astype(np.float32)
    codes, _ = ix.query(q)
    order, _ = _expected_order(ix.dump(0), codes[0])
    cum = np.cumsum(ix.dump(0)["cnt"][order])
    for k in (0, 3, 10, 25):
        _, _, tr = ix.select(q, 64, n_cand=int(cum[k]))
        assert tr["cands"] == int(cum[k])
        _, _, tr = ix.select(q, 64, n_cand=int(cum[k]) + 1)
        assert tr["cands"] == int(cum[k + 1])


# --------------------------------------------------------------------------
# Exact top-k (Table 1 "TOP-k": the k keys with the largest inner product with
# the query), the reference of the recall report.
# --------------------------------------------------------------------------
def test_exact_topk_is_fp64_argsort_with_ties(oracle_mod):
    from oracle.oracle import OracleIndex
    rng = np.random.default_rng(46)
    base = _clustered(rng, 150, 128, 6)
    K = np.concatenate([base, base[:50]])  # tokens t and 150 + t tie exactly for t < 50
    ix = OracleIndex(128, 8, 1, 16, 46).build(K, K)
    for G in (1, 4):
        q = (base[3] + 0.3 * rng.standard_normal((G, 128))).astype(np.float32)
        acc = q[0].copy()
        for h in range(1, G):
            acc = (acc + q[h]).astype(np.float32)
        s = K.astype(np.float64) @ acc.astype(np.float64)
        ref = np.lexsort((np.arange(len(s)), -s))  # score desc, then token asc
        for k in (1, 7, 64, 200):
            got = ix.exact_topk(q, k)
            assert np.array_equal(got, ref[:k]), (G, k)
        # a tied pair ranks the lower token first
        top = ix.exact_topk(q, 200)
        pos = {int(t): i for i, t in enumerate(top)}
        for t in range(50):
            assert pos[t] < pos[150 + t]
    # scores that fp32 cannot separate: q . k1 = 1 and q . k2 = 1 + 2^-30 are
    # distinct in fp64, so token 1 ranks before token 0
    K2 = np.zeros((3, 128), np.float32)
    K2[0, 0] = 1.0
    K2[1, 0], K2[1, 1] = 1.0, 1.0
    K2[2, 0] = -1.0
    q2 = np.zeros((1, 128), np.float32)
    q2[0, 0], q2[0, 1] = 1.0, 2.0 ** -30
    ix2 = OracleIndex(128, 8, 1, 16, 47).build(K2, K2)
    assert ix2.exact_topk(q2, 3).tolist() == [1, 0, 2]

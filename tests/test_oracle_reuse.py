"""Pins of the oracle's selection reuse across steps (the IceCache(r) reading):
the decision follows the query codes and the reuse count, and the pages and the
attention are those of the plain selection of the step that selected."""
import numpy as np
import pytest

from oracle import oracle as O


@pytest.fixture(scope="module")
def unit():
    rng = np.random.default_rng(21)
    centres = rng.standard_normal((16, 128))
    asg = rng.integers(0, 16, 900)
    K = (centres[asg] + 0.3 * rng.standard_normal((900, 128))).astype(np.float32)
    V = rng.standard_normal((900, 128)).astype(np.float32)
    q = (centres[3] + 0.3 * rng.standard_normal((4, 128))).astype(np.float32)
    return K, V, q


def _index(K, V):
    ix = O.OracleIndex(128, 8, 2, 16, 5)
    ix.build(K, V)
    return ix


def test_r0_selects_every_step(unit):
    K, V, q = unit
    ix = _index(K, V)
    ro = O.ReuseOracle(ix, 0)
    for s in range(4):
        qs = q * (1.0 + 0.01 * s)
        ids, npg, resel, out = ro.step(qs, 128)
        ids2, npg2, _ = ix.select(qs, 128)
        assert resel and npg == npg2 and np.array_equal(ids, ids2)
        assert np.allclose(out, ix.attn(qs, ids2, npg2))


def test_same_query_reselects_every_r_plus_one_steps(unit):
    K, V, q = unit
    ix = _index(K, V)
    ro = O.ReuseOracle(ix, 3)
    first = ix.select(q, 128)
    pattern = []
    for _ in range(9):
        ids, npg, resel, _ = ro.step(q, 128)
        pattern.append(resel)
        assert npg == first[1] and np.array_equal(ids, first[0])
    assert pattern == [True, False, False, False, True, False, False, False, True]


def test_changed_codes_or_budget_reselect(unit):
    K, V, q = unit
    ix = _index(K, V)
    ro = O.ReuseOracle(ix, 10)
    ro.step(q, 128)
    q2 = -q  # the opposite direction: every projection changes sign
    c1, _ = ix.query(q)
    c2, _ = ix.query(q2)
    assert not np.array_equal(c1, c2)
    ids, npg, resel, _ = ro.step(q2, 128)
    assert resel
    ids2, npg2, _ = ix.select(q2, 128)
    assert npg == npg2 and np.array_equal(ids, ids2)
    assert not ro.step(q2, 128)[2]
    assert ro.step(q2, 64)[2]  # another budget


def test_reused_pages_see_inserted_tokens(unit):
    K, V, q = unit
    ix = _index(K, V)
    ro = O.ReuseOracle(ix, 5)
    ids, npg, _, _ = ro.step(q, 128)
    rng = np.random.default_rng(3)
    for _ in range(40):
        ix.insert(K[rng.integers(0, 900)] + 0.01 * rng.standard_normal(128).astype(np.float32),
                  rng.standard_normal(128).astype(np.float32))
    ids_r, npg_r, resel, out = ro.step(q, 128)
    assert not resel  # the query codes do not depend on the index content
    assert np.array_equal(ids_r, ids) and npg_r == npg
    assert np.allclose(out, ix.attn(q, ids, npg))
    c_before, _ = ix.query(q)
    assert np.array_equal(c_before, ro.codes)


def test_select_heads_union(unit):
    """Per-head selection: one head equals the plain selection; identical heads
    give one list; the union holds every head's pages once, head 0's first."""
    K, V, q = unit
    ix = _index(K, V)
    ids1, n1, _ = ix.select(q[:1], 128)
    u, n, heads = O.select_heads(ix, q[:1], 128)
    assert n == n1 and np.array_equal(u, ids1[:n1])
    same = np.repeat(q[:1], 4, axis=0)
    u, n, heads = O.select_heads(ix, same, 128)
    assert n == n1 and np.array_equal(u, ids1[:n1])
    u, n, heads = O.select_heads(ix, q, 128)
    assert len(set(u.tolist())) == n
    assert np.array_equal(u[:heads[0][1]], heads[0][0][:heads[0][1]])
    for ids, m in heads:
        assert set(ids[:m].tolist()) <= set(u.tolist())

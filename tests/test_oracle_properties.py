"""Property tests of the oracle on small generated inputs (hypothesis): the
partition invariants hold for any keys, page size and composite count, and
inserting tokens one by one gives the same canonical index as building from
all of them with the frozen scale."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from tests.test_oracle_pins import _canonical, _check_partition  # noqa: E402


def _keys(seed, n, centres, spread, dup):
    rng = np.random.default_rng(seed)
    mu = rng.standard_normal((centres, 128))
    K = (mu[rng.integers(0, centres, n)] + spread * rng.standard_normal((n, 128))).astype(np.float32)
    if dup and n > 1:  # repeated keys: the partition must split on token bits
        K[rng.integers(0, n, n // 3)] = K[0]
    return K


@settings(max_examples=25, deadline=None)
@given(seed=st.integers(0, 2 ** 31 - 1), n=st.integers(1, 220), P=st.sampled_from([1, 2, 4, 16, 64]),
       L=st.integers(1, 2), centres=st.integers(1, 16), spread=st.sampled_from([0.0, 0.05, 0.3, 1.0]),
       dup=st.booleans())
def test_partition_invariants_hold(oracle_mod, seed, n, P, L, centres, spread, dup):
    from oracle.oracle import OracleIndex
    K = _keys(seed, n, centres, spread, dup)
    ix = OracleIndex(128, 8, L, P, seed % 1000).build(K, K)
    for l in range(L):
        _check_partition(ix, l, P)


@settings(max_examples=15, deadline=None)
@given(seed=st.integers(0, 2 ** 31 - 1), n0=st.integers(0, 80), steps=st.integers(1, 60),
       P=st.sampled_from([2, 4, 16]), centres=st.integers(1, 8), dup=st.booleans())
def test_insert_equals_build(oracle_mod, seed, n0, steps, P, centres, dup):
    from oracle.oracle import OracleIndex
    K = _keys(seed, n0 + steps, centres, 0.3, dup)
    V = np.zeros_like(K)
    dyn = OracleIndex(128, 8, 2, P, 9).build(K[:n0], V[:n0])
    e = dyn.e
    for s in range(steps):
        dyn.insert(K[n0 + s], V[n0 + s])
    fresh = OracleIndex(128, 8, 2, P, 9).build(K, V, forced_e=e)
    for l in range(2):
        assert _canonical(dyn, l) == _canonical(fresh, l)
        _check_partition(dyn, l, P)

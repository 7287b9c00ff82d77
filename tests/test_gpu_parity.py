"""GPU path (through the C ABI binding) against the CPU oracle, element by element.

Covers the build (codes, sorted keys, leaf tables, page contents), selection
(page ids bit-exact), attention (2e-2 bf16 / 1e-5 fp32), insertion, and the
edge cases of the method: n < P, n = P, n = P + 1, equal and duplicated keys,
a budget larger than the context, an index built empty and grown by inserts.
"""
import numpy as np
import pytest
import torch

from tests.parity_helpers import (check_select_attn, compare_index, compare_pages,
                                  oracle_for_unit, q_of_unit)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from semantic_paged_kv_head_gb300 import build
    build.build_lib()
    from semantic_paged_kv_head_gb300 import ice as m
    return m


def _synth():
    from semantic_paged_kv_head_gb300 import synth
    return synth


def _run(ice, w, keys, values, q, max_tokens=None, kv_host=False):
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, n_proj=w.n_proj,
                             seed=w.seed, max_tokens=max_tokens, kv_host=kv_host,
                             dir_kind=w.dir_kind)
    qd = q.cuda().contiguous()
    stats = torch.zeros((gix.n_units, 4), dtype=torch.int32, device="cuda")
    ids, npg = gix.select(qd, w.budget, stats=stats)
    out = gix.sparse_attn(qd, ids, npg)
    # the fused call selects the same pages; its attention is checked against the
    # oracle by the callers through `out_f` on the same tolerance
    stats_f = torch.zeros_like(stats)
    out_f, ids_f, npg_f = gix.select_attn(qd, w.budget, stats=stats_f)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    assert torch.equal(ids_f, ids) and torch.equal(npg_f, npg) and torch.equal(stats_f, stats)
    d = (out_f.float() - out.float()).abs().max().item() if out.numel() else 0.0
    assert d <= (4e-2 if w.dtype == torch.bfloat16 else 2e-5), d
    gix._last_fused_out = out_f
    return gix, ids, npg, out, stats


def _full_check(ice, w, units=None, max_pages=8, kv_host=False):
    synth = _synth()
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    gix, ids, npg, out, stats = _run(ice, w, keys, values, q, kv_host=kv_host)
    units = range(w.n_units) if units is None else units
    errs = []
    for u in units:
        orc = oracle_for_unit(w, keys, values, u)
        gd = gix.dump(u)
        compare_index(gd, orc, f"unit {u}")
        compare_pages(gix, w, keys, values, gd, u, max_pages)
        qu = q_of_unit(w, q, u)
        G = w.group
        err, _ = check_select_attn(w, orc, qu, ids[u], npg[u], out.view(-1, G, w.d)[u], stats[u],
                                   f"unit {u}")
        errs.append(err)
        check_select_attn(w, orc, qu, ids[u], npg[u], gix._last_fused_out.view(-1, G, w.d)[u],
                          None, f"unit {u} fused")
    return errs


def test_tiny_fp32_4k_workload(ice):
    """The 4096-token fp32 single-unit workload, compared in full."""
    w = _synth().WORKLOADS["tiny_fp32_4k"]
    _full_check(ice, w)


@pytest.mark.parametrize("n,P,L,G,dtype,budget", [
    (3001, 16, 2, 4, torch.bfloat16, 256),   # several tiles + ragged tail
    (2049, 32, 2, 4, torch.bfloat16, 1024),  # P = 32, large budget
    (5000, 16, 1, 2, torch.float32, 256),
    (1800, 16, 1, 4, torch.bfloat16, 256),   # one composite in bf16 (tensor-core projection, 8 directions)
    (777, 8, 2, 1, torch.bfloat16, 64),
    (4097, 16, 2, 8, torch.bfloat16, 128),
    (3500, 64, 2, 4, torch.bfloat16, 1024),  # the largest page size
    (2600, 8, 2, 4, torch.bfloat16, 512),    # 64 pages: block-wide ranking instead of warp top-32
    (2600, 8, 1, 2, torch.float32, 512),
    (1200, 16, 2, 4, torch.bfloat16, 16),    # one page
])
def test_scaled_llama_shapes(ice, n, P, L, G, dtype, budget):
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, group=G,
                     n_tokens=n, dtype=dtype, page_size=P, n_composite=L, budget=budget,
                     n_centers=32, seed=n)
    _full_check(ice, w)


@pytest.mark.parametrize("mult", [2, 4])
def test_larger_candidate_counts(ice, mult):
    """n_cand = 2 and 4 x the budget (the recall curve's settings)."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=2, n_tokens=3000,
                     n_centers=24, seed=53 + mult)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    n_cand = mult * w.budget
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             n_cand=n_cand)
    stats = torch.zeros((gix.n_units, 4), dtype=torch.int32, device="cuda")
    out, ids, npg = gix.select_attn(q.cuda(), w.budget, stats=stats)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    for u in range(w.n_units):
        orc = oracle_for_unit(w, keys, values, u)
        qu = q_of_unit(w, q, u)
        rid, rn, tr = orc.select(qu, w.budget, n_cand)
        assert int(npg[u]) == rn and np.array_equal(ids[u].cpu().numpy(), rid)
        assert int(stats[u, 1]) == tr["cands"] and int(stats[u, 0]) == tr["leaves"]
        err = np.max(np.abs(out.view(-1, w.group, w.d)[u].float().cpu().numpy() - orc.attn(qu, rid, rn)))
        assert err <= 2e-2


@pytest.mark.parametrize("n", [1, 15, 16, 17, 40])
def test_small_contexts(ice, n):
    """n < P, n = P, n = P + 1: one page or a first split; budget > context."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=2, n_tokens=n,
                     n_centers=4, budget=64, seed=7 + n)
    _full_check(ice, w)


def test_equal_and_duplicate_keys(ice):
    """All keys equal (splits on token bits only) and heavily duplicated keys."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=2, n_tokens=600,
                     n_centers=4, budget=128, seed=3)
    keys, values, centers = synth.make_kv(w)
    keys[0, 0, 0] = keys[0, 0, 0, :1]            # unit 0: every key equal
    keys[0, 0, 1] = keys[0, 0, 1, torch.arange(600) % 7]  # unit 1: 7 distinct keys
    q = synth.make_queries(w, centers)
    gix, ids, npg, out, stats = _run(ice, w, keys, values, q)
    for u in range(2):
        orc = oracle_for_unit(w, keys, values, u)
        compare_index(gix.dump(u), orc, f"unit {u}")
        check_select_attn(w, orc, q_of_unit(w, q, u), ids[u], npg[u],
                          out.view(-1, w.group, w.d)[u], stats[u], f"unit {u}")


def test_full_budget_is_dense_attention(ice):
    """Budget and candidates covering every page: sparse == dense attention."""
    from oracle import oracle as O
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["tiny_fp32_4k"], n_tokens=300, n_centers=8)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    orc = oracle_for_unit(w, keys, values, 0)
    budget = w.page_size * orc.n_leaves(0)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, n_cand=300,
                             seed=w.seed)
    ids, npg = gix.select(q.cuda(), budget)
    out = gix.sparse_attn(q.cuda(), ids, npg)
    assert int(npg[0]) == orc.n_leaves(0)
    dense = O.dense_attn(q[0, 0], keys[0, 0, 0], values[0, 0, 0])
    assert np.max(np.abs(out[0, 0].cpu().numpy() - dense)) <= 1e-5


def test_insert_matches_oracle(ice):
    """Inserts without rebuild: tables, ids and selections follow the oracle."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=3, n_tokens=700,
                     n_insert=300, n_centers=16, seed=5)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             max_tokens=w.n_tokens + w.n_insert)
    orcs = [oracle_for_unit(w, keys, values, u) for u in range(w.n_units)]
    for s in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, s)
        if s == 137:
            k = k * 3  # one key beyond the frozen norm bound (tail clamps to 0)
        gix.insert(k.cuda(), v.cuda())
        for u in range(w.n_units):
            orcs[u].insert(k.view(-1, w.d)[u], v.view(-1, w.d)[u])
        if s % 60 == 59 or s == w.n_insert - 1:
            q = synth.make_queries(w, centers, step=s, drift_deltas=deltas)
            ids, npg = gix.select(q.cuda(), w.budget)
            out = gix.sparse_attn(q.cuda(), ids, npg)
            torch.cuda.synchronize()
            assert gix.get_error() == 0
            for u in range(w.n_units):
                compare_index(gix.dump(u), orcs[u], f"step {s} unit {u}")
                check_select_attn(w, orcs[u], q_of_unit(w, q, u), ids[u], npg[u],
                                  out.view(-1, w.group, w.d)[u], None, f"step {s} unit {u}")


@pytest.mark.parametrize("G, dtype", [(4, torch.bfloat16), (2, torch.float32)])
def test_select_heads_union(ice, G, dtype):
    """Per-query-head selection with a union over the group: per-head lists and
    the union bit-exact against the oracle, attention over the union within
    tolerance."""
    from oracle import oracle as O
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, group=G,
                     n_tokens=2200, dtype=dtype, n_centers=24, seed=43)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    qd = q.cuda()
    ids, n, hid, hn = gix.select_heads(qd, w.budget)
    out = gix.sparse_attn(qd, ids, n)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    for u in range(w.n_units):
        orc = oracle_for_unit(w, keys, values, u)
        qu = q_of_unit(w, q, u)
        uo, no, heads = O.select_heads(orc, qu, w.budget)
        for g, (hi, hm) in enumerate(heads):
            assert int(hn[u, g]) == hm, (u, g)
            assert np.array_equal(hid[u, g, :hm].cpu().numpy(), hi[:hm]), (u, g)
        assert int(n[u]) == no
        assert np.array_equal(ids[u, :no].cpu().numpy(), uo)
        assert (ids[u, no:] == -1).all()
        ref = orc.attn(qu, uo, no)
        got = out.view(-1, w.group, w.d)[u].float().cpu().numpy()
        assert np.max(np.abs(got - ref)) <= (2e-2 if dtype == torch.bfloat16 else 1e-5)


@pytest.mark.parametrize("L", [1, 2])
def test_gaussian_directions(ice, L):
    """The Gaussian-direction variant of the index: same build tables, pages and
    attention as the oracle with the same directions."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, n_tokens=2500,
                     n_composite=L, n_centers=32, seed=41, dir_kind=1)
    _full_check(ice, w)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_host_resident_pool(ice, dtype):
    """Page pool in pinned host memory (the offloaded KV tier): same index, same
    pages and the same attention as the oracle; the pool bytes are on the host."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, n_tokens=3001,
                     dtype=dtype, n_centers=32, seed=11)
    _full_check(ice, w, kv_host=True)
    keys, values, centers = synth.make_kv(w)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             kv_host=True)
    inf = gix.info()
    assert inf.kv_location == ice.KV_HOST
    es = 2 if dtype == torch.bfloat16 else 4
    assert inf.host_bytes >= 2 * gix.n_units * inf.list_capacity * w.page_size * w.d * es


def test_host_resident_pool_inserts(ice):
    """Inserts write the new rows into the host pool; selections follow the oracle."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=2, n_tokens=500,
                     n_insert=120, n_centers=16, seed=15)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             max_tokens=w.n_tokens + w.n_insert, kv_host=True)
    orcs = [oracle_for_unit(w, keys, values, u) for u in range(w.n_units)]
    for s in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, s)
        gix.insert(k.cuda(), v.cuda())
        for u in range(w.n_units):
            orcs[u].insert(k.view(-1, w.d)[u], v.view(-1, w.d)[u])
    q = synth.make_queries(w, centers, step=w.n_insert, drift_deltas=deltas)
    out, ids, npg = gix.select_attn(q.cuda(), w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    for u in range(w.n_units):
        gd = gix.dump(u)
        compare_index(gd, orcs[u], f"unit {u}")
        check_select_attn(w, orcs[u], q_of_unit(w, q, u), ids[u], npg[u],
                          out.view(-1, w.group, w.d)[u], None, f"unit {u}")


def test_empty_build_then_inserts(ice):
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=2, n_tokens=0, n_insert=50,
                     n_centers=4, budget=32, seed=9)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             max_tokens=50)
    orcs = [oracle_for_unit(w, keys, values, u) for u in range(w.n_units)]
    for s in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, s)
        gix.insert(k.cuda(), v.cuda())
        for u in range(w.n_units):
            orcs[u].insert(k.view(-1, w.d)[u], v.view(-1, w.d)[u])
    q = synth.make_queries(w, centers)
    ids, npg = gix.select(q.cuda(), w.budget)
    out = gix.sparse_attn(q.cuda(), ids, npg)
    torch.cuda.synchronize()
    for u in range(w.n_units):
        compare_index(gix.dump(u), orcs[u], f"unit {u}")
        check_select_attn(w, orcs[u], q_of_unit(w, q, u), ids[u], npg[u],
                          out.view(-1, w.group, w.d)[u], None, f"unit {u}")
    # capacity: the 51st token is refused on the host
    k, v = synth.make_insert_token(w, centers, deltas, 99)
    with pytest.raises(ice.IceError) as ei:
        gix.insert(k.cuda(), v.cuda())
    assert ei.value.code == ice.ICE_ERR_CAPACITY


def test_determinism(ice):
    """Two runs on the same inputs give bit-identical page ids and outputs."""
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=4, n_tokens=3000,
                     n_centers=32, seed=11)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    _, ids1, n1, o1, _ = _run(ice, w, keys, values, q)
    _, ids2, n2, o2, _ = _run(ice, w, keys, values, q)
    assert torch.equal(ids1, ids2) and torch.equal(n1, n2) and torch.equal(o1, o2)


def test_bad_page_ids_report_bounds(ice):
    synth = _synth()
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=2, n_tokens=500,
                     n_centers=8, seed=13)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers).cuda()
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=16, n_q_heads=w.n_q_heads,
                             n_composite=2)
    ids, npg = gix.select(q, 256)
    ids[0, 0] = 10_000_000
    out = gix.sparse_attn(q, ids, npg)
    assert gix.get_error() == ice.ICE_ERR_BOUNDS
    assert gix.get_error() == 0  # cleared
    assert torch.isfinite(out.float()).all()
    npg[1] = 999  # more pages than the row holds
    gix.sparse_attn(q, ids, npg)
    assert gix.get_error() == ice.ICE_ERR_BOUNDS


@pytest.mark.parametrize("name,units", [("llama8b_36k", [0, 77, 130, 255]),
                                        ("llama8b_batch16_32k", [0, 64, 127]),
                                        ("mistral7b_gen8k", [0, 7]),
                                        ("qwen3_4b_250k", [0, 143, 287])])
def test_full_size_sampled_units(ice, name, units):
    """Full-size workloads in the launch configuration the benchmark times;
    sampled units are compared with the oracle in full."""
    synth = _synth()
    w = synth.WORKLOADS[name]
    keys, values, centers = synth.make_kv(w, device="cuda")
    q = synth.make_queries(w, centers)
    gix, ids, npg, out, stats = _run(ice, w, keys, values, q)
    for u in units:
        orc = oracle_for_unit(w, keys, values, u)
        gd = gix.dump(u)
        compare_index(gd, orc, f"unit {u}")
        compare_pages(gix, w, keys, values, gd, u, 4)
        check_select_attn(w, orc, q_of_unit(w, q, u), ids[u], npg[u],
                          out.view(-1, w.group, w.d)[u], stats[u], f"unit {u}")
    # properties at any size: page ids unique, in range, n_pages <= n_sel
    n_sel = w.budget // w.page_size
    idn = ids.cpu().numpy()
    for u in range(w.n_units):
        k = int(npg[u])
        assert 1 <= k <= n_sel
        assert len(set(idn[u, :k].tolist())) == k and (idn[u, k:] == -1).all()

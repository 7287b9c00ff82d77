"""The selection spread over a thread-block cluster of K blocks per unit
(ice_set_cluster_size), against the CPU oracle: page ids and the byte counters
bit-exact, attention within 2e-2 (bf16) / 1e-5 (fp32), for every cluster size,
one and two composites, fp32 and bf16, the largest n_sel of the cluster path,
a one-page budget, and a single unit whose leaf tables exceed what one block
can hold in shared memory."""
import numpy as np
import pytest
import torch

from tests.parity_helpers import check_select_attn, oracle_for_unit, q_of_unit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from semantic_paged_kv_head_gb300 import build
    build.build_lib()
    from semantic_paged_kv_head_gb300 import ice as m
    return m


def _check_all(ice, gix, w, keys, values, q, label):
    qd = q.cuda().contiguous()
    U = gix.n_units
    stats = torch.zeros((U, 4), dtype=torch.int32, device="cuda")
    ids, npg = gix.select(qd, w.budget, stats=stats)
    stats_f = torch.zeros_like(stats)
    out_f, ids_f, npg_f = gix.select_attn(qd, w.budget, stats=stats_f)
    torch.cuda.synchronize()
    assert gix.get_error() == 0, label
    assert torch.equal(ids_f, ids) and torch.equal(npg_f, npg) and torch.equal(stats_f, stats), label
    G = w.group
    for u in range(U):
        orc = oracle_for_unit(w, keys, values, u)
        check_select_attn(w, orc, q_of_unit(w, q, u), ids[u], npg[u], out_f.view(-1, G, w.d)[u],
                          stats[u], f"{label} unit {u}")
    return out_f


@pytest.mark.parametrize("n,P,L,G,dtype,budget", [
    (3001, 16, 2, 4, torch.bfloat16, 256),
    (2049, 32, 2, 4, torch.bfloat16, 1024),  # n_sel = 32, the largest of the cluster path
    (5000, 16, 1, 2, torch.float32, 256),
    (1200, 16, 2, 4, torch.bfloat16, 16),    # one page
    (700, 8, 2, 8, torch.bfloat16, 64),
])
def test_every_cluster_size_matches_oracle(ice, n, P, L, G, dtype, budget):
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, group=G, n_tokens=n,
                     dtype=dtype, page_size=P, n_composite=L, budget=budget, n_centers=24,
                     seed=n + 7)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    outs = {}
    for K in (1, 2, 4, 8, 16):
        gix.set_cluster_size(K)
        outs[K] = _check_all(ice, gix, w, keys, values, q, f"K={K}")
    gix.set_cluster_size(0)
    _check_all(ice, gix, w, keys, values, q, "auto")
    ref = outs[max(outs)]
    for K, o in outs.items():  # the cluster size changes the merge order only
        d = float((o.float() - ref.float()).abs().max())
        assert d <= (4e-2 if dtype == torch.bfloat16 else 2e-5), (K, d)
    gix.destroy()


def test_unit_beyond_one_block_tables(ice):
    """One unit of 120,000 tokens at page size 4 has about 49k leaves per
    composite: one block cannot hold its scan tables (the one-block kernel is
    refused), a cluster splits them and selects exactly what the oracle does."""
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=1, n_tokens=120000,
                     page_size=4, budget=64, n_centers=256, seed=77)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    assert gix.dump(0)["n_leaf"][0] > 45000
    gix.set_cluster_size(1)
    with pytest.raises(ice.IceError) as ei:
        gix.select_attn(q.cuda(), w.budget)
    assert ei.value.code == ice.ICE_ERR_UNSUPPORTED
    for K in (0, 8, 16):
        gix.set_cluster_size(K)
        _check_all(ice, gix, w, keys, values, q, f"K={K}")
    gix.destroy()


def test_forced_timeout_in_a_cluster(ice):
    """The bounded page wait of one block of a cluster runs out (test flag): the
    cluster reports the timeout, writes zeros, and the next call is exact."""
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=2, n_tokens=2000,
                     n_centers=8, seed=91)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers).cuda()
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    gix.set_cluster_size(4)
    ref, ids_ref, npg_ref = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    gix.debug_set_flags(ice.DEBUG_STALL_ATTN)
    out, ids, npg = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == ice.ICE_ERR_TIMEOUT
    assert torch.equal(ids, ids_ref) and torch.equal(npg, npg_ref)
    assert float(out.float().abs().max()) == 0.0
    gix.debug_set_flags(0)
    out2, _, _ = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    assert torch.equal(out2, ref)
    gix.destroy()


def test_selection_reads_the_index_after_an_insert(ice):
    """The cluster selection reads the index before its wait on the previous kernel of
    the stream, except right after an insert on that stream. A selection right after
    an insert must see the inserted token; one right after another selection reads
    early and must agree with it; a decode step (insert, then selection) and the
    selection after it agree too. No synchronisation between the calls: only the
    stream orders them. Page ids follow the oracle after every insert."""
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=2, n_tokens=600,
                     n_insert=24, n_centers=12, seed=17)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             max_tokens=w.n_tokens + w.n_insert)
    U, G, n_sel = gix.n_units, w.group, w.budget // w.page_size
    orcs = [oracle_for_unit(w, keys, values, u) for u in range(U)]
    results = []
    for s in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, s)
        q = synth.make_queries(w, centers, step=s, drift_deltas=deltas).cuda()
        if s % 2 == 0:
            gix.insert(k.cuda(), v.cuda())
            first = gix.select_attn(q, w.budget)   # right after the insert: waits first
        else:
            ids = torch.empty((U, n_sel), dtype=torch.int32, device="cuda")
            npg = torch.empty((U,), dtype=torch.int32, device="cuda")
            out = torch.empty_like(q)
            gix.decode_step(k.cuda(), v.cuda(), q, w.budget, ids, npg, out)
            first = (out, ids, npg)
        second = gix.select_attn(q, w.budget)      # right after a selection: reads early
        for u in range(U):
            orcs[u].insert(k.view(-1, w.d)[u], v.view(-1, w.d)[u])
        results.append((s, q, first, second))
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    for s, q, (o1, i1, n1), (o2, i2, n2) in results:
        assert torch.equal(i1, i2) and torch.equal(n1, n2), s
        assert torch.equal(o1, o2), s
    # the last step against the oracle (the index holds every insert by then)
    s, q, (o1, i1, n1), _ = results[-1]
    for u in range(U):
        check_select_attn(w, orcs[u], q_of_unit(w, q.cpu(), u), i1[u], n1[u],
                          o1.view(-1, G, w.d)[u], None, f"step {s} unit {u}")

"""A decode step (insert + select + attention) captured once in a CUDA graph and
replayed gives, step by step, the pages, outputs and final index of the same
steps run eagerly; replays past the token capacity report it on the device."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from semantic_paged_kv_head_gb300 import build
    build.build_lib()
    from semantic_paged_kv_head_gb300 import ice as m
    return m


def _dump_equal(a, b):
    """The meaningful parts of two dumps are equal: the first n_leaf leaf records,
    the first next_id lists, and in each list the slots below its count (the
    rest of the capacity is never written and holds whatever the allocation did)."""
    assert a["n"] == b["n"] and a["n_leaf"] == b["n_leaf"] and a["next_id"] == b["next_id"]
    for l, (ca, cb) in enumerate(zip(a["comp"], b["comp"])):
        N, NL = a["n_leaf"][l], a["next_id"][l]
        for key in ("pm", "pt", "t", "lo", "id", "cnt"):
            assert np.array_equal(ca[key][:N], cb[key][:N]), key
        assert np.array_equal(ca["list_cnt"][:NL], cb["list_cnt"][:NL])
        used = np.arange(a["P"])[None, :] < ca["list_cnt"][:NL, None]
        for key in ("slot_tok", "slot_key"):
            assert np.array_equal(ca[key][:NL][used], cb[key][:NL][used]), key
    assert np.array_equal(a["tok_loc"], b["tok_loc"])


def test_graph_replay_equals_eager(ice):
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=3, n_tokens=600, n_insert=40,
                     n_centers=12, seed=47)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    steps = []
    for t in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, t)
        q = synth.make_queries(w, centers, step=t, drift_deltas=deltas)
        steps.append((k.cuda(), v.cuda(), q.cuda()))
    cap = w.n_tokens + w.n_insert

    def index():
        return ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                                  n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                                  max_tokens=cap)

    U, n_sel = w.n_units, w.budget // w.page_size
    eager, graphed = index(), index()
    ids_e = torch.empty((U, n_sel), dtype=torch.int32, device="cuda")
    npg_e = torch.empty((U,), dtype=torch.int32, device="cuda")
    out_e = torch.empty_like(steps[0][2])
    ks, vs, qs = (torch.empty_like(x) for x in steps[0])
    ids_g, npg_g, out_g = torch.empty_like(ids_e), torch.empty_like(npg_e), torch.empty_like(out_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.decode_step(ks, vs, qs, w.budget, ids_g, npg_g, out_g)
    for t, (k, v, q) in enumerate(steps):
        eager.decode_step(k, v, q, w.budget, ids_e, npg_e, out_e)
        ks.copy_(k)
        vs.copy_(v)
        qs.copy_(q)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(npg_g, npg_e) and torch.equal(ids_g, ids_e), t
        assert torch.equal(out_g, out_e), t
    assert eager.get_error() == 0 and graphed.get_error() == 0
    for u in range(U):
        _dump_equal(graphed.dump(u), eager.dump(u))
    assert graphed.info().n_tokens == cap
    # past the capacity: the device count stops, the index is unchanged, the status says so
    before = [graphed.dump(u) for u in range(U)]
    g.replay()
    torch.cuda.synchronize()
    assert graphed.get_error() == ice.ICE_ERR_CAPACITY
    for u in range(U):
        _dump_equal(graphed.dump(u), before[u])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fused_decode_step_equals_separate_calls(ice, dtype):
    """The one-launch decode step (each block inserts its unit's token, then
    selects and attends) gives the index, pages and outputs of ice_insert
    followed by ice_select_attn, and the oracle's pages."""
    from oracle import oracle as O  # noqa: F401
    from semantic_paged_kv_head_gb300 import synth
    from tests.parity_helpers import check_select_attn, compare_index, oracle_for_unit, q_of_unit
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=3, n_tokens=700, n_insert=90,
                     n_centers=12, dtype=dtype, seed=59)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    cap = w.n_tokens + w.n_insert

    def index():
        return ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                                  n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                                  max_tokens=cap)

    U, n_sel = w.n_units, w.budget // w.page_size
    fused, sep = index(), index()
    # one block per unit: with few units the automatic choice is the cluster selection,
    # which runs the decode step as an insert launch and a selection launch
    fused.set_cluster_size(1)
    orcs = [oracle_for_unit(w, keys, values, u) for u in range(U)]
    ids_f = torch.empty((U, n_sel), dtype=torch.int32, device="cuda")
    npg_f = torch.empty((U,), dtype=torch.int32, device="cuda")
    for t in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, t)
        q = synth.make_queries(w, centers, step=t, drift_deltas=deltas)
        kc, vc, qc = k.cuda(), v.cuda(), q.cuda()
        out_f = torch.empty_like(qc)
        fused.decode_step(kc, vc, qc, w.budget, ids_f, npg_f, out_f)
        sep.insert(kc, vc)
        out_s, ids_s, npg_s = sep.select_attn(qc, w.budget)
        for u in range(U):
            orcs[u].insert(k.view(-1, w.d)[u], v.view(-1, w.d)[u])
        torch.cuda.synchronize()
        assert torch.equal(ids_f, ids_s) and torch.equal(npg_f, npg_s), t
        # the separate call may attend with a cluster of blocks per unit, which
        # merges the softmax partials in another order
        d = float((out_f.float() - out_s.float()).abs().max())
        assert d <= (4e-2 if dtype == torch.bfloat16 else 2e-5), (t, d)
        if t % 30 == 29:
            for u in range(U):
                compare_index(fused.dump(u), orcs[u], f"step {t} unit {u}")
                check_select_attn(w, orcs[u], q_of_unit(w, q, u), ids_f[u], npg_f[u],
                                  out_f.view(-1, w.group, w.d)[u], None, f"step {t} unit {u}")
    assert fused.get_error() == 0 and sep.get_error() == 0
